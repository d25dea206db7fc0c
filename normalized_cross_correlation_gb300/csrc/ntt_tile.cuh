// ntt_tile.cuh -- the number-theoretic transform of one 256 x 256 tile, the
// arithmetic of the FFT numerator (correlate_ntt.cu).
//
// The CUDA Handbook, section 15.8 ("The Denominator: Summed Area Tables"),
// names the FFT as the other way to form the numerator SumIT for every shift
// at once.  Over the complex numbers the rounded result is exact only within
// an error bound; over the integers modulo a prime p the transform is exact:
// the cyclic correlation of the centered image tile with the centered
// template, computed with transforms, products and inverse transforms modulo
// p, equals the true integer correlation C modulo p, and C is recovered
// because |C| <= 2^14 * wT * hT < p / 2.
//
// The prime is p = 119 * 2^23 + 1 (3 generates its multiplicative group), so
// 256th roots of unity exist and 4p < 2^32: values are reduced only lazily --
// the forward passes keep them in [0, 2p), the inverse passes in [0, 4p) --
// and no sum overflows 32 bits.
// Multiplication by a known factor w uses its precomputed companion
// wq = floor(w * 2^32 / p) (Shoup's method): q = hi32(x * wq) and
// x * w - q * p lies in [0, 2p) for any 32-bit x.
//
// Tile transform.  A 256 x 256 tile is transformed along x (rows, 256
// points) and along y (columns).  The first radix-2 step along y splits the
// spectrum into even and odd frequencies:
//     X[2m]   = sum_{r<128} (x[r] + x[r+128])         w_128^(rm)
//     X[2m+1] = sum_{r<128} (x[r] - x[r+128]) w_256^r w_128^(rm)
// so each half is a 128-row problem (136 KB of shared memory), done one after
// the other ("even pass", "odd pass").  The inverse combines the halves:
//     y[r] = e[r] + w_256^(-r) o[r],   y[r+128] = e[r] - w_256^(-r) o[r].
// Each axis is done in radix-16 register passes (256 = 16 * 16 along x,
// 128 = 16 * 8 along y).  The forward transforms are decimation in frequency
// (natural order in, digit-reversed order out) and the inverse transforms
// decimation in time (digit-reversed in, natural out), so the spectrum is
// never reordered: the template's spectrum is produced by the same code in
// the same order.
//
// Shared-memory layout: the 128 x 256 words of a half pass, row stride 272
// words, column c stored at 16*(c/16) + ((c%16) xor (c/16)).  With that
// swizzle and the stride (16 mod 32), every pass's accesses -- 16 lanes along
// a row at stride 16, 16 lanes each reading 16 consecutive words, 32 lanes
// along a column -- fall on 32 distinct banks.
//
// Every function here is __host__ __device__: the kernels call each pass
// with their thread index between barriers, and the same passes run on the
// host for checking.  Within a pass the threads touch disjoint words.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

namespace ncc {
namespace ntt {

constexpr uint32_t kP = 998244353u;  // 119 * 2^23 + 1
constexpr uint32_t kP2 = 2u * kP;    // values live in [0, 2p); 4p < 2^32
constexpr int kL = 256;              // tile side
constexpr int kHalf = 128;           // rows of a half pass
constexpr int kStride = 272;         // words per buffer row (256 + 16)
constexpr int kThreads = 512;        // threads per CTA
constexpr int kBufWords = kHalf * kStride;
// |C| <= 2^14 N must stay below p/2: N = wT * hT at most 30000 (2 * 2^14 *
// 30000 = 983040000 < p).
constexpr int kMaxPixels = 30000;

__host__ __device__ constexpr uint32_t mul_c(uint32_t a, uint32_t b) {
    return (uint32_t)((uint64_t)a * b % kP);
}
__host__ __device__ constexpr uint32_t pow_c(uint32_t b, uint32_t e) {
    uint32_t r = 1;
    while (e) {
        if (e & 1u) r = mul_c(r, b);
        b = mul_c(b, b);
        e >>= 1;
    }
    return r;
}
__host__ __device__ constexpr uint32_t shoup_c(uint32_t w) {
    return (uint32_t)(((uint64_t)w << 32) / kP);
}

constexpr uint32_t kW256 = pow_c(3u, (kP - 1) / 256);  // a primitive 256th root of unity
constexpr uint32_t kW256Inv = pow_c(kW256, kP - 2);
constexpr uint32_t kW16 = pow_c(kW256, 16);
constexpr uint32_t kW16Inv = pow_c(kW256Inv, 16);
constexpr uint32_t kScale = pow_c(65536u, kP - 2);  // 1 / (256 * 256): both inverses unnormalized
static_assert(pow_c(kW256, 128) == kP - 1, "w_256 must have order 256");

__host__ __device__ __forceinline__ uint32_t mulhi(uint32_t a, uint32_t b) {
#ifdef __CUDA_ARCH__
    return __umulhi(a, b);
#else
    return (uint32_t)(((uint64_t)a * b) >> 32);
#endif
}
__host__ __device__ __forceinline__ uint32_t umin32(uint32_t a, uint32_t b) { return a < b ? a : b; }
// [0, 4p) -> [0, 2p)
__host__ __device__ __forceinline__ uint32_t red2(uint32_t s) { return umin32(s, s - kP2); }
// [0, 2p) -> [0, p)
__host__ __device__ __forceinline__ uint32_t red1(uint32_t s) { return umin32(s, s - kP); }
// x * w mod p in [0, 2p) for any 32-bit x, w < p, wq = floor(w 2^32 / p)
__host__ __device__ __forceinline__ uint32_t mulw(uint32_t x, uint32_t w, uint32_t wq) {
    return x * w - mulhi(x, wq) * kP;
}
__host__ __device__ __forceinline__ uint32_t mulw(uint32_t x, uint2 w) { return mulw(x, w.x, w.y); }

// compile-time loop: f(integral_constant<int, I>) for I in [B, E)
template <int B, int E, class F>
__host__ __device__ __forceinline__ void cfor(F &&f) {
    if constexpr (B < E) {
        f(std::integral_constant<int, B>{});
        cfor<B + 1, E>(f);
    }
}

// N-point transform (N = 8 or 16), decimation in frequency: natural order in,
// bit-reversed order out (register i holds frequency rev(i)).  In and out in
// [0, 2p).
template <int N>
__host__ __device__ __forceinline__ void dif(uint32_t (&v)[N]) {
    static_assert(N == 8 || N == 16, "8 or 16 points");
    cfor<0, (N == 16 ? 4 : 3)>([&](auto S) {
        constexpr int h = N >> (decltype(S)::value + 1);
        cfor<0, N / (2 * h)>([&](auto Bk) {
            cfor<0, h>([&](auto J) {
                constexpr int j = decltype(J)::value;
                constexpr int a = decltype(Bk)::value * 2 * h + j, b = a + h;
                constexpr uint32_t w = pow_c(kW16, (uint32_t)(j * (8 / h)));  // w_(2h)^j
                const uint32_t u = v[a], t = v[b];
                v[a] = red2(u + t);
                if constexpr (j == 0)
                    v[b] = red2(u - t + kP2);
                else
                    v[b] = mulw(u - t + kP2, w, shoup_c(w));
            });
        });
    });
}

// The inverse (unnormalized: N times the inverse transform), decimation in
// time: bit-reversed order in, natural order out.  Inputs and outputs in
// [0, 4p): a butterfly reduces its first input to [0, 2p), multiplies the
// second (any 32-bit value) to [0, 2p), and leaves the sum and the
// difference + 2p unreduced.
template <int N>
__host__ __device__ __forceinline__ void dit_inv(uint32_t (&v)[N]) {
    static_assert(N == 8 || N == 16, "8 or 16 points");
    cfor<0, (N == 16 ? 4 : 3)>([&](auto S) {
        constexpr int h = 1 << decltype(S)::value;
        cfor<0, N / (2 * h)>([&](auto Bk) {
            cfor<0, h>([&](auto J) {
                constexpr int j = decltype(J)::value;
                constexpr int a = decltype(Bk)::value * 2 * h + j, b = a + h;
                constexpr uint32_t w = pow_c(kW16Inv, (uint32_t)(j * (8 / h)));  // w_(2h)^-j
                const uint32_t u = red2(v[a]);
                uint32_t t;
                if constexpr (j == 0)
                    t = red2(v[b]);
                else
                    t = mulw(v[b], w, shoup_c(w));
                v[a] = u + t;
                v[b] = u - t + kP2;
            });
        });
    });
}

__host__ __device__ __forceinline__ int rev4(int i) {
    return ((i & 1) << 3) | ((i & 2) << 1) | ((i & 4) >> 1) | ((i & 8) >> 3);
}
// word offset of logical column c within a buffer row
__host__ __device__ __forceinline__ int swz(int c) { return (c & ~15) + ((c & 15) ^ (c >> 4)); }

// The shared-memory working set of a CTA.
struct Tile {
    uint32_t *buf;       // [128][kStride]
    uint2 *twR, *twRi;   // [16 i][16 n2]: w_256^(+-n2 rev4(i))
    uint2 *twC, *twCi;   // [16 i][8 n2]:  w_128^(+-n2 rev4(i))
    uint2 *rowF, *rowFi; // [128 r]:       w_256^(+-r)
};
constexpr int kTableWords = 2 * (2 * 256 + 2 * 128 + 2 * 128);  // uint2 entries above, in words
constexpr size_t kSmemBytes = (size_t)(kBufWords + kTableWords) * 4;
// The image kernel also stages the tile's 256 x 256 pixels, rows 320 bytes
// apart (16 mod 32 words: lanes reading rows r and r+1 use different banks).
constexpr int kImgStride = 320;
constexpr size_t kImgSmemBytes = kSmemBytes + (size_t)kL * kImgStride;

__host__ __device__ __forceinline__ Tile carve(uint32_t *smem) {
    Tile t;
    t.buf = smem;
    uint2 *tw = reinterpret_cast<uint2 *>(smem + kBufWords);
    t.twR = tw;
    t.twRi = tw + 256;
    t.twC = tw + 512;
    t.twCi = tw + 640;
    t.rowF = tw + 768;
    t.rowFi = tw + 896;
    return t;
}

__host__ __device__ __forceinline__ uint2 factor(uint32_t w) { return make_uint2(w, shoup_c(w)); }

// The twiddle tables; thread tid of nthreads fills its share.
__host__ __device__ inline void fill_tables(int tid, int nthreads, const Tile &t) {
    for (int e = tid; e < 256; e += nthreads) {
        const int i = e >> 4, n2 = e & 15;
        const uint32_t k = (uint32_t)(n2 * rev4(i));
        t.twR[e] = factor(pow_c(kW256, k));
        t.twRi[e] = factor(pow_c(kW256Inv, k));
    }
    for (int e = tid; e < 128; e += nthreads) {
        const int i = e >> 3, n2 = e & 7;
        const uint32_t k = (uint32_t)(2 * n2 * rev4(i));  // w_128 = w_256^2
        t.twC[e] = factor(pow_c(kW256, k));
        t.twCi[e] = factor(pow_c(kW256Inv, k));
        t.rowF[e] = factor(pow_c(kW256, (uint32_t)e));
        t.rowFi[e] = factor(pow_c(kW256Inv, (uint32_t)e));
    }
}

// ---- the passes of a half (kOdd: the odd-frequency half) ----

// (1) rows, first radix-16 pass, fused with forming the half from tile rows
// r and r+128: load(row, col) gives the centered tile value in [0, p).
template <bool kOdd, class Load>
__host__ __device__ __forceinline__ void rows_fwd1(int tid, const Tile &t, Load &&load) {
#pragma unroll 1
    for (int k = 0; k < 4; ++k) {
        const int idx = tid + kThreads * k, r = idx >> 4, n2 = idx & 15;
        uint32_t v[16];
#pragma unroll
        for (int a = 0; a < 16; ++a) {
            const uint32_t top = load(r, 16 * a + n2), bot = load(r + kHalf, 16 * a + n2);
            v[a] = kOdd ? mulw(top - bot + kP, t.rowF[r]) : top + bot;
        }
        dif<16>(v);
        uint32_t *row = t.buf + r * kStride;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t x = i ? mulw(v[i], t.twR[i * 16 + n2]) : v[i];
            row[16 * i + (n2 ^ i)] = x;
        }
    }
}

// (2) rows, second radix-16 pass (16 consecutive columns).  The forward
// passes keep values in [0, 2p); the inverse passes take [0, 4p).
__host__ __device__ __forceinline__ void rows_fwd2(int tid, const Tile &t) {
#pragma unroll 1
    for (int k = 0; k < 4; ++k) {
        const int idx = tid + kThreads * k, r = idx >> 4, i = idx & 15;
        uint32_t *g = t.buf + r * kStride + 16 * i;
        uint32_t v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = g[j ^ i];
        dif<16>(v);
#pragma unroll
        for (int j = 0; j < 16; ++j) g[j ^ i] = v[j];
    }
}

// (3) columns, first pass: 16 points at row stride 8
__host__ __device__ __forceinline__ void cols_fwd1(int tid, const Tile &t) {
#pragma unroll 1
    for (int k = 0; k < 4; ++k) {
        const int idx = tid + kThreads * k, c = idx & 255, n2 = idx >> 8;
        uint32_t *col = t.buf + swz(c) + n2 * kStride;
        uint32_t v[16];
#pragma unroll
        for (int a = 0; a < 16; ++a) v[a] = col[8 * a * kStride];
        dif<16>(v);
#pragma unroll
        for (int i = 0; i < 16; ++i) col[8 * i * kStride] = i ? mulw(v[i], t.twC[i * 8 + n2]) : v[i];
    }
}

// (4) columns, second pass (8 consecutive rows), the product with the
// template's spectrum H ([128 rows][256 columns], value and companion) and
// the first inverse pass, in registers.  The spectrum of the next item is
// loaded while this one is computed.
__host__ __device__ __forceinline__ void cols_mul(int tid, const Tile &t, const uint2 *H) {
    uint2 hv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) hv[j] = H[(size_t)(8 * (tid >> 8) + j) * kL + (tid & 255)];
#pragma unroll 1
    for (int k = 0; k < 8; ++k) {
        const int idx = tid + kThreads * k, c = idx & 255, i = idx >> 8;
        uint2 hn[8];
        if (k < 7) {
            const int nx = idx + kThreads;
#pragma unroll
            for (int j = 0; j < 8; ++j) hn[j] = H[(size_t)(8 * (nx >> 8) + j) * kL + (nx & 255)];
        }
        uint32_t *col = t.buf + swz(c) + 8 * i * kStride;
        uint32_t v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = col[j * kStride];
        dif<8>(v);
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = mulw(v[j], hv[j]);
        dit_inv<8>(v);
#pragma unroll
        for (int j = 0; j < 8; ++j) col[j * kStride] = v[j];
        if (k < 7) {
#pragma unroll
            for (int j = 0; j < 8; ++j) hv[j] = hn[j];
        }
    }
}

// (4') the template's spectrum instead: second column pass, scaled by
// 1/65536, reduced to [0, p) and stored with its companion
__host__ __device__ __forceinline__ void cols_spectrum(int tid, const Tile &t, uint2 *H) {
#pragma unroll 1
    for (int k = 0; k < 8; ++k) {
        const int idx = tid + kThreads * k, c = idx & 255, i = idx >> 8;
        const uint32_t *col = t.buf + swz(c) + 8 * i * kStride;
        uint32_t v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = col[j * kStride];
        dif<8>(v);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t s = red1(mulw(v[j], kScale, shoup_c(kScale)));
            H[(size_t)(8 * i + j) * kL + c] = factor(s);
        }
    }
}

// (5) columns, last inverse pass: 16 points at row stride 8, back to natural rows
__host__ __device__ __forceinline__ void cols_inv(int tid, const Tile &t) {
#pragma unroll 1
    for (int k = 0; k < 4; ++k) {
        const int idx = tid + kThreads * k, c = idx & 255, n2 = idx >> 8;
        uint32_t *col = t.buf + swz(c) + n2 * kStride;
        uint32_t v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t x = col[8 * i * kStride];
            v[i] = i ? mulw(x, t.twCi[i * 8 + n2]) : x;
        }
        dit_inv<16>(v);
#pragma unroll
        for (int a = 0; a < 16; ++a) col[8 * a * kStride] = v[a];
    }
}

// (6) rows, first inverse pass (16 consecutive columns)
__host__ __device__ __forceinline__ void rows_inv1(int tid, const Tile &t) {
#pragma unroll 1
    for (int k = 0; k < 4; ++k) {
        const int idx = tid + kThreads * k, r = idx >> 4, i = idx & 15;
        uint32_t *g = t.buf + r * kStride + 16 * i;
        uint32_t v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = g[j ^ i];
        dit_inv<16>(v);
#pragma unroll
        for (int j = 0; j < 16; ++j) g[j ^ i] = v[j];
    }
}

// (7) rows, last inverse pass for item k of this thread (row r = idx/16,
// columns 16a + idx%16): out[a] in [0, 4p), natural order
__host__ __device__ __forceinline__ void rows_inv2(int tid, int k, const Tile &t, uint32_t (&out)[16]) {
    const int idx = tid + kThreads * k, r = idx >> 4, n2 = idx & 15;
    const uint32_t *row = t.buf + r * kStride;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t x = row[16 * i + (n2 ^ i)];
        out[i] = i ? mulw(x, t.twRi[i * 16 + n2]) : x;
    }
    dit_inv<16>(out);
}

// Centered integer from a residue in [0, 4p) of a value |C| < p/2.  (The
// inverse passes leave values in [0, 4p); products by a factor are in
// [0, 2p); a sum of the two needs its first term reduced first.)
__host__ __device__ __forceinline__ int32_t centered(uint32_t s) {
    s = red1(red2(s));
    return s > (kP >> 1) ? (int32_t)(s - kP) : (int32_t)s;
}

}  // namespace ntt
}  // namespace ncc
