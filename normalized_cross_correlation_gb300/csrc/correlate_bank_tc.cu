// correlate_bank_tc.cu -- a bank of nT templates against every valid shift of
// an 8-bit image, with the numerator on the 5th-generation tensor cores
// (tcgen05.mma kind::f16, fp32 accumulation in tensor memory) and a fused
// epilogue that reads the window moments from the summed-area tables once
// per shift and writes the fp32 coefficients of every template.
//
// Follows The CUDA Handbook, chapter 15: section 15.8 (one SAT pair serves
// every template of a bank; the four-corner box sum) and "Image in shared
// memory", Listing 15-5 (the per-shift SumIT).  For a bank the numerator is
// a dense contraction: for output row y and the 128 shifts x0..x0+127,
//     D[m][n] = sum_j sum_i I[y+j][x0+m+i] * T_n[j][i],
// i.e. for each template row j one MMA with M = 128 shifts, N = templates,
// K = 16 template columns (more K chunks for wider templates).
//
// Operands (no im2col): the A operand of image row r is MN-major with both
// core-matrix strides 128 bytes over a buffer holding eight copies of the
// row segment shifted by 0..7 pixels (block b, copy s, element e = pixel
// 8b+s+e), so element (m, k) sits at pixel m+k: one 2.2 KB buffer per image
// row serves all hT output rows that use it.  B is K-major, template row j,
// all templates.  Pixels 0..255 are exact in f16 and every product and
// partial sum is an integer below 2^24, so the fp32 accumulation is exact
// while a template group has at most 258 pixels; taller templates are
// split into row groups with separate accumulators, summed as integers.
//
// Warp roles (persistent CTAs, 2 per SM):
//   warp 0     allocates tensor memory; one thread issues the MMAs and the
//              commits (tcgen05.commit -> mbarrier),
//   warps 1-3  convert image rows (u8 -> f16 shifted copies) into a ring of
//              A buffers in shared memory, each warp every third row,
//   warps 4-11 epilogue: two warps per tensor-memory lane quarter (one per
//              half of the template columns); tcgen05.ld of the accumulator
//              row of its shift, box sums from S and Q once per shift
//              (prefetched a row ahead), the coefficient of every template
//              and coalesced fp32 stores.  With one exact fp32 group the
//              numerator N*SumIT - SumI*SumT is formed without rounding
//              error before its final rounding: both products are split
//              exactly by fma and their high parts cancel exactly
//              (Sterbenz) whenever the difference is small.
// All hand-offs are mbarriers; every wait is bounded and a wait that runs out
// records NCC_ERR_TIMEOUT and lets the CTA finish (never a hang).
#include "ncc_common.cuh"

#include <cuda_fp16.h>

namespace ncc {
namespace {

template <bool B>
struct BoolTag {
    static constexpr bool value = B;
};

constexpr int kThreads = 384;
constexpr int kM = 128;               // shifts per tile (MMA M)
constexpr int kTY = 32;               // output rows per tile
constexpr int kProducers = 96;        // warps 1-3
constexpr int kEpi0 = 128;            // first epilogue thread (warps 4-11)
constexpr int kEpiThreads = kThreads - kEpi0;
constexpr int kMaxExactPixels = 258;  // 258 * 255^2 < 2^24: exact fp32 accumulation
constexpr int kMaxSmem = 110 * 1024;  // two CTAs per SM
constexpr int kMaxTmemCols = 256;     // per CTA (two CTAs share 512 columns)

struct BankGeom {
    bool pair;      // two output rows per accumulator (see the pair mode below)
    int nTpad;      // templates padded to a multiple of 32 (MMA N; 32-column TMEM loads)
    int nK16;       // 16-column template chunks (MMA K steps per template row)
    int G;          // template rows per exact accumulator group
    int nG;         // groups
    int accCols;    // tensor-memory columns per accumulator (nTpad * nG)
    int na;         // accumulator stages
    int tmemCols;   // allocated columns (power of two >= na * accCols)
    int xBlocks;    // 8-pixel blocks per A buffer
    int xBytes;     // bytes per A buffer
    int nx;         // A buffers in the ring
    int bBytes;     // B operand bytes (all template rows and chunks)
    int offB, offX, offSt, offBar, smemBytes;
};

int pow2_at_least(int v) {
    int p = 32;
    while (p < v) p <<= 1;
    return p;
}

// Pair mode (one exact group, nTpad <= 64): one accumulator holds output rows
// y and y+1 of every template (N = 2*nTpad).  Image row y+d meets template
// row d for output row y and template row d-1 for output row y+1, so one MMA
// per image row d = 0..hT serves both rows: hT+1 MMAs per two output rows
// instead of 2*hT.  B is stored with the template rows upside down between
// two zero blocks -- block b holds template row hT-b, blocks 0 and hT+1 are
// zero -- in the layout [K chunk][K half][block][template][8 k], so the
// operand of image row d is the two consecutive blocks hT-d, hT-d+1.
bool make_geom(int wT, int hT, int nT, bool pair, BankGeom &g) {
    if (wT > kMaxExactPixels) return false;
    g.pair = pair;
    g.nTpad = (nT + 31) / 32 * 32;
    if (g.nTpad > 256) return false;
    g.nK16 = (wT + 15) / 16;
    g.G = kMaxExactPixels / wT;
    if (g.G > hT) g.G = hT;
    g.nG = (hT + g.G - 1) / g.G;
    if (pair && (g.nG != 1 || g.nTpad > 64)) return false;
    g.accCols = g.nTpad * g.nG * (pair ? 2 : 1);
    if (g.accCols > kMaxTmemCols) return false;
    g.na = kMaxTmemCols / g.accCols;
    if (g.na > 4) g.na = 4;
    g.tmemCols = pow2_at_least(g.na * g.accCols);
    if (g.tmemCols > kMaxTmemCols) return false;
    g.xBlocks = 15 + 2 * g.nK16;
    g.xBytes = g.xBlocks * 128;
    g.bBytes = pair ? g.nK16 * 2 * (hT + 2) * g.nTpad * 16 : hT * g.nK16 * g.nTpad * 32;
    g.offB = 0;
    g.offX = (g.bBytes + 1023) / 1024 * 1024;
    // The ring of converted image rows: an accumulator uses hT+1 of them at
    // once, so the converters run ahead by nx - hT - 1 rows.  As many spare
    // rows as fit (up to 16), at least 3.
    for (g.nx = hT + 16; g.nx >= hT + 4; --g.nx) {
        g.offSt = g.offX + g.nx * g.xBytes;
        const int stBytes = g.nTpad * 8;   // float2 {SumT, 1/sqrt(vT)} per template
        g.offBar = (g.offSt + stBytes + 15) / 16 * 16;
        const int barBytes = (2 * g.nx + 2 * g.na) * 8 + 16;
        g.smemBytes = g.offBar + barBytes + 1024;  // + alignment slack
        if (g.smemBytes <= kMaxSmem) return true;
    }
    return false;
}

struct BParams {
    const uint8_t *img;
    int W, H;
    const uint8_t *tmpl;
    int wT, hT, nT;
    const long long *S, *Q;
    float *out;
    long long *sumI, *sumI2, *sumIT;
    int *status;
    int Ox, Oy, ntx, ntiles;
    BankGeom g;
};

__device__ __forceinline__ uint32_t saddr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ float u64_to_f32(unsigned long long a) {
    return fmaf(__uint2float_rn((unsigned)(a >> 32)), 4294967296.0f, __uint2float_rn((unsigned)a));
}

// 1/sqrt(v) from the hardware approximation (relative error about 2^-22.9),
// flushing subnormals: v is an integer >= 1 here.
__device__ __forceinline__ float rsqrt_approx(float v) {
    float r;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ float i64_to_f32(long long v) {
    const float f = u64_to_f32(v < 0 ? (unsigned long long)(-v) : (unsigned long long)v);
    return v < 0 ? -f : f;
}

// shared-memory matrix descriptor, no swizzle (tcgen05 version field = 1)
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)(lbo >> 4) << 16) |
           ((uint64_t)(sbo >> 4) << 32) | (1ull << 46);
}

__device__ __forceinline__ void mbar_init(unsigned long long *b, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(b)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(unsigned long long *b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(b)) : "memory");
}

// Bounded wait for the phase with the given parity.  After the first wait
// that runs out, *abort short-circuits every later wait of the CTA.
__device__ __forceinline__ void mbar_wait(unsigned long long *b, uint32_t parity, int *abort,
                                          int *status) {
    uint32_t done = 0;
    asm volatile(
        "{ .reg .pred P; mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2; selp.u32 %0, 1, 0, P; }"
        : "=r"(done) : "r"(saddr(b)), "r"(parity) : "memory");
    if (done || *(volatile int *)abort) return;  // fast path: no timer read
    const uint64_t t0 = global_timer_ns();
    for (unsigned it = 0; !done; ++it) {
        asm volatile(
            "{ .reg .pred P; mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2; selp.u32 %0, 1, 0, P; }"
            : "=r"(done) : "r"(saddr(b)), "r"(parity) : "memory");
        if (!done && (it & 1023u) == 1023u) {
            if (*(volatile int *)abort) return;
            if (global_timer_ns() - t0 > 2000000000ull || it > (1u << 26)) {
                *(volatile int *)abort = 1;
                record_status(status, NCC_ERR_TIMEOUT);
                return;
            }
        }
    }
}

// The same for a whole warp: one lane polls, the answer is shuffled to the
// others (one barrier access instead of 32; the warp's control flow stays
// uniform).
__device__ __forceinline__ void mbar_wait_warp(unsigned long long *b, uint32_t parity, int *abort,
                                               int *status) {
    uint32_t done = 0;
    if ((threadIdx.x & 31u) == 0)
        asm volatile(
            "{ .reg .pred P; mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2; selp.u32 %0, 1, 0, P; }"
            : "=r"(done) : "r"(saddr(b)), "r"(parity) : "memory");
    if (!__shfl_sync(0xffffffffu, done, 0)) mbar_wait(b, parity, abort, status);
}

// Non-blocking test of a phase: its result can be consumed later, so the
// test's latency overlaps whatever the thread issues meanwhile.
__device__ __forceinline__ uint32_t mbar_test(unsigned long long *b, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred P; mbarrier.test_wait.parity.shared::cta.b64 P, [%1], %2; selp.u32 %0, 1, 0, P; }"
        : "=r"(done) : "r"(saddr(b)), "r"(parity) : "memory");
    return done;
}

// Bounded wait by one thread (mbar_wait's loop without the warp exchange).
__device__ __forceinline__ void mbar_wait_lane(unsigned long long *b, uint32_t parity, int *abort,
                                               int *status) {
    mbar_wait(b, parity, abort, status);
}

__device__ __forceinline__ void tc_commit(unsigned long long *b) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(saddr(b)) : "memory");
}

__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
    asm volatile("{ .reg .pred p; setp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
                 ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
          "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
          "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
}

// Two pixels (bytes lo, hi of `w` selected by `sel`) as exact f16x2: the
// byte is placed in the mantissa of 1024.0h and 1024 is subtracted.
__device__ __forceinline__ uint32_t bytes_to_h2(uint32_t w, uint32_t sel) {
    const uint32_t biased = __byte_perm(w, 0x64646464u, sel);
    __half2 h = *reinterpret_cast<const __half2 *>(&biased);
    h = __hsub2(h, __halves2half2(__float2half(1024.f), __float2half(1024.f)));
    return *reinterpret_cast<uint32_t *>(&h);
}

template <bool kMoments, bool kOneGroup, bool kPair>
__global__ void __launch_bounds__(kThreads, 2) bank_tc_kernel(const BParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    const BankGeom &g = p.g;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    float2 *sts = reinterpret_cast<float2 *>(smem + g.offSt);  // [nTpad] {SumT, 1/sqrt(vT)}
    unsigned long long *bar = reinterpret_cast<unsigned long long *>(smem + g.offBar);
    unsigned long long *xfull = bar, *xempty = bar + g.nx;
    unsigned long long *afull = bar + 2 * g.nx, *aempty = afull + g.na;

    // --- prologue: B operand, template statistics, barriers, tensor memory ---
    {
        const int perRow = g.nK16 * g.nTpad * 16;  // f16 elements per template row
        const int total = (kPair ? p.hT + 2 : p.hT) * perRow;
        for (int e = tid; e < total; e += kThreads) {
            const int jb = e / perRow, rem = e - jb * perRow;
            const int c = rem / (g.nTpad * 16), r2 = rem - c * g.nTpad * 16;
            const int n = r2 >> 4, k = r2 & 15;
            const int col = 16 * c + k;
            // pair mode: block jb holds template row hT - jb (blocks 0, hT+1 zero)
            const int j = kPair ? p.hT - jb : jb;
            const float v = (j >= 0 && j < p.hT && n < p.nT && col < p.wT)
                                ? (float)__ldg(p.tmpl + ((size_t)n * p.hT + j) * p.wT + col) : 0.f;
            // K-major core matrices: (k/8) * (K-half stride) + (n/8) * 128 + (n%8) * 16 + (k%8) * 2
            const int off = kPair ? ((c * 2 + (k >> 3)) * (p.hT + 2) + jb) * g.nTpad * 16 +
                                        (n >> 3) * 128 + (n & 7) * 16 + (k & 7) * 2
                                  : (jb * g.nK16 + c) * g.nTpad * 32 + (k >> 3) * g.nTpad * 16 +
                                        (n >> 3) * 128 + (n & 7) * 16 + (k & 7) * 2;
            if (NCC_BOUNDS(off >= 0 && off + 2 <= g.bBytes, p.status))
                *reinterpret_cast<__half *>(smem + g.offB + off) = __float2half(v);
        }
        const long long N = (long long)p.wT * p.hT;
        for (int n = tid; n < g.nTpad; n += kThreads) {
            unsigned a = 0, b = 0;
            if (n < p.nT) {
                const uint8_t *t = p.tmpl + (size_t)n * p.wT * p.hT;
                for (int i = 0; i < p.wT * p.hT; ++i) {
                    const unsigned v = __ldg(t + i);
                    a += v;
                    b += v * v;
                }
            }
            const long long v2 = N * (long long)b - (long long)a * (long long)a;
            sts[n] = make_float2((float)a,  // SumT < 2^25: exact
                                 (n < p.nT && v2 > 0) ? __frsqrt_rn(u64_to_f32((unsigned long long)v2)) : 0.f);
        }
        if (tid == 0) {
            for (int i = 0; i < g.nx; ++i) { mbar_init(&xfull[i], 1); mbar_init(&xempty[i], 1); }
            for (int i = 0; i < g.na; ++i) { mbar_init(&afull[i], 1); mbar_init(&aempty[i], kEpiThreads / 32); }
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            s_abort = 0;
        }
        if (warp == 0) {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                         ::"r"(saddr(&s_tmem)), "r"(g.tmemCols) : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    }
    const uint32_t tmem = s_tmem;
    const long long N = (long long)p.wT * p.hT;
    // instruction descriptor: D f32, A/B f16, A MN-major, B K-major, N, M = 128
    const uint32_t mmaN = kPair ? 2 * g.nTpad : g.nTpad;
    const uint32_t idesc = (1u << 4) | (1u << 15) | ((mmaN >> 3) << 17) | ((uint32_t)(kM >> 4) << 24);

    // image rows / output rows / accumulators (rows or row pairs) handled so far (all tiles)
    uint32_t rowSeq = 0, accSeq = 0;
    for (int tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x) {
        const int xt = tile % p.ntx, yb = tile / p.ntx;
        const int x0 = xt * kM, y0 = yb * kTY;
        const int ty = min(kTY, p.Oy - y0);
        const int nrows = ty + p.hT - 1;

        if (warp >= 1 && warp <= 3) {
            // ---- producers: image rows -> f16 shifted-copy A buffers.  Each of
            // the three warps converts every third row on its own, with all of
            // a row's loads issued before its conversions, so that three rows
            // are in flight at once (a row done by all three warps together
            // was latency-bound, one global load round trip per row) ----
            const int cw = warp - 1;
            const bool aligned8 = (p.W % 8 == 0) && ((uintptr_t)p.img % 8 == 0);
            constexpr int kMaxChunks = 8;  // chunk rows per lane: (15 + 2*nK16)*8 / 32
            const int nChunkRows = g.xBlocks * 8;
            for (int rl = cw; rl < nrows; rl += kProducers / 32) {
                const uint32_t q = rowSeq + rl, slot = q % g.nx, k = q / g.nx;
                if (k > 0) mbar_wait_warp(&xempty[slot], (k - 1) & 1, &s_abort, p.status);
                uint8_t *X = smem + g.offX + slot * g.xBytes;
                const uint8_t *src = p.img + (size_t)(y0 + rl) * p.W;
                for (int r0 = 0; r0 < nChunkRows; r0 += 32 * kMaxChunks) {
                    uint2 lo[kMaxChunks], hi[kMaxChunks];
#pragma unroll
                    for (int i = 0; i < kMaxChunks; ++i) {
                        const int row = r0 + lane + 32 * i;
                        const int xb = x0 + 8 * (row >> 3);
                        lo[i] = hi[i] = make_uint2(0, 0);
                        if (row < nChunkRows && aligned8 && xb + 16 <= p.W) {
                            lo[i] = __ldg(reinterpret_cast<const uint2 *>(src + xb));
                            hi[i] = __ldg(reinterpret_cast<const uint2 *>(src + xb + 8));
                        }
                    }
#pragma unroll
                    for (int i = 0; i < kMaxChunks; ++i) {
                        const int row = r0 + lane + 32 * i;
                        if (row >= nChunkRows) break;
                        const int xb = x0 + 8 * (row >> 3), sh = row & 7;
                        const int c0 = xb + sh;  // pixel of element 0
                        uint32_t w0 = 0, w1 = 0;
                        if (aligned8 && xb + 16 <= p.W) {
                            // a funnel shift by sh bytes of the two aligned 8-byte loads
                            const bool up = sh >= 4;
                            const uint32_t a0 = up ? lo[i].y : lo[i].x, a1 = up ? hi[i].x : lo[i].y,
                                           a2 = up ? hi[i].y : hi[i].x;
                            w0 = __funnelshift_r(a0, a1, 8u * (uint32_t)(sh & 3));
                            w1 = __funnelshift_r(a1, a2, 8u * (uint32_t)(sh & 3));
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                if (c0 + e < p.W) w0 |= (uint32_t)__ldg(src + c0 + e) << (8 * e);
                                if (c0 + 4 + e < p.W) w1 |= (uint32_t)__ldg(src + c0 + 4 + e) << (8 * e);
                            }
                        }
                        uint4 h;
                        h.x = bytes_to_h2(w0, 0x4140);
                        h.y = bytes_to_h2(w0, 0x4342);
                        h.z = bytes_to_h2(w1, 0x4140);
                        h.w = bytes_to_h2(w1, 0x4342);
                        if (NCC_BOUNDS(slot < (uint32_t)g.nx && row * 16 + 16 <= g.xBytes, p.status))
                            *reinterpret_cast<uint4 *>(X + row * 16) = h;
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&xfull[slot]);
            }
        } else if (warp == 0) {
            // ---- MMA issuer: lane 0 alone.  The tensor pipe accepts an MMA
            // only about one instruction ahead of the one it executes, so a
            // wait between MMAs leaves it idle (a test of even a completed
            // mbarrier takes some 200 cycles).  Before it issues an
            // accumulator's MMAs, the issuer therefore tests (without
            // blocking) the barriers of the next accumulator -- its
            // accumulator stage and the image rows it needs -- and after them
            // waits only for what the tests did not find complete.
            // Descriptors are linear in the shared address (field = addr >> 4)
            // and slots and phases advance incrementally: no divisions. ----
            if (lane == 0) {
                const uint64_t adesc0 = smem_desc(saddr(smem + g.offX), 128, 128);
                const uint64_t bdesc0 = smem_desc(saddr(smem + g.offB), g.nTpad * 16, 128);
                const uint32_t xStep = (uint32_t)g.xBytes >> 4;                 // next A buffer
                const uint32_t bRow = (uint32_t)(g.nK16 * g.nTpad * 32) >> 4;  // next template row
                const uint32_t bChunk = (uint32_t)(g.nTpad * 32) >> 4;         // next K chunk
                const uint32_t nx = (uint32_t)g.nx, na = (uint32_t)g.na;
                const uint32_t slot0 = rowSeq % nx;                             // slot of image row y0
                // next image row to confirm (this tile's row `ready`), its slot and phase
                int ready = 0;
                uint32_t rSlot = slot0, rPhase = (rowSeq / nx) & 1;
                // rows [ready, tested) were found complete by a look-ahead test
                int tested = 0;
                // stage of the current accumulator, how often the stage was used
                // before (aK) and aK's parity
                uint32_t aSlot = accSeq % na, aK = accSeq / na, aPhase = aK & 1;
                bool aTested = false;
                // confirms this tile's image rows up to `need` (waiting for those no test saw)
                auto confirm_rows = [&](int need) {
                    while (ready <= need) {
                        if (ready >= tested)
                            mbar_wait_lane(&xfull[rSlot], rPhase, &s_abort, p.status);
                        ++ready;
                        if (++rSlot == nx) { rSlot = 0; rPhase ^= 1u; }
                    }
                };
                // tests the image rows (ready, need] after the confirmed ones, in order
                auto test_rows = [&](int need) {
                    int r = max(ready, tested);
                    uint32_t s = rSlot, ph = rPhase;
                    for (int k = ready; k < r; ++k) { if (++s == nx) { s = 0; ph ^= 1u; } }
                    for (; r <= need && r < nrows; ++r) {
                        if (!mbar_test(&xfull[s], ph)) break;
                        tested = r + 1;
                        if (++s == nx) { s = 0; ph ^= 1u; }
                    }
                };
                auto next_acc = [&]() {
                    if (++aSlot == na) { aSlot = 0; aPhase ^= 1u; ++aK; }
                };
                const int accPerTile = kPair ? (ty + 1) >> 1 : ty;
                uint32_t ySlot = slot0;  // slot of image row y0 + yl
                for (int ai = 0; ai < accPerTile; ++ai) {
                    const int yl = kPair ? 2 * ai : ai;
                    // this accumulator: its stage free, its image rows converted
                    if (aK > 0 && !aTested)
                        mbar_wait_lane(&aempty[aSlot], aPhase ^ 1u, &s_abort, p.status);
                    const int dmax = kPair ? (yl + 1 < ty ? p.hT : p.hT - 1) : p.hT - 1;
                    confirm_rows(yl + dmax);
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    // look-ahead for the next accumulator (results used after the MMAs)
                    const uint32_t nSlot = aSlot + 1 == na ? 0u : aSlot + 1;
                    const uint32_t nK = aSlot + 1 == na ? aK + 1 : aK;
                    aTested = nK == 0 || mbar_test(&aempty[nSlot], (nK & 1u) ^ 1u);
                    if (ai + 1 < accPerTile) {
                        const int yn = kPair ? yl + 2 : yl + 1;
                        const int dn = kPair ? (yn + 1 < ty ? p.hT : p.hT - 1) : p.hT - 1;
                        test_rows(yn + dn);
                    }
                    uint32_t s = ySlot;
                    const uint32_t d0 = tmem + aSlot * g.accCols;
                    if (kPair) {
                        // B window of image row d: blocks hT-d and hT-d+1 (see make_geom)
                        const uint64_t bdescP = smem_desc(saddr(smem + g.offB), (uint32_t)((p.hT + 2) * g.nTpad * 16), 128);
                        const uint32_t bBlk = (uint32_t)(g.nTpad * 16) >> 4;
                        const uint32_t bChunkP = (uint32_t)(2 * (p.hT + 2) * g.nTpad * 16) >> 4;
                        for (int dd = 0; dd <= dmax; ++dd) {
                            // A slot in the ring; B blocks hT-dd and hT-dd+1 of hT+2;
                            // N = 2*nTpad columns of this accumulator stage
                            if (!NCC_BOUNDS(s < nx && p.hT - dd >= 0 && p.hT - dd + 1 <= p.hT + 1 &&
                                                (aSlot + 1) * (uint32_t)g.accCols <= (uint32_t)g.tmemCols,
                                            p.status)) {
                                if (++s == nx) s = 0;
                                continue;
                            }
                            const uint64_t ad = adesc0 + (uint64_t)(s * xStep);
                            const uint64_t bd = bdescP + (uint64_t)((p.hT - dd) * bBlk);
                            for (int c = 0; c < g.nK16; ++c)
                                tc_mma(d0, ad + 16u * c, bd + c * bChunkP, idesc,
                                       (dd != 0 || c != 0) ? 1u : 0u);
                            if (++s == nx) s = 0;
                        }
                        tc_commit(&afull[aSlot]);
                        tc_commit(&xempty[ySlot]);  // image rows y0+yl, y0+yl+1 done
                        if (yl + 1 < ty) tc_commit(&xempty[ySlot + 1 == nx ? 0 : ySlot + 1]);
                    } else {
                        uint32_t d = d0;
                        uint64_t bd = bdesc0;
                        int inGroup = 0;
                        for (int j = 0; j < p.hT; ++j) {
                            const uint64_t ad = adesc0 + (uint64_t)(s * xStep);
                            if (NCC_BOUNDS(s < nx && d + (uint32_t)g.nTpad <= tmem + (aSlot + 1) * (uint32_t)g.accCols,
                                           p.status))
                            for (int c = 0; c < g.nK16; ++c)
                                tc_mma(d, ad + 16u * c, bd + c * bChunk, idesc,
                                       (inGroup != 0 || c != 0) ? 1u : 0u);
                            bd += bRow;
                            if (++s == nx) s = 0;
                            if (++inGroup == g.G) { inGroup = 0; d += g.nTpad; }
                        }
                        tc_commit(&afull[aSlot]);
                        tc_commit(&xempty[ySlot]);  // image row y0+yl is done
                    }
                    next_acc();
                    for (int k = 0; k < (kPair ? 2 : 1); ++k)
                        if (++ySlot == nx) ySlot = 0;
                }
                for (int rl = ty; rl < nrows; ++rl) {
                    uint32_t e0 = (slot0 + (uint32_t)rl) % nx;
                    tc_commit(&xempty[e0]);
                }
            }
            __syncwarp();
        } else {
            // ---- epilogue: thread = shift x0 + 32*sp + lane; the two warps of a
            // lane quarter split the work: template chunks ci = ch (mod 2) of
            // every row, or (pair mode) every chunk of row ch of each pair, so
            // that no row's corners are loaded twice ----
            const int sp = warp & 3, ch = (warp - 4) >> 2;
            const int x = x0 + 32 * sp + lane;
            const uint32_t lane_base = (uint32_t)(32 * sp) << 16;
            const bool xin = x < p.Ox;
            const size_t W = (size_t)p.W, plane = (size_t)p.Oy * p.Ox;
            const int xl = x - 1, xr = x + p.wT - 1;
            const float Nf = (float)N;  // < 2^17: exact
            long long cS[4], cQ[4];     // corners of the current row: br, tr, bl, tl
            auto load_corners = [&](int y) {
                const int yt = y - 1, ybm = y + p.hT - 1;
                cS[0] = cS[1] = cS[2] = cS[3] = 0;
                cQ[0] = cQ[1] = cQ[2] = cQ[3] = 0;
                if (!xin) return;
                cS[0] = __ldg(p.S + (size_t)ybm * W + xr);
                cQ[0] = __ldg(p.Q + (size_t)ybm * W + xr);
                if (yt >= 0) { cS[1] = __ldg(p.S + (size_t)yt * W + xr); cQ[1] = __ldg(p.Q + (size_t)yt * W + xr); }
                if (xl >= 0) { cS[2] = __ldg(p.S + (size_t)ybm * W + xl); cQ[2] = __ldg(p.Q + (size_t)ybm * W + xl); }
                if (xl >= 0 && yt >= 0) { cS[3] = __ldg(p.S + (size_t)yt * W + xl); cQ[3] = __ldg(p.Q + (size_t)yt * W + xl); }
            };
            // pair mode: rows yl = ch, ch+2, ... (accumulator yl/2, row ch of
            // its two), all template chunks; otherwise every row, chunks ch, ch+2
            const int rowStep = kPair ? 2 : 1, yFirst = kPair ? ch : 0;
            const int ciStart = kPair ? 0 : ch, ciStep = kPair ? 1 : 2;
            const int nIter = kPair ? (ty + 1) >> 1 : ty;
            const uint32_t colq = kPair ? (uint32_t)ch * g.nTpad : 0u;
            if (yFirst < ty) load_corners(y0 + yFirst);
            for (int it = 0; it < nIter; ++it) {
                const int yl = yFirst + it * rowStep, y = y0 + yl;
                const bool valid = yl < ty;  // false only for row ch = 1 of a last single-row pair
                const uint32_t o = accSeq + (uint32_t)it, a = o % g.na, ka = o / g.na;
                const long long sI = cS[0] - cS[1] - cS[2] + cS[3];
                const long long sI2 = cQ[0] - cQ[1] - cQ[2] + cQ[3];
                if (yl + rowStep < ty) load_corners(y + rowStep);  // next row's corners, in flight meanwhile
                const long long vI = (long long)((unsigned long long)N * (unsigned)sI2) -
                                     (long long)((int)sI) * (long long)((int)sI);
                const float rsI = vI > 0 ? rsqrt_approx(u64_to_f32((unsigned long long)vI)) : 0.f;
                const float sIf = (float)(int)sI;  // < 2^25: exact
                // wait for the accumulator even for an invalid row: this warp's
                // aempty arrival below must not land before the stage's
                // previous use is complete, or it would count toward that use
                // and let the issuer overwrite the stage while the other warp
                // of the lane quarter still reads it
                mbar_wait_warp(&afull[a], ka & 1, &s_abort, p.status);
                if (valid) {
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const size_t obase = (size_t)y * p.Ox + x;
                // lanes whose output (or window) a check finds outside the
                // map store nothing; the warp-wide loads still run in step
                const bool xok = xin && NCC_BOUNDS(y < p.Oy && x < p.Ox && y + p.hT - 1 < p.H &&
                                                       x + p.wT - 1 < p.W, p.status);
                if (kMoments && xok && (kPair || ch == 0)) {
                    p.sumI[obase] = sI;
                    p.sumI2[obase] = sI2;
                }
                for (int ci = ciStart; ci * 32 < g.nTpad; ci += ciStep) {
                    const int cc = 32 * ci;
                    uint32_t v[32];
                    tc_ld32(tmem + lane_base + a * g.accCols + colq + cc, v);
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                    if (!kOneGroup) {
                        // several exact groups: sum their integer values
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = __float2uint_rn(__uint_as_float(v[i]));
                        for (int gi = 1; gi < g.nG; ++gi) {
                            uint32_t w[32];
                            tc_ld32(tmem + lane_base + a * g.accCols + gi * g.nTpad + cc, w);
                            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] += __float2uint_rn(__uint_as_float(w[i]));
                        }
                    }
                    if (!xok) continue;
                    if constexpr (!kMoments && kOneGroup) {
                        // r = (N*SumIT - SumI*SumT) / sqrt(vI*vT) with the numerator
                        // exact up to its last rounding: p2 = fl(SumI*SumT), e2 its
                        // exact error (fma), fma(N, SumIT, -p2) a single rounding of
                        // N*SumIT - p2 (exact whenever it is small).  The output
                        // pointer steps one template plane per coefficient.
                        float *op = p.out + obase + (size_t)cc * plane;
                        const float4 *st4 = reinterpret_cast<const float4 *>(sts + cc);
                        auto run = [&](auto fullTag) {
                            constexpr bool kFullChunk = decltype(fullTag)::value;
                            const int nHere = p.nT - cc;
#pragma unroll
                            for (int i = 0; i < 32; i += 2) {
                                const float4 s2 = st4[i / 2];
#pragma unroll
                                for (int j = 0; j < 2; ++j) {
                                    if (!kFullChunk && i + j >= nHere) continue;
                                    const float sT = j ? s2.z : s2.x, rT = j ? s2.w : s2.y;
                                    const float sit = __uint_as_float(v[i + j]);  // exact integer < 2^24
                                    const float p2 = sIf * sT, e2 = fmaf(sIf, sT, -p2);
                                    const float num = fmaf(Nf, sit, -p2) - e2;
                                    float r = num * (rsI * rT);
                                    r = fminf(1.0f, fmaxf(-1.0f, r));
                                    __stcs(op, r);
                                    op += plane;
                                }
                            }
                        };
                        if (cc + 32 <= p.nT) run(BoolTag<true>{});
                        else run(BoolTag<false>{});
                    } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int t = cc + i;
                        if (t >= p.nT) continue;
                        const size_t oo = obase + (size_t)t * plane;
                        const float2 st = sts[t];
                        if (kMoments) {
                            p.sumIT[oo] = kOneGroup ? (long long)__float2uint_rn(__uint_as_float(v[i]))
                                                    : (long long)v[i];
                            continue;
                        }
                        float num;
                        if (kOneGroup) {
                            // exact N*SumIT - SumI*SumT up to the final rounding
                            const float sit = __uint_as_float(v[i]);  // exact integer < 2^24
                            const float p1 = Nf * sit, e1 = fmaf(Nf, sit, -p1);
                            const float p2 = sIf * st.x, e2 = fmaf(sIf, st.x, -p2);
                            num = (p1 - p2) + (e1 - e2);
                        } else {
                            num = i64_to_f32((long long)((unsigned long long)N * v[i]) -
                                             (long long)((int)sI) * (long long)st.x);
                        }
                        float r = num * (rsI * st.y);
                        r = fminf(1.0f, fmaxf(-1.0f, r));
                        __stcs(p.out + oo, r);
                    }
                    }
                }
                }
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&aempty[a]);
            }
        }
        rowSeq += nrows;
        accSeq += kPair ? (uint32_t)((ty + 1) >> 1) : (uint32_t)ty;
    }

    // --- teardown: every accumulator has been drained by the epilogue ---
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     ::"r"(tmem), "r"(g.tmemCols) : "memory");
}

int g_num_sms[64] = {};

}  // namespace

bool bank_tc_supported(int W, int H, int wT, int hT, int nT) {
    (void)W;
    (void)H;
    BankGeom g;
    return nT >= 2 && (make_geom(wT, hT, nT, true, g) || make_geom(wT, hT, nT, false, g));
}

cudaError_t bank_tc_launch(const BankArgs &a, cudaStream_t stream) {
    BParams p;
    p.img = a.img; p.W = a.W; p.H = a.H;
    p.tmpl = a.tmpl; p.wT = a.wT; p.hT = a.hT; p.nT = a.nT;
    p.S = reinterpret_cast<const long long *>(a.S);
    p.Q = reinterpret_cast<const long long *>(a.Q);
    p.out = a.out;
    p.sumI = reinterpret_cast<long long *>(a.sumI);
    p.sumI2 = reinterpret_cast<long long *>(a.sumI2);
    p.sumIT = reinterpret_cast<long long *>(a.sumIT);
    p.status = a.status;
    p.Ox = a.W - a.wT + 1;
    p.Oy = a.H - a.hT + 1;
    p.ntx = (p.Ox + kM - 1) / kM;
    p.ntiles = p.ntx * ((p.Oy + kTY - 1) / kTY);
    if (!make_geom(a.wT, a.hT, a.nT, true, p.g) && !make_geom(a.wT, a.hT, a.nT, false, p.g))
        return cudaErrorNotSupported;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!g_num_sms[dev]) {
        e = cudaDeviceGetAttribute(&g_num_sms[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    const int grid = p.ntiles < 2 * g_num_sms[dev] ? p.ntiles : 2 * g_num_sms[dev];
    const size_t smem = (size_t)p.g.smemBytes;
#define NCC_BANK(M, G1, PR)                                                                   \
    do {                                                                                         \
        e = cudaFuncSetAttribute(bank_tc_kernel<M, G1, PR>,                                      \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);        \
        if (e != cudaSuccess) return e;                                                          \
        bank_tc_kernel<M, G1, PR><<<grid, kThreads, smem, stream>>>(p);                          \
    } while (0)
    const bool one = p.g.nG == 1, pair = p.g.pair;
    if (a.sumIT) {
        if (pair) NCC_BANK(true, true, true);
        else if (one) NCC_BANK(true, true, false);
        else NCC_BANK(true, false, false);
    } else {
        if (pair) NCC_BANK(false, true, true);
        else if (one) NCC_BANK(false, true, false);
        else NCC_BANK(false, false, false);
    }
#undef NCC_BANK
    return cudaGetLastError();
}

}  // namespace ncc
