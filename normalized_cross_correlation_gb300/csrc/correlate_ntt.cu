// correlate_ntt.cu -- one template against every valid shift of an 8-bit
// image, with the numerator SumIT formed by number-theoretic transforms of
// 256 x 256 image tiles (exact: the FFT over the integers modulo a prime),
// and the epilogue of the other single-template kernels: window moments from
// the summed-area tables (four-corner box sums) and fp32 coefficients.
//
// The CUDA Handbook, section 15.8 ("The Denominator: Summed Area Tables"),
// names the FFT numerator as the alternative the tables serve; chapter 15's
// "Image in shared memory" (Listing 15-5) defines the per-shift sum it
// replaces.  The transform arithmetic is in ntt_tile.cuh.
//
// Overlap-save tiling: tile (ty, tx) covers image rows ty*Vy .. +255 and
// columns tx*Vx .. +255 (zeros beyond the image), with Vy = 257 - hT and
// Vx = 257 - wT rounded down to a multiple of 16 (aligned tile columns).
// Its cyclic correlation with the template equals the true correlation at
// the Vy x Vx shifts whose windows do not wrap, and those shifts tile the
// output map.  The values are centered (I - 128, T - 128),
// so |C| <= 2^14 * wT * hT, and
//     SumIT = C + 128 * SumI + 128 * SumT - 16384 * N     (mod 2^32, exact).
//
// Kernels:
//   ntt_spectrum_kernel  two CTAs: the even and odd halves of the template's
//                        spectrum (the reversed, centered template in a
//                        256 x 256 tile, transformed like an image tile),
//                        scaled by 1/65536, with Shoup companions (512 KB);
//   ntt_corr_kernel      persistent, one CTA of 512 threads per SM: per tile
//                        the pixels staged in shared memory (64 KB), the even
//                        half (transform, product, inverse) parked in tensor
//                        memory (tcgen05.st; no MMA), then the odd half, then
//                        the combination y[r] = e[r] + w^-r o[r] (written
//                        back into the buffer) and y[r+128] = e[r] - w^-r o[r]
//                        (parked), and the epilogue of each half from the
//                        buffer, one output row per warp.
//                        Every step is a barrier-separated pass over the
//                        136 KB shared buffer; no waits other than
//                        __syncthreads.
#include "ncc_common.cuh"
#include "ntt_tile.cuh"

namespace ncc {
namespace {

using ntt::kHalf;
using ntt::kL;
using ntt::kP;
using ntt::kP2;
using ntt::kThreads;

constexpr int kMaxSide = 224;  // at least 33 valid rows and columns per tile
constexpr uint32_t kTmemCols = 256;  // 16 warps x 64 words per thread, parked between passes

__device__ __forceinline__ uint32_t centered_pixel(uint32_t v) {
    return (uint32_t)((int)v - 128) + (v < 128u ? kP : 0u);
}

__device__ __forceinline__ float u64_to_f32(unsigned long long a) {
    return fmaf(__uint2float_rn((unsigned)(a >> 32)), 4294967296.0f, __uint2float_rn((unsigned)a));
}

__device__ __forceinline__ float i64_to_f32(long long v) {
    const float f = u64_to_f32(v < 0 ? (unsigned long long)(-v) : (unsigned long long)v);
    return v < 0 ? -f : f;
}

// Tensor memory as parking space for a warp's 32 x 16 words: lane = the
// thread's lane within its warp's quarter, 16 consecutive columns.
__device__ __forceinline__ void tm_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
          "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ void tm_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tm_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tm_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 1/sqrt(v) from the hardware approximation, flushing subnormals: v >= 1 here
__device__ __forceinline__ float rsqrt_approx(float v) {
    float r;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// The template's spectrum: CTA 0 the even half, CTA 1 the odd half.  The
// template enters reversed (cyclically: tile entry (a, b) holds template
// pixel ((-a) mod 256, (-b) mod 256)) so that the product of spectra gives
// the correlation, not the convolution.
__global__ void __launch_bounds__(kThreads, 1)
ntt_spectrum_kernel(const uint8_t *__restrict__ tmpl, int wT, int hT, uint2 *__restrict__ H) {
    extern __shared__ __align__(16) uint32_t smem[];
    const ntt::Tile t = ntt::carve(smem);
    const int tid = threadIdx.x;
    ntt::fill_tables(tid, kThreads, t);
    __syncthreads();
    auto load = [&](int a, int b) -> uint32_t {
        const int j = (kL - a) & (kL - 1), i = (kL - b) & (kL - 1);
        return (j < hT && i < wT) ? centered_pixel(__ldg(tmpl + (size_t)j * wT + i)) : 0u;
    };
    if (blockIdx.x == 0)
        ntt::rows_fwd1<false>(tid, t, load);
    else
        ntt::rows_fwd1<true>(tid, t, load);
    __syncthreads();
    ntt::rows_fwd2(tid, t);
    __syncthreads();
    ntt::cols_fwd1(tid, t);
    __syncthreads();
    ntt::cols_spectrum(tid, t, H + (size_t)blockIdx.x * kHalf * kL);
}

struct NttParams {
    const uint8_t *img;
    int W, H;
    const uint8_t *tmpl;
    int wT, hT;
    const uint2 *spec;  // [2][128][256] from ntt_spectrum_kernel
    const long long *S, *Q;
    float *out;
    long long *sumI, *sumI2, *sumIT;
    int *status;
    int Ox, Oy, Vx, Vy, ntx, ntiles;
    int vec16;  // img 16-byte aligned and W % 16 == 0: the tile rows load as 16-byte vectors
};

// forward transform, product with the template's half spectrum and inverse,
// up to the last inverse pass (which the caller runs into registers)
template <bool kOdd, class Load>
__device__ __forceinline__ void half_pass(int tid, const ntt::Tile &t, const uint2 *spec, Load &&load) {
    ntt::rows_fwd1<kOdd>(tid, t, load);
    __syncthreads();
    ntt::rows_fwd2(tid, t);
    __syncthreads();
    ntt::cols_fwd1(tid, t);
    __syncthreads();
    ntt::cols_mul(tid, t, spec + (kOdd ? (size_t)kHalf * kL : 0));
    __syncthreads();
    ntt::cols_inv(tid, t);
    __syncthreads();
    ntt::rows_inv1(tid, t);
    __syncthreads();
}

// Stages the tile's pixels (rows ty0.., columns tx0.., zeros outside the
// image) in shared memory, rows kImgStride bytes apart.  tx0 is a multiple of
// 16, so with vec16 every 16-byte chunk lies wholly inside or outside a row.
__device__ __forceinline__ void stage_tile(const NttParams &p, int ty0, int tx0, uint8_t *img_s) {
    const int tid = threadIdx.x;
    const size_t W = (size_t)p.W;
    if (p.vec16) {
#pragma unroll
        for (int k = 0; k < kL * kL / 16 / kThreads; ++k) {
            const int q = tid + kThreads * k, rr = q >> 4, ch = q & 15;
            const int y = ty0 + rr, x = tx0 + 16 * ch;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (y < p.H && x < p.W) v = __ldg(reinterpret_cast<const uint4 *>(p.img + (size_t)y * W + x));
            *reinterpret_cast<uint4 *>(img_s + rr * ntt::kImgStride + 16 * ch) = v;
        }
    } else {
#pragma unroll 4
        for (int k = 0; k < kL * kL / 4 / kThreads; ++k) {
            const int q = tid + kThreads * k, rr = q >> 6, wd = q & 63;
            const int y = ty0 + rr, x = tx0 + 4 * wd;
            uint32_t v = 0;
            if (y < p.H) {
                const uint8_t *src = p.img + (size_t)y * W;
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    if (x + b < p.W) v |= (uint32_t)__ldg(src + x + b) << (8 * b);
            }
            *reinterpret_cast<uint32_t *>(img_s + rr * ntt::kImgStride + 4 * wd) = v;
        }
    }
}

// The epilogue of one half of a tile's output rows (u0 = 0 or 128): the
// centered correlations C sit in the buffer, row u - u0, logical column
// x - tx0; a warp takes a row, its lanes consecutive shifts (coalesced box
// sums and stores).  The table reads of four 32-shift chunks are issued
// before any is used; their addresses are clamped into the row, so every
// read is in bounds and only the stores are conditional.
template <bool kMoments>
__device__ __forceinline__ void epilogue_half(const NttParams &p, const ntt::Tile &t, int ty0, int tx0,
                                              int u0, long long N, unsigned sT, uint32_t cT,
                                              float invSqrtVT) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rows = min(min(kHalf, p.Vy - u0), p.Oy - (ty0 + u0));
    const int cols = min(p.Vx, p.Ox - tx0);
    const size_t W = (size_t)p.W;
    for (int rr = warp; rr < rows; rr += kThreads / 32) {
        const int y = ty0 + u0 + rr;
        const unsigned *Sb = reinterpret_cast<const unsigned *>(p.S + (size_t)(y + p.hT - 1) * W);
        const unsigned *Qb = reinterpret_cast<const unsigned *>(p.Q + (size_t)(y + p.hT - 1) * W);
        const unsigned *St = reinterpret_cast<const unsigned *>(p.S + (size_t)(y > 0 ? y - 1 : 0) * W);
        const unsigned *Qt = reinterpret_cast<const unsigned *>(p.Q + (size_t)(y > 0 ? y - 1 : 0) * W);
        const uint32_t ym = y > 0 ? 0xffffffffu : 0u;
        const uint32_t *brow = t.buf + rr * ntt::kStride;
        for (int c0 = 0; c0 * 32 < cols; c0 += 4) {
            uint32_t v[4][8];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int x = tx0 + min(lane + 32 * (c0 + u), cols - 1);
                const size_t xr = (size_t)(x + p.wT - 1), xl = (size_t)(x > 0 ? x - 1 : 0);
                v[u][0] = __ldg(Sb + 2 * xr);
                v[u][1] = __ldg(Qb + 2 * xr);
                v[u][2] = __ldg(Sb + 2 * xl);
                v[u][3] = __ldg(Qb + 2 * xl);
                v[u][4] = __ldg(St + 2 * xr);
                v[u][5] = __ldg(Qt + 2 * xr);
                v[u][6] = __ldg(St + 2 * xl);
                v[u][7] = __ldg(Qt + 2 * xl);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int xo = lane + 32 * (c0 + u), x = tx0 + xo;
                if (xo >= cols) continue;
                if (!NCC_BOUNDS(y + p.hT - 1 < p.H && x + p.wT - 1 < p.W &&
                                    (size_t)y * p.Ox + x < (size_t)p.Oy * p.Ox, p.status))
                    continue;
                const int32_t c = (int32_t)brow[ntt::swz(xo)];
                // box sums from the low 32 bits of S and Q (below 2^32, so the
                // wrapping differences are exact)
                const uint32_t xm = x > 0 ? 0xffffffffu : 0u;
                const uint32_t sI = v[u][0] - (v[u][2] & xm) - (v[u][4] & ym) + (v[u][6] & xm & ym);
                const uint32_t sI2 = v[u][1] - (v[u][3] & xm) - (v[u][5] & ym) + (v[u][7] & xm & ym);
                const uint32_t sumIT = (uint32_t)c + 128u * sI + cT;
                const size_t oi = (size_t)y * p.Ox + x;
                if (kMoments) {
                    p.sumI[oi] = (long long)sI;
                    p.sumI2[oi] = (long long)sI2;
                    p.sumIT[oi] = (long long)sumIT;
                } else {
                    const long long numi =
                        (long long)((unsigned long long)N * sumIT) - (long long)sI * (long long)sT;
                    const long long vI =
                        (long long)((unsigned long long)N * sI2) - (long long)sI * (long long)sI;
                    const float num = i64_to_f32(numi);
                    const float vIf = u64_to_f32((unsigned long long)max(vI, 1ll));
                    // a zero-variance window has num = 0 exactly; invSqrtVT is
                    // 0 for a zero-variance template
                    const float r = num * rsqrt_approx(vIf) * invSqrtVT;
                    __stcs(p.out + oi, fminf(1.0f, fmaxf(-1.0f, r)));
                }
            }
        }
    }
}

template <bool kMoments>
__global__ void __launch_bounds__(kThreads, 1) ntt_corr_kernel(const NttParams p) {
    extern __shared__ __align__(16) uint32_t smem[];
    __shared__ unsigned st[2];
    __shared__ uint32_t s_tmem;
    const ntt::Tile t = ntt::carve(smem);
    uint8_t *img_s = reinterpret_cast<uint8_t *>(smem + ntt::kBufWords + ntt::kTableWords);
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid < 2) st[tid] = 0;
    if (warp == 0) {
        // one CTA per SM (its shared memory), so the columns are free
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"((uint32_t)__cvta_generic_to_shared(&s_tmem)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    ntt::fill_tables(tid, kThreads, t);
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    // this warp's parking columns: lane quarter warp % 4, 64 columns per warp
    const uint32_t tm = s_tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(64 * (warp >> 2));
    {
        // template sums (both below 2^32)
        const int N = p.wT * p.hT;
        unsigned s = 0, s2 = 0;
        for (int i = tid; i < N; i += kThreads) {
            const unsigned v = __ldg(p.tmpl + i);
            s += v;
            s2 += v * v;
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            s += __shfl_xor_sync(0xffffffffu, s, o);
            s2 += __shfl_xor_sync(0xffffffffu, s2, o);
        }
        if ((tid & 31) == 0) {
            atomicAdd(&st[0], s);
            atomicAdd(&st[1], s2);
        }
    }
    __syncthreads();
    const long long N = (long long)p.wT * p.hT;
    const unsigned sT = st[0], sT2 = st[1];
    const long long vT = N * (long long)sT2 - (long long)sT * (long long)sT;
    const float invSqrtVT = vT > 0 ? __frsqrt_rn(u64_to_f32((unsigned long long)vT)) : 0.0f;
    const uint32_t cT = 128u * sT - 16384u * (uint32_t)N;  // SumIT = C + 128 SumI + cT (mod 2^32)

    for (int tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x) {
        const int ty0 = (tile / p.ntx) * p.Vy, tx0 = (tile % p.ntx) * p.Vx;
        stage_tile(p, ty0, tx0, img_s);
        __syncthreads();
        auto load = [&](int r, int c) -> uint32_t {
            return centered_pixel(img_s[r * ntt::kImgStride + c]);
        };
        // even half: its last inverse pass goes to tensor memory
        half_pass<false>(tid, t, p.spec, load);
#pragma unroll 1
        for (int k = 0; k < 4; ++k) {
            uint32_t e[16];
            ntt::rows_inv2(tid, k, t, e);
            tm_st16(tm + 16 * k, e);
        }
        tm_wait_st();
        __syncthreads();  // read before the odd half overwrites the buffer
        half_pass<true>(tid, t, p.spec, load);
        // y[r] = e[r] + w^-r o[r] goes back into the buffer in place (each
        // thread rewrites exactly the words its last pass read);
        // y[r+128] = e[r] - w^-r o[r] goes to tensor memory
#pragma unroll 1
        for (int k = 0; k < 4; ++k) {
            uint32_t o[16], e[16];
            tm_ld16(tm + 16 * k, e);
            ntt::rows_inv2(tid, k, t, o);
            tm_wait_ld();
            const int idx = tid + kThreads * k, r = idx >> 4, n2 = idx & 15;
            const uint2 rf = t.rowFi[r];
            uint32_t *row = t.buf + r * ntt::kStride;
#pragma unroll
            for (int a = 0; a < 16; ++a) {
                const uint32_t ov = ntt::mulw(o[a], rf), ev = ntt::red2(e[a]);  // both in [0, 2p)
                row[16 * a + (n2 ^ a)] = (uint32_t)ntt::centered(ev + ov);
                e[a] = (uint32_t)ntt::centered(ev - ov + kP2);
            }
            tm_st16(tm + 16 * k, e);
        }
        tm_wait_st();
        __syncthreads();
        epilogue_half<kMoments>(p, t, ty0, tx0, 0, N, sT, cT, invSqrtVT);
        __syncthreads();
#pragma unroll 1
        for (int k = 0; k < 4; ++k) {
            uint32_t b[16];
            tm_ld16(tm + 16 * k, b);
            tm_wait_ld();
            const int idx = tid + kThreads * k, r = idx >> 4, n2 = idx & 15;
            uint32_t *row = t.buf + r * ntt::kStride;
#pragma unroll
            for (int a = 0; a < 16; ++a) row[16 * a + (n2 ^ a)] = b[a];
        }
        __syncthreads();
        epilogue_half<kMoments>(p, t, ty0, tx0, kHalf, N, sT, cT, invSqrtVT);
        __syncthreads();  // read before the next tile's staging and passes overwrite it
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(s_tmem), "r"(kTmemCols)
                     : "memory");
}

}  // namespace

bool corr_ntt_supported(int wT, int hT) {
    return wT >= 1 && hT >= 1 && wT <= kMaxSide && hT <= kMaxSide &&
           (long long)wT * hT <= ntt::kMaxPixels;
}

cudaError_t corr_ntt_launch(const CorrArgs &a, cudaStream_t stream) {
    if (!corr_ntt_supported(a.wT, a.hT) || a.direct) return cudaErrorNotSupported;
    NttParams p;
    p.img = a.img; p.W = a.W; p.H = a.H;
    p.tmpl = a.tmpl; p.wT = a.wT; p.hT = a.hT;
    p.S = reinterpret_cast<const long long *>(a.S);
    p.Q = reinterpret_cast<const long long *>(a.Q);
    p.out = a.out;
    p.sumI = reinterpret_cast<long long *>(a.sumI);
    p.sumI2 = reinterpret_cast<long long *>(a.sumI2);
    p.sumIT = reinterpret_cast<long long *>(a.sumIT);
    p.status = a.status;
    p.Ox = a.W - a.wT + 1;
    p.Oy = a.H - a.hT + 1;
    p.Vx = (kL + 1 - a.wT) & ~15;  // a multiple of 16: tile columns start 16-byte aligned
    p.Vy = kL + 1 - a.hT;
    p.ntx = (p.Ox + p.Vx - 1) / p.Vx;
    const long long ntiles = (long long)p.ntx * ((p.Oy + p.Vy - 1) / p.Vy);
    if (ntiles >= (1ll << 31)) return cudaErrorNotSupported;
    p.ntiles = (int)ntiles;
    p.vec16 = ((uintptr_t)a.img % 16 == 0 && a.W % 16 == 0) ? 1 : 0;
    const size_t smem = ntt::kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(ntt_spectrum_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    auto corr = a.sumIT ? ntt_corr_kernel<true> : ntt_corr_kernel<false>;
    e = cudaFuncSetAttribute(corr, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ntt::kImgSmemBytes);
    if (e != cudaSuccess) return e;
    uint2 *spec = nullptr;
    e = pool_alloc(reinterpret_cast<void **>(&spec), (size_t)2 * kHalf * kL * sizeof(uint2), stream);
    if (e != cudaSuccess) return e;
    p.spec = spec;
    ntt_spectrum_kernel<<<2, kThreads, smem, stream>>>(a.tmpl, a.wT, a.hT, spec);
    e = cudaGetLastError();
    if (e == cudaSuccess) {
        const int nsm = sm_count();
        const int grid = p.ntiles < nsm ? p.ntiles : nsm;
        corr<<<grid, kThreads, ntt::kImgSmemBytes, stream>>>(p);
        e = cudaGetLastError();
    }
    const cudaError_t ef = cudaFreeAsync(spec, stream);  // stream-ordered: after both kernels
    return e != cudaSuccess ? e : ef;
}

}  // namespace ncc
