// correlate_toeplitz_tc.cu -- one large template against every valid shift of
// an 8-bit image, with the numerator on the 5th-generation tensor cores
// (tcgen05.mma kind::f16, fp32 accumulation in tensor memory) in Toeplitz
// form, and an epilogue that takes the window moments from the summed-area
// tables (four-corner box sums) and writes the fp32 coefficients.
//
// Follows The CUDA Handbook, chapter 15: "Image in shared memory", Listing
// 15-5 (the per-shift sum of pixel-template products, and the staged image
// tile it reuses), and section 15.8 (the box sums of S and Q).  One template
// is a matrix-vector product per shift; written for 64 consecutive shifts at
// once it becomes a matrix product with a Toeplitz factor.  For the output
// tile of rows y0..y0+127 and shifts x0..x0+63, template row j adds
//     D[m][n] += sum_k I[y0+m+j][x0+k] * T[j][k-n],   k in [0, Kp)
// (T zero outside its columns), i.e. one MMA chain with M = 128 output rows,
// N = 64 shifts, K = Kp = 64 + wT - 1 rounded up to 16.  Each product is
// computed about Kp/wT times over (zeros of the Toeplitz factor) -- twice
// for a 64-wide template -- in exchange for the tensor pipe's rate.
//
// Operands, both K-major without swizzle, built by descriptor arithmetic:
//   A  the image tile, rows y0..y0+R-1 with R = 128 + hT - 1, columns
//      x0..x0+Kp-1 stored in reverse order: element (r, c') at
//      (c'/8)*R*16 + r*16 + (c'%8)*2.  Rows are 16 bytes apart, so template
//      row j is the same descriptor started 16*j bytes later (LBO = R*16,
//      SBO = 128).
//   B  with the columns reversed (k' = Kp-1-k) the Toeplitz factor becomes
//      a Hankel matrix, B[n][k'] = g_j[n + k'] with g_j[t] = T[j][Kp-1-t].
//      Its K-major rows are the 16-byte windows g_j[t..t+7] at t*16 bytes
//      (t = n + 8*kc), so one buffer of 56 + 16*Kp/16 rows per template row
//      serves every K chunk with LBO = SBO = 128.
// Exactness: pixels and template values enter centered, I-128 and T-128,
// both in [-128, 127] and exact in f16.  A product is at most 2^14 in
// magnitude, so every partial sum of at most 1024 products is an integer of
// magnitude at most 2^24, exact in fp32.  Template rows go in groups of
// G = floor(1024 / wT) rows, each group into its own accumulator columns;
// the epilogue converts the groups to integers and adds them, then
//     SumIT = C + 128*SumI + 128*SumT - 16384*N,   C = sum (I-128)(T-128),
// which is exact in wrapping 32-bit arithmetic because SumIT < 2^32.
//
// Warp roles (persistent CTAs, one per SM, 512 threads; the image tile and
// the accumulator are double-buffered, so one tile's MMAs overlap the next
// tile's image conversion and the previous tile's epilogue):
//   warp 0      allocates tensor memory (2 x 256 columns); one lane issues
//               the MMAs and commits,
//   warps 1-4   the image tiles: u8 -> centered f16, columns reversed,
//   warps 5-7   per template row, its Hankel buffer in a ring,
//   warps 8-15  epilogue: two warps per tensor-memory lane quarter (one per
//               32-shift half).  While the MMAs run, an L2 prefetch of the
//               block's table rows; then tcgen05.ld of every group and
//               integer sums; the warp's 32 x 32 block goes through shared
//               memory, so the box sums from S and Q and the fp32 stores run
//               along x (coalesced), one output row at a time.
// The tensor pipe accepts an MMA only about one instruction ahead of the one
// it executes, so the issuing thread must not wait between MMAs: Hankel
// buffers go back and forth in groups of up to 8 template rows (64 MMAs per
// hand-off), and the next group's barrier is tested before the current
// group is issued.
// All hand-offs are mbarriers (tcgen05.commit for MMA completion); every
// wait is bounded and a wait that runs out records NCC_ERR_TIMEOUT and lets
// the CTA finish.  Launched with programmatic stream serialization (not done
// by the library at present) the kernel may start while the table build is
// still running: only the epilogue reads S and Q, after waiting on the grid
// dependency.
#include "ncc_common.cuh"

#include <cuda_fp16.h>

namespace ncc {
namespace {

constexpr int kThreads = 512;
constexpr int kM = 128;               // output rows per tile (MMA M)
constexpr int kN = 64;                // shifts per tile (MMA N)
constexpr int kAWarps = 4;            // warps 1-4: image tiles
constexpr int kHWarps = 3;            // warps 5-7: Hankel buffers
constexpr int kEpi0 = 8;              // first epilogue warp
constexpr int kEpiWarps = 8;          // warps 8-15
constexpr int kMaxSmem = 227 * 1024;  // one CTA per SM
constexpr int kAccCols = 256;         // columns per accumulator buffer
constexpr int kTmemCols = 512;        // two accumulator buffers
constexpr int kMaxGroupProducts = 1024;  // 1024 * 2^14 = 2^24: exact fp32 partial sums
constexpr int kXpose = 32 * 33;       // ints per epilogue warp's transpose block

struct TGeom {
    int Kp;        // K per template row, a multiple of 16 (>= 64 + wT - 1)
    int nK16;      // MMA K steps per template row
    int R;         // image rows per tile (128 + hT - 1)
    int hRows;     // 16-byte rows per Hankel buffer (56 + 16 * nK16)
    int pLen;      // f16 entries per row of the centered, reversed template table
    int G;         // template rows per exact accumulator group
    int nG;        // groups (accumulator columns nG * 64)
    int hg;        // template rows per Hankel group (one barrier hand-off per group)
    int nH;        // Hankel buffers in the ring (two groups)
    int aBytes;    // one image tile
    int offA, offH, offP, offX, offSt, offBar, smemBytes;
};

bool make_geom(int wT, int hT, TGeom &g) {
    if (wT < 1 || hT < 1 || wT > 65) return false;
    g.Kp = (kN + wT - 1 + 15) / 16 * 16;
    g.nK16 = g.Kp / 16;
    g.R = kM + hT - 1;
    g.hRows = 56 + 16 * g.nK16;
    g.pLen = (g.hRows + 8 + 7) / 8 * 8;
    g.G = kMaxGroupProducts / wT;
    if (g.G > hT) g.G = hT;
    g.nG = (hT + g.G - 1) / g.G;
    if (g.nG * kN > kAccCols) return false;
    g.aBytes = g.nK16 * 2 * g.R * 16;
    for (g.hg = 8; g.hg >= 2; g.hg /= 2) {
        g.nH = 2 * g.hg;
        g.offA = 0;
        g.offH = g.offA + 2 * g.aBytes;
        g.offP = g.offH + g.nH * g.hRows * 16;
        g.offX = g.offP + (hT * g.pLen * 2 + 15) / 16 * 16;
        g.offSt = g.offX + kEpiWarps * kXpose * 4;
        g.offBar = (g.offSt + 16 + 15) / 16 * 16;
        const int barBytes = (2 * 2 + 2 * 2 + 2 * 2 + 1) * 8;
        g.smemBytes = g.offBar + barBytes + 128;  // + alignment slack
        if (g.smemBytes <= kMaxSmem) return true;
    }
    return false;
}

struct TParams {
    const uint8_t *img;
    int W, H;
    const uint8_t *tmpl;
    int wT, hT;
    const long long *S, *Q;
    float *out;
    long long *sumI, *sumI2, *sumIT;
    int *status;
    int Ox, Oy, ntx, ntiles;
    int waitPrev;  // launched behind the table build: wait on the grid before reading S, Q
    TGeom g;
};

__device__ __forceinline__ uint32_t saddr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ float u64_to_f32(unsigned long long a) {
    return fmaf(__uint2float_rn((unsigned)(a >> 32)), 4294967296.0f, __uint2float_rn((unsigned)a));
}

__device__ __forceinline__ float i64_to_f32(long long v) {
    const float f = u64_to_f32(v < 0 ? (unsigned long long)(-v) : (unsigned long long)v);
    return v < 0 ? -f : f;
}

// 1/sqrt(v) from the hardware approximation (relative error about 2^-22.9),
// flushing subnormals: v is an integer >= 1 here.
__device__ __forceinline__ float rsqrt_approx(float v) {
    float r;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
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

__device__ __forceinline__ uint32_t mbar_try(unsigned long long *b, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred P; mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2; selp.u32 %0, 1, 0, P; }"
        : "=r"(done) : "r"(saddr(b)), "r"(parity) : "memory");
    return done;
}

// Bounded wait for the phase with the given parity, by the whole warp (one
// lane polls; the warp's control flow stays uniform).  After the first wait
// that runs out, *abort short-circuits every later wait of the CTA.
__device__ __forceinline__ void mbar_wait_warp(unsigned long long *b, uint32_t parity, int *abort,
                                               int *status) {
    uint32_t done = 0;
    if ((threadIdx.x & 31u) == 0) {
        done = mbar_try(b, parity);
        if (!done && !*(volatile int *)abort) {
            const uint64_t t0 = global_timer_ns();
            for (unsigned it = 0; !done; ++it) {
                done = mbar_try(b, parity);
                if (!done && (it & 1023u) == 1023u) {
                    if (*(volatile int *)abort) break;
                    if (global_timer_ns() - t0 > 2000000000ull || it > (1u << 26)) {
                        *(volatile int *)abort = 1;
                        record_status(status, NCC_ERR_TIMEOUT);
                        break;
                    }
                }
            }
        }
    }
    __syncwarp();
}

// Non-blocking test of a phase: the result can be consumed later, so the
// test's latency overlaps whatever the thread issues meanwhile.
__device__ __forceinline__ uint32_t mbar_test(unsigned long long *b, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred P; mbarrier.test_wait.parity.shared::cta.b64 P, [%1], %2; selp.u32 %0, 1, 0, P; }"
        : "=r"(done) : "r"(saddr(b)), "r"(parity) : "memory");
    return done;
}

// Bounded wait by one thread.  After the first wait that runs out, *abort
// short-circuits every later wait of the CTA.
__device__ __forceinline__ void mbar_wait_lane(unsigned long long *b, uint32_t parity, int *abort,
                                               int *status) {
    if (mbar_try(b, parity) || *(volatile int *)abort) return;
    const uint64_t t0 = global_timer_ns();
    for (unsigned it = 0; !mbar_try(b, parity); ++it)
        if ((it & 1023u) == 1023u) {
            if (*(volatile int *)abort) return;
            if (global_timer_ns() - t0 > 2000000000ull || it > (1u << 26)) {
                *(volatile int *)abort = 1;
                record_status(status, NCC_ERR_TIMEOUT);
                return;
            }
        }
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

// 16 consecutive accumulator columns of this thread's lane
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
}

// Two pixels of `w` (bytes chosen by `sel`, the lower f16 first) as exact
// centered f16x2: the byte goes into the mantissa of 1024.0h and 1152 is
// subtracted, leaving byte - 128.
__device__ __forceinline__ uint32_t bytes_to_centered_h2(uint32_t w, uint32_t sel) {
    const uint32_t biased = __byte_perm(w, 0x64646464u, sel);
    __half2 h = *reinterpret_cast<const __half2 *>(&biased);
    h = __hsub2(h, __halves2half2(__float2half(1152.f), __float2half(1152.f)));
    return *reinterpret_cast<uint32_t *>(&h);
}

// kNK: MMA K steps per template row when fixed at compile time (the inner
// loop unrolls), else 0.
template <bool kMoments, int kNK>
__global__ void __launch_bounds__(kThreads, 1) toeplitz_tc_kernel(const TParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ unsigned s_red[kThreads / 32][2];
    const TGeom &g = p.g;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    uint16_t *P = reinterpret_cast<uint16_t *>(smem + g.offP);  // [hT][pLen] centered, reversed
    unsigned *st = reinterpret_cast<unsigned *>(smem + g.offSt);   // SumT, SumT2
    unsigned long long *bar = reinterpret_cast<unsigned long long *>(smem + g.offBar);
    unsigned long long *aFull = bar, *aEmpty = bar + 2;            // per image-tile buffer
    unsigned long long *accFull = bar + 4, *accEmpty = bar + 6;    // per accumulator buffer
    unsigned long long *hFull = bar + 8, *hEmpty = bar + 10;  // per Hankel group of the ring
    unsigned long long *mmaDone = bar + 12;

    // --- prologue: template table, template sums, barriers, tensor memory ---
    {
        // P[j][t] = T[j][Kp-1-t] - 128 where that column exists, else 0
        const int total = p.hT * g.pLen;
        for (int e = tid; e < total; e += kThreads) {
            const int j = e / g.pLen, t = e - j * g.pLen;
            const int col = g.Kp - 1 - t;
            __half v = __float2half(0.f);
            if (col >= 0 && col < p.wT)
                v = __float2half((float)((int)__ldg(p.tmpl + (size_t)j * p.wT + col) - 128));
            P[e] = __half_as_ushort(v);
        }
        unsigned a = 0, b = 0;
        for (int i = tid; i < p.wT * p.hT; i += kThreads) {
            const unsigned v = __ldg(p.tmpl + i);
            a += v;
            b += v * v;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            a += __shfl_xor_sync(0xffffffffu, a, o);
            b += __shfl_xor_sync(0xffffffffu, b, o);
        }
        if (lane == 0) { s_red[warp][0] = a; s_red[warp][1] = b; }
        if (tid == 0) {
            for (int i = 0; i < 2; ++i) {
                mbar_init(&aFull[i], kAWarps);
                mbar_init(&aEmpty[i], 1);
                mbar_init(&accFull[i], 1);
                mbar_init(&accEmpty[i], kEpiWarps);
            }
            for (int i = 0; i < 2; ++i) { mbar_init(&hFull[i], kHWarps); mbar_init(&hEmpty[i], 1); }
            mbar_init(mmaDone, 1);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            s_abort = 0;
        }
        if (warp == 0) {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                         ::"r"(saddr(&s_tmem)), "r"(kTmemCols) : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
        __syncthreads();
        if (tid == 0) {
            unsigned sa = 0, sb = 0;
            for (int w = 0; w < kThreads / 32; ++w) { sa += s_red[w][0]; sb += s_red[w][1]; }
            st[0] = sa;
            st[1] = sb;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    }
    const uint32_t tmem = s_tmem;

    if (warp >= 1 && warp <= kAWarps) {
        // ---- image tiles: chunk (r, q) holds reversed columns c' = 8q..8q+7,
        // i.e. image columns x0+Kp-8-8q .. x0+Kp-1-8q, last first ----
        const int pt = tid - 32;
        constexpr int kPT = kAWarps * 32;
        constexpr int kBatch = 8;  // loads in flight per thread
        const bool aligned8 = (p.W % 8 == 0) && ((uintptr_t)p.img % 8 == 0);
        const int q8 = g.Kp / 8;  // 16-byte chunks per tile row
        const int nChunks = g.R * q8;
        uint32_t it = 0;
        for (int tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x, ++it) {
            const int x0 = (tile % p.ntx) * kN, y0 = (tile / p.ntx) * kM;
            const uint32_t ab = it & 1;
            if (it >= 2) mbar_wait_warp(&aEmpty[ab], ((it >> 1) - 1) & 1, &s_abort, p.status);
            uint8_t *A = smem + g.offA + ab * g.aBytes;
            for (int e0 = pt; e0 < nChunks; e0 += kPT * kBatch) {
                uint2 v[kBatch];
#pragma unroll
                for (int k = 0; k < kBatch; ++k) {
                    const int e = e0 + k * kPT;
                    v[k] = make_uint2(0, 0);
                    if (e < nChunks) {
                        const int r = e / q8, qq = e - r * q8;
                        const int y = y0 + r, col0 = x0 + g.Kp - 8 - 8 * qq;
                        if (y < p.H && col0 < p.W) {
                            const uint8_t *src = p.img + (size_t)y * p.W + col0;
                            if (aligned8 && col0 + 8 <= p.W) {
                                v[k] = __ldg(reinterpret_cast<const uint2 *>(src));
                            } else {
#pragma unroll
                                for (int bb = 0; bb < 4; ++bb) {
                                    if (col0 + bb < p.W) v[k].x |= (uint32_t)__ldg(src + bb) << (8 * bb);
                                    if (col0 + 4 + bb < p.W) v[k].y |= (uint32_t)__ldg(src + 4 + bb) << (8 * bb);
                                }
                            }
                        }
                    }
                }
#pragma unroll
                for (int k = 0; k < kBatch; ++k) {
                    const int e = e0 + k * kPT;
                    if (e >= nChunks) break;
                    const int r = e / q8, qq = e - r * q8;
                    const bool inside = y0 + r < p.H && x0 + g.Kp - 8 - 8 * qq < p.W;
                    uint4 h;  // elements 0..7 = bytes 7..0 of the loaded columns
                    h.x = bytes_to_centered_h2(v[k].y, 0x4243);
                    h.y = bytes_to_centered_h2(v[k].y, 0x4041);
                    h.z = bytes_to_centered_h2(v[k].x, 0x4243);
                    h.w = bytes_to_centered_h2(v[k].x, 0x4041);
                    if (!inside) h = make_uint4(0, 0, 0, 0);
                    const size_t off = (size_t)qq * g.R * 16 + (size_t)r * 16;
                    if (NCC_BOUNDS(off + 16 <= (size_t)g.aBytes, p.status))
                        *reinterpret_cast<uint4 *>(A + off) = h;
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&aFull[ab]);
        }
    } else if (warp > kAWarps && warp < kEpi0) {
        // ---- Hankel buffers: row t of template row j is P[j][t..t+7].  The
        // ring holds two groups of g.hg template rows; a group is handed to
        // the MMA thread (and back) with one barrier each way ----
        const int pt = tid - 32 * (kAWarps + 1);
        constexpr int kPT = kHWarps * 32;
        uint32_t q = 0;  // groups handed over so far (all tiles)
        for (int tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x) {
            for (int j0 = 0; j0 < p.hT; j0 += g.hg, ++q) {
                const uint32_t gs = q & 1;
                if (q >= 2) mbar_wait_warp(&hEmpty[gs], ((q >> 1) - 1) & 1, &s_abort, p.status);
                const int rows = min(g.hg, p.hT - j0);
                for (int e = pt; e < rows * g.hRows; e += kPT) {
                    const int jj = e / g.hRows, t = e - jj * g.hRows;
                    if (!NCC_BOUNDS((j0 + jj) * g.pLen + t + 8 <= p.hT * g.pLen &&
                                        gs * g.hg + jj < g.nH, p.status))
                        continue;
                    const uint16_t *Pj = P + (j0 + jj) * g.pLen;
                    uint4 h;
                    h.x = (uint32_t)Pj[t] | ((uint32_t)Pj[t + 1] << 16);
                    h.y = (uint32_t)Pj[t + 2] | ((uint32_t)Pj[t + 3] << 16);
                    h.z = (uint32_t)Pj[t + 4] | ((uint32_t)Pj[t + 5] << 16);
                    h.w = (uint32_t)Pj[t + 6] | ((uint32_t)Pj[t + 7] << 16);
                    *reinterpret_cast<uint4 *>(smem + g.offH + ((gs * g.hg + jj) * g.hRows + t) * 16) = h;
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&hFull[gs]);
            }
        }
    } else if (warp == 0) {
        // ---- MMA issuer: lane 0 alone.  The tensor pipe accepts an MMA only
        // about one instruction ahead of the one it executes, so any wait
        // between MMAs leaves it idle: the issuer hands Hankel buffers back
        // once per group of g.hg rows, and tests the next group's barrier
        // before it issues the current group, so that the test's latency
        // passes under the MMAs ----
        if (lane == 0) {
            // D f32, A and B f16, both K-major, N = 64, M = 128
            const uint32_t idesc = (1u << 4) | ((uint32_t)(kN >> 3) << 17) | ((uint32_t)(kM >> 4) << 24);
            const uint64_t aDesc0 = smem_desc(saddr(smem + g.offA), (uint32_t)g.R * 16, 128);
            const uint64_t hDesc0 = smem_desc(saddr(smem + g.offH), 128, 128);
            const uint32_t aChunk = (uint32_t)(2 * g.R * 16) >> 4;  // next K chunk of A
            const uint32_t aBuf = (uint32_t)g.aBytes >> 4;          // next image-tile buffer
            const uint32_t hRow = (uint32_t)(g.hRows * 16) >> 4;    // next Hankel buffer
            const int nK16 = kNK ? kNK : g.nK16;
            uint32_t q = 0, it = 0;
            uint32_t nextReady = mbar_test(&hFull[0], 0);
            for (int tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x, ++it) {
                const uint32_t ab = it & 1;
                mbar_wait_lane(&aFull[ab], (it >> 1) & 1, &s_abort, p.status);
                if (it >= 2) mbar_wait_lane(&accEmpty[ab], ((it >> 1) - 1) & 1, &s_abort, p.status);
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t dTile = tmem + ab * kAccCols;
                const uint64_t aTile = aDesc0 + (uint64_t)(ab * aBuf);
                int inGroup = 0, accGroup = 0;
                for (int j0 = 0; j0 < p.hT; j0 += g.hg, ++q) {
                    const uint32_t gs = q & 1;
                    if (!nextReady) mbar_wait_lane(&hFull[gs], (q >> 1) & 1, &s_abort, p.status);
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    nextReady = mbar_test(&hFull[gs ^ 1u], ((q + 1) >> 1) & 1);
                    const int rows = min(g.hg, p.hT - j0);
                    for (int jj = 0; jj < rows; ++jj) {
                        const int j = j0 + jj;
                        // A rows j..j+127 of the tile, Hankel rows up to
                        // 16*(nK16-1)+71, accumulator columns of the group
                        if (!NCC_BOUNDS(j + kM <= g.R && (int)(gs * g.hg) + jj < g.nH &&
                                            16 * (nK16 - 1) + 72 <= g.hRows &&
                                            (accGroup + 1) * kN <= kAccCols, p.status))
                            continue;
                        const uint32_t d = dTile + (uint32_t)(accGroup * kN);
                        const uint64_t a = aTile + (uint64_t)j;  // 16 bytes per template row
                        const uint64_t b = hDesc0 + (uint64_t)((gs * g.hg + jj) * hRow);
                        const uint32_t first = inGroup == 0 ? 0u : 1u;
                        if (kNK) {
#pragma unroll
                            for (int c = 0; c < kNK; ++c)
                                tc_mma(d, a + (uint64_t)(c * aChunk), b + (uint64_t)(c * 16), idesc,
                                       c ? 1u : first);
                        } else {
                            for (int c = 0; c < nK16; ++c)
                                tc_mma(d, a + (uint64_t)(c * aChunk), b + (uint64_t)(c * 16), idesc,
                                       c ? 1u : first);
                        }
                        if (++inGroup == g.G) { inGroup = 0; ++accGroup; }
                    }
                    tc_commit(&hEmpty[gs]);
                }
                tc_commit(&accFull[ab]);
                // the image warps wait on this only before the tile two
                // ahead; no arrive may land once the CTA has left
                if (tile + 2 * (int)gridDim.x < p.ntiles) tc_commit(&aEmpty[ab]);
            }
            // every MMA (and every commit before this one) has completed
            // before tensor memory is freed, even when a wait ran out
            tc_commit(mmaDone);
            const uint64_t t0 = global_timer_ns();
            for (unsigned n = 0; !mbar_try(mmaDone, 0); ++n)
                if (global_timer_ns() - t0 > 200000000ull || n > (1u << 26)) {
                    record_status(p.status, NCC_ERR_TIMEOUT);
                    break;
                }
        }
        __syncwarp();
    } else {
        // ---- epilogue: warp = (lane quarter qd, shift half hf); its block is
        // output rows y0 + 32*qd .. +31 by shifts x0 + 32*hf .. +31 ----
        const int ew = warp - kEpi0;
        const int qd = warp & 3, hf = ew >> 2;
        const uint32_t laneBase = (uint32_t)(32 * qd) << 16;
        int *X = reinterpret_cast<int *>(smem + g.offX) + ew * kXpose;  // [32 rows][33]
        const long long N = (long long)p.wT * p.hT;
        const unsigned sT = st[0], sT2 = st[1];
        const long long vT = N * (long long)sT2 - (long long)sT * (long long)sT;
        const float invSqrtVT = vT > 0 ? __frsqrt_rn(u64_to_f32((unsigned long long)vT)) : 0.0f;
        // SumIT = C + 128*SumI + (128*SumT - 16384*N), all mod 2^32
        const uint32_t cT = 128u * sT - 16384u * (uint32_t)N;
        const size_t W = (size_t)p.W;
        if (p.waitPrev) asm volatile("griddepcontrol.wait;" ::: "memory");
        uint32_t it = 0;
        for (int tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x, ++it) {
            const int x0 = (tile % p.ntx) * kN, y0 = (tile / p.ntx) * kM;
            const uint32_t ab = it & 1;
            {
                // While the MMAs run, pull this block's table rows into L2: per
                // output row, 8 segments of 32 entries (rows y-1 and y+hT-1,
                // columns x-1.. and x+wT-1.., of S and Q), two 128-byte lines
                // each, one line per lane of lanes 0-15.
                const int rr = min(32, p.Oy - (y0 + 32 * qd));
                const int seg = lane >> 1, line = lane & 1;
                for (int r = 0; r < rr && lane < 16; ++r) {
                    const int y = y0 + 32 * qd + r;
                    const int yy = (seg & 2) ? y + p.hT - 1 : y - 1;
                    if (yy < 0) continue;
                    const int xx = (seg & 1) ? x0 + 32 * hf + p.wT - 1 : x0 + 32 * hf - 1;
                    const long long *tb = (seg & 4) ? p.Q : p.S;
                    const int col = min(max(xx, 0) + 16 * line, p.W - 1);  // inside the table
                    const long long *ptr = tb + (size_t)yy * W + col;
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
                }
            }
            mbar_wait_warp(&accFull[ab], (it >> 1) & 1, &s_abort, p.status);
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            // (1) this lane's row: the integer sum of every group, 32 shifts,
            // into the transpose block X[row = lane][shift]
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                int acc[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[i] = 0;
                for (int gi = 0; gi < g.nG; ++gi) {
                    uint32_t v[16];
                    // a warp-uniform check: the load is a whole-warp instruction
                    if (!NCC_BOUNDS(gi * kN + 32 * hf + 16 * half + 16 <= kAccCols, p.status)) continue;
                    tc_ld16(tmem + laneBase + ab * kAccCols + (uint32_t)(gi * kN + 32 * hf + 16 * half), v);
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[i] += __float2int_rn(__uint_as_float(v[i]));
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) X[lane * 33 + 16 * half + i] = acc[i];
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&accEmpty[ab]);
            // (2) one output row at a time, lane = shift: coalesced box sums
            // from the low 32 bits of S and Q (the box sums are below 2^32,
            // so wrapping differences are exact) and coalesced stores.  The
            // table reads of four rows are issued before any is used; their
            // addresses are clamped into the tables (x to the last shift, the
            // rows above row 0 to row 0, masked out), so every read is in
            // bounds and only the stores are conditional.
            const int x = x0 + 32 * hf + lane;
            const bool xin = x < p.Ox;
            const int xc = min(x, p.Ox - 1);
            const size_t xr2 = 2 * (size_t)(xc + p.wT - 1), xl2 = 2 * (size_t)(xc > 0 ? xc - 1 : 0);
            const uint32_t xm = xc > 0 ? 0xffffffffu : 0u;
            const int rows = min(32, p.Oy - (y0 + 32 * qd));
            for (int r0 = 0; r0 < rows; r0 += 4) {
                uint32_t v[4][8];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int y = y0 + 32 * qd + min(r0 + u, rows - 1);
                    const unsigned *Sb = reinterpret_cast<const unsigned *>(p.S + (size_t)(y + p.hT - 1) * W);
                    const unsigned *Qb = reinterpret_cast<const unsigned *>(p.Q + (size_t)(y + p.hT - 1) * W);
                    const unsigned *St = reinterpret_cast<const unsigned *>(p.S + (size_t)(y > 0 ? y - 1 : 0) * W);
                    const unsigned *Qt = reinterpret_cast<const unsigned *>(p.Q + (size_t)(y > 0 ? y - 1 : 0) * W);
                    v[u][0] = __ldg(Sb + xr2);
                    v[u][1] = __ldg(Qb + xr2);
                    v[u][2] = __ldg(Sb + xl2);
                    v[u][3] = __ldg(Qb + xl2);
                    v[u][4] = __ldg(St + xr2);
                    v[u][5] = __ldg(Qt + xr2);
                    v[u][6] = __ldg(St + xl2);
                    v[u][7] = __ldg(Qt + xl2);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int r = r0 + u;
                    if (r >= rows) break;
                    const int y = y0 + 32 * qd + r;
                    const int c = X[r * 33 + lane];
                    if (!xin) continue;
                    if (!NCC_BOUNDS(y + p.hT - 1 < p.H && x + p.wT - 1 < p.W && (size_t)y * p.Ox + x <
                                        (size_t)p.Oy * p.Ox, p.status))
                        continue;
                    const uint32_t ym = y > 0 ? 0xffffffffu : 0u;
                    const uint32_t sI = v[u][0] - (v[u][2] & xm) - (v[u][4] & ym) + (v[u][6] & xm & ym);
                    const uint32_t sI2 = v[u][1] - (v[u][3] & xm) - (v[u][5] & ym) + (v[u][7] & xm & ym);
                    const uint32_t sumIT = (uint32_t)c + 128u * sI + cT;
                    const size_t o = (size_t)y * p.Ox + x;
                    if (kMoments) {
                        p.sumI[o] = (long long)sI;
                        p.sumI2[o] = (long long)sI2;
                        p.sumIT[o] = (long long)sumIT;
                    } else {
                        const long long numi = (long long)((unsigned long long)N * sumIT) -
                                               (long long)sI * (long long)sT;
                        const long long vI = (long long)((unsigned long long)N * sI2) -
                                             (long long)sI * (long long)sI;
                        const float num = i64_to_f32(numi);
                        const float vIf = u64_to_f32((unsigned long long)max(vI, 1ll));
                        // a zero-variance window has num = 0 exactly; invSqrtVT is
                        // 0 for a zero-variance template
                        const float rr = num * rsqrt_approx(vIf) * invSqrtVT;
                        __stcs(p.out + o, fminf(1.0f, fmaxf(-1.0f, rr)));
                    }
                }
            }
            __syncwarp();  // the block is read before the next tile overwrites it
        }
    }

    // --- teardown: every accumulator has been drained by the epilogue ---
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     ::"r"(tmem), "r"(kTmemCols) : "memory");
}

int g_num_sms[64] = {};

}  // namespace

bool corr_toeplitz_supported(int wT, int hT) {
    TGeom g;
    return make_geom(wT, hT, g);
}

cudaError_t corr_toeplitz_launch(const CorrArgs &a, cudaStream_t stream) {
    TParams p;
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
    p.ntx = (p.Ox + kN - 1) / kN;
    p.ntiles = p.ntx * ((p.Oy + kM - 1) / kM);
    p.waitPrev = a.overlap_prev ? 1 : 0;
    if (!make_geom(a.wT, a.hT, p.g)) return cudaErrorNotSupported;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!g_num_sms[dev]) {
        e = cudaDeviceGetAttribute(&g_num_sms[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    const int grid = p.ntiles < g_num_sms[dev] ? p.ntiles : g_num_sms[dev];
    const size_t smem = (size_t)p.g.smemBytes;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.overlap_prev ? 1 : 0;
    auto launch = [&](auto kernel) -> cudaError_t {
        cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)smem);
        if (err != cudaSuccess) return err;
        return cudaLaunchKernelEx(&cfg, kernel, p);
    };
    const int nk = p.g.nK16;
    if (a.sumIT)
        e = nk == 8 ? launch(toeplitz_tc_kernel<true, 8>)
                    : nk == 7 ? launch(toeplitz_tc_kernel<true, 7>) : launch(toeplitz_tc_kernel<true, 0>);
    else
        e = nk == 8 ? launch(toeplitz_tc_kernel<false, 8>)
                    : nk == 7 ? launch(toeplitz_tc_kernel<false, 7>) : launch(toeplitz_tc_kernel<false, 0>);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace ncc
