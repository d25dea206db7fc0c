// correlate_tc.cu -- one template against every valid shift of an 8-bit
// image, with the numerator on the 5th-generation tensor cores and a fused
// epilogue that reads the window moments from the summed-area tables and
// writes the fp32 coefficient.
//
// Follows The CUDA Handbook, chapter 15: "Image in shared memory" (Listing
// 15-5: SumIT of every window, with the image staged on chip and reused by
// all the windows that overlap it) and section 15.8 (SumI and SumI2 of every
// window from S and Q by the four-corner box sum).
//
// The numerator as accumulated matrix products.  Output rows are taken in
// blocks of 16 (yb .. yb+15) over a strip of 128 shifts (x0 .. x0+127).  For
// every image row r = yb + d that reaches the block (d = 0 .. hT+14) one MMA
// with M = 128 shifts, N = 16 output rows, K = 16 template columns adds
//     D[m][n] += sum_i I[r][x0+m+i] * T[d-n][i]        (T rows outside 0..hT-1 are 0)
// to the block's fp32 accumulator in tensor memory, so that after the last
// row D[m][n] = SumIT(x0+m, yb+n).  The B operand of image row r is a
// 16-row window, starting at row hT+14-d, of the template stored upside down
// between zero rows: one small array serves every d by moving the
// descriptor's start address (K-major, rows 16 bytes apart).  Each image row
// meets at most two blocks.  Pixels 0..255 and all partial sums are integers
// below 2^24 while wT*hT <= 258, so the f16 products and the fp32
// accumulation are exact.
//
// A operand (no im2col): MN-major with both core-matrix strides 128 bytes
// over a buffer holding eight copies of the row segment shifted by 0..7
// pixels (block b, copy s, element e = pixel 8b+s+e), so element (m, k) sits
// at pixel m+k.
//
// Pipelines move four rows per stage (one barrier operation per four rows of
// work: the per-row cost of a barrier is what limits a pipeline of tiny
// stages).  Warp roles (persistent CTAs, 2 per SM, each owning a contiguous
// run of (strip, output row) units):
//   warps 0, 9 one thread each issues the MMAs (warp 0 those of even
//              blocks, warp 9 of odd blocks) and commits them to mbarriers;
//              warp 0 also allocates tensor memory,
//   warps 1-2  convert image rows into f16 shifted-copy A buffers (warp 1 the
//              first four rows of every image box, warp 2 the last four),
//   warp 3     one thread streams the S and Q row segments (columns
//              x0-2 .. x0+wT+127) by TMA, four table rows per stage; each row
//              serves as the bottom corners of output row y-hT+1 and the top
//              corners of output row y+1, so every table row is loaded once,
//   warp 4     one thread streams image rows by TMA (8 rows per box),
//   warps 5-8  epilogue (one per tensor-memory lane quarter), four output
//              rows per step: their SumIT from one 4-column tensor-memory
//              load, their moments from the table rows.
// Every wait is bounded: a wait that runs out records NCC_ERR_TIMEOUT and the
// CTA finishes without hanging.
#include "ncc_common.cuh"

#include <cuda_fp16.h>
#include <string.h>

namespace ncc {
namespace {

constexpr int kThreads = 320;
constexpr int kM = 128;               // shifts per strip (MMA M, tensor-memory lanes)
constexpr int kBR = 16;               // output rows per block (MMA N)
constexpr int kMaxHT = 16;            // template rows supported
constexpr int kSR = 4;                // rows per pipeline stage
constexpr int kAS = 2;                // A stages in the ring (kAS * kSR buffers)
constexpr int kND = 8;                // accumulator blocks in tensor memory
constexpr int kNI = 4;                // image boxes in the ring
constexpr int kImgRows = 8;           // image rows per TMA box (two stages)
constexpr int kNQSmax = 16;           // table-row stages in the ring, at most
constexpr int kMaxExactPixels = 258;  // 258 * 255^2 < 2^24
constexpr int kMaxSmem = 112 * 1024;  // two CTAs per SM
constexpr int kMaxBox = 256;          // TMA box extent limit
// Warp roles.  Warp w runs on scheduler w % 4; the epilogue warps (5-8) must
// cover the four tensor-memory lane quarters, so the converters go to
// schedulers 1 and 2 and the MMA issuer shares scheduler 0 only with light
// warps.
constexpr int kWarpMma = 0, kWarpConv0 = 1, kWarpConv1 = 2, kWarpTable = 3, kWarpImage = 4;
constexpr int kWarpMma1 = 9;          // second MMA issuer (odd blocks)
constexpr int kEpi0 = 160;
static_assert(kWarpConv1 == kWarpConv0 + 1 && kEpi0 == 5 * 32, "warp role layout");
static_assert(kImgRows == kAS * kSR, "one image box feeds one stage per converter warp");

struct TcGeom {
    int nK16;       // 16-column template chunks (MMA K steps per image row and block)
    int xBlocks;    // 8-pixel blocks per A buffer
    int xBytes;     // bytes per A buffer
    int imgBW;      // image box width in bytes (pixels x0 .. x0+imgBW-1)
    int rowBW;      // table-row segment in elements: columns x0-2 .. x0-2+rowBW-1
    int qOff;       // bytes from a table stage's S rows to its Q rows (128-aligned)
    int stageBytes; // one table stage: kSR S rows, then kSR Q rows at qOff
    int nqsLog2;    // table stages in the ring (a power of two)
    int bRows;      // rows of the upside-down template array (multiple of 8)
    int offB, offX, offI, offQ, offBar, smemBytes;
};

bool make_geom(int wT, int hT, TcGeom &g) {
    if (hT > kMaxHT || wT * hT > kMaxExactPixels) return false;
    g.nK16 = (wT + 15) / 16;
    g.xBlocks = 15 + 2 * g.nK16;
    g.xBytes = g.xBlocks * 128;
    g.imgBW = 8 * g.xBlocks + 8;                 // = 128 + 16 * nK16, a multiple of 16
    g.rowBW = (kM + wT + 2 + 1) & ~1;            // even: 16-byte TMA boxes of int64
    if (g.imgBW > kMaxBox || g.rowBW > kMaxBox) return false;
    g.qOff = (kSR * g.rowBW * 8 + 127) / 128 * 128;   // TMA destinations 128-byte aligned
    g.stageBytes = 2 * g.qOff;
    g.bRows = (hT + 2 * kBR - 2 + 7) / 8 * 8;    // 15 zero rows, hT rows, 15 zero rows
    g.offB = 0;
    const int bBytes = g.nK16 * 2 * g.bRows * 16;
    g.offX = (bBytes + 1023) / 1024 * 1024;
    g.offI = g.offX + kAS * kSR * g.xBytes;
    g.offQ = (g.offI + kNI * kImgRows * g.imgBW + 127) / 128 * 128;
    const int barBytes = (2 * kAS + 2 * kND + 2 * kNI + 2 * kNQSmax) * 8;
    // table stages: a group of four output rows needs the stages of its top
    // rows and of its bottom rows hT further (ceil((hT+3)/4) + 1 stages), one
    // more stage to refill, and more lookahead where shared memory allows
    const int need = (hT + 3 + kSR - 1) / kSR + 2;
    int lgMin = 0;
    while ((1 << lgMin) < need) ++lgMin;
    for (int lg = lgMin + 1; lg >= lgMin; --lg) {
        if ((1 << lg) > kNQSmax) continue;
        g.nqsLog2 = lg;
        g.offBar = g.offQ + (1 << lg) * g.stageBytes;
        g.smemBytes = g.offBar + barBytes + 1024;  // + alignment slack
        if (g.smemBytes <= kMaxSmem) return true;
    }
    return false;
}

struct TParams {
    int W, H, wT, hT;
    const uint8_t *tmpl;
    float *out;
    long long *sumI, *sumI2, *sumIT;
    int *status;
    int Ox, Oy, nStrips;
    long long units;  // nStrips * Oy
    TcGeom g;
};

__device__ __forceinline__ uint32_t saddr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ float u64_to_f32(unsigned long long a) {
    return fmaf(__uint2float_rn((unsigned)(a >> 32)), 4294967296.0f, __uint2float_rn((unsigned)a));
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

__device__ __forceinline__ void mbar_expect_tx(unsigned long long *b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 ::"r"(saddr(b)), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint32_t mbar_try(unsigned long long *b, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred P; mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2; selp.u32 %0, 1, 0, P; }"
        : "=r"(done) : "r"(saddr(b)), "r"(parity) : "memory");
    return done;
}

// Bounded wait for the phase with the given parity: one poll inline, the
// rest out of line (keeps the hot loops small).  After the first wait that
// runs out, *abort short-circuits every later wait of the CTA.  A nonzero
// `nap` (ns) sleeps between polls so that waiting warps leave the issue slots
// to the warps doing work.
__device__ __noinline__ void mbar_wait_slow(unsigned long long *b, uint32_t parity, int *abort,
                                            int *status, unsigned nap) {
    if (*(volatile int *)abort) return;
    const uint64_t t0 = global_timer_ns();
    for (unsigned it = 0;; ++it) {
        if (nap) __nanosleep(nap);
        if (mbar_try(b, parity)) return;
        if ((it & 255u) == 255u) {
            if (*(volatile int *)abort) return;
            if (global_timer_ns() - t0 > 2000000000ull || it > (1u << 26)) {
                *(volatile int *)abort = 1;
                record_status(status, NCC_ERR_TIMEOUT);
                return;
            }
        }
    }
}

__device__ __forceinline__ void mbar_wait(unsigned long long *b, uint32_t parity, int *abort,
                                          int *status, unsigned nap = 0) {
    if (!mbar_try(b, parity)) mbar_wait_slow(b, parity, abort, status, nap);
}

// The same for a whole warp: one lane polls and the answer is shuffled to
// the others, so the barrier sees one access instead of 32.  Lanes that
// must wait longer fall into the out-of-line loop together.
__device__ __forceinline__ void mbar_wait_warp(unsigned long long *b, uint32_t parity, int *abort,
                                               int *status, unsigned nap = 0) {
    const unsigned lane = threadIdx.x & 31u;
    uint32_t done = 0;
    if (lane == 0) done = mbar_try(b, parity);
    if (!__shfl_sync(0xffffffffu, done, 0)) mbar_wait_slow(b, parity, abort, status, nap);
}

// Bounded wait used at teardown for copies still in flight: never skipped by
// the abort flag (the CTA must not exit while a copy may still land).  All
// the drains of a thread share one deadline, so the total stays bounded.
__device__ __forceinline__ void mbar_drain(unsigned long long *b, uint32_t parity,
                                           uint64_t deadline, int *status) {
    for (unsigned it = 0; !mbar_try(b, parity); ++it) {
        if ((it & 1023u) == 1023u && (global_timer_ns() > deadline || it > (1u << 24))) {
            record_status(status, NCC_ERR_TIMEOUT);
            return;
        }
    }
}

__device__ __forceinline__ void tma_2d(const CUtensorMap *map, void *dst, int x, int y,
                                       unsigned long long *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(saddr(dst)), "l"(map), "r"(x), "r"(y), "r"(saddr(bar))
        : "memory");
}

// Issue helpers for a warp that runs the MMA loop uniformly: only the lane
// with `leader` set issues (a predicate, not a branch, so the descriptor
// arithmetic stays warp-uniform).
__device__ __forceinline__ void tc_commit_if(unsigned long long *b, bool leader) {
    asm volatile("{ .reg .pred q; setp.ne.b32 q, %1, 0;\n"
                 "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0]; }"
                 ::"r"(saddr(b)), "r"((uint32_t)leader) : "memory");
}

__device__ __forceinline__ void tc_mma_if(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t acc, bool leader) {
    asm volatile("{ .reg .pred p, q; setp.ne.b32 p, %4, 0; setp.ne.b32 q, %5, 0;\n"
                 "@q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
                 ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"((uint32_t)leader) : "memory");
}

// Two pixels (bytes selected by `sel` from `w`) as exact f16x2: the byte is
// placed in the mantissa of 1024.0h and 1024 is subtracted.
__device__ __forceinline__ uint32_t bytes_to_h2(uint32_t w, uint32_t sel) {
    const uint32_t biased = __byte_perm(w, 0x64646464u, sel);
    __half2 h = *reinterpret_cast<const __half2 *>(&biased);
    h = __hsub2(h, __halves2half2(__float2half(1024.f), __float2half(1024.f)));
    return *reinterpret_cast<uint32_t *>(&h);
}

// Ring bookkeeping: the q-th use (counted over the whole CTA) of a ring of
// K slots (K a power of two) is slot q % K, phase parity (q / K) & 1.
template <int K>
__device__ __forceinline__ uint32_t slot_of(uint32_t q) { return q % K; }
template <int K>
__device__ __forceinline__ uint32_t parity_of(uint32_t q) { return (q / K) & 1u; }
static_assert((kAS & (kAS - 1)) == 0 && (kND & (kND - 1)) == 0 && (kNI & (kNI - 1)) == 0,
              "ring sizes are powers of two");
// The same for the table ring, whose size (1 << lg stages) is chosen at launch.
__device__ __forceinline__ uint32_t qslot(uint32_t q, int lg) { return q & ((1u << lg) - 1u); }
__device__ __forceinline__ uint32_t qparity(uint32_t q, int lg) { return (q >> lg) & 1u; }

// A segment of nOut output rows: its blocks, the image rows its MMAs use,
// the image rows converted (whole boxes), and its table rows (whole stages).
__device__ __forceinline__ int seg_blocks(int nOut) { return (nOut + kBR - 1) / kBR; }
__device__ __forceinline__ int seg_image_rows(int nOut, int hT) {
    return seg_blocks(nOut) * kBR + hT - 1;
}
__device__ __forceinline__ int seg_boxes(int nOut, int hT) {
    return (seg_image_rows(nOut, hT) + kImgRows - 1) / kImgRows;
}
__device__ __forceinline__ int seg_table_stages(int nOut, int hT) {
    return (nOut + hT + kSR - 1) / kSR;  // table rows ya-1 .. ya+nOut+hT-2, rounded up
}

// The CTA's units (strip-major (strip, output row) pairs) split into
// segments of consecutive output rows of one strip.
struct SegIter {
    long long u, u1;
    int Oy;
    __device__ __forceinline__ bool next(int &strip, int &ya, int &yb) {
        if (u >= u1) return false;
        strip = (int)(u / Oy);
        ya = (int)(u - (long long)strip * Oy);
        const long long left = u1 - u;
        yb = left < (long long)(Oy - ya) ? ya + (int)left : Oy;
        u += yb - ya;
        return true;
    }
};

template <bool kMoments>
__global__ void __launch_bounds__(kThreads, 2)
corr_tc_kernel(const __grid_constant__ CUtensorMap tmI, const __grid_constant__ CUtensorMap tmS,
               const __grid_constant__ CUtensorMap tmQ, const TParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ unsigned s_red[kThreads / 32][2];
    __shared__ float s_sumT, s_invSqrtVT;
    __shared__ int s_vTpos;

    const TcGeom &g = p.g;
    const int lg = g.nqsLog2;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    unsigned long long *bar = reinterpret_cast<unsigned long long *>(smem + g.offBar);
    unsigned long long *afull = bar, *aempty = afull + kAS;
    unsigned long long *dfull = aempty + kAS, *dempty = dfull + kND;
    unsigned long long *ifull = dempty + kND, *iempty = ifull + kNI;
    unsigned long long *qfull = iempty + kNI, *qempty = qfull + kNQSmax;

    SegIter segs{(long long)blockIdx.x * p.units / gridDim.x,
                 (long long)(blockIdx.x + 1) * p.units / gridDim.x, p.Oy};

    // --- prologue: B operand, template statistics, barriers, tensor memory ---
    {
        // Upside-down template between zero rows: array row t holds template
        // row hT+14-t.  K-major, chunk c, k-group kg: rows 16 bytes apart.
        const int perChunk = g.bRows * 16;   // f16 elements per chunk
        const int total = g.nK16 * perChunk;
        unsigned sa = 0, sb = 0;
        for (int e = tid; e < total; e += kThreads) {
            const int c = e / perChunk, rem = e - c * perChunk;
            const int t = rem >> 4, k = rem & 15;
            const int j = p.hT + kBR - 2 - t, col = 16 * c + k;
            unsigned v = 0;
            if (j >= 0 && j < p.hT && col < p.wT) v = __ldg(p.tmpl + (size_t)j * p.wT + col);
            sa += v;
            sb += v * v;
            const int off = (c * 2 + (k >> 3)) * g.bRows * 16 + t * 16 + (k & 7) * 2;
            *reinterpret_cast<__half *>(smem + g.offB + off) = __uint2half_rn(v);  // exact
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            sa += __shfl_xor_sync(0xffffffffu, sa, o);
            sb += __shfl_xor_sync(0xffffffffu, sb, o);
        }
        if (lane == 0) { s_red[warp][0] = sa; s_red[warp][1] = sb; }
        if (tid == 0) {
            for (int i = 0; i < kAS; ++i) { mbar_init(&afull[i], 1); mbar_init(&aempty[i], 2); }
            for (int i = 0; i < kND; ++i) { mbar_init(&dfull[i], 1); mbar_init(&dempty[i], 4); }
            for (int i = 0; i < kNI; ++i) { mbar_init(&ifull[i], 1); mbar_init(&iempty[i], 2); }
            for (int i = 0; i < kNQSmax; ++i) { mbar_init(&qfull[i], 1); mbar_init(&qempty[i], 4); }
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            s_abort = 0;
        }
        if (warp == 0) {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                         ::"r"(saddr(&s_tmem)), "r"(kND * kBR) : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (tid == 0) {
            unsigned a = 0, b = 0;
            for (int w = 0; w < kThreads / 32; ++w) { a += s_red[w][0]; b += s_red[w][1]; }
            const long long N = (long long)p.wT * p.hT;
            const long long vT = N * (long long)b - (long long)a * (long long)a;
            s_sumT = (float)a;  // < 2^17: exact
            s_vTpos = vT > 0;
            s_invSqrtVT = vT > 0 ? __frsqrt_rn(u64_to_f32((unsigned long long)vT)) : 0.f;
        }
        __syncthreads();
    }
    const uint32_t tmem = s_tmem;

    if (warp == kWarpMma || warp == kWarpMma1) {
        // ---- MMA issuers: one A stage (four image rows) per step ----
        // Two warps share the work: warp kWarpMma the blocks of even index,
        // warp kWarpMma1 the odd ones; both consume every A stage (its empty
        // barrier counts two commits).  The whole warp runs the loop
        // (warp-uniform addresses and descriptors); lane 0 alone issues.
        {
            const bool leader = lane == 0;
            const uint32_t mine = warp == kWarpMma ? 0u : 1u;   // block parity owned
            // instruction descriptor: D f32, A/B f16, A MN-major, B K-major, N = 16, M = 128
            const uint32_t idesc = (1u << 4) | (1u << 15) | ((uint32_t)(kBR >> 3) << 17) |
                                   ((uint32_t)(kM >> 4) << 24);
            const uint64_t adesc0 = smem_desc(saddr(smem + g.offX), 128, 128);
            // the window of image-row offset d starts at array row hT+14-d
            const int dLast = p.hT + kBR - 2;  // last image-row offset of a block
            const uint64_t bdesc0 = smem_desc(saddr(smem + g.offB) + (uint32_t)dLast * 16,
                                              (uint32_t)g.bRows * 16, 128);
            const uint32_t xStep = (uint32_t)g.xBytes >> 4;
            const uint32_t bChunk = (uint32_t)(2 * g.bRows * 16) >> 4;
            uint32_t qs = 0, qb = 0;  // A stages / blocks issued so far
            int strip, ya, yb;
            while (segs.next(strip, ya, yb)) {
                const int nblk = seg_blocks(yb - ya), nr = seg_image_rows(yb - ya, p.hT);
                const int nst = seg_boxes(yb - ya, p.hT) * (kImgRows / kSR);
                for (int st = 0; st < nst; ++st, ++qs) {
                    const uint32_t as = slot_of<kAS>(qs);
                    mbar_wait_warp(&afull[as], parity_of<kAS>(qs), &s_abort, p.status);
                    bool fenced = false;
                    for (int k = 0; k < kSR; ++k) {
                        const int rr = st * kSR + k;
                        if (rr >= nr) break;
                        // blocks reached by this image row: blk*16 <= rr <= blk*16 + dLast
                        const int bhi = min(rr / kBR, nblk - 1);
                        const int blo = rr > dLast ? (rr - dLast + kBR - 1) / kBR : 0;
                        if ((rr % kBR) == 0 && rr / kBR < nblk &&
                            ((qb + (uint32_t)(rr / kBR)) & 1u) == mine) {
                            // first image row of one of this warp's blocks: its
                            // accumulator must be free
                            const uint32_t kb = qb + (uint32_t)(rr / kBR);
                            mbar_wait_warp(&dempty[slot_of<kND>(kb)], parity_of<kND>(kb) ^ 1u,
                                           &s_abort, p.status);
                            fenced = false;
                        }
                        if (!fenced) {
                            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                            fenced = true;
                        }
                        const uint64_t ad = adesc0 + (uint64_t)((as * kSR + k) * xStep);
                        for (int blk = blo; blk <= bhi; ++blk) {
                            if (((qb + (uint32_t)blk) & 1u) != mine) continue;
                            const int d = rr - blk * kBR;
                            const uint32_t ds = slot_of<kND>(qb + (uint32_t)blk);
                            const uint64_t bd = bdesc0 - (uint64_t)d;  // start moves back d rows of 16 B
                            for (int c = 0; c < g.nK16; ++c)
                                tc_mma_if(tmem + ds * kBR, ad + 16u * c, bd + c * bChunk, idesc,
                                          (d != 0 || c != 0) ? 1u : 0u, leader);
                            if (d == dLast) tc_commit_if(&dfull[ds], leader);
                        }
                    }
                    tc_commit_if(&aempty[as], leader);
                }
                qb += (uint32_t)nblk;
            }
            // the last commit to each A stage's empty barrier lands before the CTA exits
            if (leader) {
                const uint64_t deadline = global_timer_ns() + 2000000000ull;
                for (uint32_t k = qs > (uint32_t)kAS ? qs - kAS : 0u; k < qs; ++k)
                    mbar_drain(&aempty[slot_of<kAS>(k)], parity_of<kAS>(k), deadline, p.status);
            }
        }
        __syncwarp();
    } else if (warp == kWarpTable) {
        // ---- table rows: S and Q segments by TMA, kSR rows per stage ----
        if (lane == 0) {
            const uint32_t bytes = 2u * kSR * (uint32_t)g.rowBW * 8u;
            uint32_t q = 0;  // table stages issued so far
            int strip, ya, yb;
            while (segs.next(strip, ya, yb) && !*(volatile int *)&s_abort) {
                const int x = strip * kM - 2;
                const int nst = seg_table_stages(yb - ya, p.hT);  // rows ya-1 .. from stage 0
                for (int st = 0; st < nst; ++st, ++q) {
                    const uint32_t s = qslot(q, lg);
                    mbar_wait(&qempty[s], qparity(q, lg) ^ 1u, &s_abort, p.status, 256);
                    if (*(volatile int *)&s_abort) break;
                    uint8_t *dst = smem + g.offQ + s * g.stageBytes;
                    mbar_expect_tx(&qfull[s], bytes);
                    tma_2d(&tmS, dst, x, ya - 1 + st * kSR, &qfull[s]);
                    tma_2d(&tmQ, dst + g.qOff, x, ya - 1 + st * kSR, &qfull[s]);
                }
            }
            // every issued copy has landed before the CTA exits
            const uint64_t deadline = global_timer_ns() + 2000000000ull;
            const uint32_t nq = 1u << lg;
            for (uint32_t k = q > nq ? q - nq : 0u; k < q; ++k)
                mbar_drain(&qfull[qslot(k, lg)], qparity(k, lg), deadline, p.status);
        }
        __syncwarp();
    } else if (warp == kWarpImage) {
        // ---- image rows by TMA, kImgRows per box ----
        if (lane == 0) {
            const uint32_t bytes = (uint32_t)(g.imgBW * kImgRows);
            uint32_t q = 0;  // boxes issued so far
            int strip, ya, yb;
            while (segs.next(strip, ya, yb) && !*(volatile int *)&s_abort) {
                const int nbox = seg_boxes(yb - ya, p.hT);
                for (int bx = 0; bx < nbox; ++bx, ++q) {
                    const uint32_t s = slot_of<kNI>(q);
                    mbar_wait(&iempty[s], parity_of<kNI>(q) ^ 1u, &s_abort, p.status, 256);
                    if (*(volatile int *)&s_abort) break;
                    mbar_expect_tx(&ifull[s], bytes);
                    tma_2d(&tmI, smem + g.offI + s * kImgRows * g.imgBW, strip * kM,
                           ya + bx * kImgRows, &ifull[s]);
                }
            }
            const uint64_t deadline = global_timer_ns() + 2000000000ull;
            for (uint32_t k = q > (uint32_t)kNI ? q - kNI : 0u; k < q; ++k)
                mbar_drain(&ifull[slot_of<kNI>(k)], parity_of<kNI>(k), deadline, p.status);
        }
        __syncwarp();
    } else if (warp == kWarpConv0 || warp == kWarpConv1) {
        // ---- converters: image rows -> f16 shifted-copy A buffers ----
        // Warp cw converts rows 4cw .. 4cw+3 of every image box into A stage
        // slot cw (the CTA's A stages alternate between the two warps).
        const int cw = warp - kWarpConv0;
        uint32_t qi = 0;  // boxes consumed so far
        int strip, ya, yb;
        while (segs.next(strip, ya, yb)) {
            const int nbox = seg_boxes(yb - ya, p.hT);
            for (int bx = 0; bx < nbox; ++bx, ++qi) {
                const uint32_t is = slot_of<kNI>(qi);
                const uint32_t qa = 2u * qi + (uint32_t)cw;   // this warp's A stage
                mbar_wait_warp(&ifull[is], parity_of<kNI>(qi), &s_abort, p.status, 64);
                mbar_wait_warp(&aempty[cw], parity_of<kAS>(qa) ^ 1u, &s_abort, p.status, 64);
                const uint8_t *box = smem + g.offI + is * kImgRows * g.imgBW + cw * kSR * g.imgBW;
                uint8_t *X = smem + g.offX + cw * kSR * g.xBytes;
                // one 16-byte chunk (row k, block b, copy s) per lane and step:
                // consecutive lanes store consecutive chunks (no bank
                // conflicts); copy s = pixels 8b+s .. 8b+s+7
                const int perRow = 8 * g.xBlocks;
                for (int c = lane; c < kSR * perRow; c += 32) {
                    const int k = c / perRow, cc = c - k * perRow;
                    const int b = cc >> 3, s = cc & 7;
                    const uint8_t *src = box + k * g.imgBW + 8 * b;
                    const uint2 lo = *reinterpret_cast<const uint2 *>(src);
                    const uint2 hi = *reinterpret_cast<const uint2 *>(src + 8);
                    const bool up = s >= 4;
                    const uint32_t w0 = up ? lo.y : lo.x, w1 = up ? hi.x : lo.y, w2 = up ? hi.y : hi.x;
                    const uint32_t sh = 8u * (uint32_t)(s & 3);
                    const uint32_t b0 = __funnelshift_r(w0, w1, sh);  // pixels s .. s+3
                    const uint32_t b1 = __funnelshift_r(w1, w2, sh);  // pixels s+4 .. s+7
                    reinterpret_cast<uint4 *>(X + k * g.xBytes)[cc] =
                        make_uint4(bytes_to_h2(b0, 0x4140), bytes_to_h2(b0, 0x4342),
                                   bytes_to_h2(b1, 0x4140), bytes_to_h2(b1, 0x4342));
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&afull[cw]);
                    mbar_arrive(&iempty[is]);
                }
            }
        }
    } else if (tid >= kEpi0 && tid < kEpi0 + 128) {
        // ---- epilogue: thread = shift x0 + xo; four output rows per step ----
        const int qd = warp & 3;                 // tensor-memory lane quarter of this warp
        const int xo = 32 * qd + lane;
        const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
        const long long N = (long long)p.wT * p.hT;
        const float Nf = (float)N;               // <= 258: exact
        const float sTf = s_sumT, invSqrtVT = s_invSqrtVT;
        const bool vTpos = s_vTpos != 0;
        const int cl = 2 * (xo + 1), cr = 2 * (xo + p.wT + 1);  // low words of columns x-1, x+wT-1
        const uint32_t rowWords = (uint32_t)g.rowBW * 2;         // u32 words per table row
        const uint32_t qWords = (uint32_t)g.qOff / 4;            // S rows -> Q rows of a stage
        const uint32_t *qbase = reinterpret_cast<const uint32_t *>(smem + g.offQ);
        const uint32_t stageWords = (uint32_t)g.stageBytes / 4;
        uint32_t qb = 0, qq = 0;  // blocks / table stages consumed so far
        int strip, ya, yb;
        while (segs.next(strip, ya, yb)) {
            const int x = strip * kM + xo;
            const bool xin = x < p.Ox;
            const int nOut = yb - ya, nblk = seg_blocks(nOut);
            for (int blk = 0; blk < nblk; ++blk, ++qb) {
                const uint32_t ds = slot_of<kND>(qb);
                mbar_wait_warp(&dfull[ds], parity_of<kND>(qb), &s_abort, p.status, 32);
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll 1
                for (int g4 = 0; g4 < kBR / kSR; ++g4) {
                    const int o0 = blk * kBR + kSR * g4;
                    if (o0 >= nOut) break;
                    // table rows o0..o0+3 (tops, one stage) and o0+hT..o0+hT+3
                    // (bottoms, one or two stages); a top stage was already
                    // waited for as a bottom stage unless o0 < hT
                    const uint32_t tq = qq + (uint32_t)(o0 / kSR);
                    const uint32_t bq0 = qq + (uint32_t)((o0 + p.hT) / kSR);
                    const int oLast = min(o0 + kSR - 1, nOut - 1);   // last output row of the group
                    const uint32_t bq1 = qq + (uint32_t)((oLast + p.hT) / kSR);
                    if (o0 < p.hT) mbar_wait_warp(&qfull[qslot(tq, lg)], qparity(tq, lg), &s_abort, p.status);
                    mbar_wait_warp(&qfull[qslot(bq0, lg)], qparity(bq0, lg), &s_abort, p.status);
                    if (bq1 != bq0)
                        mbar_wait_warp(&qfull[qslot(bq1, lg)], qparity(bq1, lg), &s_abort, p.status);
                    // (no calls between the tensor-memory load and its wait)
                    uint32_t r4[4];
                    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                                 : "=r"(r4[0]), "=r"(r4[1]), "=r"(r4[2]), "=r"(r4[3])
                                 : "r"(tmem + lane_base + ds * kBR + kSR * g4));
                    uint32_t sI[kSR], sI2[kSR];
#pragma unroll
                    for (int k = 0; k < kSR; ++k) {
                        const uint32_t rt = qq * kSR + (uint32_t)(o0 + k);   // table row (ring count)
                        const uint32_t rb = rt + (uint32_t)p.hT;
                        const uint32_t *St = qbase + qslot(rt / kSR, lg) * stageWords + (rt % kSR) * rowWords;
                        const uint32_t *Sb = qbase + qslot(rb / kSR, lg) * stageWords + (rb % kSR) * rowWords;
                        const uint32_t *Qt = St + qWords, *Qb = Sb + qWords;
                        // low 32 bits of each corner (little-endian int64): the
                        // four-corner sums are below 2^32, so wrapping is exact.
                        // Rows past the segment read ring memory harmlessly.
                        sI[k] = Sb[cr] - St[cr] - Sb[cl] + St[cl];
                        sI2[k] = Qb[cr] - Qt[cr] - Qb[cl] + Qt[cl];
                    }
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&qempty[qslot(tq, lg)]);  // rows y-1 of o0..o0+3 done
                    if (xin) {
#pragma unroll
                        for (int k = 0; k < kSR; ++k) {
                            const int o = o0 + k;
                            if (o >= nOut) continue;
                            const size_t oi = (size_t)(ya + o) * p.Ox + x;
                            const float s = __uint_as_float(r4[k]);  // SumIT, exact
                            if (kMoments) {
                                p.sumI[oi] = (long long)sI[k];
                                p.sumI2[oi] = (long long)sI2[k];
                                p.sumIT[oi] = (long long)__float2uint_rn(s);
                            } else {
                                // exact N*SumIT - SumI*SumT and N*SumI2 - SumI^2 up
                                // to their final roundings (fma splits; the high
                                // parts cancel exactly when they are close)
                                const float sIf = (float)sI[k], sI2f = (float)sI2[k];
                                const float p1 = Nf * s, e1 = fmaf(Nf, s, -p1);
                                const float p2 = sIf * sTf, e2 = fmaf(sIf, sTf, -p2);
                                const float num = (p1 - p2) + (e1 - e2);
                                const float q1 = Nf * sI2f, f1 = fmaf(Nf, sI2f, -q1);
                                const float q2 = sIf * sIf, f2 = fmaf(sIf, sIf, -q2);
                                const float vI = (q1 - q2) + (f1 - f2);
                                float r = 0.f;
                                if (vI > 0.f && vTpos) {
                                    r = num * rsqrtf(vI) * invSqrtVT;
                                    r = fminf(1.0f, fmaxf(-1.0f, r));
                                }
                                __stcs(p.out + oi, r);
                            }
                        }
                    }
                }
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&dempty[ds]);
            }
            // table stages never freed as a top stage (from the one after the
            // last group's): make sure they landed, then free them
            const int nst = seg_table_stages(nOut, p.hT);
            for (int st = (nOut - 1) / kSR + 1; st < nst; ++st) {
                const uint32_t tq = qq + (uint32_t)st;
                mbar_wait_warp(&qfull[qslot(tq, lg)], qparity(tq, lg), &s_abort, p.status);
                if (lane == 0) mbar_arrive(&qempty[qslot(tq, lg)]);
            }
            qq += (uint32_t)nst;
        }
    }

    // --- teardown: every accumulator has been drained by the epilogue ---
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     ::"r"(tmem), "r"(kND * kBR) : "memory");
}

int g_num_sms[64] = {};

}  // namespace

bool corr_tc_supported(const CorrArgs &a) {
    TcGeom g;
    return make_geom(a.wT, a.hT, g) && a.W % 16 == 0 && (uintptr_t)a.img % 16 == 0 &&
           (uintptr_t)a.S % 16 == 0 && (uintptr_t)a.Q % 16 == 0 &&
           tensor_map_encoder() != nullptr;
}

cudaError_t corr_tc_launch(const CorrArgs &a, cudaStream_t stream) {
    TParams p;
    p.W = a.W; p.H = a.H; p.wT = a.wT; p.hT = a.hT;
    p.tmpl = a.tmpl;
    p.out = a.out;
    p.sumI = reinterpret_cast<long long *>(a.sumI);
    p.sumI2 = reinterpret_cast<long long *>(a.sumI2);
    p.sumIT = reinterpret_cast<long long *>(a.sumIT);
    p.status = a.status;
    p.Ox = a.W - a.wT + 1;
    p.Oy = a.H - a.hT + 1;
    p.nStrips = (p.Ox + kM - 1) / kM;
    p.units = (long long)p.nStrips * p.Oy;
    if (!make_geom(a.wT, a.hT, p.g)) return cudaErrorNotSupported;

    CUtensorMap tmI, tmS, tmQ;
    memset(&tmI, 0, sizeof(tmI));
    memset(&tmS, 0, sizeof(tmS));
    memset(&tmQ, 0, sizeof(tmQ));
    if (!make_tensor_map_2d(&tmI, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.img, a.W, a.H, p.g.imgBW,
                            kImgRows) ||
        !make_tensor_map_2d(&tmS, CU_TENSOR_MAP_DATA_TYPE_INT64, 8, a.S, a.W, a.H, p.g.rowBW, kSR) ||
        !make_tensor_map_2d(&tmQ, CU_TENSOR_MAP_DATA_TYPE_INT64, 8, a.Q, a.W, a.H, p.g.rowBW, kSR))
        return cudaErrorNotSupported;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!g_num_sms[dev]) {
        e = cudaDeviceGetAttribute(&g_num_sms[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    const long long maxGrid = 2ll * g_num_sms[dev];
    const int grid = (int)(p.units < maxGrid ? p.units : maxGrid);
    const size_t smem = (size_t)p.g.smemBytes;
    if (a.sumIT) {
        e = cudaFuncSetAttribute(corr_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        corr_tc_kernel<true><<<grid, kThreads, smem, stream>>>(tmI, tmS, tmQ, p);
    } else {
        e = cudaFuncSetAttribute(corr_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        corr_tc_kernel<false><<<grid, kThreads, smem, stream>>>(tmI, tmS, tmQ, p);
    }
    return cudaGetLastError();
}

}  // namespace ncc
