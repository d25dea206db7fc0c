// correlate_dp4a.cu -- one template against every valid shift of an 8-bit
// image, with the numerator on the integer dot-product pipe (__dp4a) and a
// fused epilogue that reads the window moments from the summed-area tables
// and writes the fp32 coefficient.
//
// Follows The CUDA Handbook, chapter 15: "Image in shared memory"
// (Listing 15-5: the image tile plus a template-sized overfetch is staged in
// shared memory and each thread sums I*T over its windows), and section 15.8
// (SumI and SumI2 of every window from S and Q by the four-corner box sum).
//
// GB300 design:
//   - Output tile: 128 shifts wide by 8*kRPT rows; 256 threads; each thread
//     owns kRPT rows x 4 shifts.  Lane = 4*qg + d owns the shifts
//     x0 + 16*qg + 4*k + d (k = 0..3) of rows kRPT*warp .. kRPT*warp+kRPT-1.
//     kRPT = 8 (tiles of 128 x 64, three CTAs per SM) in general; kRPT = 4
//     (128 x 32) for templates up to 16 wide, whose kernel then fits four
//     CTAs per SM, and for maps too small to give every SM two larger tiles.
//   - The tile plus its (wT-1) x (hT-1) halo is one TMA box (cp.async.bulk.
//     tensor, completion on an mbarrier).  Images whose rows are not a
//     multiple of 16 bytes, or boxes beyond the TMA limits, use plain loads.
//   - Each lane reads 32 aligned bytes of a tile row (lanes of one qg share
//     them: conflict-free broadcast loads) and moves them by d bytes with one
//     byte permute per word, so its four shifts see 32-bit groups of four
//     pixels; per tile row the cost is 2 shared loads and 7 permutes against
//     up to 128 __dp4a.
//   - The numerator loop runs in three phases -- tile rows that meet only
//     the first output rows, rows that meet all eight, rows that meet only
//     the last ones -- so no (row, output row) pair is tested at run time
//     (templates of at least 8 rows; shorter ones take a predicated loop).
//   - The template is packed into 32-bit words in shared memory, in chunks of
//     16 pixels, zero-padded to a multiple of 16 (the zero bytes cancel any
//     pixels read past the window).
//   - SumIT accumulates in uint32 (exact while wT*hT*255^2 < 2^32).  16-row
//     templates get an instantiation with the height fixed at compile time.
//   - Epilogue: the SumIT tile is transposed through shared memory (over the
//     dead image tile, columns swizzled so that neither the stores nor the
//     row reads conflict); the CTA then walks its output rows four at a
//     time, one shift and two rows per thread.  The table rows a step needs
//     (S and Q at rows y-1.. and y+hT-1.., columns x0-2 .. x0+wT+127) arrive
//     as four TMA boxes of four rows each into a two-stage ring -- few, large
//     requests, since each TMA request costs about a hundred cycles to
//     issue.  The first two stages are requested right after the image tile
//     (one SM's requests are served in order); a stage is refilled as soon
//     as every warp has read it.  Steps go in pairs, one per ring stage, so
//     the staged-row addresses are compile-time offsets.  TMA's zero fill
//     outside the tables implements the four-corner rule's row -1 / column
//     -1 = 0.
//   - Launched after the SAT build with programmatic stream serialization
//     (ncc_match), the kernel may start before the tables are complete: it
//     waits on the grid dependency before the first table-row request (the
//     first wave of CTAs makes that request after its numerator).
//   - Direct moments (kDirect): SumI and SumI2 come from the staged tile
//     instead of S and Q, by sliding column sums and row prefixes in shared
//     memory, 16 output rows per pass.  (Tables whose rows are not a multiple of 16 bytes, or
//     templates wider than 127, read the corners with global loads.)  The
//     four-corner sums use the low 32 bits of the table entries (exact: the
//     sums are below 2^32); templates of at most 363 pixels form the
//     coefficient's numerator and variance terms exactly in 32-bit integers
//     (their magnitude is at most N^2 * 127.5^2 < 2^31), larger ones in
//     exact int64; each term is rounded to fp32 once.
#include "ncc_common.cuh"

#include <cuda.h>
#include <string.h>

namespace ncc {
namespace {

constexpr int kOutW = 128;
constexpr int kRowsPerThread = 8;
constexpr int kWarps = 8;
constexpr int kOutH = kWarps * kRowsPerThread;  // 64
constexpr int kSmallRPT = 4;   // rows per thread of the 128 x 32 tiles
static_assert(kCorrBandRows % kOutH == 0 && kCorrBandRows % (kWarps * kSmallRPT) == 0,
              "row bands must consist of whole tiles");
constexpr int kQuadMaxHT = 64; // narrow templates up to this height run four CTAs per SM
constexpr int kThreads = kWarps * 32;
constexpr int kMaxCtasPerSm = 3;   // resident CTAs per SM (launch bound)
constexpr int kMaxTmaBox = 256;        // TMA box extent limit per dimension
constexpr int kMaxSmem = 227 * 1024;   // opt-in shared memory per CTA

constexpr int kEpiStages = 2;          // table-row staging ring depth
constexpr int kEpiRowsPerStep = 4;     // output rows per epilogue step (rows per TMA box)
constexpr int kEpiBufs = 4;            // boxes per stage: S top, S bottom, Q top, Q bottom
// Templates at most kNarrowT wide share one table-row segment width, so the
// kernel instantiated for them addresses the staged rows with immediate
// offsets.
constexpr int kNarrowT = 16;
constexpr int kNarrowBW = (kOutW + kNarrowT + 2) & ~1;                        // 146 columns
constexpr int kNarrowBuf = (kEpiRowsPerStep * kNarrowBW * 8 + 127) / 128 * 128;  // bytes per box
// Templates of at most this many pixels form the coefficient's numerator
// N*SumIT - SumI*SumT and variance term N*SumI2 - SumI^2 in 32-bit integers:
// both are N^2 times a covariance or variance of values in 0..255, so at
// most N^2 * 127.5^2 < 2^31 in magnitude.
constexpr long long kMaxInt32N = 363;
// Direct moments: output rows per pass of the column-sum / row-prefix
// buffers (two tables of kDirRows rows in shared memory at a time).
constexpr int kDirRows = 16;
// Direct moments: tile columns one thread per column covers.
constexpr int kDirMaxCols = kThreads;

struct Geom {
    int nch;         // 16-pixel template chunks
    int boxW;        // staged tile width in bytes = kOutW + 16*nch
    int boxH;        // staged tile height = output rows + hT - 1
    int tmplOff;     // offset of the packed template (after the tile / SumIT region)
    int epiBW;       // table-row segment length (int64 elements), even
    int epiBuf;      // bytes per box (kEpiRowsPerStep table-row segments, 128-aligned)
    int epiOff;      // offset of the staging ring
    int sumOff;      // offset of the SumIT transpose (0: over the dead tile)
    int cpOff;       // direct moments: offset of the column-sum / row-prefix buffers
    int cPitch;      // direct moments: u32 words per buffer row (odd, > kOutW + wT - 1)
    int smemBytes;   // dynamic shared memory (plus 128 bytes of alignment slack)
};

// direct: the window moments come from the staged tile (the tile outlives
// the numerator, so the SumIT transpose gets its own space) instead of from
// the summed-area tables.
Geom make_geom(int wT, int hT, bool direct = false, int tileH = kOutH) {
    Geom g;
    g.nch = (wT + 15) / 16;
    g.boxW = kOutW + 16 * g.nch;
    g.boxH = tileH + hT - 1;
    const int tileBytes = (g.boxW * g.boxH + 127) / 128 * 128;
    const int sumBytes = tileH * kOutW * 4;  // the SumIT transpose reuses the tile's space
    if (direct) {
        g.tmplOff = tileBytes;
        g.sumOff = (g.tmplOff + hT * g.nch * 16 + 127) / 128 * 128;
        g.cpOff = g.sumOff + sumBytes;
        g.cPitch = (kOutW + wT) | 1;
        g.epiBW = g.epiBuf = 0;
        g.epiOff = g.cpOff;
        g.smemBytes = g.cpOff + 2 * kDirRows * g.cPitch * 4 + 128;
        return g;
    }
    g.sumOff = g.cpOff = g.cPitch = 0;
    g.tmplOff = tileBytes > sumBytes ? tileBytes : sumBytes;
    g.epiBW = (kOutW + wT + 2) & ~1;   // columns x0-2 .. x0+wT+127, rounded up to even
    if (wT <= kNarrowT) g.epiBW = kNarrowBW;  // one fixed layout for narrow templates
    g.epiBuf = (kEpiRowsPerStep * g.epiBW * 8 + 127) / 128 * 128;
    g.epiOff = (g.tmplOff + hT * g.nch * 16 + 127) / 128 * 128;
    g.smemBytes = g.epiOff + kEpiStages * kEpiBufs * g.epiBuf + 128;
    return g;
}

struct KParams {
    const uint8_t *img;
    int W, H;
    const uint8_t *tmpl;
    int wT, hT;
    const long long *S, *Q;
    float *out;
    long long *sumI, *sumI2, *sumIT;
    int *status;
    int Ox, Oy;
    int lateWave;    // CTAs (linear id) that request their first table rows after the numerator
    int tileRow0;    // first tile row of the launch (a band of output rows; 0 for the whole map)
    Geom g;
};

template <bool B>
struct BoolTag {
    static constexpr bool value = B;
};

template <int I>
struct IntTag {
    static constexpr int value = I;
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// fp32 value of a non-negative 64-bit integer below 2^56, rounded once:
// hi * 2^32 + fl(lo) in one fma (the error of fl(lo) is below 2^-25 of the
// total whenever hi > 0).
__device__ __forceinline__ float u64_to_f32(unsigned long long a) {
    return fmaf(__uint2float_rn((unsigned)(a >> 32)), 4294967296.0f,
                __uint2float_rn((unsigned)a));
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

__device__ __forceinline__ void tma_2d(const CUtensorMap *map, void *dst, int x, int y,
                                       unsigned long long *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Waits until the grid this kernel depends on programmatically has finished
// and its writes are visible; returns at once for an ordinary launch.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ uint32_t mbar_try(unsigned long long *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred P; mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2; selp.u32 %0, 1, 0, P; }"
        : "=r"(done) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return done;
}

__device__ __forceinline__ void mbar_arrive(unsigned long long *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Bounded wait on an mbarrier phase; gives up (recording the status) rather
// than hang if a transfer never lands.
__device__ __forceinline__ void mbar_wait(unsigned long long *bar, uint32_t parity, int *status) {
    uint32_t done = 0;
    for (unsigned it = 0; !done; ++it) {
        asm volatile(
            "{ .reg .pred P; mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2; selp.u32 %0, 1, 0, P; }"
            : "=r"(done) : "r"(smem_u32(bar)), "r"(parity) : "memory");
        if (it > (1u << 24)) {
            record_status(status, NCC_ERR_TIMEOUT);
            break;
        }
    }
}

// kNarrow: the template is at most kNarrowT wide (fixed staged layout; with
// kDirect, a fixed row-prefix pass).
// kHT: the template height when fixed at compile time (0: run time).
// kDirect: window moments from the staged tile, not from S and Q.
// kRPT: output rows per thread (8; 4 for maps too small to fill the GPU).
template <bool kTma, bool kMoments, bool kTmaEpi, bool kNarrow, int kHT, bool kDirect, int kRPT>
__global__ void __launch_bounds__(kThreads, (kRPT == kSmallRPT && kNarrow) ? 4 : kMaxCtasPerSm)
corr_dp4a_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmS,
                 const __grid_constant__ CUtensorMap tmQ, const KParams p) {
    constexpr int kTileH = kWarps * kRPT;  // output rows per tile
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    __shared__ __align__(8) unsigned long long s_bar;
    __shared__ __align__(8) unsigned long long s_ebar[kEpiStages];
    __shared__ __align__(8) unsigned long long s_efree[kEpiStages];
    __shared__ unsigned s_red[kWarps][2];
    __shared__ long long s_sumT, s_vT;
    __shared__ float s_invSqrtVT;

    const Geom &g = p.g;
    const int epiBW = kNarrow ? kNarrowBW : g.epiBW, epiBuf = kNarrow ? kNarrowBuf : g.epiBuf;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // tile rows bottom-up: the table build writes its tables top-down, so
    // the last rows it wrote -- still in L2 -- are read first; a launch over
    // a band of output rows starts at tile row p.tileRow0
    const int x0 = blockIdx.x * kOutW, y0 = (p.tileRow0 + (int)gridDim.y - 1 - (int)blockIdx.y) * kTileH;
    const int epiSteps = (min(kTileH, p.Oy - y0) + kEpiRowsPerStep - 1) / kEpiRowsPerStep;
    uint8_t *epi = smem + g.epiOff;
    // table-row segments of epilogue step t: rows y0+2t+h, buffers
    // [stage][h][S top, S bottom, Q top, Q bottom]
    auto issue_epi = [&](int t) {
        const int st = t % kEpiStages;
        const int y = y0 + kEpiRowsPerStep * t;  // first output row of the step
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                     ::"r"(smem_u32(&s_ebar[st])),
                       "r"((uint32_t)(kEpiBufs * kEpiRowsPerStep * epiBW * 8))
                     : "memory");
        uint8_t *b = epi + st * kEpiBufs * epiBuf;
        tma_2d(&tmS, b, x0 - 2, y - 1, &s_ebar[st]);                      // rows y-1 ..
        tma_2d(&tmS, b + epiBuf, x0 - 2, y + p.hT - 1, &s_ebar[st]);      // rows y+hT-1 ..
        tma_2d(&tmQ, b + 2 * epiBuf, x0 - 2, y - 1, &s_ebar[st]);
        tma_2d(&tmQ, b + 3 * epiBuf, x0 - 2, y + p.hT - 1, &s_ebar[st]);
    };

    if (kTmaEpi && tid == 0) {
        for (int i = 0; i < kEpiStages; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&s_ebar[i])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;"
                         ::"r"(smem_u32(&s_efree[i])), "r"(kWarps));
        }
        asm volatile("fence.mbarrier_init.release.cluster;");
        asm volatile("fence.proxy.async.shared::cta;");
    }

    // --- stage the image tile (copy 0) ---------------------------------
    if (kTma) {
        if (tid == 0) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&s_bar)));
            asm volatile("fence.mbarrier_init.release.cluster;");
            asm volatile("fence.proxy.async.shared::cta;");
            const uint32_t bytes = (uint32_t)(g.boxW * g.boxH);
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                         ::"r"(smem_u32(&s_bar)), "r"(bytes) : "memory");
            asm volatile(
                "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                " [%0], [%1, {%2, %3}], [%4];"
                ::"r"(smem_u32(smem)), "l"(&tmap), "r"(x0), "r"(y0), "r"(smem_u32(&s_bar))
                : "memory");
        }
    }
    // The first table-row stages are requested after the image tile: this
    // SM's copies are served in order, and the tile is needed first.  The
    // CTAs of the first wave of an overlapped launch may start before the
    // tables are complete: they request them after their numerator.
    const bool lateIssue = (int)(blockIdx.y * gridDim.x + blockIdx.x) < p.lateWave;
    if (kTmaEpi && tid == 0 && !lateIssue) {
        grid_dependency_wait();
        for (int t = 0; t < kEpiStages && t < epiSteps; ++t) issue_epi(t);
    }
    if (!kTma) {
        for (int idx = tid; idx < g.boxW * g.boxH; idx += kThreads) {
            const int r = idx / g.boxW, c = idx - r * g.boxW;
            const int y = y0 + r, x = x0 + c;
            smem[idx] = (y < p.H && x < p.W) ? __ldg(p.img + (size_t)y * p.W + x) : (uint8_t)0;
        }
    }

    // --- pack the template, template statistics (overlaps the TMA) -------
    uint32_t *tw = reinterpret_cast<uint32_t *>(smem + g.tmplOff);
    const int nWords = p.hT * g.nch * 4;
    unsigned sa = 0, sb = 0;    // SumT < 2^25 and SumT2 < 2^32 (wT*hT <= 66051)
    for (int wi = tid; wi < nWords; wi += kThreads) {
        const int j = wi / (g.nch * 4), cw = wi - j * g.nch * 4;
        const int slot = ((cw >> 2) * p.hT + j) * 4 + (cw & 3);  // chunk-major
        uint32_t v = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int i = 4 * cw + b;
            if (i < p.wT) {
                const unsigned t = __ldg(p.tmpl + (size_t)j * p.wT + i);
                v |= t << (8 * b);
                sa += t;
                sb += t * t;
            }
        }
        tw[slot] = v;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        sa += __shfl_xor_sync(0xffffffffu, sa, o);
        sb += __shfl_xor_sync(0xffffffffu, sb, o);
    }
    if (lane == 0) { s_red[warp][0] = sa; s_red[warp][1] = sb; }
    __syncthreads();
    if (tid == 0) {
        unsigned a = 0, b = 0;
        for (int w = 0; w < kWarps; ++w) { a += s_red[w][0]; b += s_red[w][1]; }
        const long long N = (long long)p.wT * p.hT;
        const long long vT = N * (long long)b - (long long)a * (long long)a;
        s_sumT = a;
        s_vT = vT;
        s_invSqrtVT = vT > 0 ? __frsqrt_rn(u64_to_f32((unsigned long long)vT)) : 0.0f;
    }
    if (kTma) mbar_wait(&s_bar, 0, p.status);  // every thread: the tile has landed
    __syncthreads();

    // --- numerator: SumIT for 8 rows x 4 shifts per thread -----------------
    // Lane 4*qg + d reads 32 aligned bytes at 16*qg (+16 per chunk) and
    // moves them by d bytes with one byte permute per word, so each of its
    // shifts x0 + 16*qg + 4*k + d sees 32-bit groups of four pixels.
    const int hT = kHT ? kHT : p.hT;
    const int qg = lane >> 2, d = lane & 3;
    const uint32_t sel = 0x3210u + 0x1111u * (uint32_t)d;
    const uint8_t *cp = smem + 16 * qg;
    uint32_t acc[kRPT][4];
#pragma unroll
    for (int i = 0; i < kRPT; ++i)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[i][k] = 0u;

    for (int c = 0; c < g.nch; ++c) {
        const uint8_t *cc = cp + 16 * c + warp * kRPT * g.boxW;
        const uint4 *tc = reinterpret_cast<const uint4 *>(tw) + c * hT;  // chunk c of row j at tc[j]
        // the d-shifted words of tile row r of this warp
        auto row_words = [&](int r, uint32_t (&v)[7]) {
            const uint8_t *rp = cc + r * g.boxW;
            const uint4 a = *reinterpret_cast<const uint4 *>(rp);
            const uint4 b = *reinterpret_cast<const uint4 *>(rp + 16);
            v[0] = __byte_perm(a.x, a.y, sel); v[1] = __byte_perm(a.y, a.z, sel);
            v[2] = __byte_perm(a.z, a.w, sel); v[3] = __byte_perm(a.w, b.x, sel);
            v[4] = __byte_perm(b.x, b.y, sel); v[5] = __byte_perm(b.y, b.z, sel);
            v[6] = __byte_perm(b.z, b.w, sel);
        };
        // output row i of the thread += image row (i + j) x template row j
        auto mac = [&](uint32_t (&a)[4], const uint32_t (&v)[7], const uint4 t) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t s = a[k];
                s = __dp4a(v[k + 0], t.x, s);
                s = __dp4a(v[k + 1], t.y, s);
                s = __dp4a(v[k + 2], t.z, s);
                s = __dp4a(v[k + 3], t.w, s);
                a[k] = s;
            }
        };
        if (hT >= kRPT) {
            // tile row r meets output rows i = max(0, r-hT+1) .. min(7, r):
            // ramp-up rows, full rows and ramp-down rows, without branches
#pragma unroll
            for (int r = 0; r < kRPT - 1; ++r) {
                uint32_t v[7];
                row_words(r, v);
#pragma unroll
                for (int i = 0; i <= r; ++i) mac(acc[i], v, tc[r - i]);
            }
            auto full_row = [&](int r) {
                uint32_t v[7];
                row_words(r, v);
#pragma unroll
                for (int i = 0; i < kRPT; ++i) mac(acc[i], v, tc[r - i]);
            };
            if constexpr (kHT != 0) {
                // fixed height: the phase unrolls and the template rows it
                // reads stay in registers from one tile row to the next
#pragma unroll
                for (int r = kRPT - 1; r < kHT; ++r) full_row(r);
            } else {
                for (int r = kRPT - 1; r < hT; ++r) full_row(r);
            }
#pragma unroll
            for (int m = 0; m < kRPT - 1; ++m) {
                const int r = hT + m;
                uint32_t v[7];
                row_words(r, v);
#pragma unroll
                for (int i = m + 1; i < kRPT; ++i) mac(acc[i], v, tc[r - i]);
            }
        } else {
            const int rows = kRPT + hT - 1;
            for (int r = 0; r < rows; ++r) {
                uint32_t v[7];
                row_words(r, v);
#pragma unroll
                for (int i = 0; i < kRPT; ++i) {
                    const int j = r - i;
                    if (j >= 0 && j < hT) mac(acc[i], v, tc[j]);
                }
            }
        }
    }

    if (kTmaEpi && tid == 0 && lateIssue) {
        grid_dependency_wait();
        for (int t = 0; t < kEpiStages && t < epiSteps; ++t) issue_epi(t);
    }

    // --- transpose SumIT through shared memory ------------------------------
    __syncthreads();  // every warp is done with the staged copies
    // [kTileH][kOutW], column c stored at c ^ (((c >> 5) & 3) << 2): the
    // 32 lanes of one store (columns 16*qg + 4*k + d) then fall in 32
    // different banks, and a row read of 32 consecutive columns still does.
    uint32_t *sIT = reinterpret_cast<uint32_t *>(smem + (kDirect ? g.sumOff : 0));
    {
        uint32_t *sw = sIT + 16 * qg + d;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int ck = 4 * (k ^ (qg >> 1));
#pragma unroll
            for (int i = 0; i < kRPT; ++i)
                sw[(warp * kRPT + i) * kOutW + ck] = acc[i][k];
        }
    }
    __syncthreads();

    // --- epilogue: moments from S and Q, coefficient -----------------------
    // The four-corner sums are below 2^32, so they are formed from the low
    // 32 bits of the table entries with wrapping arithmetic, exactly.  For
    // templates of at most kMaxInt32N pixels the numerator and variance
    // terms are exact 32-bit integers; larger templates take exact 64-bit
    // integers.
    const long long N = (long long)p.wT * p.hT;
    // S and Q are complete: the plain-load epilogue reads them in every
    // thread (with TMA only thread 0's requests do, after its own wait)
    if constexpr (!kTmaEpi && !kDirect) grid_dependency_wait();
    const long long sT = s_sumT, vT = s_vT;
    const float invSqrtVT = s_invSqrtVT;
    const bool smallN = N <= kMaxInt32N;
    const uint32_t Nu = (uint32_t)N, sTu = (uint32_t)sT;
    const int h = warp >> 2, xo = (warp & 3) * 32 + lane, x = x0 + xo;
    const int xs = xo ^ ((warp & 3) << 2);                     // column xo in the SumIT layout
    const int segWords = epiBW * 2;                            // u32 words per table-row segment
    const int cl = 2 * (xo + 1), cr = 2 * (xo + p.wT + 1);      // low words of x-1, x+wT-1
    // the loop is instantiated per coefficient path and for full tiles
    // (every output row and column valid: no per-output bounds checks)
    auto epilogue = [&](auto smallTag, auto fullTag) {
    constexpr bool kSmall = decltype(smallTag)::value, kFull = decltype(fullTag)::value;
    const size_t ox2 = 2 * (size_t)p.Ox, ox4 = 2 * ox2;
    float *outRow = p.out + (size_t)(y0 + h) * p.Ox + x;   // row y0 + 4t + h, column x
    auto step = [&](int t, auto stTag) {
        constexpr int st = decltype(stTag)::value;
        const uint32_t par = (uint32_t)((t / kEpiStages) & 1);
        // this thread's output rows of the step: h and h + 2
        uint32_t sIv[2] = {0, 0}, sI2v[2] = {0, 0};
        if (kTmaEpi) {
            // the whole warp polls the stage's barrier (a uniform wait)
            if (!mbar_try(&s_ebar[st], par)) mbar_wait(&s_ebar[st], par, p.status);
            const uint32_t *b = reinterpret_cast<const uint32_t *>(epi + st * kEpiBufs * epiBuf);
            const int box = epiBuf / 4;                            // u32 words per box
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int o = (h + 2 * q) * segWords;
                const uint32_t *St = b + o, *Sb = b + box + o, *Qt = b + 2 * box + o, *Qb = b + 3 * box + o;
                // both corners inside the staged segment, the segment inside its box
                if (!NCC_BOUNDS(cl >= 0 && cr < segWords && o + segWords <= box, p.status)) continue;
                sIv[q] = Sb[cr] - St[cr] - Sb[cl] + St[cl];
                sI2v[q] = Qb[cr] - Qt[cr] - Qb[cl] + Qt[cl];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_efree[st]);           // this warp is done with the stage
            // the refill of this stage for step t+2 goes out as soon as every
            // warp has read it, before this step's arithmetic
            if (tid == 0 && t + kEpiStages < epiSteps) {
                mbar_wait(&s_efree[st], par, p.status);          // all warps released the stage
                issue_epi(t + kEpiStages);
            }
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
        const int row = kEpiRowsPerStep * t + h + 2 * q, y = y0 + row;
        uint32_t sI = sIv[q], sI2 = sI2v[q];
        if (!kTmaEpi && y < p.Oy && x < p.Ox) {
            const size_t W = (size_t)p.W;
            const long long *St = p.S + (size_t)(y - 1) * W, *Sb = p.S + (size_t)(y + p.hT - 1) * W;
            const long long *Qt = p.Q + (size_t)(y - 1) * W, *Qb = p.Q + (size_t)(y + p.hT - 1) * W;
            const int xl = x - 1, xr = x + p.wT - 1;
            sI = (uint32_t)__ldg(Sb + xr);
            sI2 = (uint32_t)__ldg(Qb + xr);
            if (y > 0) { sI -= (uint32_t)__ldg(St + xr); sI2 -= (uint32_t)__ldg(Qt + xr); }
            if (x > 0) { sI -= (uint32_t)__ldg(Sb + xl); sI2 -= (uint32_t)__ldg(Qb + xl); }
            if (x > 0 && y > 0) { sI += (uint32_t)__ldg(St + xl); sI2 += (uint32_t)__ldg(Qt + xl); }
        }
        if (kFull || (y < p.Oy && x < p.Ox)) {
            const unsigned sumIT = sIT[row * kOutW + xs];
            const size_t o = (size_t)y * p.Ox + x;
            float *const op = outRow + (q ? ox2 : (size_t)0);
            // the output inside the map; the stepped row pointer at its address
            if (!NCC_BOUNDS(y < p.Oy && x < p.Ox && (kMoments || op == p.out + o), p.status)) continue;
            if (kMoments) {
                p.sumI[o] = (long long)sI;
                p.sumI2[o] = (long long)sI2;
                p.sumIT[o] = (long long)sumIT;
            } else {
                float num, vIf;
                if (kSmall) {
                    // both terms exactly by wrapping 32-bit products, then
                    // one rounding each
                    num = (float)(int)(Nu * sumIT - sI * sTu);
                    const uint32_t vIu = Nu * sI2 - sI * sI;
                    vIf = (float)max(vIu, 1u);
                } else {
                    // SumI < 2^25 and SumT < 2^25; SumI2 < 2^32
                    const long long numi = (long long)((unsigned long long)N * sumIT) -
                                           (long long)sI * (long long)sT;
                    const long long vI = (long long)((unsigned long long)N * sI2) -
                                         (long long)sI * (long long)sI;
                    num = i64_to_f32(numi);
                    vIf = u64_to_f32((unsigned long long)max(vI, 1ll));
                }
                // A window of zero variance has num = 0 exactly (all its pixels
                // are equal), so with vIf >= 1 its coefficient is +0 without
                // a select; invSqrtVT is 0 for a zero-variance template.
                const float rr = num * rsqrt_approx(vIf) * invSqrtVT;
                __stcs(op, fminf(1.0f, fmaxf(-1.0f, rr)));
            }
        }
        }
        outRow += ox4;
    };
    // steps in pairs, so that each step's ring stage (and with it every
    // staged-row address) is a compile-time constant
    static_assert(kEpiStages == 2, "steps go in pairs, one per ring stage");
    for (int t = 0; t < epiSteps; t += 2) {
        step(t, IntTag<0>{});
        if (t + 1 < epiSteps) step(t + 1, IntTag<1>{});
    }
    };
    // Direct moments.  Per pass of kDirRows output rows: (1) thread t keeps
    // the sums of I and I^2 over hT tile rows of tile column t, sliding down
    // one row at a time, and stores them; (2) each stored row is replaced by
    // its exclusive prefix over the columns; (3) SumI of the window at
    // column c is prefix[c + wT] - prefix[c], and the same for SumI2.  The
    // u32 arithmetic wraps, which is exact: both sums are below 2^32.
    auto direct_epilogue = [&](auto smallTag, auto fullTag) {
    constexpr bool kSmall = decltype(smallTag)::value, kFull = decltype(fullTag)::value;
    const int ncols = kOutW + p.wT - 1;         // tile columns the windows cover
    const int cP = g.cPitch;
    uint32_t *P1 = reinterpret_cast<uint32_t *>(smem + g.cpOff), *P2 = P1 + kDirRows * cP;
    const uint8_t *col = smem + tid;              // this thread's tile column
    const bool colOwner = tid < ncols;
    uint32_t c1 = 0, c2 = 0;
    if (colOwner)
        for (int j = 0; j < p.hT; ++j) {
            const uint32_t v = col[j * g.boxW];
            c1 += v;
            c2 += v * v;
        }
    const int rowsValid = min(kTileH, p.Oy - y0);
    const int per = (ncols + 31) >> 5;            // columns per lane in the prefix pass (<= 8)
    for (int yb = 0; yb < rowsValid; yb += kDirRows) {
        // (1) column sums of the pass's rows
        if (colOwner) {
#pragma unroll 4
            for (int r = 0; r < kDirRows; ++r) {
                const int yr = yb + r;
                P1[r * cP + tid] = c1;
                P2[r * cP + tid] = c2;
                if (yr + 1 < kTileH) {                 // the tile holds rows 0 .. kTileH + hT - 2
                    const uint32_t a = col[(yr + p.hT) * g.boxW], b = col[yr * g.boxW];
                    c1 += a - b;
                    c2 += a * a - b * b;
                }
            }
        }
        __syncthreads();
        // (2) exclusive prefix of every stored row, in place: entry e holds
        //     the sum of columns 0 .. e-1 (entry ncols the whole row)
        if constexpr (kNarrow) {
            // at most kOutW + kNarrowT - 1 columns: 5 per lane, both tables
            // of a row in one pass
            constexpr int kPer = (kOutW + kNarrowT - 1 + 31) / 32;
            for (int rr = warp; rr < kDirRows; rr += kWarps) {
                uint32_t *r1 = P1 + rr * cP, *r2 = P2 + rr * cP;
                uint32_t a[kPer], b[kPer], ra = 0, rb = 0;
#pragma unroll
                for (int j = 0; j < kPer; ++j) {
                    const int c = lane * kPer + j;
                    const bool in = c < ncols;
                    ra += in ? r1[c] : 0u;
                    rb += in ? r2[c] : 0u;
                    a[j] = ra;
                    b[j] = rb;
                }
                uint32_t ia = ra, ib = rb;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t ua = __shfl_up_sync(0xffffffffu, ia, o);
                    const uint32_t ub = __shfl_up_sync(0xffffffffu, ib, o);
                    if (lane >= o) { ia += ua; ib += ub; }
                }
                ia -= ra;
                ib -= rb;
                __syncwarp();                         // every lane has read its columns
#pragma unroll
                for (int j = 0; j < kPer; ++j) {
                    const int c = lane * kPer + j;
                    if (c < ncols) {
                        r1[c + 1] = ia + a[j];
                        r2[c + 1] = ib + b[j];
                    }
                }
                if (lane == 0) { r1[0] = 0u; r2[0] = 0u; }
            }
        } else
        for (int task = warp; task < 2 * kDirRows; task += kWarps) {
            uint32_t *rowp = (task < kDirRows ? P1 : P2) + (task % kDirRows) * cP;
            uint32_t s[8];
            uint32_t run = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int c = lane * per + j;
                run += (j < per && c < ncols) ? rowp[c] : 0u;
                s[j] = run;
            }
            uint32_t incl = run;                      // inclusive scan of the lane totals
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            const uint32_t base = incl - run;
            __syncwarp();                             // every lane has read its columns
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int c = lane * per + j;
                if (j < per && c < ncols) rowp[c + 1] = base + s[j];
            }
            if (lane == 0) rowp[0] = 0u;
        }
        __syncthreads();
        // (3) coefficients of the pass's rows: thread = column xo, rows h, h+2, ..
        float *const outPass = p.out + (size_t)(y0 + yb + h) * p.Ox + x;
        const size_t ox2 = 2 * (size_t)p.Ox;
#pragma unroll 2
        for (int i = 0; i < kDirRows / 2; ++i) {
            const int r = h + 2 * i, row = yb + r, y = y0 + row;
            if (kFull || (y < p.Oy && x < p.Ox)) {
                // the prefix entries inside the pass's buffers; the output in the map
                if (!NCC_BOUNDS(xo + p.wT < cP && y < p.Oy && x < p.Ox &&
                                    (kMoments || outPass + (size_t)i * ox2 == p.out + (size_t)y * p.Ox + x),
                                p.status))
                    continue;
                const uint32_t sI = P1[r * cP + xo + p.wT] - P1[r * cP + xo];
                const uint32_t sI2 = P2[r * cP + xo + p.wT] - P2[r * cP + xo];
                const unsigned sumIT = sIT[row * kOutW + xs];
                const size_t o = (size_t)y * p.Ox + x;
                if (kMoments) {
                    p.sumI[o] = (long long)sI;
                    p.sumI2[o] = (long long)sI2;
                    p.sumIT[o] = (long long)sumIT;
                } else {
                    float num, vIf;
                    if (kSmall) {
                        num = (float)(int)(Nu * sumIT - sI * sTu);
                        const uint32_t vIu = Nu * sI2 - sI * sI;
                        vIf = (float)max(vIu, 1u);
                    } else {
                        const long long numi = (long long)((unsigned long long)N * sumIT) -
                                               (long long)sI * (long long)sT;
                        const long long vI = (long long)((unsigned long long)N * sI2) -
                                             (long long)sI * (long long)sI;
                        num = i64_to_f32(numi);
                        vIf = u64_to_f32((unsigned long long)max(vI, 1ll));
                    }
                    const float rr = num * rsqrt_approx(vIf) * invSqrtVT;
                    __stcs(outPass + (size_t)i * ox2, fminf(1.0f, fmaxf(-1.0f, rr)));
                }
            }
        }
        __syncthreads();                              // before the next pass overwrites the buffers
    }
    };
    const bool full = y0 + kTileH <= p.Oy && x0 + kOutW <= p.Ox;
    if constexpr (kDirect) {
        if (smallN && full) direct_epilogue(BoolTag<true>{}, BoolTag<true>{});
        else if (smallN) direct_epilogue(BoolTag<true>{}, BoolTag<false>{});
        else direct_epilogue(BoolTag<false>{}, BoolTag<false>{});
    } else {
        if (smallN && full) epilogue(BoolTag<true>{}, BoolTag<true>{});
        else if (smallN) epilogue(BoolTag<true>{}, BoolTag<false>{});
        else epilogue(BoolTag<false>{}, BoolTag<false>{});
    }
}

}  // namespace

bool corr_dp4a_supported(int wT, int hT) {
    return wT >= 1 && hT >= 1 && make_geom(wT, hT).smemBytes <= kMaxSmem;
}

bool corr_dp4a_direct_supported(int wT, int hT) {
    return wT >= 1 && hT >= 1 && kOutW + wT - 1 <= kDirMaxCols &&
           make_geom(wT, hT, true).smemBytes <= kMaxSmem;
}

cudaError_t corr_dp4a_launch(const CorrArgs &a, cudaStream_t stream) {
    KParams p;
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
    if (a.direct && !corr_dp4a_direct_supported(a.wT, a.hT)) return cudaErrorNotSupported;
    // Tiles of 128 x 32 (four output rows per thread) on the all-TMA path:
    //   - for templates up to 16 wide and kQuadMaxHT high, whose kernel fits
    //     four CTAs on an SM (64 registers, under 56 KB of shared memory);
    //   - for maps too small to give every SM two tiles of 128 x 64.
    const long long tiles64 =
        (long long)((p.Ox + kOutW - 1) / kOutW) * ((p.Oy + kOutH - 1) / kOutH);
    const bool allTma = !a.direct && a.W % 16 == 0 && (uintptr_t)a.img % 16 == 0 &&
                        (uintptr_t)a.S % 16 == 0 && (uintptr_t)a.Q % 16 == 0;
    const bool quad = allTma && a.wT <= kNarrowT && a.hT <= kQuadMaxHT;
    const bool small = quad || (allTma && tiles64 < 2ll * sm_count() && a.wT <= 126 && a.hT <= 225);
    const int tileH = small ? kWarps * kSmallRPT : kOutH;
    // the CTAs resident at once: four per SM for the narrow 128 x 32 kernels
    p.lateWave = a.overlap_prev ? (quad ? 4 : kMaxCtasPerSm) * sm_count() : 0;
    p.g = make_geom(a.wT, a.hT, a.direct, tileH);

    CUtensorMap tmap;
    memset(&tmap, 0, sizeof(tmap));
    bool tma = (a.W % 16 == 0) && ((uintptr_t)a.img % 16 == 0) && p.g.boxW <= kMaxTmaBox &&
               p.g.boxH <= kMaxTmaBox;
    EncodeTiledFn enc = tma ? tensor_map_encoder() : nullptr;
    if (enc) {
        const cuuint64_t dims[2] = {(cuuint64_t)a.W, (cuuint64_t)a.H};
        const cuuint64_t strides[1] = {(cuuint64_t)a.W};
        const cuuint32_t box[2] = {(cuuint32_t)p.g.boxW, (cuuint32_t)p.g.boxH};
        const cuuint32_t estr[2] = {1, 1};
        CUresult r = enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(a.img), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        tma = (r == CUDA_SUCCESS);
    } else {
        tma = false;
    }
    const bool moments = a.sumIT != nullptr;
    CUtensorMap tmS, tmQ;
    memset(&tmS, 0, sizeof(tmS));
    memset(&tmQ, 0, sizeof(tmQ));
    bool tmaEpi = !a.direct && (a.W % 2 == 0) && ((uintptr_t)a.S % 16 == 0) &&
                  ((uintptr_t)a.Q % 16 == 0) && p.g.epiBW <= kMaxTmaBox;
    if (tmaEpi) enc = tensor_map_encoder();
    if (tmaEpi && enc) {
        const cuuint64_t dims[2] = {(cuuint64_t)a.W, (cuuint64_t)a.H};
        const cuuint64_t strides[1] = {(cuuint64_t)a.W * 8};
        const cuuint32_t box[2] = {(cuuint32_t)p.g.epiBW, (cuuint32_t)kEpiRowsPerStep};
        const cuuint32_t estr[2] = {1, 1};
        CUresult r1 = enc(&tmS, CU_TENSOR_MAP_DATA_TYPE_INT64, 2, const_cast<int64_t *>(a.S), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        CUresult r2 = enc(&tmQ, CU_TENSOR_MAP_DATA_TYPE_INT64, 2, const_cast<int64_t *>(a.Q), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        tmaEpi = (r1 == CUDA_SUCCESS && r2 == CUDA_SUCCESS);
    } else {
        tmaEpi = false;
    }
    if (small && !(tma && tmaEpi)) return cudaErrorNotSupported;  // the checks above exclude it
    // a band of output rows [rowBegin, rowEnd): whole tiles only, so that no
    // tile belongs to two bands (kCorrBandRows is a multiple of both heights)
    const int rowEnd = a.rowEnd > 0 ? a.rowEnd : p.Oy;
    if (a.rowBegin < 0 || a.rowBegin % tileH != 0 || rowEnd > p.Oy || a.rowBegin >= rowEnd ||
        (rowEnd % tileH != 0 && rowEnd != p.Oy))
        return cudaErrorInvalidValue;
    p.tileRow0 = a.rowBegin / tileH;
    const dim3 grid((p.Ox + kOutW - 1) / kOutW, (rowEnd + tileH - 1) / tileH - p.tileRow0);
    const dim3 block(kThreads);
    const size_t smem = (size_t)p.g.smemBytes;
    cudaError_t e;
#define NCC_LAUNCH(T, M, E, NW, HT, D, R)                                                    \
    do {                                                                                     \
        e = cudaFuncSetAttribute(corr_dp4a_kernel<T, M, E, NW, HT, D, R>,                    \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);    \
        if (e != cudaSuccess) return e;                                                      \
        if (a.overlap_prev) {                                                                \
            cudaLaunchConfig_t cfg = {};                                                     \
            cfg.gridDim = grid;                                                              \
            cfg.blockDim = block;                                                            \
            cfg.dynamicSmemBytes = smem;                                                     \
            cfg.stream = stream;                                                             \
            cudaLaunchAttribute attr[1];                                                     \
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;                 \
            attr[0].val.programmaticStreamSerializationAllowed = 1;                          \
            cfg.attrs = attr;                                                                \
            cfg.numAttrs = 1;                                                                \
            e = cudaLaunchKernelEx(&cfg, corr_dp4a_kernel<T, M, E, NW, HT, D, R>, tmap, tmS, tmQ, p); \
            if (e != cudaSuccess) return e;                                                  \
        } else {                                                                             \
            corr_dp4a_kernel<T, M, E, NW, HT, D, R><<<grid, block, smem, stream>>>(tmap, tmS, tmQ, p); \
        }                                                                                    \
    } while (0)
    // the fixed narrow layout only where the rows are staged by TMA; a
    // compile-time height for the common 16-row templates on that path
    const bool narrow = a.wT <= kNarrowT;
#define NCC_LAUNCH_E(T, M)                                                         \
    do {                                                                           \
        if (a.direct && narrow && a.hT == 16) NCC_LAUNCH(T, M, false, true, 16, true, 8); \
        else if (a.direct && narrow) NCC_LAUNCH(T, M, false, true, 0, true, 8);    \
        else if (a.direct) NCC_LAUNCH(T, M, false, false, 0, true, 8);             \
        else if (tmaEpi && narrow && a.hT == 16) NCC_LAUNCH(T, M, true, true, 16, false, 8); \
        else if (tmaEpi && narrow) NCC_LAUNCH(T, M, true, true, 0, false, 8);      \
        else if (tmaEpi) NCC_LAUNCH(T, M, true, false, 0, false, 8);               \
        else NCC_LAUNCH(T, M, false, false, 0, false, 8);                          \
    } while (0)
    // 128 x 32 tiles: the all-TMA kernels with four rows per thread
#define NCC_LAUNCH_S(M)                                                                    \
    do {                                                                                   \
        if (narrow && a.hT == 16) NCC_LAUNCH(true, M, true, true, 16, false, kSmallRPT);   \
        else if (narrow) NCC_LAUNCH(true, M, true, true, 0, false, kSmallRPT);             \
        else NCC_LAUNCH(true, M, true, false, 0, false, kSmallRPT);                        \
    } while (0)
    if (small && moments) NCC_LAUNCH_S(true);
    else if (small) NCC_LAUNCH_S(false);
    else if (tma && moments) NCC_LAUNCH_E(true, true);
    else if (tma) NCC_LAUNCH_E(true, false);
    else if (moments) NCC_LAUNCH_E(false, true);
    else NCC_LAUNCH_E(false, false);
#undef NCC_LAUNCH_S
#undef NCC_LAUNCH_E
#undef NCC_LAUNCH
    return cudaGetLastError();
}

}  // namespace ncc
