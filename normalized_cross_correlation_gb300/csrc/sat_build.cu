// sat_build.cu -- single-pass builder of the two summed-area tables
// S = SAT(I) and Q = SAT(I^2), inclusive, int64 (The CUDA Handbook,
// section 15.8, "The Denominator: Summed Area Tables").
//
// Design (GB300).  The image is cut into tiles of 128 columns by 128 rows,
// handed out by an atomic ticket in row-major order to a persistent grid
// (three CTAs on every SM).  Each CTA runs two warp groups over a
// double-buffered shared-memory stage:
//   - producer warps 0-3 take a ticket, load the tile's pixels with one TMA
//     box per tile, issued a tile ahead into a three-slot pixel ring (plain
//     loads when rows are not 16-byte multiples).  Thread pt owns row pt and
//     column pt: it sums its row with byte dot products (in uint32: a row's
//     running sum of squares is at most W*255^2 < 2^32 for W <= 66051) and
//     publishes it at once, then forms the column sums of the warp-local
//     row prefixes while its first look-back loads are in flight, and gets
//     the row's carry from the tiles to its left and the column's carry from
//     the tiles above by decoupled look-backs -- the section's three-state
//     protocol (empty / aggregate published / inclusive prefix published).
//     The stage receives the row carries and each writer group's starting
//     column sums;
//   - writer warps 4-7 rebuild the rows from the pixels, four rows at a
//     time so that their warp scans overlap, and stream S and Q out as
//     int64 with 32-byte stores.
// The look-back latency of one tile thus overlaps the writes of the
// previous one inside every CTA.
//
// Sharing the tiles.  One SM stores at most about 28 bytes per clock,
// whatever its warps or store instructions, and the tables are 16 of the
// 17 bytes per pixel, so an SM that writes one tile more than the others
// ends one tile's store time later.  The ticket rule therefore evens out
// tiles per SM, not per CTA: a CTA draws only while its SM holds fewer than
// ceil(tiles / SMs) tiles and no more than its share of the tiles drawn so
// far; otherwise it naps (at most kShareWaitNs) until the tiles run out.
// The last CTA to finish returns the ticket and the SM counters to zero.
//
// Look-back words.  Every published value is one 64-bit word holding
// {epoch:5, state:2, value:57}, written and read with single-copy-atomic
// relaxed GPU-scope accesses: the state travels with its value, so a
// publication needs no separate flag or fence.  Row words pack the row's
// sum of I (25 bits) and of I^2 (32 bits) -- both fit for W <= 66051 and
// their sums never carry across fields.  Column words carry S (< 2^39) or
// Q (< 2^47) of one column, one word each.  A waiting thread reads a
// window of predecessors with independent loads per round, and a producer
// thread keeps its row's window and its column's windows in flight together:
// the column look-back reads only the tiles above, so it runs during the row
// look-back, and only this tile's own column publication waits for the row
// carries (its column sums include them).  The epoch tag
// lets the workspace be reused without clearing it: a word from an earlier
// call reads as empty.
//
// Tickets are taken in row-major order and every wait points at a tile with
// a smaller ticket, whose CTA is already running: the look-backs cannot
// deadlock.  Every wait is bounded (timeout and iteration cap); a wait that
// runs out records NCC_ERR_TIMEOUT, raises the call's abort word, and the
// CTA stops without writing that tile.
#include "ncc_common.cuh"

#include <cuda.h>
#include <mutex>
#include <string.h>

namespace ncc {
namespace {

constexpr int kTileW = 128;           // tile width: 32 lanes x 4 columns
constexpr int kGroups = 4;            // producer warps = writer warps = row groups per tile
constexpr int kProducers = kGroups * 32;
constexpr int kThreads = 2 * kProducers;
constexpr int kRowsPerWarp = 32;
constexpr int kTileH = kGroups * kRowsPerWarp;  // 128
constexpr int kCtasPerSm = 3;
constexpr int kMaxSmIds = 1024;       // per-SM tile counters (indexed by %smid)
constexpr uint64_t kShareWaitNs = 40000;  // longest nap of a CTA whose SM is ahead of its share
constexpr int kShareQ = 4;            // an SM may run ahead of its share by kShareQ/4 tile
constexpr int kStageDone = -1, kStageAbort = -2;
constexpr int kColWords = 2 * kTileW;          // S and Q word per column
constexpr int kRowWindow = 8;         // row predecessors read per look-back round
constexpr int kColWindowEarly = 4;    // column predecessors read alongside the row look-back
constexpr int kColWindow = 8;         // column predecessors read per round afterwards

constexpr int kEpochShift = 59, kStateShift = 57;
constexpr uint64_t kValueMask = (1ull << kStateShift) - 1;
constexpr int kRowQShift = 25;        // row word: I in bits 0..24, I^2 in 25..56
constexpr uint32_t kMaxEpoch = 31;

struct SatWs {
    unsigned long long *ticket;  // tile dispenser (ticket = tile index); 0 between launches
    unsigned *abort;             // holds the epoch of a call whose wait ran out
    unsigned *done;              // CTAs finished; the last one resets the counters
    unsigned *smTiles;           // [kMaxSmIds] tiles drawn by the CTAs of each SM
    uint64_t *row;               // [ntiles][kTileH] row words
    uint64_t *col;               // [ntiles][kColWords] column words (S part, then Q part)
};

__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t *p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_u64(uint64_t *p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t make_word(uint32_t epoch, uint32_t state, uint64_t value) {
    return ((uint64_t)epoch << kEpochShift) | ((uint64_t)state << kStateShift) | value;
}

__device__ __forceinline__ uint32_t word_state(uint64_t w, uint32_t epoch) {
    return ((uint32_t)(w >> kEpochShift) == epoch) ? (uint32_t)(w >> kStateShift) & 3u
                                                    : FLAG_EMPTY;
}

// Inclusive scans of kScanRows 128-pixel row segments, four bytes per lane:
// p[j][c] / s[j][c] = sum of pixels / of squared pixels of row j from the
// warp's first column up to this lane's column c (uint32).  The lane-local
// prefixes come from byte dot products; the sums over the lanes to the left
// come from one shuffle scan in which two rows' pixel sums share a word
// (each at most 128 * 255 < 2^16), so the rows' chains run side by side.
constexpr int kScanRows = 4;
__device__ __forceinline__ void row_scan_rows(const uint32_t (&px)[kScanRows], int lane,
                                              uint32_t (&p)[kScanRows][4],
                                              uint32_t (&s)[kScanRows][4]) {
    uint32_t tI[kScanRows / 2], tQ[kScanRows];
#pragma unroll
    for (int j = 0; j < kScanRows; ++j) {
        const uint32_t v = px[j];
        p[j][0] = v & 0xffu;
        p[j][1] = __dp4a(v, 0x00000101u, 0u);
        p[j][2] = __dp4a(v, 0x00010101u, 0u);
        p[j][3] = __dp4a(v, 0x01010101u, 0u);
        s[j][0] = __dp4a(v, v & 0x000000ffu, 0u);
        s[j][1] = __dp4a(v, v & 0x0000ffffu, 0u);
        s[j][2] = __dp4a(v, v & 0x00ffffffu, 0u);
        s[j][3] = __dp4a(v, v, 0u);
        tQ[j] = s[j][3];
    }
#pragma unroll
    for (int h = 0; h < kScanRows / 2; ++h) tI[h] = p[2 * h][3] | (p[2 * h + 1][3] << 16);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t uI[kScanRows / 2], uQ[kScanRows];
#pragma unroll
        for (int h = 0; h < kScanRows / 2; ++h) uI[h] = __shfl_up_sync(0xffffffffu, tI[h], o);
#pragma unroll
        for (int j = 0; j < kScanRows; ++j) uQ[j] = __shfl_up_sync(0xffffffffu, tQ[j], o);
        if (lane >= o) {
#pragma unroll
            for (int h = 0; h < kScanRows / 2; ++h) tI[h] += uI[h];
#pragma unroll
            for (int j = 0; j < kScanRows; ++j) tQ[j] += uQ[j];
        }
    }
#pragma unroll
    for (int h = 0; h < kScanRows / 2; ++h) {
        // exclusive = inclusive - own; neither half borrows (each half's
        // inclusive sum includes its own term)
        const uint32_t e = tI[h] - (p[2 * h][3] | (p[2 * h + 1][3] << 16));
        const uint32_t e0 = e & 0xffffu, e1 = e >> 16;
#pragma unroll
        for (int c = 0; c < 4; ++c) { p[2 * h][c] += e0; p[2 * h + 1][c] += e1; }
    }
#pragma unroll
    for (int j = 0; j < kScanRows; ++j) {
        const uint32_t e = tQ[j] - s[j][3];
#pragma unroll
        for (int c = 0; c < 4; ++c) s[j][c] += e;
    }
}

struct WaitCtx {
    unsigned *abort;
    int *status;
    uint32_t epoch;
    uint64_t t0, timeout_ns;
};

// One decoupled look-back in progress: the predecessors' words of one
// element sit at p0 + i*delta, i = 0..count-1 (nearest first).  `acc`
// gathers the values of consecutive published predecessors; the chain is
// done at the first inclusive prefix or after the last predecessor.  Loads
// and examination are separate steps so that a thread can keep several
// chains' windows in flight in one round trip.
struct Chain {
    const uint64_t *p0;
    long long delta;
    int count, next;
    uint64_t acc;
    bool done;
};

__device__ __forceinline__ Chain make_chain(const uint64_t *p0, long long delta, int count) {
    Chain c;
    c.p0 = p0;
    c.delta = delta;
    c.count = count;
    c.next = 0;
    c.acc = 0;
    c.done = count <= 0;
    return c;
}

template <int N>
__device__ __forceinline__ void chain_load(const Chain &c, uint64_t (&w)[N]) {
#pragma unroll
    for (int i = 0; i < N; ++i)
        w[i] = (!c.done && c.next + i < c.count) ? ld_relaxed_u64(c.p0 + (long long)(c.next + i) * c.delta)
                                                 : 0ull;
}

// Consumes the loaded window up to the first empty word; returns whether
// anything was consumed.
template <int N>
__device__ __forceinline__ bool chain_take(Chain &c, const uint64_t (&w)[N], uint32_t epoch) {
    if (c.done) return false;
    int used = 0;
    bool prefix = false;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        if (used == i && !prefix && c.next + i < c.count) {
            const uint32_t st = word_state(w[i], epoch);
            if (st != FLAG_EMPTY) {
                c.acc += w[i] & kValueMask;
                used = i + 1;
                prefix = (st == FLAG_PREFIX);
            }
        }
    }
    c.next += used;
    if (prefix || c.next >= c.count) c.done = true;
    return used > 0;
}

// Back-off between polls that found nothing new.  Returns false when the
// wait ran out (recorded as NCC_ERR_TIMEOUT, and the call's abort word
// raised) or another CTA of the call aborted.
struct Backoff {
    unsigned ns = 32, polls = 0;
    __device__ __forceinline__ bool wait(const WaitCtx &cx) {
        __nanosleep(ns);
        if (ns < 256) ns <<= 1;
        if ((++polls & 7u) == 0u) {
            if (ld_relaxed_gpu(cx.abort) == cx.epoch) return false;
            if (global_timer_ns() - cx.t0 > cx.timeout_ns || polls > (1u << 26)) {
                atomicExch(cx.abort, cx.epoch);
                record_status(cx.status, NCC_ERR_TIMEOUT);
                return false;
            }
        }
        return true;
    }
};

// 32 contiguous bytes (four int64) in one 256-bit store: a lane fills one
// whole L2 sector, a warp 1 KB.
__device__ __forceinline__ void st_v4_b64(long long *p, long long a, long long b, long long c,
                                          long long d) {
#ifdef NCC_SAT_STREAMING_STORES
    asm volatile("st.global.cs.v4.b64 [%0], {%1, %2, %3, %4};" ::"l"(p), "l"(a), "l"(b), "l"(c), "l"(d)
                 : "memory");
#else
    asm volatile("st.global.v4.b64 [%0], {%1, %2, %3, %4};" ::"l"(p), "l"(a), "l"(b), "l"(c), "l"(d)
                 : "memory");
#endif
}

__device__ __forceinline__ void named_bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void named_bar_arrive(int id, int n) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ unsigned sm_id() {
    unsigned r;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
    return r;
}

// One double-buffered hand-off from the producer warps to the writer warps.
struct Stage {
    uint2 rowCarry[kTileH];                 // row sums left of the tile (I, I^2)
    long long colStart[kGroups][2][kTileW]; // S / Q just above each writer group's first row
    int tile;                               // tile index; kStageDone / kStageAbort to stop
    int pix;                                // pixel-ring slot holding the tile's pixels
};

// Producer barrier (warps 0-3 only) and the stage hand-off barriers.
constexpr int kBarProd = 1, kBarFull0 = 2, kBarEmpty0 = 4;
constexpr int kPixSlots = 3;            // pixel ring: one tile ahead + two stages

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// kStore: 2 = 32-byte stores (W % 4 == 0, tables 32-byte aligned),
// 1 = 16-byte stores (W even, tables 16-byte aligned), 0 = 8-byte stores.
template <bool kTma, bool kAligned4, int kStore>
__global__ void __launch_bounds__(kThreads, 3)
sat_build_kernel(const __grid_constant__ CUtensorMap tmap, const uint8_t *__restrict__ img,
                 int W, int H, long long *__restrict__ S, long long *__restrict__ Q, SatWs ws,
                 int ntx, int ntiles, uint32_t epoch, int nsm, int smCap, int shareQ,
                 int *status, uint64_t timeout_ns, int fault_tile) {
    extern __shared__ __align__(128) uint8_t s_dyn[];
    uint8_t (*s_pix)[kTileH][kTileW] = reinterpret_cast<uint8_t (*)[kTileH][kTileW]>(
        (reinterpret_cast<uintptr_t>(s_dyn) + 127) & ~uintptr_t(127));
    __shared__ __align__(16) Stage st[2];
    __shared__ __align__(16) uint2 s_colPart[kGroups][kTileW];  // per-warp column sums of warp-local prefixes
    __shared__ long long s_warpCarry[kGroups][2];               // per-warp sums of the row carries
    __shared__ __align__(8) unsigned long long s_pbar[kPixSlots];
    __shared__ unsigned s_tile, s_next;
    __shared__ int s_fail, s_last;

    // A kernel launched after this one with programmatic serialization may
    // be scheduled as this grid's CTAs retire (it waits on this grid before
    // it reads the tables).
    asm volatile("griddepcontrol.launch_dependents;");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (warp < kGroups) {
        // ================= producer warps: tiles, scans, look-backs =================
        const int pt = tid;  // 0..127
        // Next tile.  One SM's store rate is what bounds the build, so the
        // tiles are shared out evenly over the SMs rather than the CTAs: a
        // CTA draws only while its SM holds fewer than smCap tiles and no
        // more than its share of the tiles drawn so far (plus shareQ/4 of a
        // tile); otherwise it naps, so that SMs behind draw first, until the
        // tiles run out.  The naps end after kShareWaitNs at the latest:
        // correctness never depends on other CTAs being resident.
        auto grab = [&]() -> unsigned {
            const unsigned smSlot = sm_id() % kMaxSmIds;
            const uint64_t w0 = global_timer_ns();
            for (;;) {
                // reserve the SM's next slot first, so that CTAs of one SM
                // deciding at once see each other; hand it back on a nap
                const unsigned c = atomicAdd(ws.smTiles + smSlot, 1u);
                const unsigned long long t = ld_relaxed_u64(reinterpret_cast<const uint64_t *>(ws.ticket));
                if (t >= (unsigned long long)ntiles || c < (unsigned)kCtasPerSm ||
                    (c < (unsigned)smCap &&
                     4ull * c * (unsigned)nsm <= 4ull * t + (unsigned long long)shareQ * (unsigned)nsm) ||
                    global_timer_ns() - w0 > kShareWaitNs)
                    break;
                atomicSub(ws.smTiles + smSlot, 1u);
                __nanosleep(256);
            }
            const unsigned long long t = atomicAdd(ws.ticket, 1ull);
            return t < (unsigned long long)ntiles ? (unsigned)t : (unsigned)ntiles;
        };
        // pixels of `tile` into ring slot `slot`: one TMA box (completion on
        // s_pbar[slot]); tiles past the image edge read zeros
        auto issue_pixels = [&](unsigned tile, int slot) {
            const int tx = (int)(tile % (unsigned)ntx), ty = (int)(tile / (unsigned)ntx);
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                         ::"r"(smem_addr(&s_pbar[slot])), "r"((uint32_t)(kTileH * kTileW)) : "memory");
            asm volatile(
                "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                " [%0], [%1, {%2, %3}], [%4];"
                ::"r"(smem_addr(&s_pix[slot][0][0])), "l"(&tmap), "r"(tx * kTileW), "r"(ty * kTileH),
                  "r"(smem_addr(&s_pbar[slot]))
                : "memory");
        };
        if (pt == 0) {
            if (kTma) {
                for (int k = 0; k < kPixSlots; ++k)
                    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&s_pbar[k])));
                asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            }
            s_next = grab();
            if (kTma && s_next < (unsigned)ntiles) issue_pixels(s_next, 0);
        }
        bool pending = kTma;  // a pixel load may be in flight into slot (i % 3)
        int i = 0;
        for (;; ++i) {
            const int sb = i & 1, ps = i % kPixSlots;
            Stage &S_ = st[sb];
            if (i >= 2) named_bar_sync(kBarEmpty0 + sb, kThreads);  // writers are done with tile i-2
            if (pt == 0) {
                const unsigned cur = s_next;
                s_tile = cur;
                s_fail = 0;
                if (cur < (unsigned)ntiles) {
                    s_next = grab();  // prefetch the next ticket and its pixels
                    if (kTma && s_next < (unsigned)ntiles) issue_pixels(s_next, (i + 1) % kPixSlots);
                }
            }
            named_bar_sync(kBarProd, kProducers);
            const unsigned tile = s_tile;
            if (tile >= (unsigned)ntiles) {
                if (pt == 0) S_.tile = kStageDone;
                named_bar_arrive(kBarFull0 + sb, kThreads);
                pending = false;
                break;
            }
            const WaitCtx cx{ws.abort, status, epoch, global_timer_ns(), timeout_ns};
            const int tx = (int)(tile % (unsigned)ntx), ty = (int)(tile / (unsigned)ntx);
            const int xl = tx * kTileW + 4 * lane;
            const int row0 = ty * kTileH + warp * kRowsPerWarp;
            const bool publish = (int)tile != fault_tile;

            // 1. pixels (four columns per lane), in the ring slot
            if (kTma) {
                // bounded wait for this slot's TMA (its (i/3)-th completion)
                uint32_t done = 0;
                for (unsigned it = 0; !done; ++it) {
                    asm volatile(
                        "{ .reg .pred P; mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2; selp.u32 %0, 1, 0, P; }"
                        : "=r"(done) : "r"(smem_addr(&s_pbar[ps])), "r"((uint32_t)((i / kPixSlots) & 1)) : "memory");
                    if (!done && it > (1u << 22)) { record_status(status, NCC_ERR_TIMEOUT); break; }
                }
            } else {
                for (int k = 0; k < kRowsPerWarp; ++k) {
                    const int y = row0 + k;
                    uint32_t v = 0;
                    if (y < H) {
                        const uint8_t *rp = img + (size_t)y * W;
                        if (kAligned4 && xl + 3 < W) {
                            v = __ldg(reinterpret_cast<const unsigned *>(rp + xl));
                        } else {
#pragma unroll
                            for (int b = 0; b < 4; ++b)
                                if (xl + b < W) v |= (uint32_t)__ldg(rp + xl + b) << (8 * b);
                        }
                    }
                    *reinterpret_cast<uint32_t *>(&s_pix[ps][warp * kRowsPerWarp + k][4 * lane]) = v;
                }
                __syncwarp();
            }
            // 2. this thread's row total (row pt, read with the word order
            //    rotated by the lane so that a warp's 32 rows hit 32 banks),
            //    published at once as the row's aggregate
            const uint8_t *myRow = &s_pix[ps][pt][0];
            uint32_t rowI = 0, rowQ = 0;
#pragma unroll 8
            for (int j = 0; j < kTileW / 4; ++j) {
                const uint32_t v = *reinterpret_cast<const uint32_t *>(myRow + 4 * ((j + lane) & 31));
                rowI = __dp4a(v, 0x01010101u, rowI);
                rowQ = __dp4a(v, v, rowQ);
            }
            const uint64_t rowV = (uint64_t)rowI | ((uint64_t)rowQ << kRowQShift);
            uint64_t *rowMine = ws.row + (size_t)tile * kTileH + pt;
            if (publish && NCC_BOUNDS(tile < ntiles && pt < kTileH, status))
                st_relaxed_u64(rowMine, make_word(epoch, tx == 0 ? FLAG_PREFIX : FLAG_AGGREGATE, rowV));

            // 3. row carry by look-back to the left.  The column look-back
            //    (thread pt also owns column pt) reads only the tiles above,
            //    so its windows ride along in the same round trips; it
            //    finishes in step 5, once this tile's column sums are known.
            //    The first windows are in flight while the column sums of
            //    the warp-local row prefixes are formed.
            Chain row = make_chain(rowMine - kTileH, -(long long)kTileH, tx);
            Chain colS = make_chain(ws.col + (long long)((int)tile - ntx) * kColWords + pt,
                                    -(long long)ntx * kColWords, ty);
            Chain colQ = make_chain(ws.col + (long long)((int)tile - ntx) * kColWords + kTileW + pt,
                                    -(long long)ntx * kColWords, ty);
            Backoff bo;
            bool ok = true;
            {
                uint64_t wr[kRowWindow], w0[kColWindowEarly], w1[kColWindowEarly];
                chain_load(row, wr);
                chain_load(colS, w0);
                chain_load(colQ, w1);
                // Column sums over the warp's 32 rows of the row prefixes
                // within the warp's part of the tile: the prefix at (row k,
                // lane L, column c) is (sum of row k's lanes < L) + (lane L's
                // pixels up to c), so its sum over the rows is one exclusive
                // lane scan of the lanes' 32-row totals plus the prefix sums
                // of the lane's per-column totals.  Per-column totals of two
                // byte lanes share a 32-bit word (at most 32 * 255 each).
                uint32_t b02 = 0, b13 = 0, q0 = 0, q1 = 0, q2 = 0, q3 = 0;
#pragma unroll 8
                for (int k = 0; k < kRowsPerWarp; ++k) {
                    const uint32_t v =
                        *reinterpret_cast<const uint32_t *>(&s_pix[ps][warp * kRowsPerWarp + k][4 * lane]);
                    b02 += __byte_perm(v, 0u, 0x4240);
                    b13 += __byte_perm(v, 0u, 0x4341);
                    const uint32_t x0 = v & 255u, x1 = (v >> 8) & 255u, x2 = (v >> 16) & 255u, x3 = v >> 24;
                    q0 += x0 * x0; q1 += x1 * x1; q2 += x2 * x2; q3 += x3 * x3;
                }
                uint32_t cI[4], cQ[4];
                cI[0] = b02 & 0xffffu;
                cI[1] = cI[0] + (b13 & 0xffffu);
                cI[2] = cI[1] + (b02 >> 16);
                cI[3] = cI[2] + (b13 >> 16);
                cQ[0] = q0; cQ[1] = q0 + q1; cQ[2] = cQ[1] + q2; cQ[3] = cQ[2] + q3;
                uint32_t eI = cI[3], eQ = cQ[3];  // inclusive lane scan, then exclusive
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t tI = __shfl_up_sync(0xffffffffu, eI, o);
                    const uint32_t tQ = __shfl_up_sync(0xffffffffu, eQ, o);
                    if (lane >= o) { eI += tI; eQ += tQ; }
                }
                eI -= cI[3];
                eQ -= cQ[3];
                // the lane-local prefix is summed over 32 rows; the lanes to
                // the left contribute their 32-row totals to every column
                uint4 *dst = reinterpret_cast<uint4 *>(&s_colPart[warp][4 * lane]);
                dst[0] = make_uint4(cI[0] + eI, cQ[0] + eQ, cI[1] + eI, cQ[1] + eQ);
                dst[1] = make_uint4(cI[2] + eI, cQ[2] + eQ, cI[3] + eI, cQ[3] + eQ);
                const bool moved = chain_take(row, wr, epoch);
                chain_take(colS, w0, epoch);
                chain_take(colQ, w1, epoch);
                if (!row.done && !moved) ok = bo.wait(cx);
            }
            while (ok && !row.done) {
                uint64_t wr[kRowWindow], w0[kColWindowEarly], w1[kColWindowEarly];
                chain_load(row, wr);
                chain_load(colS, w0);
                chain_load(colQ, w1);
                const bool moved = chain_take(row, wr, epoch);
                chain_take(colS, w0, epoch);
                chain_take(colQ, w1, epoch);
                if (!row.done && !moved) ok = bo.wait(cx);
            }
            if (!ok) s_fail = 1;
            else if (tx > 0 && publish) st_relaxed_u64(rowMine, make_word(epoch, FLAG_PREFIX, row.acc + rowV));
            {
                const uint64_t carry = ok ? row.acc : 0ull;
                const uint32_t rcI = (uint32_t)(carry & ((1u << kRowQShift) - 1u));
                const uint32_t rcQ = (uint32_t)(carry >> kRowQShift);
                S_.rowCarry[pt] = make_uint2(rcI, rcQ);
                // 4. per-warp sums of the row carries
                long long a = rcI, b = rcQ;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    a += __shfl_xor_sync(0xffffffffu, a, o);
                    b += __shfl_xor_sync(0xffffffffu, b, o);
                }
                if (lane == 0) { s_warpCarry[warp][0] = a; s_warpCarry[warp][1] = b; }
            }
            named_bar_sync(kBarProd, kProducers);
            if (s_fail) {
                if (pt == 0) S_.tile = kStageAbort;
                named_bar_arrive(kBarFull0 + sb, kThreads);
                break;
            }
            // 5. column carries: thread = column, both tables together.  The
            //    column sums include the row carries, so they are published
            //    only now: as an inclusive prefix when the look-back above
            //    already ended, else as an aggregate until it does.
            {
                const int c = pt;
                long long agg[2] = {0, 0};
#pragma unroll
                for (int w = 0; w < kGroups; ++w) {
                    const uint2 cp = s_colPart[w][c];
                    agg[0] += (long long)cp.x + s_warpCarry[w][0];
                    agg[1] += (long long)cp.y + s_warpCarry[w][1];
                }
                uint64_t *mine = ws.col + (size_t)tile * kColWords + c;
                const bool early = colS.done && colQ.done;  // ty == 0 included
                if (publish && NCC_BOUNDS(tile < ntiles && c + kTileW < kColWords, status)) {
                    const uint32_t state = early ? FLAG_PREFIX : FLAG_AGGREGATE;
                    const uint64_t b0 = early ? colS.acc : 0ull, b1 = early ? colQ.acc : 0ull;
                    st_relaxed_u64(mine, make_word(epoch, state, b0 + (uint64_t)agg[0]));
                    st_relaxed_u64(mine + kTileW, make_word(epoch, state, b1 + (uint64_t)agg[1]));
                }
                bool ok = true;
                while (!colS.done || !colQ.done) {
                    uint64_t w0[kColWindow], w1[kColWindow];
                    chain_load(colS, w0);
                    chain_load(colQ, w1);
                    const bool moved = chain_take(colS, w0, epoch) | chain_take(colQ, w1, epoch);
                    if ((!colS.done || !colQ.done) && !moved && !bo.wait(cx)) { ok = false; break; }
                }
                if (!ok) {
                    s_fail = 1;
                } else if (!early && publish) {
                    st_relaxed_u64(mine, make_word(epoch, FLAG_PREFIX, colS.acc + (uint64_t)agg[0]));
                    st_relaxed_u64(mine + kTileW, make_word(epoch, FLAG_PREFIX, colQ.acc + (uint64_t)agg[1]));
                }
                long long run0 = (long long)colS.acc, run1 = (long long)colQ.acc;
#pragma unroll
                for (int g = 0; g < kGroups; ++g) {
                    S_.colStart[g][0][c] = run0;
                    S_.colStart[g][1][c] = run1;
                    const uint2 cp = s_colPart[g][c];
                    run0 += (long long)cp.x + s_warpCarry[g][0];
                    run1 += (long long)cp.y + s_warpCarry[g][1];
                }
            }
            named_bar_sync(kBarProd, kProducers);
            const bool failed = s_fail != 0;
            if (pt == 0) {
                S_.tile = failed ? kStageAbort : (int)tile;
                S_.pix = ps;
            }
            named_bar_arrive(kBarFull0 + sb, kThreads);  // hand the stage to the writers
            if (failed) break;
        }
        // a pixel load issued for a tile this CTA will not process must land
        // before the CTA exits
        if (kTma && pt == 0) {
            const unsigned t = s_next;
            if (t < (unsigned)ntiles && t != s_tile) {
                const int slot = (i + 1) % kPixSlots;
                uint32_t done = 0;
                for (unsigned it = 0; !done && it < (1u << 22); ++it)
                    asm volatile(
                        "{ .reg .pred P; mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2; selp.u32 %0, 1, 0, P; }"
                        : "=r"(done) : "r"(smem_addr(&s_pbar[slot])), "r"((uint32_t)(((i + 1) / kPixSlots) & 1)) : "memory");
            }
        }
        (void)pending;
        // balance the writers' last release of a stage (see the writer loop)
        if (i >= 1) named_bar_sync(kBarEmpty0 + ((i + 1) & 1), kThreads);
    } else {
        // ================= writer warps: rows of S and Q =================
        const int g = warp - kGroups;
        for (int i = 0;; ++i) {
            const int sb = i & 1;
            const Stage &S_ = st[sb];
            named_bar_sync(kBarFull0 + sb, kThreads);
            const int tile = S_.tile;
            if (tile < 0) break;  // done or aborted: no release, the producer stopped too
            const int tx = tile % ntx, ty = tile / ntx;
            int xl = tx * kTileW + 4 * lane;
#ifdef NCC_DEBUG
            // debug builds only: fault_tile == -2 sends tile 0's stores one
            // row width to the left (before the start of S and Q), for the
            // test that the check below catches it: the stores are skipped
            // and NCC_ERR_BOUNDS is recorded
            if (fault_tile == -2 && tile == 0) xl -= W;
#endif
            const int ps = S_.pix;
            long long runI[4], runQ[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                runI[c] = S_.colStart[g][0][4 * lane + c];
                runQ[c] = S_.colStart[g][1][4 * lane + c];
            }
            // four rows at a time: their lane scans are independent, so
            // their shuffle chains overlap.  Rows past the image bottom are
            // zeros in the stage and only their stores are skipped.
#pragma unroll 1
            for (int k0 = 0; k0 < kRowsPerWarp; k0 += kScanRows) {
                const int r0 = g * kRowsPerWarp + k0, y0 = ty * kTileH + r0;
                uint32_t px[kScanRows];
                uint2 rc[kScanRows];
#pragma unroll
                for (int j = 0; j < kScanRows; ++j) {
                    px[j] = *reinterpret_cast<const uint32_t *>(&s_pix[ps][r0 + j][4 * lane]);
                    rc[j] = S_.rowCarry[r0 + j];
                }
                uint32_t pI[kScanRows][4], pQ[kScanRows][4];
                row_scan_rows(px, lane, pI, pQ);
#pragma unroll
                for (int j = 0; j < kScanRows; ++j) {
                    const int y = y0 + j;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        runI[c] += (uint32_t)(rc[j].x + pI[j][c]);
                        runQ[c] += (uint32_t)(rc[j].y + pQ[j][c]);
                    }
                    if (y >= H) continue;
                    const size_t o = (size_t)y * W + xl;
                    if (!NCC_BOUNDS(tile < ntiles && xl >= 0, status)) continue;
                    if (kStore == 2 && xl + 3 < W) {
                        st_v4_b64(S + o, runI[0], runI[1], runI[2], runI[3]);
                        st_v4_b64(Q + o, runQ[0], runQ[1], runQ[2], runQ[3]);
                    } else if (kStore == 1 && xl + 3 < W) {
                        __stcs(reinterpret_cast<longlong2 *>(S + o), make_longlong2(runI[0], runI[1]));
                        __stcs(reinterpret_cast<longlong2 *>(S + o + 2), make_longlong2(runI[2], runI[3]));
                        __stcs(reinterpret_cast<longlong2 *>(Q + o), make_longlong2(runQ[0], runQ[1]));
                        __stcs(reinterpret_cast<longlong2 *>(Q + o + 2), make_longlong2(runQ[2], runQ[3]));
                    } else {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            if (xl + c < W) {
                                S[o + c] = runI[c];
                                Q[o + c] = runQ[c];
                            }
                        }
                    }
                }
            }
            named_bar_arrive(kBarEmpty0 + sb, kThreads);  // the stage may be refilled
        }
    }
    // The last CTA out returns the dispenser and the SM counters to zero for
    // the next launch on this workspace (every CTA has drawn its last ticket
    // before it counts itself done).
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        s_last = atomicAdd(ws.done, 1u) == gridDim.x - 1 ? 1 : 0;
    }
    __syncthreads();
    if (s_last) {
        __threadfence();
        for (int k = tid; k < kMaxSmIds; k += kThreads) ws.smTiles[k] = 0u;
        if (tid == 0) {
            *ws.ticket = 0ull;
            *ws.done = 0u;
        }
    }
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Workspace: ticket (8 bytes), abort word, done count; the SM counters from
// byte 256; the row words, then the column words.
constexpr size_t kHeaderBytes = 256 + kMaxSmIds * sizeof(unsigned);
static_assert(kHeaderBytes % 256 == 0, "row words stay 256-byte aligned");

// Library-owned look-back workspace, one per device.  Calls on different
// streams are ordered through `last` so they never use it concurrently; it
// is allocated, grown and cleared in stream order, without a host
// synchronization.
struct DeviceWs {
    void *ptr = nullptr;
    size_t bytes = 0;
    uint32_t epoch = 0;
    bool dirty = false;
    bool used = false;
    cudaEvent_t last = nullptr;
    cudaStream_t last_stream = nullptr;
};
constexpr int kMaxDevices = 64;
DeviceWs g_ws[kMaxDevices];
std::mutex g_ws_mutex;

}  // namespace

SatPlan sat_plan(int W, int H) {
    SatPlan p;
    p.tile_w = kTileW;
    p.tile_h = kTileH;
    p.ntx = (W + kTileW - 1) / kTileW;
    p.nty = (H + kTileH - 1) / kTileH;
    const size_t nt = (size_t)p.ntx * p.nty;
    p.zero_bytes = kHeaderBytes;  // dispenser, abort word, done count, SM counters
    p.total_bytes = kHeaderBytes + align_up(nt * kTileH * 8, 256) + align_up(nt * kColWords * 8, 256);
    return p;
}

int sm_count() {
    static int sms[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
    if (!sms[dev] && cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 1;
    return sms[dev] > 0 ? sms[dev] : 1;
}

// Persistent grid: the same number of CTAs on every SM (kCtasPerSm, or one
// CTA per tile for small images); the kernel's share rule then spreads the
// tiles evenly over the SMs.
int persistent_grid(int ntiles, int nsm) {
    const int resident = nsm * kCtasPerSm;
    return ntiles < resident ? ntiles : resident;
}

cudaError_t sat_launch(const uint8_t *img, int W, int H, int64_t *S, int64_t *Q,
                       void *workspace, const SatPlan &plan, uint32_t epoch, int *status,
                       uint64_t timeout_ns, int fault_tile, cudaStream_t stream) {
    const size_t nt = (size_t)plan.ntx * plan.nty;
    char *base = static_cast<char *>(workspace);
    SatWs ws;
    ws.ticket = reinterpret_cast<unsigned long long *>(base);
    ws.abort = reinterpret_cast<unsigned *>(base + 8);
    ws.done = reinterpret_cast<unsigned *>(base + 12);
    ws.smTiles = reinterpret_cast<unsigned *>(base + 256);
    ws.row = reinterpret_cast<uint64_t *>(base + kHeaderBytes);
    ws.col = reinterpret_cast<uint64_t *>(base + kHeaderBytes + align_up(nt * kTileH * 8, 256));

    const bool aligned4 = (W % 4 == 0) && ((uintptr_t)img % 4 == 0);
    const int store = ((W % 4 == 0) && ((uintptr_t)S % 32 == 0) && ((uintptr_t)Q % 32 == 0)) ? 2
                      : ((W % 2 == 0) && ((uintptr_t)S % 16 == 0) && ((uintptr_t)Q % 16 == 0)) ? 1
                                                                                               : 0;
    CUtensorMap tmap;
    memset(&tmap, 0, sizeof(tmap));
    bool tma = (W % 16 == 0) && ((uintptr_t)img % 16 == 0);
    EncodeTiledFn enc = tma ? tensor_map_encoder() : nullptr;
    if (enc) {
        const cuuint64_t dims[2] = {(cuuint64_t)W, (cuuint64_t)H};
        const cuuint64_t strides[1] = {(cuuint64_t)W};
        const cuuint32_t box[2] = {(cuuint32_t)kTileW, (cuuint32_t)kTileH};
        const cuuint32_t estr[2] = {1, 1};
        tma = enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(img), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    } else {
        tma = false;
    }
    const int nsm = sm_count();
    const int grid = persistent_grid((int)nt, nsm);
    const int smCap = (int)((nt + nsm - 1) / nsm);  // tiles per SM, rounded up
    long long *s = reinterpret_cast<long long *>(S), *q = reinterpret_cast<long long *>(Q);
    const int dyn = kPixSlots * kTileH * kTileW + 128;
#define NCC_SAT(T, A, V)                                                                        \
    do {                                                                                        \
        cudaError_t ea = cudaFuncSetAttribute(sat_build_kernel<T, A, V>,                         \
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, dyn); \
        if (ea != cudaSuccess) return ea;                                                       \
        sat_build_kernel<T, A, V><<<grid, kThreads, dyn, stream>>>(tmap, img, W, H, s, q, ws,   \
                                                                   plan.ntx, (int)nt, epoch,    \
                                                                   nsm, smCap, kShareQ, status, \
                                                                   timeout_ns, fault_tile);     \
    } while (0)
    if (tma && store == 2) NCC_SAT(true, true, 2);
    else if (tma && store == 1) NCC_SAT(true, true, 1);
    else if (tma) NCC_SAT(true, true, 0);
    else if (aligned4 && store == 1) NCC_SAT(false, true, 1);
    else if (aligned4) NCC_SAT(false, true, 0);
    else if (store == 1) NCC_SAT(false, false, 1);
    else NCC_SAT(false, false, 0);
#undef NCC_SAT
    return cudaGetLastError();
}

cudaError_t sat_build_run(const uint8_t *img, int W, int H, int64_t *S, int64_t *Q,
                          int *status, uint64_t timeout_ns, int fault_tile,
                          cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    const SatPlan plan = sat_plan(W, H);
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    DeviceWs &d = g_ws[dev];
    if (!d.last) {
        e = cudaEventCreateWithFlags(&d.last, cudaEventDisableTiming);
        if (e != cudaSuccess) return e;
    }
    if (d.bytes < plan.total_bytes) {
        if (d.ptr) {
            // the old workspace goes back to the pool after its last use:
            // order this stream after that use, then free in stream order
            if (d.used && d.last_stream != stream) {
                e = cudaStreamWaitEvent(stream, d.last, 0);
                if (e != cudaSuccess) return e;
            }
            e = cudaFreeAsync(d.ptr, stream);
            if (e != cudaSuccess) return e;
            d.ptr = nullptr;
            d.bytes = 0;
            d.used = false;
        }
        const size_t bytes = align_up(plan.total_bytes, 1 << 20);
        e = pool_alloc(&d.ptr, bytes, stream);
        if (e != cudaSuccess) {
            d.ptr = nullptr;
            return e;
        }
        e = cudaMemsetAsync(d.ptr, 0, bytes, stream);
        if (e != cudaSuccess) return e;
        d.bytes = bytes;
        d.epoch = 0;
        d.dirty = false;
    }
    if (d.used && d.last_stream != stream) {
        e = cudaStreamWaitEvent(stream, d.last, 0);
        if (e != cudaSuccess) return e;
    }
    if (d.epoch >= kMaxEpoch || d.dirty) {
        // epochs wrap: clear every word so no stale word can match
        e = cudaMemsetAsync(d.ptr, 0, d.bytes, stream);
        if (e != cudaSuccess) return e;
        d.epoch = 0;
        d.dirty = false;
    }
    d.epoch += 1;
    e = sat_launch(img, W, H, S, Q, d.ptr, plan, d.epoch, status, timeout_ns, fault_tile, stream);
    if (e != cudaSuccess) {
        d.dirty = true;  // whether the kernel ran is unknown: clear before the next use
        return e;
    }
    e = cudaEventRecord(d.last, stream);
    d.last_stream = stream;
    d.used = true;
    return e;
}

}  // namespace ncc
