// sat_build.cu -- single-pass builder of the two summed-area tables
// S = SAT(I) and Q = SAT(I^2), inclusive, int64 (The CUDA Handbook,
// section 15.8, "The Denominator: Summed Area Tables").
//
// Design (GB300).  The image is cut into tiles of 128 columns by 128 rows,
// handed out by an atomic ticket in row-major order to a persistent grid
// (three CTAs per SM).  Each CTA runs two warp groups over a double-buffered
// shared-memory stage:
//   - producer warps 0-3 take a ticket, load the tile's pixels with
//     one TMA box per tile, issued a tile ahead into a three-slot pixel
//     ring (plain loads when rows are not 16-byte multiples), scan each
//     row segment (four columns per lane, 32 rows per warp) in uint32 with
//     warp shuffles (a row's running
//     sum of squares is at most W*255^2 < 2^32 for W <= 66051), then get
//     each row's carry from the tiles to its left and each column's carry
//     from the tiles above by decoupled look-backs -- the section's
//     three-state protocol (empty / aggregate published / inclusive prefix
//     published) -- and leave pixels, row carries and each writer group's
//     starting column sums in the stage;
//   - writer warps 4-7 rebuild the rows from the stage and stream S and Q
//     out as int64 with 16-byte streaming stores.
// The look-back latency of one tile thus overlaps the writes of the
// previous one inside every CTA.
//
// Look-back words.  Every published value is one 64-bit word holding
// {epoch:5, state:2, value:57}, written and read with single-copy-atomic
// relaxed GPU-scope accesses: the state travels with its value, so a
// publication needs no separate flag or fence.  Row words pack the row's
// sum of I (25 bits) and of I^2 (32 bits) -- both fit for W <= 66051 and
// their sums never carry across fields.  Column words carry S (< 2^39) or
// Q (< 2^47) of one column, one word each.  A waiting thread reads up to
// kWindow predecessors with independent loads per round.  The epoch tag
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
constexpr int kStageDone = -1, kStageAbort = -2;
constexpr int kColWords = 2 * kTileW;          // S and Q word per column
constexpr int kWindow = 8;            // predecessors read per look-back round

constexpr int kEpochShift = 59, kStateShift = 57;
constexpr uint64_t kValueMask = (1ull << kStateShift) - 1;
constexpr int kRowQShift = 25;        // row word: I in bits 0..24, I^2 in 25..56
constexpr uint32_t kMaxEpoch = 31;

struct SatWs {
    unsigned long long *ticket;  // tile dispenser: ticket - ticket_base = tile index
    unsigned *abort;             // holds the epoch of a call whose wait ran out
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

// Inclusive scan of one 128-pixel row segment held as four bytes per lane:
// p[c] / s[c] = sum of pixels / of squared pixels from the warp's first
// column up to this lane's column c (uint32).  Lane 31's p[3], s[3] are the
// segment's totals.
__device__ __forceinline__ void row_scan(uint32_t px, int lane, uint32_t (&p)[4],
                                         uint32_t (&s)[4]) {
    const uint32_t b0 = px & 255u, b1 = (px >> 8) & 255u, b2 = (px >> 16) & 255u, b3 = px >> 24;
    p[0] = b0; p[1] = p[0] + b1; p[2] = p[1] + b2; p[3] = p[2] + b3;
    s[0] = b0 * b0; s[1] = s[0] + b1 * b1; s[2] = s[1] + b2 * b2; s[3] = s[2] + b3 * b3;
    uint32_t sI = p[3], sQ = s[3];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t tI = __shfl_up_sync(0xffffffffu, sI, o);
        const uint32_t tQ = __shfl_up_sync(0xffffffffu, sQ, o);
        if (lane >= o) { sI += tI; sQ += tQ; }
    }
    const uint32_t eI = sI - p[3], eQ = sQ - s[3];
#pragma unroll
    for (int c = 0; c < 4; ++c) { p[c] += eI; s[c] += eQ; }
}

struct WaitCtx {
    unsigned *abort;
    int *status;
    uint32_t epoch;
    uint64_t t0, timeout_ns;
};

// Decoupled look-back of one element over `count` predecessors whose words
// sit at words[(first - i*step) * tstride], i = 0..count-1 (nearest first).
// Adds the values of consecutive published predecessors up to and including
// the nearest inclusive prefix into `acc`.  Returns false when a wait ran
// out or another CTA of the call aborted.
__device__ __forceinline__ bool look_back(const uint64_t *words, size_t tstride, int first,
                                          int step, int count, uint64_t &acc,
                                          const WaitCtx &cx) {
    int i0 = 0;
    unsigned backoff = 32, polls = 0;
    while (i0 < count) {
        uint64_t w[kWindow];
#pragma unroll
        for (int i = 0; i < kWindow; ++i)
            w[i] = (i0 + i < count)
                       ? ld_relaxed_u64(words + (size_t)(first - (i0 + i) * step) * tstride)
                       : 0ull;
        int used = 0;
        bool done = false;
#pragma unroll
        for (int i = 0; i < kWindow; ++i) {
            if (used == i && !done && i0 + i < count) {
                const uint32_t st = word_state(w[i], cx.epoch);
                if (st != FLAG_EMPTY) {
                    acc += w[i] & kValueMask;
                    used = i + 1;
                    done = (st == FLAG_PREFIX);
                }
            }
        }
        if (done) return true;
        if (used == 0) {
            // the nearest unconsumed predecessor has not published yet
            __nanosleep(backoff);
            if (backoff < 256) backoff <<= 1;
            if ((++polls & 7u) == 0u) {
                if (ld_relaxed_gpu(cx.abort) == cx.epoch) return false;
                if (global_timer_ns() - cx.t0 > cx.timeout_ns || polls > (1u << 26)) {
                    atomicExch(cx.abort, cx.epoch);
                    record_status(cx.status, NCC_ERR_TIMEOUT);
                    return false;
                }
            }
            continue;
        }
        i0 += used;
    }
    return true;
}

// The same look-back for two independent chains at once (the S and Q words
// of one column): both windows are loaded before either is examined, so the
// two chains share each round trip.
__device__ __forceinline__ bool look_back2(const uint64_t *w0s, const uint64_t *w1s, size_t tstride,
                                           int first, int step, int count, uint64_t &acc0,
                                           uint64_t &acc1, const WaitCtx &cx) {
    int i0[2] = {0, 0};
    bool done[2] = {count == 0, count == 0};
    uint64_t acc[2] = {0, 0};
    unsigned backoff = 32, polls = 0;
    while (!done[0] || !done[1]) {
        uint64_t w[2][kWindow];
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int i = 0; i < kWindow; ++i)
                w[q][i] = (!done[q] && i0[q] + i < count)
                              ? ld_relaxed_u64((q ? w1s : w0s) + (size_t)(first - (i0[q] + i) * step) * tstride)
                              : 0ull;
        bool stalled = true;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            if (done[q]) continue;
            int used = 0;
#pragma unroll
            for (int i = 0; i < kWindow; ++i) {
                if (used == i && !done[q] && i0[q] + i < count) {
                    const uint32_t st = word_state(w[q][i], cx.epoch);
                    if (st != FLAG_EMPTY) {
                        acc[q] += w[q][i] & kValueMask;
                        used = i + 1;
                        done[q] = (st == FLAG_PREFIX);
                    }
                }
            }
            i0[q] += used;
            if (i0[q] >= count) done[q] = true;
            if (used) stalled = false;
        }
        if (stalled && (!done[0] || !done[1])) {
            __nanosleep(backoff);
            if (backoff < 256) backoff <<= 1;
            if ((++polls & 7u) == 0u) {
                if (ld_relaxed_gpu(cx.abort) == cx.epoch) return false;
                if (global_timer_ns() - cx.t0 > cx.timeout_ns || polls > (1u << 26)) {
                    atomicExch(cx.abort, cx.epoch);
                    record_status(cx.status, NCC_ERR_TIMEOUT);
                    return false;
                }
            }
        }
    }
    acc0 += acc[0];
    acc1 += acc[1];
    return true;
}

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

// After a failed wait the CTA stops, but it still draws tickets until one
// lies past the last tile, so that every launch advances the ticket counter
// by exactly ntiles + gridDim.x (the host's next ticket base relies on it).

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
                 int ntx, int ntiles, uint32_t epoch, unsigned long long ticket_base,
                 int *status, uint64_t timeout_ns, int fault_tile) {
    extern __shared__ __align__(128) uint8_t s_dyn[];
    uint8_t (*s_pix)[kTileH][kTileW] = reinterpret_cast<uint8_t (*)[kTileH][kTileW]>(
        (reinterpret_cast<uintptr_t>(s_dyn) + 127) & ~uintptr_t(127));
    __shared__ __align__(16) Stage st[2];
    __shared__ uint2 s_rowTot[kTileH];                          // tile row sums
    __shared__ uint2 s_rowCarry[kTileH];
    __shared__ __align__(16) uint2 s_colPart[kGroups][kTileW];  // per-warp column sums of warp-local prefixes
    __shared__ long long s_warpCarry[kGroups][2];               // per-warp sums of the row carries
    __shared__ __align__(8) unsigned long long s_pbar[kPixSlots];
    __shared__ unsigned s_tile, s_next;
    __shared__ int s_fail;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (warp < kGroups) {
        // ================= producer warps: tiles, scans, look-backs =================
        const int pt = tid;  // 0..127
        auto grab = [&]() -> unsigned {
            return (unsigned)(atomicAdd(ws.ticket, 1ull) - ticket_base);
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
            // 2. row totals and column sums of the warp-local row prefixes,
            //    without per-row scans: the prefix at (row k, lane L, column c)
            //    is (sum of row k's lanes < L) + (lane L's own pixels up to c),
            //    so its sum over the 32 rows is one exclusive lane scan of the
            //    lanes' 32-row totals plus the lane-local prefix sums.
            uint32_t cI[4] = {0, 0, 0, 0}, cQ[4] = {0, 0, 0, 0};
            uint32_t sumI = 0, sumQ = 0;  // this lane's total over the warp's rows
#pragma unroll 8
            for (int k = 0; k < kRowsPerWarp; ++k) {
                const uint32_t v =
                    *reinterpret_cast<const uint32_t *>(&s_pix[ps][warp * kRowsPerWarp + k][4 * lane]);
                const uint32_t b0 = v & 255u, b1 = (v >> 8) & 255u, b2 = (v >> 16) & 255u, b3 = v >> 24;
                const uint32_t i1 = b0 + b1, i2 = i1 + b2, i3 = i2 + b3;
                const uint32_t q0 = b0 * b0, q1 = q0 + b1 * b1, q2 = q1 + b2 * b2, q3 = q2 + b3 * b3;
                cI[0] += b0; cI[1] += i1; cI[2] += i2; cI[3] += i3;
                cQ[0] += q0; cQ[1] += q1; cQ[2] += q2; cQ[3] += q3;
                sumI += i3;
                sumQ += q3;
                const uint32_t totI = __reduce_add_sync(0xffffffffu, i3);
                const uint32_t totQ = __reduce_add_sync(0xffffffffu, q3);
                if (lane == 0) s_rowTot[warp * kRowsPerWarp + k] = make_uint2(totI, totQ);
            }
            {
                uint32_t eI = sumI, eQ = sumQ;  // inclusive lane scan, then exclusive
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t tI = __shfl_up_sync(0xffffffffu, eI, o);
                    const uint32_t tQ = __shfl_up_sync(0xffffffffu, eQ, o);
                    if (lane >= o) { eI += tI; eQ += tQ; }
                }
                eI -= sumI;
                eQ -= sumQ;
#pragma unroll
                for (int c = 0; c < 4; ++c) { cI[c] += eI; cQ[c] += eQ; }
            }
            {
                uint4 *dst = reinterpret_cast<uint4 *>(&s_colPart[warp][4 * lane]);
                dst[0] = make_uint4(cI[0], cQ[0], cI[1], cQ[1]);
                dst[1] = make_uint4(cI[2], cQ[2], cI[3], cQ[3]);
            }
            named_bar_sync(kBarProd, kProducers);

            // 3. row carries (one row per producer thread): publish this tile's
            //    row sums, look back to the left
            {
                const uint2 tot = s_rowTot[pt];
                const uint64_t v = (uint64_t)tot.x | ((uint64_t)tot.y << kRowQShift);
                uint64_t *mine = ws.row + (size_t)tile * kTileH + pt;
                if (publish)
                    st_relaxed_u64(mine, make_word(epoch, tx == 0 ? FLAG_PREFIX : FLAG_AGGREGATE, v));
                uint64_t carry = 0;
                if (tx > 0) {
                    if (look_back(ws.row + pt, kTileH, (int)tile - 1, 1, tx, carry, cx)) {
                        if (publish) st_relaxed_u64(mine, make_word(epoch, FLAG_PREFIX, carry + v));
                    } else {
                        s_fail = 1;
                    }
                }
                const uint2 rc = make_uint2((uint32_t)(carry & ((1u << kRowQShift) - 1u)),
                                            (uint32_t)(carry >> kRowQShift));
                s_rowCarry[pt] = rc;
                S_.rowCarry[pt] = rc;
            }
            named_bar_sync(kBarProd, kProducers);
            if (s_fail) {
                if (pt == 0) {
                    unsigned t = s_next;
                    while (t < (unsigned)ntiles) t = grab();  // keep the ticket count exact
                    S_.tile = kStageAbort;
                }
                named_bar_arrive(kBarFull0 + sb, kThreads);
                break;
            }
            // 4. per-warp sums of the row carries
            {
                long long a = 0, b = 0;
                if (lane < kRowsPerWarp) {
                    const uint2 c = s_rowCarry[warp * kRowsPerWarp + lane];
                    a = c.x;
                    b = c.y;
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    a += __shfl_xor_sync(0xffffffffu, a, o);
                    b += __shfl_xor_sync(0xffffffffu, b, o);
                }
                if (lane == 0) { s_warpCarry[warp][0] = a; s_warpCarry[warp][1] = b; }
            }
            named_bar_sync(kBarProd, kProducers);
            // 5. column carries: thread = column, both tables together
            {
                const int c = pt;
                long long part[kGroups][2];
                long long agg[2] = {0, 0};
#pragma unroll
                for (int w = 0; w < kGroups; ++w) {
                    const uint2 cp = s_colPart[w][c];
                    part[w][0] = (long long)cp.x + s_warpCarry[w][0];
                    part[w][1] = (long long)cp.y + s_warpCarry[w][1];
                    agg[0] += part[w][0];
                    agg[1] += part[w][1];
                }
                uint64_t *mine = ws.col + (size_t)tile * kColWords + c;
                if (publish) {
                    const uint32_t state = ty == 0 ? FLAG_PREFIX : FLAG_AGGREGATE;
                    st_relaxed_u64(mine, make_word(epoch, state, (uint64_t)agg[0]));
                    st_relaxed_u64(mine + kTileW, make_word(epoch, state, (uint64_t)agg[1]));
                }
                uint64_t carry0 = 0, carry1 = 0;
                if (ty > 0) {
                    if (look_back2(ws.col + c, ws.col + kTileW + c, kColWords, (int)tile - ntx, ntx,
                                   ty, carry0, carry1, cx)) {
                        if (publish) {
                            st_relaxed_u64(mine, make_word(epoch, FLAG_PREFIX, carry0 + (uint64_t)agg[0]));
                            st_relaxed_u64(mine + kTileW, make_word(epoch, FLAG_PREFIX, carry1 + (uint64_t)agg[1]));
                        }
                    } else {
                        s_fail = 1;
                    }
                }
                long long run0 = (long long)carry0, run1 = (long long)carry1;
#pragma unroll
                for (int g = 0; g < kGroups; ++g) {
                    S_.colStart[g][0][c] = run0;
                    S_.colStart[g][1][c] = run1;
                    run0 += part[g][0];
                    run1 += part[g][1];
                }
            }
            named_bar_sync(kBarProd, kProducers);
            const bool failed = s_fail != 0;
            if (pt == 0) {
                if (failed) {
                    unsigned t = s_next;
                    while (t < (unsigned)ntiles) t = grab();
                }
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
            const int xl = tx * kTileW + 4 * lane;
            const int ps = S_.pix;
            long long runI[4], runQ[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                runI[c] = S_.colStart[g][0][4 * lane + c];
                runQ[c] = S_.colStart[g][1][4 * lane + c];
            }
#pragma unroll 4
            for (int k = 0; k < kRowsPerWarp; ++k) {
                const int r = g * kRowsPerWarp + k, y = ty * kTileH + r;
                if (y >= H) break;
                const uint2 rc = S_.rowCarry[r];
                uint32_t pI[4], pQ[4];
                row_scan(*reinterpret_cast<const uint32_t *>(&s_pix[ps][r][4 * lane]), lane, pI, pQ);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    runI[c] += (uint32_t)(rc.x + pI[c]);
                    runQ[c] += (uint32_t)(rc.y + pQ[c]);
                }
                const size_t o = (size_t)y * W + xl;
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
            named_bar_arrive(kBarEmpty0 + sb, kThreads);  // the stage may be refilled
        }
    }
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Library-owned look-back workspace, one per device.  Calls on different
// streams are ordered through `last` so they never use it concurrently.
struct DeviceWs {
    void *ptr = nullptr;
    size_t bytes = 0;
    uint32_t epoch = 0;
    unsigned long long ticket_base = 0;
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
    p.zero_bytes = 256;                                       // ticket and abort word
    p.total_bytes = 256 + align_up(nt * kTileH * 8, 256) + align_up(nt * kColWords * 8, 256);
    return p;
}

// Persistent grid: as many rounds as the resident CTAs need, and the tiles
// spread evenly over them, so no CTA runs a last round alone.
int persistent_grid(int ntiles) {
    static int sms[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
    if (!sms[dev] && cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 1;
    const int resident = sms[dev] * kCtasPerSm;
    const int rounds = (ntiles + resident - 1) / resident;
    return (ntiles + rounds - 1) / rounds;
}

cudaError_t sat_launch(const uint8_t *img, int W, int H, int64_t *S, int64_t *Q,
                       void *workspace, const SatPlan &plan, uint32_t epoch,
                       unsigned long long ticket_base, int *status, uint64_t timeout_ns,
                       int fault_tile, cudaStream_t stream, unsigned long long *tickets_used) {
    const size_t nt = (size_t)plan.ntx * plan.nty;
    char *base = static_cast<char *>(workspace);
    SatWs ws;
    ws.ticket = reinterpret_cast<unsigned long long *>(base);
    ws.abort = reinterpret_cast<unsigned *>(base + 8);
    ws.row = reinterpret_cast<uint64_t *>(base + 256);
    ws.col = reinterpret_cast<uint64_t *>(base + 256 + align_up(nt * kTileH * 8, 256));

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
    const int grid = persistent_grid((int)nt);
    long long *s = reinterpret_cast<long long *>(S), *q = reinterpret_cast<long long *>(Q);
    const int dyn = kPixSlots * kTileH * kTileW + 128;
#define NCC_SAT(T, A, V)                                                                        \
    do {                                                                                        \
        cudaError_t ea = cudaFuncSetAttribute(sat_build_kernel<T, A, V>,                         \
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, dyn); \
        if (ea != cudaSuccess) return ea;                                                       \
        sat_build_kernel<T, A, V><<<grid, kThreads, dyn, stream>>>(tmap, img, W, H, s, q, ws,   \
                                                                   plan.ntx, (int)nt, epoch,    \
                                                                   ticket_base, status,         \
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
    // every CTA takes tickets until it draws one past the last tile
    if (tickets_used) *tickets_used = (unsigned long long)nt + (unsigned long long)grid;
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
            if (d.used) cudaEventSynchronize(d.last);
            cudaFree(d.ptr);
            d.ptr = nullptr;
            d.bytes = 0;
        }
        const size_t bytes = align_up(plan.total_bytes, 1 << 20);
        e = cudaMalloc(&d.ptr, bytes);
        if (e != cudaSuccess) return e;
        e = cudaMemset(d.ptr, 0, bytes);
        if (e != cudaSuccess) return e;
        d.bytes = bytes;
        d.epoch = 0;
        d.ticket_base = 0;
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
        d.ticket_base = 0;
        d.dirty = false;
    }
    d.epoch += 1;
    unsigned long long used = 0;
    e = sat_launch(img, W, H, S, Q, d.ptr, plan, d.epoch, d.ticket_base, status, timeout_ns,
                   fault_tile, stream, &used);
    if (e != cudaSuccess) {
        d.dirty = true;  // the ticket count is unknown: clear before the next use
        return e;
    }
    d.ticket_base += used;
    e = cudaEventRecord(d.last, stream);
    d.last_stream = stream;
    d.used = true;
    return e;
}

}  // namespace ncc
