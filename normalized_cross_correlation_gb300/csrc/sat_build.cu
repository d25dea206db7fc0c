// sat_build.cu -- single-pass builder of the two summed-area tables
// S = SAT(I) and Q = SAT(I^2), inclusive, int64 (The CUDA Handbook,
// section 15.8, "The Denominator: Summed Area Tables").
//
// Design (GB300): the image is cut into tiles of kTileW = 128 columns by
// kTileH = 64 rows, one CTA of 256 threads per tile.  A CTA
//   1. loads its pixels with coalesced 4-byte loads (one warp spans the tile
//      width, four columns per lane, eight rows per warp),
//   2. scans each row segment in uint32 with warp shuffles (a row's running
//      sum of squares is at most W*255^2 < 2^32 for W <= 66051),
//   3. gets each row's carry from the tiles to its left, then each column's
//      carry from the tiles above, by decoupled look-backs that follow the
//      section's three-state protocol (empty / aggregate published /
//      inclusive prefix published), and
//   4. writes S and Q as int64 with 16-byte streaming stores.
//
// Look-back words.  Every published value is one 64-bit word holding
// {epoch:5, state:2, value:57}, written and read with single-copy-atomic
// relaxed GPU-scope accesses: the state travels with its value, so a
// publication needs no separate flag, fence or CTA barrier.  Row words pack
// the row's sum of I (25 bits) and of I^2 (32 bits) -- both fit for
// W <= 66051 and their sums never carry across fields.  Column words carry
// S (< 2^39) or Q (< 2^47) of one column, one word each, so the two tables'
// column look-backs run independently.  A waiting thread reads up to kWindow
// predecessors with independent loads per round.  The epoch tag lets the
// workspace be reused without clearing it: a word from an earlier call
// reads as empty.
//
// Tiles are handed out by an atomic ticket in row-major order, so every
// wait points at a tile whose CTA is already running and the look-backs
// cannot deadlock.  Every wait is bounded (timeout and iteration cap); a wait
// that runs out records NCC_ERR_TIMEOUT, raises the call's abort word and
// the CTA leaves without writing.
#include "ncc_common.cuh"

#include <mutex>

namespace ncc {
namespace {

constexpr int kTileW = 128;           // tile width: 32 lanes x 4 columns
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerWarp = 8;
constexpr int kTileH = kWarps * kRowsPerWarp;  // 64
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

template <bool kAligned4, bool kVecStore>
__global__ void __launch_bounds__(kThreads, 4)
sat_build_kernel(const uint8_t *__restrict__ img, int W, int H, long long *__restrict__ S,
                 long long *__restrict__ Q, SatWs ws, int ntx, uint32_t epoch,
                 unsigned long long ticket_base, int *status, uint64_t timeout_ns,
                 int fault_tile) {
    __shared__ unsigned s_tile;
    __shared__ uint2 s_rowTot[kTileH];                          // tile row sums
    __shared__ uint2 s_rowCarry[kTileH];                        // row sums left of the tile
    __shared__ __align__(16) uint2 s_colPart[kWarps][kTileW];   // per-warp column sums of warp-local prefixes
    __shared__ long long s_warpCarry[kWarps][2];                // per-warp sums of s_rowCarry
    __shared__ long long s_colCarry[2][kTileW];                 // S and Q column sums above the tile

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const WaitCtx cx{ws.abort, status, epoch, global_timer_ns(), timeout_ns};
    if (tid == 0) s_tile = (unsigned)(atomicAdd(ws.ticket, 1ull) - ticket_base);
    __syncthreads();
    const unsigned tile = s_tile;
    const int tx = (int)(tile % (unsigned)ntx), ty = (int)(tile / (unsigned)ntx);
    const int xl = tx * kTileW + 4 * lane;           // this lane's first column
    const int row0 = ty * kTileH + warp * kRowsPerWarp;
    const bool publish = (int)tile != fault_tile;

    // 1. pixels: four columns per lane, kRowsPerWarp rows per warp.
    uint32_t px[kRowsPerWarp];
#pragma unroll
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
        px[k] = v;
    }

    // 2. warp-local row scans; the column sums of the warp-local prefixes
    //    feed the tile's column aggregate.  (The output pass repeats the
    //    scans instead of keeping them in registers.)
    uint32_t cI[4] = {0, 0, 0, 0}, cQ[4] = {0, 0, 0, 0};
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
        uint32_t pI[4], pQ[4];
        row_scan(px[k], lane, pI, pQ);
#pragma unroll
        for (int c = 0; c < 4; ++c) { cI[c] += pI[c]; cQ[c] += pQ[c]; }
        if (lane == 31) s_rowTot[warp * kRowsPerWarp + k] = make_uint2(pI[3], pQ[3]);
    }
    {
        uint4 *dst = reinterpret_cast<uint4 *>(&s_colPart[warp][4 * lane]);
        dst[0] = make_uint4(cI[0], cQ[0], cI[1], cQ[1]);
        dst[1] = make_uint4(cI[2], cQ[2], cI[3], cQ[3]);
    }
    __syncthreads();

    // 3. row carries: publish this tile's row sums, look back to the left.
    bool ok = true;
    if (tid < kTileH) {
        const uint2 tot = s_rowTot[tid];
        const uint64_t v = (uint64_t)tot.x | ((uint64_t)tot.y << kRowQShift);
        uint64_t *mine = ws.row + (size_t)tile * kTileH + tid;
        if (publish)
            st_relaxed_u64(mine, make_word(epoch, tx == 0 ? FLAG_PREFIX : FLAG_AGGREGATE, v));
        uint64_t carry = 0;
        if (tx > 0) {
            ok = look_back(ws.row + tid, kTileH, (int)tile - 1, 1, tx, carry, cx);
            if (ok && publish) st_relaxed_u64(mine, make_word(epoch, FLAG_PREFIX, carry + v));
        }
        s_rowCarry[tid] = make_uint2((uint32_t)(carry & ((1u << kRowQShift) - 1u)),
                                     (uint32_t)(carry >> kRowQShift));
    }
    if (__syncthreads_or(!ok)) return;

    // 4. column carries.  The tile's column aggregate is the sum over its
    //    rows of the full row prefixes = per-warp column partials + the sum
    //    of the row carries.  Thread t handles column t % 128 of table t / 128.
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
    __syncthreads();
    {
        const int c = tid & (kTileW - 1), part = tid >> 7;
        long long agg = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const uint2 cp = s_colPart[w][c];
            agg += (long long)(part ? cp.y : cp.x) + s_warpCarry[w][part];
        }
        uint64_t *mine = ws.col + (size_t)tile * kColWords + tid;
        if (publish)
            st_relaxed_u64(mine, make_word(epoch, ty == 0 ? FLAG_PREFIX : FLAG_AGGREGATE,
                                           (uint64_t)agg));
        uint64_t carry = 0;
        if (ty > 0) {
            ok = look_back(ws.col + tid, kColWords, (int)tile - ntx, ntx, ty, carry, cx);
            if (ok && publish)
                st_relaxed_u64(mine, make_word(epoch, FLAG_PREFIX, carry + (uint64_t)agg));
        }
        s_colCarry[part][c] = (long long)carry;
    }
    if (__syncthreads_or(!ok)) return;

    // 5. outputs: running column sums from the carry above, down this warp's rows.
    long long runI[4], runQ[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        runI[c] = s_colCarry[0][4 * lane + c];
        runQ[c] = s_colCarry[1][4 * lane + c];
    }
    for (int w = 0; w < warp; ++w) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint2 p = s_colPart[w][4 * lane + c];
            runI[c] += (long long)p.x + s_warpCarry[w][0];
            runQ[c] += (long long)p.y + s_warpCarry[w][1];
        }
    }
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
        const int y = row0 + k;
        if (y >= H) break;
        const uint2 rc = s_rowCarry[warp * kRowsPerWarp + k];
        uint32_t pI[4], pQ[4];
        row_scan(px[k], lane, pI, pQ);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            runI[c] += (uint32_t)(rc.x + pI[c]);
            runQ[c] += (uint32_t)(rc.y + pQ[c]);
        }
        const size_t o = (size_t)y * W + xl;
        if (kVecStore && xl + 3 < W) {
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

cudaError_t sat_launch(const uint8_t *img, int W, int H, int64_t *S, int64_t *Q,
                       void *workspace, const SatPlan &plan, uint32_t epoch,
                       unsigned long long ticket_base, int *status, uint64_t timeout_ns,
                       int fault_tile, cudaStream_t stream) {
    const size_t nt = (size_t)plan.ntx * plan.nty;
    char *base = static_cast<char *>(workspace);
    SatWs ws;
    ws.ticket = reinterpret_cast<unsigned long long *>(base);
    ws.abort = reinterpret_cast<unsigned *>(base + 8);
    ws.row = reinterpret_cast<uint64_t *>(base + 256);
    ws.col = reinterpret_cast<uint64_t *>(base + 256 + align_up(nt * kTileH * 8, 256));

    const bool aligned4 = (W % 4 == 0) && ((uintptr_t)img % 4 == 0);
    const bool vec = (W % 2 == 0) && ((uintptr_t)S % 16 == 0) && ((uintptr_t)Q % 16 == 0);
    const dim3 grid((unsigned)nt), block(kThreads);
    long long *s = reinterpret_cast<long long *>(S), *q = reinterpret_cast<long long *>(Q);
#define NCC_SAT(A, V)                                                                  \
    sat_build_kernel<A, V><<<grid, block, 0, stream>>>(img, W, H, s, q, ws, plan.ntx,  \
                                                       epoch, ticket_base, status,     \
                                                       timeout_ns, fault_tile)
    if (aligned4 && vec) NCC_SAT(true, true);
    else if (aligned4) NCC_SAT(true, false);
    else if (vec) NCC_SAT(false, true);
    else NCC_SAT(false, false);
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
    e = sat_launch(img, W, H, S, Q, d.ptr, plan, d.epoch, d.ticket_base, status, timeout_ns,
                   fault_tile, stream);
    if (e != cudaSuccess) {
        d.dirty = true;  // the ticket count is unknown: clear before the next use
        return e;
    }
    d.ticket_base += (unsigned long long)plan.ntx * plan.nty;
    e = cudaEventRecord(d.last, stream);
    d.last_stream = stream;
    d.used = true;
    return e;
}

}  // namespace ncc
