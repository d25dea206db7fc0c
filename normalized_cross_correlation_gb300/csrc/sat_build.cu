// sat_build.cu -- single-pass builder of the two summed-area tables
// S = SAT(I) and Q = SAT(I^2), inclusive, int64 (The CUDA Handbook,
// section 15.8, "The Denominator: Summed Area Tables").
//
// Design (GB300): the image is cut into tiles of kTileW = 128 columns by
// TH rows.  A tile's CTA
//   1. loads its pixels with coalesced 4-byte loads (one warp spans the tile
//      width, four columns per lane),
//   2. scans each row in uint32 with warp shuffles (a row's running sum of
//      squares is at most W*255^2, which fits uint32 for W <= 66051),
//   3. gets each row's carry from the tiles to its left and each column's
//      carry from the tiles above with decoupled look-backs (the section's
//      three-state flag: 0 empty, 1 aggregate published, 2 inclusive prefix
//      published), and
//   4. writes S and Q as int64 with 16-byte streaming stores.
// Tiles are handed out by an atomic ticket in row-major order, so every wait
// points at a tile whose CTA is already running: the look-backs cannot
// deadlock.  Every wait is bounded (see wait_flag); a wait that runs out
// records NCC_ERR_TIMEOUT and the CTA leaves without publishing.
#include "ncc_common.cuh"

namespace ncc {
namespace {

constexpr int kTileW = 128;           // tile width: 32 lanes x 4 columns
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerWarp = 16;      // tile height TH = kWarps * kRowsPerWarp
constexpr int kTileH = kWarps * kRowsPerWarp;
constexpr int kWindow = 4;            // predecessors examined per look-back round

struct SatWs {
    unsigned *ticket;   // tile dispenser (row-major order)
    unsigned *abort;    // raised by the first CTA whose wait ran out
    unsigned *flagH;    // [ntiles] state of the row-carry results
    unsigned *flagV;    // [ntiles] state of the column-carry results
    uint2 *hAgg;        // [ntiles][kTileH] row sums over the tile (I, I^2)
    uint2 *hPref;       // [ntiles][kTileH] row sums from column 0 to the tile's right edge
    longlong2 *vAgg;    // [ntiles][kTileW] column sums of full row prefixes over the tile
    longlong2 *vPref;   // [ntiles][kTileW] the same from row 0 to the tile's bottom edge
};

__device__ __forceinline__ void add_to(uint2 &a, const uint2 &b) { a.x += b.x; a.y += b.y; }
__device__ __forceinline__ void add_to(longlong2 &a, const longlong2 &b) { a.x += b.x; a.y += b.y; }

// Inclusive scan of one 128-pixel row segment held as four bytes per lane:
// p[c] / s[c] = sum of pixels / of squared pixels from the warp's first
// column up to this lane's column c (uint32).  Lane 31's p[3], s[3] are the
// segment's totals.
__device__ __forceinline__ void row_scan(uint32_t px, int lane, uint32_t (&p)[4], uint32_t (&s)[4]) {
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

// Decoupled look-back over the predecessors first, first - step, ..., 0
// (flag indices), accumulating their published values for element `elem`.
// Reads up to kWindow flags per round with independent acquire loads, then
// the values of every ready predecessor up to and including the nearest
// inclusive prefix with independent loads.  Returns false when a wait ran
// out (or another CTA aborted).
template <typename V>
__device__ __forceinline__ bool look_back(const unsigned *flags, int first, int step,
                                          int count, const V *agg, const V *pref,
                                          int vstride, int elem, V &acc, unsigned *abort,
                                          int *status, uint64_t t0, uint64_t timeout_ns) {
    int i0 = 0;  // predecessors consumed so far
    while (i0 < count) {
        unsigned f[kWindow];
#pragma unroll
        for (int i = 0; i < kWindow; ++i)
            f[i] = (i0 + i < count) ? ld_acquire_gpu(&flags[first - (i0 + i) * step]) : FLAG_EMPTY;
        if (f[0] == FLAG_EMPTY) {
            f[0] = wait_flag(&flags[first - i0 * step], abort, status, t0, timeout_ns);
            if (f[0] == FLAG_EMPTY) return false;
        }
        // ready run: consecutive non-empty flags, ending at the first prefix
        int run = 0;
        bool found = false;
#pragma unroll
        for (int i = 0; i < kWindow; ++i) {
            if (run == i && !found && i0 + i < count && f[i] != FLAG_EMPTY) {
                ++run;
                found = (f[i] == FLAG_PREFIX);
            }
        }
#pragma unroll
        for (int i = 0; i < kWindow; ++i) {
            if (i < run) {
                const size_t idx = (size_t)(first - (i0 + i) * step) * vstride + elem;
                add_to(acc, __ldcg(f[i] == FLAG_PREFIX ? &pref[idx] : &agg[idx]));
            }
        }
        if (found) return true;
        i0 += run;
    }
    return true;
}

template <bool kAligned4, bool kVecStore>
__global__ void __launch_bounds__(kThreads, 2)
sat_build_kernel(const uint8_t *__restrict__ img, int W, int H, long long *__restrict__ S,
                 long long *__restrict__ Q, SatWs ws, int ntx, int *status,
                 uint64_t timeout_ns, int fault_tile) {
    __shared__ unsigned s_tile;
    __shared__ uint2 s_rowTot[kTileH];               // tile row sums
    __shared__ uint2 s_rowCarry[kTileH];             // row sums left of the tile
    __shared__ __align__(16) uint2 s_colPart[kWarps][kTileW];  // per-warp column sums of warp-local prefixes
    __shared__ long long s_warpCarry[kWarps][2];     // per-warp sums of s_rowCarry
    __shared__ longlong2 s_colCarry[kTileW];         // column sums above the tile

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint64_t t0 = global_timer_ns();
    if (tid == 0) s_tile = atomicAdd(ws.ticket, 1u);
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

    // 2. warp-local row scans in uint32; the column sums of the warp-local
    //    prefixes feed the tile's column aggregate.  (The output pass
    //    repeats the scans instead of keeping them in registers.)
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

    // 3. row carries: publish the tile's row sums, look back to the left.
    bool ok = true;
    if (tid < kTileH) {
        const size_t slot = (size_t)tile * kTileH + tid;
        if (tx == 0) ws.hPref[slot] = s_rowTot[tid];
        else ws.hAgg[slot] = s_rowTot[tid];
        __threadfence();
    }
    __syncthreads();
    if (tid == 0 && publish) st_release_gpu(&ws.flagH[tile], tx == 0 ? FLAG_PREFIX : FLAG_AGGREGATE);
    if (tid < kTileH) {
        uint2 carry = make_uint2(0u, 0u);
        ok = look_back(ws.flagH, (int)tile - 1, 1, tx, ws.hAgg, ws.hPref, kTileH, tid, carry,
                       ws.abort, status, t0, timeout_ns);
        s_rowCarry[tid] = carry;
        if (ok && tx > 0) {
            const uint2 tot = s_rowTot[tid];
            ws.hPref[(size_t)tile * kTileH + tid] = make_uint2(carry.x + tot.x, carry.y + tot.y);
            __threadfence();
        }
    }
    if (__syncthreads_or(!ok)) return;
    if (tid == 0 && tx > 0 && publish) st_release_gpu(&ws.flagH[tile], FLAG_PREFIX);

    // 4. column carries: the tile's column aggregate is the sum over its rows
    //    of the full row prefixes = per-warp column partials + row carries.
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
    longlong2 colAgg = make_longlong2(0, 0);
    if (tid < kTileW) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const uint2 c = s_colPart[w][tid];
            colAgg.x += (long long)c.x + s_warpCarry[w][0];
            colAgg.y += (long long)c.y + s_warpCarry[w][1];
        }
        const size_t slot = (size_t)tile * kTileW + tid;
        if (ty == 0) ws.vPref[slot] = colAgg;
        else ws.vAgg[slot] = colAgg;
        __threadfence();
    }
    __syncthreads();
    if (tid == 0 && publish) st_release_gpu(&ws.flagV[tile], ty == 0 ? FLAG_PREFIX : FLAG_AGGREGATE);
    if (tid < kTileW) {
        longlong2 carry = make_longlong2(0, 0);
        ok = look_back(ws.flagV, (int)tile - ntx, ntx, ty, ws.vAgg, ws.vPref, kTileW, tid, carry,
                       ws.abort, status, t0, timeout_ns);
        s_colCarry[tid] = carry;
        if (ok && ty > 0) {
            ws.vPref[(size_t)tile * kTileW + tid] =
                make_longlong2(carry.x + colAgg.x, carry.y + colAgg.y);
            __threadfence();
        }
    }
    if (__syncthreads_or(!ok)) return;
    if (tid == 0 && ty > 0 && publish) st_release_gpu(&ws.flagV[tile], FLAG_PREFIX);

    // 5. outputs: running column sums from the carry above, down this warp's rows.
    long long runI[4], runQ[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const longlong2 cc = s_colCarry[4 * lane + c];
        runI[c] = cc.x;
        runQ[c] = cc.y;
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

}  // namespace

SatPlan sat_plan(int W, int H) {
    SatPlan p;
    p.tile_w = kTileW;
    p.tile_h = kTileH;
    p.ntx = (W + kTileW - 1) / kTileW;
    p.nty = (H + kTileH - 1) / kTileH;
    const size_t nt = (size_t)p.ntx * p.nty;
    size_t off = 256;                                  // ticket, abort
    off += align_up(nt * sizeof(unsigned), 256);       // flagH
    off += align_up(nt * sizeof(unsigned), 256);       // flagV
    p.zero_bytes = off;
    off += 2 * align_up(nt * kTileH * sizeof(uint2), 256);      // hAgg, hPref
    off += 2 * align_up(nt * kTileW * sizeof(longlong2), 256);  // vAgg, vPref
    p.total_bytes = off;
    return p;
}

cudaError_t sat_launch(const uint8_t *img, int W, int H, int64_t *S, int64_t *Q,
                       void *workspace, const SatPlan &plan, int *status,
                       uint64_t timeout_ns, int fault_tile, cudaStream_t stream) {
    const size_t nt = (size_t)plan.ntx * plan.nty;
    char *base = static_cast<char *>(workspace);
    SatWs ws;
    size_t off = 0;
    ws.ticket = reinterpret_cast<unsigned *>(base);
    ws.abort = reinterpret_cast<unsigned *>(base + 4);
    off = 256;
    ws.flagH = reinterpret_cast<unsigned *>(base + off);
    off += align_up(nt * sizeof(unsigned), 256);
    ws.flagV = reinterpret_cast<unsigned *>(base + off);
    off += align_up(nt * sizeof(unsigned), 256);
    ws.hAgg = reinterpret_cast<uint2 *>(base + off);
    off += align_up(nt * kTileH * sizeof(uint2), 256);
    ws.hPref = reinterpret_cast<uint2 *>(base + off);
    off += align_up(nt * kTileH * sizeof(uint2), 256);
    ws.vAgg = reinterpret_cast<longlong2 *>(base + off);
    off += align_up(nt * kTileW * sizeof(longlong2), 256);
    ws.vPref = reinterpret_cast<longlong2 *>(base + off);

    const bool aligned4 = (W % 4 == 0) && ((uintptr_t)img % 4 == 0);
    const bool vec = (W % 2 == 0) && ((uintptr_t)S % 16 == 0) && ((uintptr_t)Q % 16 == 0);
    const dim3 grid((unsigned)nt), block(kThreads);
    long long *s = reinterpret_cast<long long *>(S), *q = reinterpret_cast<long long *>(Q);
    if (aligned4 && vec)
        sat_build_kernel<true, true><<<grid, block, 0, stream>>>(img, W, H, s, q, ws, plan.ntx, status, timeout_ns, fault_tile);
    else if (aligned4)
        sat_build_kernel<true, false><<<grid, block, 0, stream>>>(img, W, H, s, q, ws, plan.ntx, status, timeout_ns, fault_tile);
    else if (vec)
        sat_build_kernel<false, true><<<grid, block, 0, stream>>>(img, W, H, s, q, ws, plan.ntx, status, timeout_ns, fault_tile);
    else
        sat_build_kernel<false, false><<<grid, block, 0, stream>>>(img, W, H, s, q, ws, plan.ntx, status, timeout_ns, fault_tile);
    return cudaGetLastError();
}

}  // namespace ncc
