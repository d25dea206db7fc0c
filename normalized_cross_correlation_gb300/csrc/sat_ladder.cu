// sat_ladder.cu -- the two slower builders of the summed-area tables that
// The CUDA Handbook, section 15.8 ("The Denominator: Summed Area Tables")
// sets against the fused single pass, written for this GPU so the
// comparison of Figures 15-8 and 15-9 can be measured here.  The product
// path is sat_build.cu; these builders exist for the measured ladder and
// produce the same inclusive int64 tables S = SAT(I), Q = SAT(I^2).
//
//   naive     one thread per image row runs the row's running sums of I and
//             I^2 straight into S and Q; then one thread per column adds
//             down its column in place (the section's one-thread-per-line
//             build).
//   two-pass  the section's transpose-free two-pass build: first the rows'
//             running sums go to a uint32 intermediate (a row's sum of
//             squares is at most W*255^2 < 2^32), one warp per row, 128
//             pixels per step; then a column scan reads the intermediate and
//             writes S and Q.  In the column scan each block owns a strip of
//             128 columns and a stripe of 128 rows, taken by an atomic
//             ticket in row-major order: it sums its columns, publishes the
//             sums, looks back over the stripes above for each column's
//             carry (three states: empty / aggregate / inclusive prefix, one
//             64-bit word per column), publishes its inclusive prefix and
//             writes its stripe.  Every wait points at a smaller ticket and
//             is bounded.
#include "ncc_common.cuh"

#include <mutex>

namespace ncc {
namespace {

constexpr int kStrip = 128;         // columns per column-scan block (one thread each)
constexpr int kStripe = 128;        // rows per column-scan block
constexpr int kRowWarps = 8;        // rows per block in the row pass (one warp each)
constexpr int kStateShift = 62;
constexpr uint64_t kValueMask = (1ull << kStateShift) - 1;

// ---------------------------------------------------------------- naive --

// The one-thread-per-line build of section 15.8: each thread owns one line
// of the tables and walks it from its first element to its last, replacing
// every element by the running total of the line so far, for S and Q in the
// same walk.  The build is two launches of this kernel.  Along rows the
// values walked are the pixels and their squares; along columns they are
// what the row launch left in S and Q, so after the column launch every
// element holds its whole upper-left rectangle.  Rows are walked with unit
// stride but the threads of a warp sit W elements apart, so that launch is
// uncoalesced by construction -- the cost the section measures.
template <bool kAlongRows>
__global__ void naive_line_kernel(const uint8_t *__restrict__ img, int W, int H,
                                  long long *__restrict__ S, long long *__restrict__ Q) {
    const int line = blockIdx.x * blockDim.x + threadIdx.x;
    if (line >= (kAlongRows ? H : W)) return;
    const size_t step = kAlongRows ? 1 : (size_t)W;
    const size_t begin = kAlongRows ? (size_t)line * W : (size_t)line;
    const size_t end = begin + step * (size_t)(kAlongRows ? W : H);
    long long total = 0, total_sq = 0;
    for (size_t o = begin; o != end; o += step) {
        if constexpr (kAlongRows) {
            const long long v = img[o];
            total += v;
            total_sq += v * v;
        } else {
            total += S[o];
            total_sq += Q[o];
        }
        S[o] = total;
        Q[o] = total_sq;
    }
}

// ------------------------------------------------------------- two-pass --

// Pass 1: row running sums into uint32 rowS / rowQ, one warp per row; each
// lane takes four consecutive pixels of every 128-pixel step.
__global__ void __launch_bounds__(kRowWarps * 32)
rows_u32_kernel(const uint8_t *__restrict__ img, int W, int H, uint32_t *__restrict__ rowS,
                uint32_t *__restrict__ rowQ) {
    const int lane = threadIdx.x & 31;
    const int y = blockIdx.x * kRowWarps + (threadIdx.x >> 5);
    if (y >= H) return;  // warp-uniform
    const uint8_t *row = img + (size_t)y * W;
    uint32_t *sr = rowS + (size_t)y * W, *qr = rowQ + (size_t)y * W;
    uint32_t carryI = 0, carryQ = 0;
    for (int x0 = 0; x0 < W; x0 += 128) {
        const int x = x0 + 4 * lane;
        uint32_t p[4], s[4];
        uint32_t a = 0, b = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t v = x + c < W ? row[x + c] : 0u;
            a += v;
            b += v * v;
            p[c] = a;
            s[c] = b;
        }
        uint32_t tI = a, tQ = b;  // inclusive scan of the lanes' totals
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t uI = __shfl_up_sync(0xffffffffu, tI, o);
            const uint32_t uQ = __shfl_up_sync(0xffffffffu, tQ, o);
            if (lane >= o) { tI += uI; tQ += uQ; }
        }
        const uint32_t eI = carryI + tI - a, eQ = carryQ + tQ - b;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (x + c < W) {
                sr[x + c] = eI + p[c];
                qr[x + c] = eQ + s[c];
            }
        }
        carryI += __shfl_sync(0xffffffffu, tI, 31);
        carryQ += __shfl_sync(0xffffffffu, tQ, 31);
    }
}

struct ColWs {
    unsigned *ticket;  // tile dispenser (zeroed before each build)
    uint64_t *words;   // [ntiles][2 * kStrip]: S word, then Q word, per column
};

__device__ __forceinline__ uint64_t ld_word(const uint64_t *p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_word(uint64_t *p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Pass 2: column scan of the intermediate with a decoupled look-back over
// the stripes above.  One thread per column.
__global__ void __launch_bounds__(kStrip)
cols_dlb_kernel(const uint32_t *__restrict__ rowS, const uint32_t *__restrict__ rowQ, int W, int H,
                long long *__restrict__ S, long long *__restrict__ Q, ColWs ws, int ntx,
                int *status, uint64_t timeout_ns) {
    __shared__ unsigned s_tile;
    if (threadIdx.x == 0) s_tile = atomicAdd(ws.ticket, 1u);
    __syncthreads();
    const int tile = (int)s_tile, tx = tile % ntx, ty = tile / ntx;
    const int x = tx * kStrip + (int)threadIdx.x, y0 = ty * kStripe;
    const int rows = min(kStripe, H - y0);
    const bool xin = x < W;

    // column sums of this stripe
    long long aggS = 0, aggQ = 0;
    if (xin)
        for (int r = 0; r < rows; ++r) {
            const size_t o = (size_t)(y0 + r) * W + x;
            aggS += rowS[o];
            aggQ += rowQ[o];
        }
    uint64_t *mine = ws.words + (size_t)tile * 2 * kStrip + threadIdx.x;
    const uint64_t state0 = ty == 0 ? 2ull : 1ull;
    st_word(mine, (state0 << kStateShift) | (uint64_t)aggS);
    st_word(mine + kStrip, (state0 << kStateShift) | (uint64_t)aggQ);

    // carries from the stripes above: add aggregates until an inclusive prefix
    long long carryS = 0, carryQ = 0;
    bool doneS = ty == 0, doneQ = ty == 0;
    const uint64_t t0 = global_timer_ns();
    unsigned polls = 0;
    for (int prev = tile - ntx; !(doneS && doneQ) && prev >= 0;) {
        const uint64_t *w = ws.words + (size_t)prev * 2 * kStrip + threadIdx.x;
        const uint64_t a = doneS ? 0ull : ld_word(w), b = doneQ ? 0ull : ld_word(w + kStrip);
        const uint32_t sa = (uint32_t)(a >> kStateShift), sb = (uint32_t)(b >> kStateShift);
        if ((!doneS && sa == 0u) || (!doneQ && sb == 0u)) {
            // the stripe above has not published yet
            __nanosleep(64);
            if ((++polls & 63u) == 0u &&
                (global_timer_ns() - t0 > timeout_ns || polls > (1u << 26))) {
                record_status(status, NCC_ERR_TIMEOUT);
                break;
            }
            continue;
        }
        if (!doneS) {
            carryS += (long long)(a & kValueMask);
            doneS = sa == 2u;
        }
        if (!doneQ) {
            carryQ += (long long)(b & kValueMask);
            doneQ = sb == 2u;
        }
        prev -= ntx;
    }
    if (ty > 0) {
        st_word(mine, (2ull << kStateShift) | (uint64_t)(carryS + aggS));
        st_word(mine + kStrip, (2ull << kStateShift) | (uint64_t)(carryQ + aggQ));
    }

    // the stripe's table entries
    if (xin) {
        long long s = carryS, q = carryQ;
        for (int r = 0; r < rows; ++r) {
            const size_t o = (size_t)(y0 + r) * W + x;
            s += rowS[o];
            q += rowQ[o];
            S[o] = s;
            Q[o] = q;
        }
    }
}

// Library-owned intermediate and look-back words, one set per device.
struct LadderWs {
    void *ptr = nullptr;
    size_t bytes = 0;
};
constexpr int kMaxDevices = 64;
LadderWs g_lws[kMaxDevices];
std::mutex g_lws_mutex;

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

cudaError_t sat_ladder_run(int variant, const uint8_t *img, int W, int H, int64_t *S, int64_t *Q,
                           int *status, uint64_t timeout_ns, cudaStream_t stream) {
    long long *s = reinterpret_cast<long long *>(S), *q = reinterpret_cast<long long *>(Q);
    if (variant == NCC_SAT_NAIVE) {
        naive_line_kernel<true><<<(H + 127) / 128, 128, 0, stream>>>(img, W, H, s, q);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        naive_line_kernel<false><<<(W + 127) / 128, 128, 0, stream>>>(img, W, H, s, q);
        return cudaGetLastError();
    }
    if (variant != NCC_SAT_TWO_PASS) return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    const int ntx = (W + kStrip - 1) / kStrip, nty = (H + kStripe - 1) / kStripe;
    const size_t ntiles = (size_t)ntx * nty;
    const size_t inter = round_up((size_t)W * H * 4, 256);
    const size_t head = 256, wordBytes = round_up(ntiles * 2 * kStrip * 8, 256);
    const size_t need = head + wordBytes + 2 * inter;
    std::lock_guard<std::mutex> lock(g_lws_mutex);
    LadderWs &d = g_lws[dev];
    if (d.bytes < need) {
        if (d.ptr) {
            e = cudaDeviceSynchronize();  // the old workspace may still be in use
            if (e != cudaSuccess) return e;
            cudaFree(d.ptr);
            d.ptr = nullptr;
            d.bytes = 0;
        }
        e = cudaMalloc(&d.ptr, need);
        if (e != cudaSuccess) return e;
        d.bytes = need;
    }
    char *base = static_cast<char *>(d.ptr);
    ColWs ws;
    ws.ticket = reinterpret_cast<unsigned *>(base);
    ws.words = reinterpret_cast<uint64_t *>(base + head);
    uint32_t *rowS = reinterpret_cast<uint32_t *>(base + head + wordBytes);
    uint32_t *rowQ = reinterpret_cast<uint32_t *>(base + head + wordBytes + inter);
    // ticket and look-back words start empty on every build
    e = cudaMemsetAsync(base, 0, head + wordBytes, stream);
    if (e != cudaSuccess) return e;
    rows_u32_kernel<<<(H + kRowWarps - 1) / kRowWarps, kRowWarps * 32, 0, stream>>>(img, W, H, rowS, rowQ);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cols_dlb_kernel<<<(unsigned)ntiles, kStrip, 0, stream>>>(rowS, rowQ, W, H, s, q, ws, ntx, status,
                                                            timeout_ns);
    return cudaGetLastError();
}

}  // namespace ncc
