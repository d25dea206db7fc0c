// ncc_api.cu -- the library's C ABI (declared in include/ncc.h, the test
// hooks in include/ncc_debug.h): argument checks, the stream-ordered device
// memory pool, kernel selection and the per-device status word.
#include "ncc_common.cuh"

#include <atomic>
#include <mutex>
#include <string.h>

namespace {

// Per-device status word written by kernels (first error wins).
__device__ int g_ncc_status = 0;
// Where ncc_sync_status's read-and-clear kernel leaves the word it took.
__device__ int g_ncc_status_taken = 0;

// Takes the status word and leaves zero in one atomic step, so an error
// recorded at any moment is either returned now or kept for the next call.
__global__ void take_status_kernel(int *status, int *taken) { *taken = atomicExch(status, 0); }

constexpr int kMaxDevices = 64;
int *g_status_ptr[kMaxDevices] = {};
std::mutex g_mutex;

// Test hook state (ncc_debug_set_fault, ncc_debug_set_path,
// ncc_debug_fail_alloc), guarded by g_mutex except the failure count.
int g_fault_tile = -1;
uint64_t g_timeout_ns = 1000000000ull;
int g_path = 0;
int g_last_path = NCC_PATH_NONE;
std::atomic<int> g_fail_allocs{0};
std::mutex g_take_mutex;  // one read-and-clear at a time (shared landing word)
int *g_taken_ptr[kMaxDevices] = {};

void set_last_path(int path) {
    std::lock_guard<std::mutex> lock(g_mutex);
    g_last_path = path;
}

constexpr int kMaxW = 66051;  // 66051 * 255^2 < 2^32: a row's running sum of squares fits uint32
// Automatic selection of the single-template numerator, from a sweep of all
// three kernels on this GPU (one call each, 16x16 to 64x64 templates on
// 1024^2 to 8192^2 images):
//   - the Toeplitz tensor-core kernel's time hardly depends on the template
//     (its box-sum epilogue binds), dp4a's grows with ceil(wT/4)*hT; on maps
//     of at least 4M shifts they cross between 16x16 (64 dp4a per output:
//     4096^2 dp4a 100 us, Toeplitz 181 us) and 20x20 (100: 212 against
//     188 us);
//   - on smaller maps they tie up to 32x32 (1024^2: 33 us each), where dp4a
//     keeps the templates below 320 dp4a per output, since inside ncc_match
//     only it overlaps the table build;
//   - the transform kernel is slower than the Toeplitz kernel for every
//     template the latter takes (8192^2, 64x64: 1316 against 1224 us), and
//     takes the wider ones from 320 dp4a per output on.
constexpr long long kToeplitzMinDp4a = 96;
constexpr long long kToeplitzMinOutputs = 4000000;
constexpr long long kToeplitzMinDp4aSmall = 320;
constexpr long long kNttMinDp4a = 320;
constexpr long long kMaxN = 66051;  // wT*hT*255^2 < 2^32: SumIT fits uint32
// The host-buffer path bands a single-template dp4a map from 8 MB of
// coefficients on, into at most 8 bands (6 to 8 bands of a 66 MB map
// measured best: 0.57 ms per call against 0.64 ms with the kernels storing
// straight into page-locked memory).
constexpr size_t kBandedMinBytes = 8u << 20;
constexpr int kMaxBands = 8;

int status_ptr(int **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NCC_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_ncc_status) != cudaSuccess) return NCC_ERR_CUDA;
        g_status_ptr[dev] = static_cast<int *>(p);
    }
    *out = g_status_ptr[dev];
    return NCC_OK;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const char *pa = static_cast<const char *>(a), *pb = static_cast<const char *>(b);
    return pa < pb + nb && pb < pa + na;
}

int check_image(const uint8_t *img, int W, int H) {
    if (!img || W <= 0 || H <= 0) return NCC_ERR_INVALID_ARG;
    if (W > kMaxW || (long long)W * H >= (1ll << 31)) return NCC_ERR_UNSUPPORTED;
    return NCC_OK;
}

int check_correlate(const uint8_t *img, int W, int H, const uint8_t *tmpl, int wT, int hT,
                    int nT, const int64_t *S, const int64_t *Q) {
    int rc = check_image(img, W, H);
    if (rc != NCC_OK) return rc;
    if (!tmpl || !S || !Q || wT < 1 || hT < 1 || nT < 1 || wT > W || hT > H)
        return NCC_ERR_INVALID_ARG;
    if ((uintptr_t)S % 8 || (uintptr_t)Q % 8) return NCC_ERR_INVALID_ARG;
    if ((long long)wT * hT > kMaxN) return NCC_ERR_UNSUPPORTED;
    if ((long long)nT * (W - wT + 1) * (long long)(H - hT + 1) >= (1ll << 40))
        return NCC_ERR_UNSUPPORTED;
    return NCC_OK;
}

// Stream-ordered pool for the library's device memory (the SAT builder's
// look-back workspace, the host-buffer path's buffers), one per device.  Its
// release threshold keeps freed memory reserved, so repeated calls reuse it
// instead of mapping it afresh after every synchronization (what the default
// pool, which releases at each synchronization, would do).
cudaMemPool_t g_host_pool[kMaxDevices] = {};

int host_path_pool(cudaMemPool_t *out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NCC_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_host_pool[dev]) {
        cudaMemPoolProps props;
        memset(&props, 0, sizeof(props));
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return NCC_ERR_CUDA;
        uint64_t keep = ~0ull;
        if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) {
            cudaMemPoolDestroy(pool);
            return NCC_ERR_CUDA;
        }
        g_host_pool[dev] = pool;
    }
    *out = g_host_pool[dev];
    return NCC_OK;
}

// Arguments of the direct-moment calls (no tables).
int check_direct(const uint8_t *img, int W, int H, const uint8_t *tmpl, int wT, int hT, int nT) {
    int rc = check_image(img, W, H);
    if (rc != NCC_OK) return rc;
    if (!tmpl || wT < 1 || hT < 1 || nT < 1 || wT > W || hT > H) return NCC_ERR_INVALID_ARG;
    if ((long long)wT * hT > kMaxN) return NCC_ERR_UNSUPPORTED;
    if ((long long)nT * (W - wT + 1) * (long long)(H - hT + 1) >= (1ll << 40))
        return NCC_ERR_UNSUPPORTED;
    if (!ncc::corr_dp4a_direct_supported(wT, hT)) return NCC_ERR_UNSUPPORTED;
    return NCC_OK;
}

int to_status(cudaError_t e) {
    if (e == cudaSuccess) return NCC_OK;
    if (e == cudaErrorMemoryAllocation) return NCC_ERR_NOMEM;
    if (e == cudaErrorNotSupported) return NCC_ERR_UNSUPPORTED;
    return NCC_ERR_CUDA;
}

// The numerator kernel for these sizes: NCC_PATH_BANK for a bank the
// tensor-core bank kernel takes; otherwise the single-template kernel,
// forced by `path` (ncc_debug_set_path) or picked automatically -- the
// Toeplitz tensor-core product for templates whose numerator dominates, the
// transform kernel for templates that product cannot take, dp4a for smaller
// templates.  NCC_ERR_UNSUPPORTED when the forced or needed kernel cannot
// take the sizes.
int pick_kernel(int W, int H, int wT, int hT, int nT, int path, bool direct) {
    if (!direct && nT > 1 && ncc::bank_tc_supported(W, H, wT, hT, nT)) return NCC_PATH_BANK;
    if (direct) path = NCC_PATH_DP4A;  // the direct moments exist on the dp4a kernel only
    const long long plane = (long long)(W - wT + 1) * (H - hT + 1);
    const long long dp4aPerOutput = (long long)((wT + 3) / 4) * hT;
    int kernel = NCC_PATH_DP4A;
    if (path == NCC_PATH_TOEPLITZ || path == NCC_PATH_NTT) {
        const bool ok = path == NCC_PATH_TOEPLITZ ? ncc::corr_toeplitz_supported(wT, hT)
                                                  : ncc::corr_ntt_supported(wT, hT);
        if (!ok) return NCC_ERR_UNSUPPORTED;
        kernel = path;
    } else if (path == 0) {
        const bool tzOk = ncc::corr_toeplitz_supported(wT, hT);
        const long long tzMin = plane >= kToeplitzMinOutputs ? kToeplitzMinDp4a : kToeplitzMinDp4aSmall;
        if (tzOk && dp4aPerOutput >= tzMin)
            kernel = NCC_PATH_TOEPLITZ;
        else if (!tzOk && ncc::corr_ntt_supported(wT, hT) && dp4aPerOutput >= kNttMinDp4a)
            kernel = NCC_PATH_NTT;
    }
    if (kernel == NCC_PATH_DP4A && !ncc::corr_dp4a_supported(wT, hT)) return NCC_ERR_UNSUPPORTED;
    return kernel;
}

int current_path() {
    std::lock_guard<std::mutex> lock(g_mutex);
    return g_path;
}

// Numerator + epilogue for nT templates, either coefficients or moments.
// after_sat: the previous kernel on the stream is this library's SAT build
// of img, so a single-template launch may overlap its tail.
// rowBegin, rowEnd: only the output rows [rowBegin, rowEnd) (both 0: all),
// on the dp4a kernel only (edges as CorrArgs requires).
int run_correlate(const uint8_t *img, int W, int H, const uint8_t *tmpl, int wT, int hT, int nT,
                  const int64_t *S, const int64_t *Q, float *out, int64_t *sumI,
                  int64_t *sumI2, int64_t *sumIT, cudaStream_t stream, bool after_sat = false,
                  bool direct = false, int rowBegin = 0, int rowEnd = 0) {
    int *status = nullptr;
    int rc = status_ptr(&status);
    if (rc != NCC_OK) return rc;
    const size_t plane = (size_t)(W - wT + 1) * (H - hT + 1);
    const int path = current_path();
    const int kernel = pick_kernel(W, H, wT, hT, nT, path, direct);
    if (kernel < 0) return kernel;
    const bool band = rowBegin != 0 || rowEnd != 0;
    if (band && kernel != NCC_PATH_DP4A) return NCC_ERR_UNSUPPORTED;
    if (kernel == NCC_PATH_BANK) {
        ncc::BankArgs b{img, W, H, tmpl, wT, hT, nT, S, Q, out, sumI, sumI2, sumIT, status};
        rc = to_status(ncc::bank_tc_launch(b, stream));
        if (rc == NCC_OK) set_last_path(NCC_PATH_BANK);
        return rc;
    }
    int used = NCC_PATH_NONE;
    for (int t = 0; t < nT; ++t) {
        ncc::CorrArgs a;
        a.img = img; a.W = W; a.H = H;
        a.tmpl = tmpl + (size_t)t * wT * hT;
        a.wT = wT; a.hT = hT; a.S = S; a.Q = Q;
        a.out = out ? out + (size_t)t * plane : nullptr;
        // the window moments do not depend on the template; every launch
        // rewrites the same SumI/SumI2 plane
        a.sumI = sumI;
        a.sumI2 = sumI2;
        a.sumIT = sumIT ? sumIT + (size_t)t * plane : nullptr;
        a.status = status;
        a.overlap_prev = after_sat && t == 0;
        a.direct = direct;
        a.rowBegin = rowBegin;
        a.rowEnd = rowEnd;
        cudaError_t e = cudaErrorNotSupported;
        if (kernel == NCC_PATH_TOEPLITZ) {
            // plain stream order: behind the table build the early start
            // measured slower for this kernel (8192x8192, 64x64: 2.19 ms per
            // image against 1.87 ms as two calls), its CTAs taking whole SMs
            a.overlap_prev = false;
            e = ncc::corr_toeplitz_launch(a, stream);
        } else if (kernel == NCC_PATH_NTT) {
            a.overlap_prev = false;
            e = ncc::corr_ntt_launch(a, stream);
        }
        if (e == cudaSuccess && kernel != NCC_PATH_DP4A) used = kernel;
        if (e == cudaErrorNotSupported || kernel == NCC_PATH_DP4A) {
            if (path == NCC_PATH_TOEPLITZ || path == NCC_PATH_NTT) return NCC_ERR_UNSUPPORTED;
            e = ncc::corr_dp4a_launch(a, stream);
            if (e == cudaSuccess) used = NCC_PATH_DP4A;
        }
        if (e != cudaSuccess)
            return band && e == cudaErrorInvalidValue ? NCC_ERR_INVALID_ARG : to_status(e);
    }
    set_last_path(used);
    return NCC_OK;
}

// The host-buffer path's copy stream, one per device (non-blocking, kept for
// the process): the coefficient bands go back to the host on it while the
// correlation of the next band runs on the caller's stream.
cudaStream_t g_copy_stream[kMaxDevices] = {};

int copy_stream(cudaStream_t *out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NCC_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_copy_stream[dev] &&
        cudaStreamCreateWithFlags(&g_copy_stream[dev], cudaStreamNonBlocking) != cudaSuccess) {
        g_copy_stream[dev] = nullptr;
        return NCC_ERR_CUDA;
    }
    *out = g_copy_stream[dev];
    return NCC_OK;
}

}  // namespace

namespace ncc {
// The per-device status word's device address, for entry points defined in
// other translation units.
int status_word(int **out) { return status_ptr(out); }

cudaError_t pool_alloc(void **ptr, size_t bytes, cudaStream_t stream) {
    int left = g_fail_allocs.load();
    while (left > 0) {
        if (g_fail_allocs.compare_exchange_weak(left, left - 1)) return cudaErrorMemoryAllocation;
    }
    cudaMemPool_t pool = nullptr;
    const int rc = host_path_pool(&pool);
    if (rc != NCC_OK) return cudaErrorInitializationError;
    return cudaMallocFromPoolAsync(ptr, bytes, pool, stream);
}
}  // namespace ncc

extern "C" {

int ncc_sat_build(const uint8_t *img, int W, int H, int64_t *S, int64_t *Q,
                  ncc_stream_t stream) {
    int rc = check_image(img, W, H);
    if (rc != NCC_OK) return rc;
    if (!S || !Q || (uintptr_t)S % 8 || (uintptr_t)Q % 8) return NCC_ERR_INVALID_ARG;
    const size_t n = (size_t)W * H;
    if (overlaps(S, n * 8, Q, n * 8) || overlaps(S, n * 8, img, n) || overlaps(Q, n * 8, img, n))
        return NCC_ERR_INVALID_ARG;
    int *status = nullptr;
    rc = status_ptr(&status);
    if (rc != NCC_OK) return rc;
    int fault;
    uint64_t timeout;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        fault = g_fault_tile;
        timeout = g_timeout_ns;
    }
    return to_status(ncc::sat_build_run(img, W, H, S, Q, status, timeout, fault,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

int ncc_sat_build_variant(const uint8_t *img, int W, int H, int64_t *S, int64_t *Q, int variant,
                          ncc_stream_t stream) {
    if (variant == NCC_SAT_FUSED) return ncc_sat_build(img, W, H, S, Q, stream);
    if (variant != NCC_SAT_NAIVE && variant != NCC_SAT_TWO_PASS) return NCC_ERR_INVALID_ARG;
    int rc = check_image(img, W, H);
    if (rc != NCC_OK) return rc;
    if (!S || !Q || (uintptr_t)S % 8 || (uintptr_t)Q % 8) return NCC_ERR_INVALID_ARG;
    const size_t n = (size_t)W * H;
    if (overlaps(S, n * 8, Q, n * 8) || overlaps(S, n * 8, img, n) || overlaps(Q, n * 8, img, n))
        return NCC_ERR_INVALID_ARG;
    int *status = nullptr;
    rc = status_ptr(&status);
    if (rc != NCC_OK) return rc;
    uint64_t timeout;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        timeout = g_timeout_ns;
    }
    return to_status(ncc::sat_ladder_run(variant, img, W, H, S, Q, status, timeout,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

int ncc_correlate(const uint8_t *img, int W, int H, const uint8_t *tmpl, int wT, int hT,
                  const int64_t *S, const int64_t *Q, float *out, ncc_stream_t stream) {
    return ncc_correlate_bank(img, W, H, tmpl, wT, hT, 1, S, Q, out, stream);
}

int ncc_correlate_bank(const uint8_t *img, int W, int H, const uint8_t *tmpl, int wT, int hT,
                       int nT, const int64_t *S, const int64_t *Q, float *out,
                       ncc_stream_t stream) {
    int rc = check_correlate(img, W, H, tmpl, wT, hT, nT, S, Q);
    if (rc != NCC_OK) return rc;
    if (!out || (uintptr_t)out % 4) return NCC_ERR_INVALID_ARG;
    const size_t n = (size_t)W * H;
    const size_t nout = (size_t)nT * (W - wT + 1) * (H - hT + 1) * sizeof(float);
    if (overlaps(out, nout, S, n * 8) || overlaps(out, nout, Q, n * 8) ||
        overlaps(out, nout, img, n) || overlaps(out, nout, tmpl, (size_t)nT * wT * hT))
        return NCC_ERR_INVALID_ARG;
    return run_correlate(img, W, H, tmpl, wT, hT, nT, S, Q, out, nullptr, nullptr, nullptr,
                         reinterpret_cast<cudaStream_t>(stream));
}

int ncc_correlate_moments(const uint8_t *img, int W, int H, const uint8_t *tmpl, int wT, int hT,
                          int nT, const int64_t *S, const int64_t *Q, int64_t *sumI,
                          int64_t *sumI2, int64_t *sumIT, ncc_stream_t stream) {
    int rc = check_correlate(img, W, H, tmpl, wT, hT, nT, S, Q);
    if (rc != NCC_OK) return rc;
    if (!sumI || !sumI2 || !sumIT || (uintptr_t)sumI % 8 || (uintptr_t)sumI2 % 8 ||
        (uintptr_t)sumIT % 8)
        return NCC_ERR_INVALID_ARG;
    const size_t plane = (size_t)(W - wT + 1) * (H - hT + 1) * 8;
    if (overlaps(sumI, plane, sumI2, plane) || overlaps(sumI, plane, sumIT, plane * nT) ||
        overlaps(sumI2, plane, sumIT, plane * nT))
        return NCC_ERR_INVALID_ARG;
    return run_correlate(img, W, H, tmpl, wT, hT, nT, S, Q, nullptr, sumI, sumI2, sumIT,
                         reinterpret_cast<cudaStream_t>(stream));
}

int ncc_correlate_direct(const uint8_t *img, int W, int H, const uint8_t *tmpl, int wT, int hT,
                         int nT, float *out, ncc_stream_t stream) {
    int rc = check_direct(img, W, H, tmpl, wT, hT, nT);
    if (rc != NCC_OK) return rc;
    if (!out || (uintptr_t)out % 4) return NCC_ERR_INVALID_ARG;
    const size_t nout = (size_t)nT * (W - wT + 1) * (H - hT + 1) * sizeof(float);
    if (overlaps(out, nout, img, (size_t)W * H) || overlaps(out, nout, tmpl, (size_t)nT * wT * hT))
        return NCC_ERR_INVALID_ARG;
    return run_correlate(img, W, H, tmpl, wT, hT, nT, nullptr, nullptr, out, nullptr, nullptr,
                         nullptr, reinterpret_cast<cudaStream_t>(stream), false, true);
}

int ncc_correlate_direct_moments(const uint8_t *img, int W, int H, const uint8_t *tmpl, int wT,
                                 int hT, int nT, int64_t *sumI, int64_t *sumI2, int64_t *sumIT,
                                 ncc_stream_t stream) {
    int rc = check_direct(img, W, H, tmpl, wT, hT, nT);
    if (rc != NCC_OK) return rc;
    if (!sumI || !sumI2 || !sumIT || (uintptr_t)sumI % 8 || (uintptr_t)sumI2 % 8 ||
        (uintptr_t)sumIT % 8)
        return NCC_ERR_INVALID_ARG;
    const size_t plane = (size_t)(W - wT + 1) * (H - hT + 1) * 8;
    if (overlaps(sumI, plane, sumI2, plane) || overlaps(sumI, plane, sumIT, plane * nT) ||
        overlaps(sumI2, plane, sumIT, plane * nT))
        return NCC_ERR_INVALID_ARG;
    return run_correlate(img, W, H, tmpl, wT, hT, nT, nullptr, nullptr, nullptr, sumI, sumI2,
                         sumIT, reinterpret_cast<cudaStream_t>(stream), false, true);
}

int ncc_match(const uint8_t *img, int W, int H, const uint8_t *tmpl, int wT, int hT, int nT,
              int64_t *S, int64_t *Q, float *out, ncc_stream_t stream) {
    int rc = check_correlate(img, W, H, tmpl, wT, hT, nT, S, Q);
    if (rc != NCC_OK) return rc;
    if (!out || (uintptr_t)out % 4) return NCC_ERR_INVALID_ARG;
    const size_t n = (size_t)W * H;
    const size_t nout = (size_t)nT * (W - wT + 1) * (H - hT + 1) * sizeof(float);
    if (overlaps(out, nout, S, n * 8) || overlaps(out, nout, Q, n * 8) ||
        overlaps(out, nout, img, n) || overlaps(out, nout, tmpl, (size_t)nT * wT * hT) ||
        overlaps(S, n * 8, tmpl, (size_t)nT * wT * hT) || overlaps(Q, n * 8, tmpl, (size_t)nT * wT * hT))
        return NCC_ERR_INVALID_ARG;
    rc = ncc_sat_build(img, W, H, S, Q, stream);   // checks S, Q against img and each other
    if (rc != NCC_OK) return rc;
    // the overlap only behind the fused builder, which lets its dependents start
    return run_correlate(img, W, H, tmpl, wT, hT, nT, S, Q, out, nullptr, nullptr, nullptr,
                         reinterpret_cast<cudaStream_t>(stream), true);
}

int ncc_match_host(const uint8_t *img, int W, int H, const uint8_t *tmpl, int wT, int hT,
                   int nT, float *out, ncc_stream_t stream) {
    int rc = check_image(img, W, H);
    if (rc != NCC_OK) return rc;
    if (!tmpl || !out || wT < 1 || hT < 1 || nT < 1 || wT > W || hT > H)
        return NCC_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t n = (size_t)W * H, nt = (size_t)nT * wT * hT;
    const int Ox = W - wT + 1, Oy = H - hT + 1;
    const size_t nout = (size_t)nT * Ox * Oy;
    // A large single-template map on the dp4a kernel is correlated in bands
    // of output rows, each copied back on the library's copy stream while
    // the next band is correlated: the copy over the host link is the
    // longest step (about 190 GB/s), and this hides all but the first
    // band's correlation behind it.  Other maps: page-locked output that
    // the device can address is written by the kernels directly over the
    // link; otherwise a device buffer and one copy.
    const bool banded = nT == 1 && nout * 4 >= kBandedMinBytes &&
                        pick_kernel(W, H, wT, hT, nT, current_path(), false) == NCC_PATH_DP4A;
    float *direct = nullptr;
    if (!banded) {
        cudaPointerAttributes pa;
        if (cudaPointerGetAttributes(&pa, out) == cudaSuccess && pa.type == cudaMemoryTypeHost &&
            pa.devicePointer && (uintptr_t)pa.devicePointer % 4 == 0)
            direct = static_cast<float *>(pa.devicePointer);
        else
            (void)cudaGetLastError();  // pageable memory: clear the query's error, if any
    }
    cudaStream_t cs = nullptr;
    if (banded && (rc = copy_stream(&cs)) != NCC_OK) return rc;
    // one device block: tables first (8-byte aligned), then out, image, templates
    const size_t outBytes = direct ? 0 : nout * 4;
    const size_t offQ = n * 8, offOut = 2 * n * 8, offImg = (offOut + outBytes + 255) / 256 * 256;
    const size_t offT = (offImg + n + 255) / 256 * 256, total = offT + nt;
    char *d = nullptr;
    cudaError_t e = ncc::pool_alloc(reinterpret_cast<void **>(&d), total, st);
    if (e != cudaSuccess) return e == cudaErrorMemoryAllocation ? NCC_ERR_NOMEM : NCC_ERR_CUDA;
    int64_t *S = reinterpret_cast<int64_t *>(d), *Q = reinterpret_cast<int64_t *>(d + offQ);
    float *dout = direct ? direct : reinterpret_cast<float *>(d + offOut);
    uint8_t *dimg = reinterpret_cast<uint8_t *>(d + offImg), *dt = reinterpret_cast<uint8_t *>(d + offT);
    rc = NCC_OK;
    if (cudaMemcpyAsync(dimg, img, n, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(dt, tmpl, nt, cudaMemcpyHostToDevice, st) != cudaSuccess)
        rc = NCC_ERR_CUDA;
    if (!banded) {
        if (rc == NCC_OK) rc = ncc_match(dimg, W, H, dt, wT, hT, nT, S, Q, dout, stream);
        if (rc == NCC_OK && !direct &&
            cudaMemcpyAsync(out, dout, nout * 4, cudaMemcpyDeviceToHost, st) != cudaSuccess)
            rc = NCC_ERR_CUDA;
    } else {
        // at most kMaxBands bands of whole tiles, the bottom one first (the
        // build writes the tables top-down, so its last rows are still in
        // L2); the first band's launch overlaps the build's tail
        const int per = (Oy + kMaxBands - 1) / kMaxBands;
        const int bandRows = (per + ncc::kCorrBandRows - 1) / ncc::kCorrBandRows * ncc::kCorrBandRows;
        const int nb = (Oy + bandRows - 1) / bandRows;
        cudaEvent_t ev[kMaxBands + 1] = {};
        int made = 0;
        for (; made <= nb; ++made)
            if (cudaEventCreateWithFlags(&ev[made], cudaEventDisableTiming) != cudaSuccess) break;
        if (made <= nb) rc = NCC_ERR_CUDA;
        if (rc == NCC_OK) rc = check_correlate(dimg, W, H, dt, wT, hT, nT, S, Q);
        if (rc == NCC_OK) rc = ncc_sat_build(dimg, W, H, S, Q, stream);
        // every band's kernel is enqueued before any copy: a copy into
        // pageable memory returns only once it is done
        int launched = 0;
        for (int k = 0; k < nb && rc == NCC_OK; ++k, ++launched) {
            const int b = nb - 1 - k, y0 = b * bandRows, y1 = y0 + bandRows < Oy ? y0 + bandRows : Oy;
            rc = run_correlate(dimg, W, H, dt, wT, hT, 1, S, Q, dout, nullptr, nullptr, nullptr, st,
                               k == 0, false, y0, y1);
            if (rc == NCC_OK && cudaEventRecord(ev[k], st) != cudaSuccess) rc = NCC_ERR_CUDA;
        }
        for (int k = 0; k < launched && rc == NCC_OK; ++k) {
            const int b = nb - 1 - k, y0 = b * bandRows, y1 = y0 + bandRows < Oy ? y0 + bandRows : Oy;
            const size_t off = (size_t)y0 * Ox, cnt = (size_t)(y1 - y0) * Ox;
            if (cudaStreamWaitEvent(cs, ev[k], 0) != cudaSuccess ||
                cudaMemcpyAsync(out + off, dout + off, cnt * 4, cudaMemcpyDeviceToHost, cs) != cudaSuccess)
                rc = NCC_ERR_CUDA;
        }
        // the caller's stream (and the buffers' release below) waits for the copies
        if (made > nb && (cudaEventRecord(ev[nb], cs) != cudaSuccess ||
                          cudaStreamWaitEvent(st, ev[nb], 0) != cudaSuccess) && rc == NCC_OK)
            rc = NCC_ERR_CUDA;
        for (int k = 0; k < made; ++k) cudaEventDestroy(ev[k]);
    }
    cudaFreeAsync(d, st);
    const int rs = ncc_sync_status(stream);
    return rc != NCC_OK ? rc : rs;
}

int ncc_sync_status(ncc_stream_t stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return NCC_ERR_CUDA;
    int *status = nullptr;
    int rc = status_ptr(&status);
    if (rc != NCC_OK) return rc;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NCC_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_take_mutex);
    if (!g_taken_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_ncc_status_taken) != cudaSuccess) return NCC_ERR_CUDA;
        g_taken_ptr[dev] = static_cast<int *>(p);
    }
    // read and clear in one atomic exchange on the device, then fetch the
    // value it took; both in stream order after the work just synchronized
    take_status_kernel<<<1, 1, 0, st>>>(status, g_taken_ptr[dev]);
    if (cudaGetLastError() != cudaSuccess) return NCC_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyAsync(&v, g_taken_ptr[dev], sizeof(int), cudaMemcpyDeviceToHost, st) !=
            cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return NCC_ERR_CUDA;
    return v;
}

const char *ncc_status_string(int status) {
    switch (status) {
        case NCC_OK: return "ok";
        case NCC_ERR_INVALID_ARG: return "invalid argument";
        case NCC_ERR_UNSUPPORTED: return "unsupported size or shape";
        case NCC_ERR_CUDA: return "CUDA runtime error";
        case NCC_ERR_TIMEOUT: return "look-back wait timed out";
        case NCC_ERR_NOMEM: return "device workspace allocation failed";
        case NCC_ERR_BOUNDS: return "index check failed (debug build)";
        default: return "unknown status";
    }
}

int ncc_version(void) { return (0 << 16) | 1; }

int ncc_debug_set_path(int path) {
    if (path != 0 && path != NCC_PATH_DP4A && path != NCC_PATH_TOEPLITZ && path != NCC_PATH_NTT)
        return NCC_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_mutex);
    g_path = path;
    return NCC_OK;
}

int ncc_debug_last_path(void) {
    std::lock_guard<std::mutex> lock(g_mutex);
    return g_last_path;
}

int ncc_debug_fail_alloc(int count) {
    if (count < 0) return NCC_ERR_INVALID_ARG;
    g_fail_allocs.store(count);
    return NCC_OK;
}

int ncc_debug_set_fault(int suppress_tile, uint64_t timeout_ns) {
#ifdef NCC_DEBUG
    if (suppress_tile < -2) return NCC_ERR_INVALID_ARG;  // -2: the index-check test
#else
    if (suppress_tile < -1) return NCC_ERR_INVALID_ARG;
#endif
    std::lock_guard<std::mutex> lock(g_mutex);
    g_fault_tile = suppress_tile;
    g_timeout_ns = timeout_ns ? timeout_ns : 1000000000ull;
    return NCC_OK;
}

}  // extern "C"
