// sat_build_noalloc.cu -- ncc_sat_build_noalloc: the summed-area-table
// builder for callers that must not allocate device memory.
//
// Who needs it: code that runs where a cudaMalloc is not allowed or not
// wanted -- a host callback or a real-time loop that must not block
// (cudaMalloc and cudaFree can synchronize the whole device), or a host
// framework that owns all device memory through its own pool and budget,
// where a hidden allocation would fail or fragment it.  The regular
// ncc_sat_build allocates its look-back workspace on first use; this entry
// point instead uses a fixed scratch array compiled into the library.
//
// The scratch is one file-scope __device__ array of kScratchBytes (8 MiB).
// Every GPU that loads the library holds one copy until the process exits.
// Host code cannot use the array's name as a device address, so the first
// call on each device looks the address up with cudaGetSymbolAddress (that
// call allocates nothing) and caches it.  All calls on a device share the array and it keeps the
// last call's contents, so each call clears the part the kernel needs to
// start at zero; calls whose kernels overlap on the GPU (different streams,
// no ordering between them) race on the array and must be ordered by the
// caller.
#include "ncc_common.cuh"

#include <mutex>

namespace {

constexpr size_t kScratchBytes = 8u << 20;
static __device__ __align__(256) unsigned char g_sat_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

constexpr int kMaxW = 66051;        // a row's running sum of squares must fit uint32
constexpr uint64_t kTimeoutNs = 1000000000ull;

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const char *pa = static_cast<const char *>(a), *pb = static_cast<const char *>(b);
    return pa < pb + nb && pb < pa + na;
}

// Device address of the scratch array on the current device (looked up once
// per device).
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_sat_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

namespace ncc {
int status_word(int **out);  // defined with the other entry points
}

extern "C" int ncc_sat_build_noalloc(const uint8_t *img, int W, int H, int64_t *S, int64_t *Q,
                                     ncc_stream_t stream) {
    if (!img || !S || !Q || W <= 0 || H <= 0) return NCC_ERR_INVALID_ARG;
    if (W > kMaxW || (long long)W * H >= (1ll << 31)) return NCC_ERR_UNSUPPORTED;
    if ((uintptr_t)S % 8 || (uintptr_t)Q % 8) return NCC_ERR_INVALID_ARG;
    const size_t n = (size_t)W * H;
    if (overlaps(S, n * 8, Q, n * 8) || overlaps(S, n * 8, img, n) || overlaps(Q, n * 8, img, n))
        return NCC_ERR_INVALID_ARG;
    const ncc::SatPlan plan = ncc::sat_plan(W, H);
    if (plan.total_bytes > kScratchBytes) return NCC_ERR_UNSUPPORTED;  // beyond the fixed scratch

    int *status = nullptr;
    int rc = ncc::status_word(&status);
    if (rc != NCC_OK) return rc;
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return NCC_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // The previous call's look-back words are still in the array: clear the
    // whole region this image uses so every word reads as not yet published.
    if (cudaMemsetAsync(scratch, 0, plan.total_bytes, st) != cudaSuccess) return NCC_ERR_CUDA;
    const cudaError_t e = ncc::sat_launch(img, W, H, S, Q, scratch, plan, /*epoch=*/1u, status,
                                          kTimeoutNs, /*fault_tile=*/-1, st);
    return e == cudaSuccess ? NCC_OK : NCC_ERR_CUDA;
}
