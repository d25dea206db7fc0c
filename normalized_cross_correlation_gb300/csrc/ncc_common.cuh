// ncc_common.cuh -- small device helpers and launch interfaces shared by the
// library's translation units (inline PTX for the memory-model operations,
// the bounded look-back wait, and the host launchers' declarations).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ncc.h"
#include "../../include/ncc_debug.h"

namespace ncc {

// ---------------------------------------------------------------------------
// Memory-model helpers (PTX ISA: ld.acquire / st.release at GPU scope).
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned ld_relaxed_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Records the first error of a launch sequence in the per-device status word.
__device__ __forceinline__ void record_status(int *status, int code) {
    atomicCAS(status, 0, code);
}

// Index checks of the debug build (compiled with -DNCC_DEBUG): NCC_BOUNDS(c,
// status) is true when c holds; when it does not, it records NCC_ERR_BOUNDS
// in the status word and is false, so the caller skips the access.  In the
// regular build it is the constant true and costs nothing.
#ifdef NCC_DEBUG
#define NCC_BOUNDS(cond, status) \
    ((cond) ? true : (::ncc::record_status((status), NCC_ERR_BOUNDS), false))
#else
#define NCC_BOUNDS(cond, status) true
#endif

// Look-back flag states (section 15.8's three-state protocol).
enum : unsigned { FLAG_EMPTY = 0u, FLAG_AGGREGATE = 1u, FLAG_PREFIX = 2u };

// Waits until *flag leaves FLAG_EMPTY and returns its state.  The wait is
// bounded twice: by `timeout_ns` of %globaltimer since `t0`, and by an
// iteration cap.  It also gives up when another CTA has raised *abort.  On
// giving up it raises *abort, records NCC_ERR_TIMEOUT and returns
// FLAG_EMPTY, so the caller can leave without publishing anything.
__device__ __forceinline__ unsigned wait_flag(const unsigned *flag, unsigned *abort,
                                              int *status, uint64_t t0,
                                              uint64_t timeout_ns) {
    unsigned f = ld_acquire_gpu(flag);
    if (f != FLAG_EMPTY) return f;
    unsigned backoff = 32;
    for (unsigned it = 1;; ++it) {
        __nanosleep(backoff);
        if (backoff < 256) backoff <<= 1;
        f = ld_acquire_gpu(flag);
        if (f != FLAG_EMPTY) return f;
        if ((it & 7u) == 0u) {
            if (ld_relaxed_gpu(abort) != 0u) return FLAG_EMPTY;
            if (global_timer_ns() - t0 > timeout_ns || it > (1u << 26)) {
                atomicExch(abort, 1u);
                record_status(status, NCC_ERR_TIMEOUT);
                return FLAG_EMPTY;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Tensor maps for TMA: the driver's cuTensorMapEncodeTiled, looked up once
// through the runtime (null when the driver does not provide it).
// ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn tensor_map_encoder() {
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(ptr);
        return nullptr;
    }();
    return fn;
}

// A 2-D row-major tensor map: `elem` bytes per element, dims {W, H}, row
// stride W*elem bytes, box {boxW, boxH}, no swizzle, zero fill outside.
inline bool make_tensor_map_2d(CUtensorMap *map, CUtensorMapDataType type, int elem,
                               const void *base, int W, int H, int boxW, int boxH) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)W, (cuuint64_t)H};
    const cuuint64_t strides[1] = {(cuuint64_t)W * (cuuint64_t)elem};
    const cuuint32_t box[2] = {(cuuint32_t)boxW, (cuuint32_t)boxH};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, type, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// Library-owned device memory (defined in ncc_api.cu).
// ---------------------------------------------------------------------------

// Stream-ordered allocation from the library's per-device pool, whose
// release threshold keeps freed memory reserved for the next request.  While
// the allocation-failure test hook (ncc_debug_fail_alloc) has failures left,
// it fails with cudaErrorMemoryAllocation as an exhausted device would.
cudaError_t pool_alloc(void **ptr, size_t bytes, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Host launchers (defined in the kernel translation units).
// ---------------------------------------------------------------------------

// Summed-area tables: tiling and look-back workspace size for an image.
struct SatPlan {
    int tile_w, tile_h;     // tile shape in pixels
    int ntx, nty;           // tiles per row / per column
    size_t zero_bytes;      // leading bytes of the workspace that must start at zero
    size_t total_bytes;     // whole workspace
};
SatPlan sat_plan(int W, int H);
// One launch of the builder on a caller-provided workspace whose first
// zero_bytes are zero (a launch leaves them zero again when it ends).
// `epoch` (1..31) tags this call's look-back words.
cudaError_t sat_launch(const uint8_t *img, int W, int H, int64_t *S, int64_t *Q,
                       void *workspace, const SatPlan &plan, uint32_t epoch, int *status,
                       uint64_t timeout_ns, int fault_tile, cudaStream_t stream);
// The naive and two-pass builders of the SAT ladder (variant NCC_SAT_NAIVE
// or NCC_SAT_TWO_PASS), on their own per-device workspace.
cudaError_t sat_ladder_run(int variant, const uint8_t *img, int W, int H, int64_t *S, int64_t *Q,
                           int *status, uint64_t timeout_ns, cudaStream_t stream);
// The builder on the library's per-device workspace (allocated on first use).
cudaError_t sat_build_run(const uint8_t *img, int W, int H, int64_t *S, int64_t *Q,
                          int *status, uint64_t timeout_ns, int fault_tile,
                          cudaStream_t stream);

// Single-template correlation (dp4a numerator + fused box-sum epilogue).
struct CorrArgs {
    const uint8_t *img;
    int W, H;
    const uint8_t *tmpl;
    int wT, hT;
    const int64_t *S, *Q;
    float *out;                 // coefficients (null when moments are requested)
    int64_t *sumI, *sumI2, *sumIT;  // moments (all null unless requested)
    int *status;                // per-device status word
    // Launch with programmatic stream serialization: the kernel may start
    // while the previous kernel on the stream (the SAT build, which lets its
    // dependents start) is still running; it reads only img and tmpl before
    // it waits on that grid, and S and Q after.  Only for a previous kernel
    // that writes neither img nor tmpl.
    bool overlap_prev = false;
    // Window moments from the staged image tile (sliding column sums and row
    // prefixes in shared memory) instead of from S and Q, which are unused.
    bool direct = false;
    // Output rows [rowBegin, rowEnd) only (rowEnd 0: through the last row);
    // dp4a kernel only.  rowBegin and, unless it is the map's last row,
    // rowEnd must be multiples of kCorrBandRows.  The tables and the image
    // are still the whole map's.
    int rowBegin = 0, rowEnd = 0;
};
// Band edges for CorrArgs::rowBegin / rowEnd: a multiple of every tile
// height of the dp4a kernel (32 and 64 rows).
constexpr int kCorrBandRows = 64;
// Multiprocessors of the current device (cached per device).
int sm_count();
bool corr_dp4a_supported(int wT, int hT);
// The same with direct window moments (CorrArgs::direct): wT <= 129.
bool corr_dp4a_direct_supported(int wT, int hT);
cudaError_t corr_dp4a_launch(const CorrArgs &a, cudaStream_t stream);
// The same as a Toeplitz matrix product on the tensor cores (tcgen05, exact
// centered f16 operands, fp32 accumulation in groups of at most 1024
// products): wT <= 65 and a tile that fits two CTAs per SM.  Honours
// CorrArgs::overlap_prev; no direct moments.
bool corr_toeplitz_supported(int wT, int hT);
cudaError_t corr_toeplitz_launch(const CorrArgs &a, cudaStream_t stream);
// The same with the numerator from number-theoretic transforms of 256 x 256
// tiles (exact modulo a prime): wT, hT <= 224 and wT * hT <= 30000.  Plain
// stream order; no direct moments.  Allocates the template's spectrum
// (512 KB) from the library's stream-ordered pool for the duration of the
// call.
bool corr_ntt_supported(int wT, int hT);
cudaError_t corr_ntt_launch(const CorrArgs &a, cudaStream_t stream);

// Template-bank correlation on the tensor cores (tcgen05, f16 operands,
// fp32 accumulation; exact while wT*hT*255^2 < 2^24).
struct BankArgs {
    const uint8_t *img;
    int W, H;
    const uint8_t *tmpl;
    int wT, hT, nT;
    const int64_t *S, *Q;
    float *out;
    int64_t *sumI, *sumI2, *sumIT;
    int *status;
};
bool bank_tc_supported(int W, int H, int wT, int hT, int nT);
cudaError_t bank_tc_launch(const BankArgs &a, cudaStream_t stream);

}  // namespace ncc
