/*
 * ncc.h -- C ABI of the GB300 (sm_103a) normalized cross-correlation library.
 *
 * Normalized cross-correlation (NCC) template matching of an 8-bit image
 * against 8-bit templates, after The CUDA Handbook, chapter 15 ("Image
 * Processing: Normalized Correlation"):
 *   - the denominators' first and second moments come from two inclusive
 *     int64 summed-area tables, S of I and Q of I^2, read with the
 *     four-corner box sum (section 15.8, "The Denominator: Summed Area
 *     Tables", Figure 15-7);
 *   - the numerator SumIT is swept over every valid shift and combined with
 *     the moments into one coefficient per shift ("Image in shared memory",
 *     Listing 15-5).
 *
 * Coefficient (the listing names the routine but does not print its body;
 * this library takes Pearson's correlation in exact-integer form):
 *     N   = wT*hT
 *     num = N*SumIT - SumI*SumT
 *     vI  = N*SumI2 - SumI^2,    vT = N*SumT2 - SumT^2
 *     r   = num / sqrt(vI*vT)    (0 when vI == 0 or vT == 0; clamped to [-1,1])
 * num, vI and vT are exact 64-bit integers; r is rounded to fp32.
 *
 * Conventions shared by every entry point:
 *   - Images are dense row-major uint8 [H][W] (row stride W bytes).
 *     Templates are dense uint8 [nT][hT][wT].  Tables are dense int64 [H][W].
 *   - Valid shifts only: Ox = W-wT+1 columns, Oy = H-hT+1 rows.  Coefficient
 *     maps are dense fp32 [nT][Oy][Ox]; out[t][y][x] belongs to the window of
 *     template t whose top-left image pixel is (x, y).
 *   - Unless an entry point says otherwise, every pointer is a DEVICE pointer
 *     owned by the caller.  The library never frees caller memory and keeps
 *     no reference to it after the call returns.
 *   - Calls are asynchronous and ordered on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) on the current CUDA device.  The return
 *     value covers argument checks, workspace allocation and launch errors
 *     only.  Errors found by a kernel while it runs (a look-back wait that
 *     ran out) are recorded in a per-device status word and reported by
 *     ncc_sync_status().
 *   - Limits: 1 <= W <= 66051 (a row's running sum of squares must fit in
 *     uint32: 66051 * 255^2 < 2^32), 1 <= H, W*H < 2^31, and
 *     wT*hT <= 66051 (the numerator is accumulated in uint32).  Larger
 *     inputs return NCC_ERR_UNSUPPORTED rather than wrong results.
 */
#ifndef NCC_GB300_H
#define NCC_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *ncc_stream_t;

/* Status codes (0 = success, negative = failure). */
enum ncc_status_code {
    NCC_OK = 0,
    NCC_ERR_INVALID_ARG = -1,  /* null/misaligned pointer, bad size, aliasing  */
    NCC_ERR_UNSUPPORTED = -2,  /* valid request outside the library's limits  */
    NCC_ERR_CUDA = -3,         /* a CUDA runtime call or launch failed         */
    NCC_ERR_TIMEOUT = -4,      /* a kernel's bounded wait ran out (device)     */
    NCC_ERR_NOMEM = -5,        /* stream-ordered workspace allocation failed   */
    NCC_ERR_BOUNDS = -6        /* a debug build's index check failed (device)  */
};

/*
 * ncc_sat_build -- the two summed-area tables of section 15.8.
 *   S[y][x] = sum_{j<=y, i<=x} I[j][i],  Q[y][x] = sum_{j<=y, i<=x} I[j][i]^2
 * (inclusive; int64 because the totals pass 2^31 by a 512x512 image; each
 * row's running sums fit uint32, as the section notes).
 *   img  device, uint8 [H][W], read only.
 *   S, Q device, int64 [H][W], written completely; 8-byte aligned; must not
 *        overlap each other or img.
 * Single pass: a decoupled look-back scan over tiles, handed out in
 * row-major order so that every wait points at an earlier tile.  The
 * look-back state lives in a per-device workspace owned by the library: it
 * is allocated (cudaMalloc) on the first call on a device and whenever a
 * larger image needs more room, and reused afterwards without clearing.  Calls on different
 * streams are ordered through an event so they never share it concurrently.
 * The build kernel lets a kernel launched after it with programmatic stream
 * serialization start before it ends (ncc_match uses this); such a kernel
 * must wait on the grid dependency before it reads S or Q.  Ordinary
 * stream order is unaffected.
 * Returns NCC_OK, NCC_ERR_INVALID_ARG, NCC_ERR_UNSUPPORTED, NCC_ERR_NOMEM or
 * NCC_ERR_CUDA.
 */
int ncc_sat_build(const uint8_t *img, int W, int H, int64_t *S, int64_t *Q,
                  ncc_stream_t stream);

/*
 * ncc_sat_build_variant -- the same tables by one of the builders that
 * section 15.8 compares (Figures 15-8 and 15-9), for measuring that
 * comparison on this GPU.  variant:
 *   NCC_SAT_FUSED     the single-pass tiled look-back of ncc_sat_build (the
 *                     product path; this call is ncc_sat_build);
 *   NCC_SAT_NAIVE     one thread per image row writes the rows' running sums
 *                     into S and Q, then one thread per column adds down its
 *                     column in place;
 *   NCC_SAT_TWO_PASS  row running sums to a uint32 intermediate, then a
 *                     column scan with a decoupled look-back over stripes of
 *                     128 rows (no transposes).
 *   Arguments, layouts and results as ncc_sat_build; NCC_ERR_INVALID_ARG for
 *   an unknown variant.  The two-pass builder allocates (cudaMalloc) a
 *   per-device workspace of 8 bytes per pixel plus its look-back words on
 *   first use and when a larger image needs more; it is kept for later calls
 *   and is not safe against concurrent calls on other streams.  Look-back
 *   waits that run out record NCC_ERR_TIMEOUT for ncc_sync_status.
 */
enum ncc_sat_variant { NCC_SAT_FUSED = 0, NCC_SAT_NAIVE = 1, NCC_SAT_TWO_PASS = 2 };
int ncc_sat_build_variant(const uint8_t *img, int W, int H, int64_t *S, int64_t *Q, int variant,
                          ncc_stream_t stream);

/*
 * ncc_sat_build_noalloc -- ncc_sat_build for callers that cannot allocate
 * device memory (the pages have no counterpart: it is an interface
 * addition).  Callers inside a host callback or a real-time loop cannot let
 * a library call cudaMalloc/cudaFree, which may synchronize the whole
 * device; a framework that owns every device allocation through its own
 * pool cannot let a library allocate behind its budget.  This
 * entry point allocates nothing: its look-back scratch is a fixed 8 MiB
 * array compiled into the library, which every GPU that loads the library
 * holds until the process exits.
 *   Arguments, layouts, results and errors as ncc_sat_build, plus:
 *   NCC_ERR_UNSUPPORTED when the image needs more scratch than 8 MiB, i.e.
 *   when ceil(W/128) * ceil(H/128) > 2729 tiles (4096x4096 fits; 8192x8192
 *   does not).
 * The first call on a device looks up the scratch array's device address
 * (cudaGetSymbolAddress, which allocates nothing).  All calls on a device
 * share the array and each clears what it needs to start at zero;
 * calls whose kernels overlap on the GPU race on it, so order them (one
 * stream, or events).
 */
int ncc_sat_build_noalloc(const uint8_t *img, int W, int H, int64_t *S,
                          int64_t *Q, ncc_stream_t stream);

/*
 * ncc_correlate -- one template, every valid shift (Listing 15-5's sums,
 * section 15.8's box sums, the coefficient above).
 *   img  device uint8 [H][W].
 *   tmpl device uint8 [hT][wT].
 *   S, Q device int64 [H][W]: must hold ncc_sat_build(img) output, ordered
 *        before this call (same stream, or an event).
 *   out  device fp32 [Oy][Ox], written completely; must not overlap inputs.
 * Kernels: the integer dot-product (dp4a) numerator; for templates up to 65
 * pixels wide whose dp4a numerator would take at least 96 dp4a per output,
 * ceil(wT/4)*hT (about 20x20 and up; 320, about 40x40, on maps of fewer than
 * 4M shifts), a tensor-core numerator (tcgen05) that writes the sums over 64
 * consecutive shifts as one matrix product with a Toeplitz factor, from exact
 * centered f16 operands (pixel and template value minus 128) accumulated in
 * fp32 groups of at most 1024 products; for templates that kernel cannot
 * take (wider than 65, or too tall for its accumulator groups) up to
 * 224 x 224 and 30000 pixels, from 320 dp4a per output, a numerator from
 * number-theoretic transforms of 256 x 256 image tiles (section 15.8's FFT
 * numerator, computed modulo the prime 998244353, which makes it exact;
 * centered values as above), which allocates the template's 512 KB spectrum
 * from the library's stream-ordered pool for the duration of the call.  All
 * produce the same integer sums and the same coefficients.
 * Returns NCC_OK, NCC_ERR_INVALID_ARG, NCC_ERR_UNSUPPORTED, NCC_ERR_NOMEM
 * (the spectrum could not be allocated) or NCC_ERR_CUDA.
 */
int ncc_correlate(const uint8_t *img, int W, int H, const uint8_t *tmpl,
                  int wT, int hT, const int64_t *S, const int64_t *Q,
                  float *out, ncc_stream_t stream);

/*
 * ncc_correlate_bank -- nT templates of one size against one image; one SAT
 * pair serves every template of the bank (section 15.8).
 *   tmpl device uint8 [nT][hT][wT];  out device fp32 [nT][Oy][Ox].
 *   Other arguments as ncc_correlate.  1 <= nT.
 * Returns as ncc_correlate.
 */
int ncc_correlate_bank(const uint8_t *img, int W, int H, const uint8_t *tmpl,
                       int wT, int hT, int nT, const int64_t *S,
                       const int64_t *Q, float *out, ncc_stream_t stream);

/*
 * ncc_correlate_moments -- the exact integer sums behind the coefficients,
 * for verification: per shift SumI and SumI2 (from S and Q by the
 * four-corner box sum) and per template and shift SumIT (Listing 15-5).
 *   sumI, sumI2 device int64 [Oy][Ox];  sumIT device int64 [nT][Oy][Ox].
 *   Other arguments as ncc_correlate_bank; the same kernels compute the
 *   numerator as in ncc_correlate (nT == 1) or ncc_correlate_bank (nT > 1).
 * Returns as ncc_correlate.
 */
int ncc_correlate_moments(const uint8_t *img, int W, int H,
                          const uint8_t *tmpl, int wT, int hT, int nT,
                          const int64_t *S, const int64_t *Q, int64_t *sumI,
                          int64_t *sumI2, int64_t *sumIT, ncc_stream_t stream);

/*
 * ncc_correlate_direct -- the coefficients of nT templates without summed-area
 * tables: the window moments SumI and SumI2 come from the image tile the
 * numerator stages in shared memory, as the shared-memory kernel of chapter
 * 15 (Listing 15-5) forms its window sums from the staged image.  Per pass of
 * 16 output rows: sliding sums of I and I^2 down each tile column over hT
 * rows, then exclusive prefix sums along each row; a window's sum is the
 * difference of two prefixes (exact in wrapping 32-bit arithmetic).
 *   img, tmpl, out, sizes and stream as ncc_correlate_bank; no S or Q.
 *   wT <= 129.  Each template is one launch of the single-template kernel.
 * The integer moments and the arithmetic are those of ncc_correlate, so for
 * one template the coefficients equal ncc_correlate's bit for bit.
 * Returns as ncc_correlate; NCC_ERR_UNSUPPORTED for wT > 129.
 */
int ncc_correlate_direct(const uint8_t *img, int W, int H, const uint8_t *tmpl,
                         int wT, int hT, int nT, float *out, ncc_stream_t stream);

/*
 * ncc_correlate_direct_moments -- the exact integer sums behind
 * ncc_correlate_direct, for verification: sumI, sumI2 device int64
 * [Oy][Ox] and sumIT device int64 [nT][Oy][Ox], as ncc_correlate_moments.
 */
int ncc_correlate_direct_moments(const uint8_t *img, int W, int H,
                                 const uint8_t *tmpl, int wT, int hT, int nT,
                                 int64_t *sumI, int64_t *sumI2, int64_t *sumIT,
                                 ncc_stream_t stream);

/*
 * ncc_match -- the whole path on device buffers: ncc_sat_build(img) into S
 * and Q, then ncc_correlate_bank of the nT templates against them, ordered
 * on `stream` (the SAT serves the denominators and the templates' numerators
 * follow, as in section 15.8).  For a single template the correlation kernel
 * is launched with programmatic stream serialization: its CTAs may start as
 * the SAT build's CTAs retire and run their numerators (which read only img
 * and tmpl), and they wait for the build to finish before they read S or Q.
 * The results are those of the two separate calls, bit for bit.
 *   S, Q device int64 [H][W], written (caller-owned, as ncc_sat_build);
 *   other arguments as ncc_correlate_bank.  S and Q must not overlap img,
 *   tmpl, out or each other.
 * Returns as ncc_correlate_bank.
 */
int ncc_match(const uint8_t *img, int W, int H, const uint8_t *tmpl, int wT,
              int hT, int nT, int64_t *S, int64_t *Q, float *out,
              ncc_stream_t stream);

/*
 * ncc_match_host -- the whole path with HOST buffers: copies img and tmpl to
 * the device, runs ncc_match on them and brings the coefficients back, all
 * ordered on `stream`, then synchronizes it.
 *   img  host uint8 [H][W];  tmpl host uint8 [nT][hT][wT];
 *   out  host fp32 [nT][Oy][Ox].  Page-locked host memory makes the copies
 *   asynchronous and fast; pageable memory also works.
 * A single template whose map has at least 8 MB of coefficients and goes to
 * the dp4a kernel is correlated in up to 8 bands of output rows; each band
 * is copied back on a non-blocking stream that the library keeps per device
 * while the next band is correlated, and `stream` waits for those copies.
 * Other maps: when `out` is page-locked memory the device can address, the
 * kernels store the coefficients into it directly; otherwise they go to a
 * device buffer that is copied back.
 * Device buffers come from a stream-ordered pool that the library keeps per
 * device (memory freed to it stays reserved for the next call) and go back
 * to it before return.  Returns the first failure among the steps, including
 * any status recorded by the kernels (as ncc_sync_status would).
 */
int ncc_match_host(const uint8_t *img, int W, int H, const uint8_t *tmpl,
                   int wT, int hT, int nT, float *out, ncc_stream_t stream);

/*
 * ncc_sync_status -- synchronizes `stream`, then returns and clears the
 * current device's status word: NCC_OK, or the first error a kernel
 * recorded since the last call (NCC_ERR_TIMEOUT when a look-back wait ran
 * out).  The word is per device, shared by all streams on it.  Returns
 * NCC_ERR_CUDA if the synchronization itself fails.
 */
int ncc_sync_status(ncc_stream_t stream);

/* Static, human-readable text for a status code. */
const char *ncc_status_string(int status);

/* Library version, (major << 16) | minor. */
int ncc_version(void);

/* Test hooks (fault and allocation-failure injection, kernel selection)
 * are declared in ncc_debug.h; they are not part of the computing path. */

#ifdef __cplusplus
}
#endif

#endif /* NCC_GB300_H */
