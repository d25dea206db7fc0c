/*
 * ncc_debug.h -- test hooks of the GB300 normalized cross-correlation
 * library (libncc_gb300.so).  None of them computes anything: they inject
 * failures on the host (a look-back tile that never publishes, an
 * allocation that fails), select between the single-template kernels, and
 * report which kernel ran, so the tests can reach paths that a correct run
 * on a healthy GPU never takes.  The computing path is declared in ncc.h.
 * These are process-wide switches, not for concurrent use with other calls.
 */
#ifndef NCC_GB300_DEBUG_H
#define NCC_GB300_DEBUG_H

#include "ncc.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * ncc_debug_set_fault -- test hook for the bounded waits.  While
 * suppress_tile >= 0, the SAT builder's tile with that row-major index never
 * publishes its look-back results, so every tile that depends on it waits
 * until its limit (timeout_ns; 0 restores the default of one second) runs
 * out and records NCC_ERR_TIMEOUT.  suppress_tile = -1 restores normal
 * operation.  In the debug build (libncc_gb300_debug.so, compiled with
 * NCC_DEBUG), suppress_tile = -2 instead sends the table stores of tile 0
 * one row width to the left, before the start of S and Q, where the build's
 * index check must stop them and record NCC_ERR_BOUNDS; the regular build
 * refuses -2.
 * Process-wide; not for concurrent use.
 */
int ncc_debug_set_fault(int suppress_tile, uint64_t timeout_ns);

/*
 * ncc_debug_fail_alloc -- test hook for allocation failure.  The next
 * `count` device allocations the library makes (the SAT builder's look-back
 * workspace when it is first allocated or grown, the host-buffer path's
 * device buffers, the transform kernel's template spectrum) fail as on an exhausted device, so the calls that need
 * them return NCC_ERR_NOMEM and launch nothing.  count = 0 cancels the
 * failures still pending.  Process-wide; not for concurrent use.
 * Returns NCC_OK, or NCC_ERR_INVALID_ARG for a negative count.
 */
int ncc_debug_fail_alloc(int count);

/* Kernels a correlate call can launch (ncc_debug_last_path). */
enum ncc_path_code {
    NCC_PATH_NONE = 0,
    NCC_PATH_DP4A = 1,     /* single template, integer dot products         */
    /* 2 is not used (it named a tensor-core kernel that has been removed) */
    NCC_PATH_BANK = 3,     /* template bank, tcgen05 tensor cores            */
    NCC_PATH_TOEPLITZ = 4, /* single large template, tcgen05 Toeplitz product */
    NCC_PATH_NTT = 5       /* single large template, number-theoretic transforms */
};

/*
 * ncc_debug_set_path -- selects the single-template kernel that
 * ncc_correlate, ncc_correlate_moments, ncc_match and ncc_correlate_bank (for
 * banks the bank kernel does not take) use.  0 = automatic (see
 * ncc_correlate in ncc.h), NCC_PATH_DP4A = dp4a, NCC_PATH_TOEPLITZ = the
 * Toeplitz tensor-core kernel, NCC_PATH_NTT = the number-theoretic-transform
 * kernel; a forced kernel that does not apply to the template's shape makes
 * the call return NCC_ERR_UNSUPPORTED.  Process-wide; not for concurrent
 * use.  Returns NCC_OK, or NCC_ERR_INVALID_ARG for another value.
 */
int ncc_debug_set_path(int path);

/*
 * ncc_debug_last_path -- the kernel (ncc_path_code) launched by the most
 * recent successful correlate call of this process; NCC_PATH_NONE before
 * the first.
 */
int ncc_debug_last_path(void);

#ifdef __cplusplus
}
#endif

#endif /* NCC_GB300_DEBUG_H */
