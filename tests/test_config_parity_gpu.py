"""Parity of every named workload at its full size, in the launch
configuration the bench uses, against the oracle over the whole output.

For each workload: every coefficient within 1e-5 absolute of the oracle's
double, and the exact integer sums behind them -- SumI and SumI2 (the
four-corner box sums of section 15.8) and SumIT (Listing 15-5's numerator)
-- bit for bit, through ncc_correlate_moments.  Outputs are written over
NaN / poison-filled buffers, so a cell no kernel writes fails.

The 64-template bank is compared 16 templates at a time to bound host
memory (the oracle keeps per-template copies of its window sums).
"""
import numpy as np
import pytest

import oracle
from gpu_util import moments, nan_map, to_dev
from normalized_cross_correlation_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = 1e-5


def check_workload(ncc, threads, w, chunk=None):
    import torch
    dimg = to_dev(w.image)
    S, Q = ncc.ncc_sat_build(dimg)
    oS, oQ = oracle.sat(w.image)
    np.testing.assert_array_equal(S.cpu().numpy(), oS)
    np.testing.assert_array_equal(Q.cpu().numpy(), oQ)
    del oS, oQ
    dt = to_dev(w.templates)
    nT = w.nT
    out = nan_map(nT, w.Oy, w.Ox)
    if nT == 1:
        ncc.ncc_correlate(dimg, dt[0], S, Q, out=out[0])
    else:
        ncc.ncc_correlate_bank(dimg, dt, S, Q, out=out)
    assert ncc.ncc_sync_status() == ncc.NCC_OK
    sI, sI2, sIT = moments(ncc, dimg, dt, S, Q)
    del S, Q
    r = out.cpu().numpy()
    del out
    sI, sI2 = sI.cpu().numpy(), sI2.cpu().numpy()
    step = chunk or nT
    for t0 in range(0, nT, step):
        t1 = min(nT, t0 + step)
        ref, oI, oI2, oIT = oracle.correlate(w.image, w.templates[t0:t1], with_sums=True,
                                             threads=threads)
        np.testing.assert_allclose(r[t0:t1], ref, rtol=0, atol=TOL)
        np.testing.assert_array_equal(sIT[t0:t1].cpu().numpy(), oIT)
        if t0 == 0:
            np.testing.assert_array_equal(sI, oI[0])
            np.testing.assert_array_equal(sI2, oI2[0])
        del ref, oI, oI2, oIT
    assert np.all(np.abs(r) <= 1.0)
    for t, x, y in w.crops:
        assert abs(r[t, y, x] - 1.0) <= TOL
    torch.cuda.empty_cache()
    return r


def test_tiny_256_t16(ncc, threads):
    r = check_workload(ncc, threads, inputs.tiny_ncc())
    assert np.argmax(r[0]) == 37 * 241 + 100


def test_smooth_1024_t32(ncc, threads):
    check_workload(ncc, threads, inputs.smooth_1024())


def test_headline_4096_t16(ncc, threads):
    check_workload(ncc, threads, inputs.headline_4096())


def test_bank_2048_64x16(ncc, threads):
    r = check_workload(ncc, threads, inputs.bank_2048(), chunk=16)
    assert r.shape == (64, 2033, 2033)


def test_large_8192_t64(ncc, threads):
    r = check_workload(ncc, threads, inputs.large_8192())
    assert r.shape == (1, 8129, 8129)
    assert ncc.ncc_debug_last_path() == ncc.NCC_PATH_TOEPLITZ


def test_wide_4096_t128(ncc, threads):
    r = check_workload(ncc, threads, inputs.wide_4096())
    assert r.shape == (1, 3969, 3969)
    assert ncc.ncc_debug_last_path() == ncc.NCC_PATH_NTT
