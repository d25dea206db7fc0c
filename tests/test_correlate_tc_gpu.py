"""GPU parity of the tensor-core single-template path (tcgen05 numerator,
diagonal sums of per-row products, box-sum epilogue) against the oracle, and
against the dp4a path on the same inputs.

Integers (SumI, SumI2, SumIT) bit-exact; coefficients within 1e-5 absolute.
Shapes cover: templates shorter than the 16-row MMA width (zero rows), wider
than one 16-column K step, a wide segment (wT = 112), one-row and
one-column templates, images narrower than one 128-shift strip, images fewer
rows tall than one 8-row image box, and CTAs whose unit ranges cross strips
and hold one-row segments.
"""
import numpy as np
import pytest

import oracle
from normalized_cross_correlation_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = 1e-5

TC_CASES = [  # (W, H, wT, hT): W a multiple of 16, hT <= 16, wT*hT <= 258, wT <= 126
    (256, 64, 16, 16), (400, 150, 8, 8), (512, 100, 16, 1), (320, 90, 1, 16),
    (480, 77, 17, 9), (1024, 40, 112, 2), (144, 300, 32, 8), (208, 5, 10, 5),
    (4096, 24, 16, 16), (2048, 300, 5, 7), (128, 129, 15, 15), (16, 20, 3, 5),
]


def to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.fixture
def path(ncc):
    """Selects the tensor-core kernel; restores automatic selection after."""
    ncc.ncc_debug_set_path(ncc.NCC_PATH_TENSOR)
    yield ncc
    ncc.ncc_debug_set_path(0)


def run(ncc, img, T, moments):
    dimg = to_dev(img)
    S, Q = ncc.ncc_sat_build(dimg)
    if moments:
        res = ncc.ncc_correlate_moments(dimg, to_dev(T), S, Q)
        assert ncc.ncc_sync_status() == 0
        return tuple(a.cpu().numpy() for a in res)
    r = ncc.ncc_correlate(dimg, to_dev(T), S, Q)
    assert ncc.ncc_sync_status() == 0
    return r.cpu().numpy()


def expect_tensor_path(ncc, W, H):
    assert ncc.ncc_debug_last_path() == ncc.NCC_PATH_TENSOR


@pytest.mark.parametrize("W,H,wT,hT", TC_CASES)
def test_tc_moments_bit_exact(path, threads, W, H, wT, hT):
    ncc = path
    w = inputs.random_case(W * 13 + H + wT, W, H, wT, hT, nT=1, n_crops=1)
    sI, sI2, sIT = run(ncc, w.image, w.templates[0], moments=True)
    expect_tensor_path(ncc, W, H)
    _, oI, oI2, oIT = oracle.correlate(w.image, w.templates[0], with_sums=True, threads=threads)
    np.testing.assert_array_equal(sI, oI)
    np.testing.assert_array_equal(sI2, oI2)
    np.testing.assert_array_equal(sIT[0], oIT)


@pytest.mark.parametrize("W,H,wT,hT", TC_CASES)
def test_tc_coefficients_match_oracle_and_dp4a(path, threads, W, H, wT, hT):
    ncc = path
    w = inputs.random_case(W * 7 + H + hT, W, H, wT, hT, nT=1, n_crops=1)
    r = run(ncc, w.image, w.templates[0], moments=False)
    expect_tensor_path(ncc, W, H)
    ref = oracle.correlate(w.image, w.templates[0], threads=threads)
    assert r.shape == ref.shape
    np.testing.assert_allclose(r, ref, rtol=0, atol=TOL)
    _, x, y = w.crops[0]
    if wT * hT > 1:
        assert abs(r[y, x] - 1.0) <= TOL
    assert np.all(np.abs(r) <= 1.0)
    ncc.ncc_debug_set_path(ncc.NCC_PATH_DP4A)
    r2 = run(ncc, w.image, w.templates[0], moments=False)
    assert ncc.ncc_debug_last_path() == ncc.NCC_PATH_DP4A
    np.testing.assert_allclose(r, r2, rtol=0, atol=TOL)
    ncc.ncc_debug_set_path(0)
    run(ncc, w.image, w.templates[0], moments=False)
    assert ncc.ncc_debug_last_path() == ncc.NCC_PATH_DP4A     # automatic choice


def test_tc_zero_variance_and_negated_crop(path):
    ncc = path
    rng = np.random.default_rng(21)
    img = rng.integers(0, 256, (200, 320), dtype=np.uint8)
    img[50:90, 64:160] = 77                           # constant patch
    T = img[120:136, 200:216].copy()
    r = run(ncc, img, T, moments=False)
    assert ncc.ncc_debug_last_path() == ncc.NCC_PATH_TENSOR
    assert np.all(r[50:75, 64:145] == 0.0)
    assert abs(r[120, 200] - 1.0) <= TOL
    rn = run(ncc, img, (255 - T).astype(np.uint8), moments=False)
    assert abs(rn[120, 200] + 1.0) <= TOL
    flat = np.full((16, 16), 5, np.uint8)
    assert np.all(run(ncc, img, flat, moments=False) == 0.0)


def test_headline_workload_on_the_tensor_path(path, threads):
    ncc = path
    w = inputs.headline_4096()
    r = run(ncc, w.image, w.templates[0], moments=False)
    assert ncc.ncc_debug_last_path() == ncc.NCC_PATH_TENSOR
    _, x, y = w.crops[0]
    assert abs(r[y, x] - 1.0) <= TOL
    rng = np.random.default_rng(31)
    rows = np.concatenate([[0, 4080], rng.integers(0, 4081, 6)])
    for yy in rows:
        ref = oracle.correlate_at(w.image, w.templates[0], np.arange(4081), np.full(4081, yy),
                                  threads=threads)
        np.testing.assert_allclose(r[yy], ref, rtol=0, atol=TOL)


def test_forced_tensor_path_rejects_shapes_it_cannot_take(path):
    import torch
    ncc = path
    img = torch.zeros((100, 300), dtype=torch.uint8, device="cuda")   # W % 16 != 0
    S, Q = ncc.ncc_sat_build(img)
    T = torch.zeros((16, 16), dtype=torch.uint8, device="cuda")
    with pytest.raises(ncc.NccError) as e:
        ncc.ncc_correlate(img, T, S, Q)
    assert e.value.code == ncc.NCC_ERR_UNSUPPORTED
    img = torch.zeros((100, 320), dtype=torch.uint8, device="cuda")
    S, Q = ncc.ncc_sat_build(img)
    T = torch.zeros((17, 16), dtype=torch.uint8, device="cuda")       # hT > 16
    with pytest.raises(ncc.NccError) as e:
        ncc.ncc_correlate(img, T, S, Q)
    assert e.value.code == ncc.NCC_ERR_UNSUPPORTED
    assert ncc.ncc_sync_status() == 0
