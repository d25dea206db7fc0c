"""GPU parity of ncc_correlate (one template) against the oracle.

Integers (SumI, SumI2, SumIT) must match bit-exactly; coefficients within
1e-5 absolute (the fp32 result against the oracle's double).  Sizes span
several output tiles (128 x 32) with ragged tails; the full-size workloads
compare every coefficient (the largest ones in test_config_parity_gpu.py),
in the launch configuration the bench uses.  Every output is written over a
NaN-filled buffer, so a skipped cell fails.
"""
import numpy as np
import pytest

import oracle
from gpu_util import moments, nan_map, to_dev
from normalized_cross_correlation_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = 1e-5


def gpu_ncc(ncc, img, T):
    """Coefficients of one template, written over a NaN-filled map."""
    dimg = to_dev(img)
    S, Q = ncc.ncc_sat_build(dimg)
    out = nan_map(img.shape[0] - T.shape[0] + 1, img.shape[1] - T.shape[1] + 1)
    r = ncc.ncc_correlate(dimg, to_dev(T), S, Q, out=out)
    assert ncc.ncc_sync_status() == 0
    return r.cpu().numpy()


def gpu_moments(ncc, img, T):
    dimg = to_dev(img)
    S, Q = ncc.ncc_sat_build(dimg)
    sI, sI2, sIT = moments(ncc, dimg, to_dev(T), S, Q)
    return sI.cpu().numpy(), sI2.cpu().numpy(), sIT.cpu().numpy()


CASES = [  # (W, H, wT, hT)
    (40, 30, 1, 1), (50, 41, 3, 5), (300, 200, 16, 16), (257, 190, 17, 9),
    (400, 333, 32, 32), (600, 300, 64, 64), (129, 77, 129, 1), (93, 150, 1, 150),
    (64, 64, 64, 64), (1000, 260, 13, 31), (272, 96, 100, 40), (513, 70, 128, 20),
    # grouped table-row loads: partial last block of 4*hT rows, views shifted by H mod hT
    (512, 300, 12, 7), (256, 157, 8, 15), (320, 133, 20, 2),
    # 16-row templates on the TMA path (compile-time height), ragged last tiles
    (528, 200, 16, 16), (256, 100, 5, 16), (1024, 131, 16, 16),
]


@pytest.mark.parametrize("W,H,wT,hT", CASES)
def test_moments_bit_exact(ncc, threads, W, H, wT, hT):
    w = inputs.random_case(W * 31 + H, W, H, wT, hT, nT=1, n_crops=1)
    sI, sI2, sIT = gpu_moments(ncc, w.image, w.templates[0])
    _, oI, oI2, oIT = oracle.correlate(w.image, w.templates[0], with_sums=True, threads=threads)
    np.testing.assert_array_equal(sI, oI)
    np.testing.assert_array_equal(sI2, oI2)
    np.testing.assert_array_equal(sIT[0], oIT)


@pytest.mark.parametrize("W,H,wT,hT", CASES)
def test_coefficients_match_oracle(ncc, threads, W, H, wT, hT):
    w = inputs.random_case(W * 17 + H, W, H, wT, hT, nT=1, n_crops=1)
    r = gpu_ncc(ncc, w.image, w.templates[0])
    ref = oracle.correlate(w.image, w.templates[0], threads=threads)
    assert r.shape == ref.shape
    np.testing.assert_allclose(r, ref, rtol=0, atol=TOL)
    _, x, y = w.crops[0]
    if wT * hT > 1:                                  # a 1-pixel template has zero variance
        assert abs(r[y, x] - 1.0) <= TOL
    assert np.all(np.abs(r) <= 1.0)


def test_tiny_workload_full_map(ncc, threads):
    w = inputs.tiny_ncc()
    r = gpu_ncc(ncc, w.image, w.templates[0])
    ref = oracle.correlate(w.image, w.templates[0], threads=threads)
    assert r.shape == (241, 241)
    np.testing.assert_allclose(r, ref, rtol=0, atol=TOL)
    assert abs(r[37, 100] - 1.0) <= TOL
    assert np.argmax(r) == 37 * 241 + 100


def test_smooth_1024_full_map(ncc, threads):
    w = inputs.smooth_1024()
    r = gpu_ncc(ncc, w.image, w.templates[0])
    ref = oracle.correlate(w.image, w.templates[0], threads=threads)
    assert r.shape == (993, 993)
    np.testing.assert_allclose(r, ref, rtol=0, atol=TOL)


def test_headline_4096_full_map(ncc, threads):
    w = inputs.headline_4096()
    r = gpu_ncc(ncc, w.image, w.templates[0])
    ref = oracle.correlate(w.image, w.templates[0], threads=threads)
    np.testing.assert_allclose(r, ref, rtol=0, atol=TOL)
    _, x, y = w.crops[0]
    assert abs(r[y, x] - 1.0) <= TOL


def test_zero_variance_windows_and_templates(ncc):
    rng = np.random.default_rng(3)
    img = rng.integers(0, 256, (200, 300), dtype=np.uint8)
    img[50:90, 60:140] = 77                          # constant patch
    T = rng.integers(0, 256, (16, 16), dtype=np.uint8)
    r = gpu_ncc(ncc, img, T)
    assert np.all(r[50:75, 60:125] == 0.0)
    flat = np.full((16, 16), 5, np.uint8)
    assert np.all(gpu_ncc(ncc, img, flat) == 0.0)


def test_negated_crop_is_minus_one(ncc):
    w = inputs.tiny_ncc()
    r = gpu_ncc(ncc, w.image, (255 - w.templates[0]).astype(np.uint8))
    assert abs(r[37, 100] + 1.0) <= TOL
    assert np.argmin(r) == 37 * 241 + 100


def test_single_shift_and_single_pixel(ncc):
    rng = np.random.default_rng(4)
    img = rng.integers(0, 256, (37, 53), dtype=np.uint8)
    r = gpu_ncc(ncc, img, img.copy())               # template = whole image: one shift
    assert r.shape == (1, 1) and abs(r[0, 0] - 1.0) <= TOL
    one = np.array([[9]], np.uint8)
    r = gpu_ncc(ncc, one, one)                       # 1-pixel image: zero variance
    assert r.shape == (1, 1) and r[0, 0] == 0.0


def test_unaligned_image_rows_use_the_fallback_loader(ncc, threads):
    # W % 16 != 0 cannot be described by a TMA tensor map
    w = inputs.random_case(8, 1001, 123, 16, 16, nT=1, n_crops=1)
    r = gpu_ncc(ncc, w.image, w.templates[0])
    ref = oracle.correlate(w.image, w.templates[0], threads=threads)
    np.testing.assert_allclose(r, ref, rtol=0, atol=TOL)


def test_unsupported_template_is_rejected_not_miscomputed(ncc):
    import torch
    img = torch.zeros((300, 300), dtype=torch.uint8, device="cuda")
    S, Q = ncc.ncc_sat_build(img)
    T = torch.zeros((300, 300), dtype=torch.uint8, device="cuda")
    with pytest.raises(ncc.NccError) as e:
        ncc.ncc_correlate(img, T, S, Q)
    assert e.value.code == ncc.NCC_ERR_UNSUPPORTED


def test_host_entry_point_matches_device_path(ncc):
    import torch
    w = inputs.random_case(77, 700, 300, 16, 16, nT=1, n_crops=1)
    dev = gpu_ncc(ncc, w.image, w.templates[0])
    img = torch.from_numpy(w.image).pin_memory()
    T = torch.from_numpy(w.templates).pin_memory()
    out = torch.empty((1,) + dev.shape, dtype=torch.float32).pin_memory()
    ncc.ncc_match_host(img, T, out)
    np.testing.assert_array_equal(out[0].numpy(), dev)
