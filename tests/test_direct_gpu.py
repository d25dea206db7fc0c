"""GPU parity of the direct-moment correlation (ncc_correlate_direct): the
window moments come from the staged image tile instead of the summed-area
tables.

SumI, SumI2 and SumIT must match the oracle bit-exactly; the coefficients
must equal ncc_correlate's (the same integers through the same arithmetic)
bit for bit, and so lie within 1e-5 absolute of the oracle's.  Shapes span
several output tiles and passes, ragged edges, the plain-load path (rows not
a multiple of 16 bytes), 1-pixel and 1-row templates and the widest template
the direct kernel takes (129).
"""
import numpy as np
import pytest

import oracle
from gpu_util import moments, nan_map, to_dev
from normalized_cross_correlation_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = 1e-5

CASES = [  # (W, H, wT, hT)
    (40, 30, 1, 1), (50, 41, 3, 5), (300, 200, 16, 16), (257, 190, 17, 9),
    (400, 333, 32, 32), (600, 300, 64, 64), (129, 77, 129, 1), (93, 150, 1, 150),
    (64, 64, 64, 64), (1000, 260, 13, 31), (272, 96, 100, 40), (513, 70, 128, 20),
    (528, 200, 16, 16), (256, 100, 5, 16), (1024, 131, 16, 16), (640, 97, 7, 3),
]


@pytest.mark.parametrize("W,H,wT,hT", CASES)
def test_direct_moments_bit_exact(ncc, threads, W, H, wT, hT):
    w = inputs.random_case(W * 13 + H, W, H, wT, hT, nT=1, n_crops=1)
    sI, sI2, sIT = moments(ncc, to_dev(w.image), to_dev(w.templates), direct=True)
    _, oI, oI2, oIT = oracle.correlate(w.image, w.templates[0], with_sums=True, threads=threads)
    np.testing.assert_array_equal(sI.cpu().numpy(), oI)
    np.testing.assert_array_equal(sI2.cpu().numpy(), oI2)
    np.testing.assert_array_equal(sIT.cpu().numpy()[0], oIT)


@pytest.mark.parametrize("W,H,wT,hT", CASES)
def test_direct_coefficients_equal_the_table_path(ncc, threads, W, H, wT, hT):
    w = inputs.random_case(W * 19 + H, W, H, wT, hT, nT=1, n_crops=1)
    dimg, dt = to_dev(w.image), to_dev(w.templates)
    r = ncc.ncc_correlate_direct(dimg, dt, out=nan_map(1, w.Oy, w.Ox))
    S, Q = ncc.ncc_sat_build(dimg)
    r0 = ncc.ncc_correlate(dimg, dt[0], S, Q, out=nan_map(w.Oy, w.Ox))
    assert ncc.ncc_sync_status() == 0
    np.testing.assert_array_equal(r.cpu().numpy()[0], r0.cpu().numpy())
    ref = oracle.correlate(w.image, w.templates[0], threads=threads)
    np.testing.assert_allclose(r.cpu().numpy()[0], ref, rtol=0, atol=TOL)
    _, x, y = w.crops[0]
    if wT * hT > 1:
        assert abs(float(r[0, y, x]) - 1.0) <= TOL


def test_direct_headline_4096_equals_the_table_path(ncc):
    """The bench's workload, in the launch configuration the bench times."""
    w = inputs.headline_4096()
    dimg, dt = to_dev(w.image), to_dev(w.templates)
    r = ncc.ncc_correlate_direct(dimg, dt, out=nan_map(1, w.Oy, w.Ox))
    S, Q, r0 = ncc.ncc_match(dimg, dt, out=nan_map(1, w.Oy, w.Ox))
    assert ncc.ncc_sync_status() == 0
    np.testing.assert_array_equal(r.cpu().numpy(), r0.cpu().numpy())


def test_direct_bank_matches_oracle(ncc, threads):
    w = inputs.random_case(31, 300, 170, 12, 10, nT=5, n_crops=2)
    r = ncc.ncc_correlate_direct(to_dev(w.image), to_dev(w.templates),
                                 out=nan_map(5, w.Oy, w.Ox)).cpu().numpy()
    assert ncc.ncc_sync_status() == 0
    for t in range(5):
        ref = oracle.correlate(w.image, w.templates[t], threads=threads)
        np.testing.assert_allclose(r[t], ref, rtol=0, atol=TOL)


def test_direct_zero_variance_and_saturated(ncc):
    """Flat windows give 0; a saturated image (sums at their largest) stays
    exact: a crop of it correlates to 1."""
    img = np.full((200, 300), 255, np.uint8)
    img[50:120, 60:200] = np.random.default_rng(5).integers(0, 256, (70, 140), dtype=np.uint8)
    T = img[60:76, 100:116].copy()
    r = ncc.ncc_correlate_direct(to_dev(img), to_dev(T), out=nan_map(1, 185, 285)).cpu().numpy()[0]
    assert ncc.ncc_sync_status() == 0
    assert r[0, 0] == 0.0                              # a window of constant 255
    assert abs(r[60, 100] - 1.0) <= TOL
    ref = oracle.correlate(img, T)
    np.testing.assert_allclose(r, ref, rtol=0, atol=TOL)


def test_direct_rejects_too_wide_templates(ncc):
    img = to_dev(np.zeros((40, 200), np.uint8))
    T = to_dev(np.zeros((4, 130), np.uint8))
    with pytest.raises(ncc.NccError) as e:
        ncc.ncc_correlate_direct(img, T)
    assert e.value.code == ncc.NCC_ERR_UNSUPPORTED
