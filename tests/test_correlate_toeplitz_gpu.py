"""GPU parity of the Toeplitz tensor-core numerator (single templates up to 65
pixels wide) against the oracle.

SumI, SumI2 and SumIT must match bit-exactly; coefficients within 1e-5
absolute.  The kernel accumulates centered products (I-128)(T-128) in fp32
groups of at most 1024 products and recovers SumIT from them, so the cases
cover several accumulator groups (ragged last group), saturated images and
templates whose group sums reach the 2^24 bound, ragged tiles (128 rows x 64
shifts), rows that are not multiples of 8 bytes (byte-wise loads), and small
templates forced onto this kernel.  Outputs are written over NaN / poison.
"""
import numpy as np
import pytest

import oracle
from gpu_util import moments, nan_map, to_dev
from normalized_cross_correlation_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = 1e-5


@pytest.fixture
def toeplitz(ncc):
    """Forces the Toeplitz kernel; restores automatic selection after."""
    ncc.ncc_debug_set_path(ncc.NCC_PATH_TOEPLITZ)
    yield ncc
    ncc.ncc_debug_set_path(0)


CASES = [  # (W, H, wT, hT)
    (300, 200, 64, 64), (257, 190, 48, 17), (500, 300, 65, 40), (129, 130, 64, 1),
    (100, 260, 50, 64), (1001, 150, 64, 64), (700, 140, 64, 33), (64, 64, 64, 64),
    (383, 255, 56, 48),
    # narrow templates forced onto the kernel: other K widths and group sizes
    (50, 41, 3, 5), (300, 200, 16, 16), (257, 190, 17, 9), (400, 333, 32, 32), (90, 70, 1, 1),
]


@pytest.mark.parametrize("W,H,wT,hT", CASES)
def test_toeplitz_moments_bit_exact(toeplitz, threads, W, H, wT, hT):
    ncc = toeplitz
    w = inputs.random_case(W * 29 + H, W, H, wT, hT, nT=1, n_crops=1)
    dimg = to_dev(w.image)
    S, Q = ncc.ncc_sat_build(dimg)
    sI, sI2, sIT = moments(ncc, dimg, to_dev(w.templates), S, Q)
    assert ncc.ncc_debug_last_path() == ncc.NCC_PATH_TOEPLITZ
    _, oI, oI2, oIT = oracle.correlate(w.image, w.templates[0], with_sums=True, threads=threads)
    np.testing.assert_array_equal(sI.cpu().numpy(), oI)
    np.testing.assert_array_equal(sI2.cpu().numpy(), oI2)
    np.testing.assert_array_equal(sIT.cpu().numpy()[0], oIT)


@pytest.mark.parametrize("W,H,wT,hT", CASES)
def test_toeplitz_coefficients_match_oracle(toeplitz, threads, W, H, wT, hT):
    ncc = toeplitz
    w = inputs.random_case(W * 23 + H, W, H, wT, hT, nT=1, n_crops=1)
    dimg = to_dev(w.image)
    S, Q = ncc.ncc_sat_build(dimg)
    r = ncc.ncc_correlate(dimg, to_dev(w.templates[0]), S, Q, out=nan_map(w.Oy, w.Ox))
    assert ncc.ncc_sync_status() == 0
    assert ncc.ncc_debug_last_path() == ncc.NCC_PATH_TOEPLITZ
    r = r.cpu().numpy()
    ref = oracle.correlate(w.image, w.templates[0], threads=threads)
    np.testing.assert_allclose(r, ref, rtol=0, atol=TOL)
    _, x, y = w.crops[0]
    if wT * hT > 1:
        assert abs(r[y, x] - 1.0) <= TOL


def saturated_case():
    """Blocks of 0 and 255 in image and template: every centered product is
    +-16384 or +-16256, so a 64x64 template's groups of 16 rows sum to
    magnitudes up to 2^24."""
    rng = np.random.default_rng(44)
    img = rng.integers(0, 256, (400, 500), dtype=np.uint8)
    img[0:200, 0:250] = 0
    img[200:400, 250:500] = 255
    img[100:300, 100:164] = (rng.random((200, 64)) < 0.5) * np.uint8(255)
    T = np.zeros((64, 64), np.uint8)
    T[32:, :] = 255
    return img, T


def test_toeplitz_saturated_group_bounds(toeplitz, threads):
    ncc = toeplitz
    img, T = saturated_case()
    dimg = to_dev(img)
    S, Q = ncc.ncc_sat_build(dimg)
    for tmpl in (T, np.zeros_like(T), np.full_like(T, 255), img[120:184, 110:174].copy()):
        sI, sI2, sIT = moments(ncc, dimg, to_dev(tmpl), S, Q)
        _, oI, oI2, oIT = oracle.correlate(img, tmpl, with_sums=True, threads=threads)
        np.testing.assert_array_equal(sIT.cpu().numpy()[0], oIT)
        np.testing.assert_array_equal(sI.cpu().numpy(), oI)
        r = ncc.ncc_correlate(dimg, to_dev(tmpl), S, Q, out=nan_map(337, 437)).cpu().numpy()
        ref = oracle.correlate(img, tmpl, threads=threads)
        np.testing.assert_allclose(r, ref, rtol=0, atol=TOL)
    assert ncc.ncc_sync_status() == 0


def test_toeplitz_zero_variance_and_negated_crop(toeplitz):
    ncc = toeplitz
    w = inputs.random_case(71, 400, 300, 64, 64, nT=1, n_crops=1)
    img = w.image.copy()
    img[10:120, 20:150] = 9                              # constant windows
    dimg = to_dev(img)
    S, Q = ncc.ncc_sat_build(dimg)
    T = w.templates[0]
    r = ncc.ncc_correlate(dimg, to_dev(T), S, Q, out=nan_map(237, 337)).cpu().numpy()
    assert np.all(r[10:57, 20:87] == 0.0)
    flat = np.full((64, 64), 200, np.uint8)
    assert np.all(ncc.ncc_correlate(dimg, to_dev(flat), S, Q).cpu().numpy() == 0.0)
    _, x, y = w.crops[0]
    neg = (255 - img[y:y + 64, x:x + 64]).astype(np.uint8)
    rn = ncc.ncc_correlate(dimg, to_dev(neg), S, Q).cpu().numpy()
    assert abs(rn[y, x] + 1.0) <= TOL
    assert ncc.ncc_sync_status() == 0


def test_automatic_selection_takes_toeplitz_for_large_templates(ncc):
    """On maps of fewer than 4M shifts: Toeplitz from ceil(wT/4)*hT >= 320
    dp4a per output (40x40 and up), dp4a below (32x32, and wide but short
    templates)."""
    w = inputs.random_case(5, 300, 200, 64, 64, nT=1, n_crops=1)
    dimg = to_dev(w.image)
    S, Q = ncc.ncc_sat_build(dimg)
    T = w.templates[0]
    for tmpl, path in ((T, ncc.NCC_PATH_TOEPLITZ), (T[:40, :40], ncc.NCC_PATH_TOEPLITZ),
                       (T[:32, :32], ncc.NCC_PATH_DP4A), (T[:16, :], ncc.NCC_PATH_DP4A),
                       (T[:, :16], ncc.NCC_PATH_DP4A)):
        ncc.ncc_correlate(dimg, to_dev(tmpl), S, Q)
        assert ncc.ncc_debug_last_path() == path, tmpl.shape
    assert ncc.ncc_sync_status() == 0


def test_automatic_selection_on_large_maps(ncc):
    """On maps of at least 4M shifts: Toeplitz from 96 dp4a per output
    (20x20: 100), dp4a below (16x16: 64; 64 x 4: 64)."""
    img = to_dev(np.zeros((2200, 2200), np.uint8))
    S, Q = ncc.ncc_sat_build(img)
    rng = np.random.default_rng(8)
    for shape, path in (((20, 20), ncc.NCC_PATH_TOEPLITZ), ((16, 16), ncc.NCC_PATH_DP4A),
                        ((4, 64), ncc.NCC_PATH_DP4A), ((24, 16), ncc.NCC_PATH_TOEPLITZ)):
        ncc.ncc_correlate(img, to_dev(rng.integers(0, 256, shape, dtype=np.uint8)), S, Q)
        assert ncc.ncc_debug_last_path() == path, shape
    assert ncc.ncc_sync_status() == 0


def test_toeplitz_equals_dp4a(ncc):
    """Both numerators give the same integers; the coefficients agree to fp32
    rounding (the same arithmetic from the same integers: bit for bit)."""
    w = inputs.random_case(606, 900, 500, 64, 64, nT=1, n_crops=1)
    dimg, dt = to_dev(w.image), to_dev(w.templates[0])
    S, Q = ncc.ncc_sat_build(dimg)
    try:
        ncc.ncc_debug_set_path(ncc.NCC_PATH_DP4A)
        r0 = ncc.ncc_correlate(dimg, dt, S, Q, out=nan_map(w.Oy, w.Ox)).cpu().numpy()
        ncc.ncc_debug_set_path(ncc.NCC_PATH_TOEPLITZ)
        r1 = ncc.ncc_correlate(dimg, dt, S, Q, out=nan_map(w.Oy, w.Ox)).cpu().numpy()
    finally:
        ncc.ncc_debug_set_path(0)
    assert ncc.ncc_sync_status() == 0
    np.testing.assert_array_equal(r1, r0)


def test_toeplitz_under_match_equals_separate_calls(ncc):
    """ncc_match runs the table build and this kernel; the results equal the
    separate calls bit for bit, call after call."""
    w = inputs.random_case(808, 1536, 700, 64, 64, nT=1, n_crops=1)
    dimg, dt = to_dev(w.image), to_dev(w.templates)
    S0, Q0 = ncc.ncc_sat_build(dimg)
    r0 = ncc.ncc_correlate(dimg, dt[0], S0, Q0, out=nan_map(w.Oy, w.Ox)).cpu().numpy()
    for _ in range(3):
        S, Q, r = ncc.ncc_match(dimg, dt, out=nan_map(1, w.Oy, w.Ox))
        assert ncc.ncc_sync_status() == 0
        assert ncc.ncc_debug_last_path() == ncc.NCC_PATH_TOEPLITZ
        np.testing.assert_array_equal(r.cpu().numpy()[0], r0)


def test_forced_toeplitz_rejects_shapes_it_cannot_take(toeplitz):
    ncc = toeplitz
    img = to_dev(np.zeros((300, 300), np.uint8))
    S, Q = ncc.ncc_sat_build(img)
    for shape in ((70, 70), (200, 64)):                  # (hT, wT): too wide; too many groups
        with pytest.raises(ncc.NccError) as e:
            ncc.ncc_correlate(img, to_dev(np.zeros(shape, np.uint8)), S, Q)
        assert e.value.code == ncc.NCC_ERR_UNSUPPORTED
