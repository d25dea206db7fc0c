"""GPU parity of the transform numerator (number-theoretic transforms of
256 x 256 tiles modulo the prime 998244353) against the oracle.

SumI, SumI2 and SumIT must match bit-exactly; coefficients within 1e-5
absolute, and bit-identical to the dp4a kernel's (the same arithmetic from
the same integers).  The cases cover several tiles in both directions with
ragged last tiles (a tile yields 257 - hT rows and 257 - wT columns of
shifts), images smaller than one tile, rows of odd widths, templates from
1 x 1 to the largest the kernel takes (224 wide; 30000 pixels), and the
extremes of the centered correlation |C| <= 2^14 * wT * hT that the prime
must exceed twice.  Outputs are written over NaN / poison.
"""
import numpy as np
import pytest

import oracle
from gpu_util import moments, nan_map, to_dev
from normalized_cross_correlation_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = 1e-5


@pytest.fixture
def ntt(ncc):
    """Forces the transform kernel; restores automatic selection after."""
    ncc.ncc_debug_set_path(ncc.NCC_PATH_NTT)
    yield ncc
    ncc.ncc_debug_set_path(0)


CASES = [  # (W, H, wT, hT)
    (600, 500, 64, 64),     # 3 x 3 tiles of 193 x 193 shifts, ragged
    (1001, 300, 100, 80),   # 6 x 2 tiles, ragged, odd row width
    (700, 700, 128, 128),   # 129 x 129 shifts per tile
    (300, 420, 173, 173),   # 29929 pixels: |C| close to its bound
    (500, 260, 224, 30),    # the widest template
    (130, 900, 20, 224),    # the tallest
    (200, 150, 1, 1),       # 256 x 256 shifts per tile; image smaller than a tile
    (257, 190, 17, 9),
    (90, 70, 3, 5),
    (4000, 10, 70, 10),     # one tile row, many tiles
]


@pytest.mark.parametrize("W,H,wT,hT", CASES)
def test_ntt_moments_bit_exact(ntt, threads, W, H, wT, hT):
    ncc = ntt
    w = inputs.random_case(W * 31 + H, W, H, wT, hT, nT=1, n_crops=1)
    dimg = to_dev(w.image)
    S, Q = ncc.ncc_sat_build(dimg)
    sI, sI2, sIT = moments(ncc, dimg, to_dev(w.templates), S, Q)
    assert ncc.ncc_debug_last_path() == ncc.NCC_PATH_NTT
    _, oI, oI2, oIT = oracle.correlate(w.image, w.templates[0], with_sums=True, threads=threads)
    np.testing.assert_array_equal(sI.cpu().numpy(), oI)
    np.testing.assert_array_equal(sI2.cpu().numpy(), oI2)
    np.testing.assert_array_equal(sIT.cpu().numpy()[0], oIT)


@pytest.mark.parametrize("W,H,wT,hT", CASES)
def test_ntt_coefficients_match_oracle(ntt, threads, W, H, wT, hT):
    ncc = ntt
    w = inputs.random_case(W * 37 + H, W, H, wT, hT, nT=1, n_crops=1)
    dimg = to_dev(w.image)
    S, Q = ncc.ncc_sat_build(dimg)
    r = ncc.ncc_correlate(dimg, to_dev(w.templates[0]), S, Q, out=nan_map(w.Oy, w.Ox))
    assert ncc.ncc_sync_status() == 0
    assert ncc.ncc_debug_last_path() == ncc.NCC_PATH_NTT
    r = r.cpu().numpy()
    ref = oracle.correlate(w.image, w.templates[0], threads=threads)
    np.testing.assert_allclose(r, ref, rtol=0, atol=TOL)
    _, x, y = w.crops[0]
    if wT * hT > 1:
        assert abs(r[y, x] - 1.0) <= TOL


@pytest.mark.parametrize("img_offset", [0, 3])
def test_ntt_image_pointer_alignment(ntt, threads, img_offset):
    """Rows a multiple of 16 bytes long: from a 16-byte-aligned image the
    tile rows are staged with 16-byte loads, from an image 3 bytes into its
    buffer byte by byte; both through the C ABI, bit for bit the same."""
    import torch
    ncc = ntt
    w = inputs.random_case(4242, 640, 480, 96, 72, nT=1, n_crops=1)
    n = w.image.size
    ibuf = torch.zeros(n + 64, dtype=torch.uint8, device="cuda")
    ibuf[img_offset:img_offset + n] = torch.from_numpy(w.image.ravel()).cuda()
    dimg = to_dev(w.image)
    S, Q = ncc.ncc_sat_build(dimg)
    out = nan_map(w.Oy, w.Ox)
    tm = to_dev(w.templates[0])
    rc = ncc.lib().ncc_correlate(ibuf.data_ptr() + img_offset, w.W, w.H, tm.data_ptr(), w.wT, w.hT,
                                 S.data_ptr(), Q.data_ptr(), out.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == 0, ncc.ncc_status_string(rc)
    assert ncc.ncc_sync_status() == 0
    assert ncc.ncc_debug_last_path() == ncc.NCC_PATH_NTT
    ref = oracle.correlate(w.image, w.templates[0], threads=threads)
    np.testing.assert_allclose(out.cpu().numpy(), ref, rtol=0, atol=TOL)


@pytest.mark.parametrize("img_v,tmpl_v", [(0, 0), (255, 0), (0, 255), (255, 255)])
def test_ntt_extreme_centered_sums(ntt, threads, img_v, tmpl_v):
    """A constant image block at 0 or 255 against a constant 173 x 173
    template at 0 or 255: every centered product is +-16384 or +-16256, so
    |C| reaches 29929 * 16384 = 4.90e8 of the 4.99e8 that the prime allows
    (SumIT checked bit for bit).  A template with noise in its lower rows
    then checks the coefficients over the same image."""
    ncc = ntt
    rng = np.random.default_rng(img_v * 3 + tmpl_v)
    img = rng.integers(0, 256, (500, 600), dtype=np.uint8)
    img[0:300, 0:350] = img_v
    dimg = to_dev(img)
    S, Q = ncc.ncc_sat_build(dimg)
    T = np.full((173, 173), tmpl_v, np.uint8)
    sI, sI2, sIT = moments(ncc, dimg, to_dev(T[None]), S, Q)
    _, oI, oI2, oIT = oracle.correlate(img, T, with_sums=True, threads=threads)
    np.testing.assert_array_equal(sIT.cpu().numpy()[0], oIT)
    np.testing.assert_array_equal(sI.cpu().numpy(), oI)
    np.testing.assert_array_equal(sI2.cpu().numpy(), oI2)
    centered = oIT - 128 * oI - 128 * int(T.sum()) + 16384 * T.size
    assert np.abs(centered).max() >= 29929 * 16129                # 127 * 127 at (255, 255)
    T[100:, :] = rng.integers(0, 256, (73, 173), dtype=np.uint8)
    r = ncc.ncc_correlate(dimg, to_dev(T), S, Q, out=nan_map(328, 428)).cpu().numpy()
    np.testing.assert_allclose(r, oracle.correlate(img, T, threads=threads), rtol=0, atol=TOL)
    assert ncc.ncc_sync_status() == 0


def test_ntt_zero_variance_and_negated_crop(ntt):
    ncc = ntt
    w = inputs.random_case(72, 700, 500, 100, 100, nT=1, n_crops=1)
    img = w.image.copy()
    img[10:200, 20:250] = 9                              # constant windows
    dimg = to_dev(img)
    S, Q = ncc.ncc_sat_build(dimg)
    T = w.templates[0]
    r = ncc.ncc_correlate(dimg, to_dev(T), S, Q, out=nan_map(401, 601)).cpu().numpy()
    assert np.all(r[10:101, 20:151] == 0.0)
    flat = np.full((100, 100), 200, np.uint8)
    assert np.all(ncc.ncc_correlate(dimg, to_dev(flat), S, Q).cpu().numpy() == 0.0)
    _, x, y = w.crops[0]
    neg = (255 - img[y:y + 100, x:x + 100]).astype(np.uint8)
    rn = ncc.ncc_correlate(dimg, to_dev(neg), S, Q).cpu().numpy()
    assert abs(rn[y, x] + 1.0) <= TOL
    assert ncc.ncc_sync_status() == 0


def test_ntt_equals_dp4a_and_toeplitz(ncc):
    """The three single-template numerators give the same integers, so the
    coefficients agree bit for bit."""
    w = inputs.random_case(607, 900, 700, 64, 64, nT=1, n_crops=1)
    dimg, dt = to_dev(w.image), to_dev(w.templates[0])
    S, Q = ncc.ncc_sat_build(dimg)
    maps = {}
    try:
        for path in (ncc.NCC_PATH_DP4A, ncc.NCC_PATH_TOEPLITZ, ncc.NCC_PATH_NTT):
            ncc.ncc_debug_set_path(path)
            maps[path] = ncc.ncc_correlate(dimg, dt, S, Q, out=nan_map(w.Oy, w.Ox)).cpu().numpy()
            assert ncc.ncc_debug_last_path() == path
    finally:
        ncc.ncc_debug_set_path(0)
    assert ncc.ncc_sync_status() == 0
    np.testing.assert_array_equal(maps[ncc.NCC_PATH_NTT], maps[ncc.NCC_PATH_DP4A])
    np.testing.assert_array_equal(maps[ncc.NCC_PATH_NTT], maps[ncc.NCC_PATH_TOEPLITZ])


def test_automatic_selection_takes_ntt_for_wide_templates(ncc):
    """Templates wider than the Toeplitz kernel takes (65) go to the
    transform kernel from the same dp4a count; narrower ones keep their
    kernels, and shapes the transform kernel cannot take stay on dp4a."""
    w = inputs.random_case(6, 900, 600, 240, 240, nT=1, n_crops=1)
    dimg = to_dev(w.image)
    S, Q = ncc.ncc_sat_build(dimg)
    T = w.templates[0]
    for tmpl, path in ((T[:80, :80], ncc.NCC_PATH_NTT), (T[:20, :128], ncc.NCC_PATH_NTT),
                       (T[:64, :64], ncc.NCC_PATH_TOEPLITZ), (T[:16, :16], ncc.NCC_PATH_DP4A),
                       (T[:6, :200], ncc.NCC_PATH_DP4A),    # 50 * 6 = 300 dp4a per output
                       (T[:200, :200], ncc.NCC_PATH_DP4A),  # 40000 pixels: beyond the prime
                       (T[:10, :240], ncc.NCC_PATH_DP4A)):  # wider than 224
        ncc.ncc_correlate(dimg, to_dev(tmpl), S, Q)
        assert ncc.ncc_debug_last_path() == path, tmpl.shape
    assert ncc.ncc_sync_status() == 0


def test_automatic_selection_at_every_image_size(ncc):
    """Templates the Toeplitz kernel takes stay on it on large images too;
    the transform kernel takes the wider ones and those too tall for the
    Toeplitz kernel's accumulator groups (40 x 200: eight groups of 25 rows)."""
    large = to_dev(np.zeros((6000, 6000), np.uint8))
    rng = np.random.default_rng(3)
    for shape, path in (((64, 64), ncc.NCC_PATH_TOEPLITZ), ((80, 80), ncc.NCC_PATH_NTT),
                        ((200, 40), ncc.NCC_PATH_NTT)):
        T = to_dev(rng.integers(0, 256, shape, dtype=np.uint8))
        S, Q = ncc.ncc_sat_build(large)
        ncc.ncc_correlate(large, T, S, Q)
        assert ncc.ncc_debug_last_path() == path, shape
        del S, Q
    assert ncc.ncc_sync_status() == 0


def test_ntt_under_match_equals_separate_calls(ncc):
    """ncc_match runs the table build and this kernel; the results equal the
    separate calls bit for bit, call after call."""
    w = inputs.random_case(809, 1300, 700, 96, 96, nT=1, n_crops=1)
    dimg, dt = to_dev(w.image), to_dev(w.templates)
    S0, Q0 = ncc.ncc_sat_build(dimg)
    r0 = ncc.ncc_correlate(dimg, dt[0], S0, Q0, out=nan_map(w.Oy, w.Ox)).cpu().numpy()
    assert ncc.ncc_debug_last_path() == ncc.NCC_PATH_NTT
    for _ in range(3):
        S, Q, r = ncc.ncc_match(dimg, dt, out=nan_map(1, w.Oy, w.Ox))
        assert ncc.ncc_sync_status() == 0
        assert ncc.ncc_debug_last_path() == ncc.NCC_PATH_NTT
        np.testing.assert_array_equal(r.cpu().numpy()[0], r0)


def test_ntt_spectrum_allocation_failure(ntt):
    """The template's spectrum comes from the library's pool; a failed
    allocation returns NCC_ERR_NOMEM and launches nothing, and the next call
    is exact."""
    ncc = ntt
    w = inputs.random_case(810, 400, 300, 64, 64, nT=1, n_crops=1)
    dimg, dt = to_dev(w.image), to_dev(w.templates[0])
    S, Q = ncc.ncc_sat_build(dimg)
    ncc.ncc_debug_fail_alloc(1)
    try:
        with pytest.raises(ncc.NccError) as e:
            ncc.ncc_correlate(dimg, dt, S, Q)
        assert e.value.code == ncc.NCC_ERR_NOMEM
    finally:
        ncc.ncc_debug_fail_alloc(0)
    r = ncc.ncc_correlate(dimg, dt, S, Q, out=nan_map(w.Oy, w.Ox)).cpu().numpy()
    assert ncc.ncc_sync_status() == 0
    np.testing.assert_allclose(r, oracle.correlate(w.image, w.templates[0]), rtol=0, atol=TOL)


def test_forced_ntt_rejects_shapes_it_cannot_take(ntt):
    ncc = ntt
    img = to_dev(np.zeros((400, 400), np.uint8))
    S, Q = ncc.ncc_sat_build(img)
    for shape in ((10, 225), (225, 10), (180, 180)):     # (hT, wT): too wide, too tall, > 30000 px
        with pytest.raises(ncc.NccError) as e:
            ncc.ncc_correlate(img, to_dev(np.zeros(shape, np.uint8)), S, Q)
        assert e.value.code == ncc.NCC_ERR_UNSUPPORTED


def test_ntt_full_size_8192_t64_equals_other_paths_and_oracle_samples(ncc, threads):
    """The 8192 x 8192 image with its 64 x 64 template (43 x 43 tiles): the
    transform kernel's coefficients equal the Toeplitz kernel's bit for bit
    (that kernel's full map is checked against the oracle elsewhere), and
    20000 random shifts plus the crop match the oracle's coefficients."""
    w = inputs.large_8192()
    dimg, dt = to_dev(w.image), to_dev(w.templates[0])
    S, Q = ncc.ncc_sat_build(dimg)
    try:
        ncc.ncc_debug_set_path(ncc.NCC_PATH_NTT)
        r = ncc.ncc_correlate(dimg, dt, S, Q, out=nan_map(w.Oy, w.Ox))
        assert ncc.ncc_debug_last_path() == ncc.NCC_PATH_NTT
        ncc.ncc_debug_set_path(ncc.NCC_PATH_TOEPLITZ)
        r2 = ncc.ncc_correlate(dimg, dt, S, Q, out=nan_map(w.Oy, w.Ox))
    finally:
        ncc.ncc_debug_set_path(0)
    assert ncc.ncc_sync_status() == 0
    assert bool((r == r2).all())
    rng = np.random.default_rng(5)
    xs = rng.integers(0, w.Ox, 20000)
    ys = rng.integers(0, w.Oy, 20000)
    _, cx, cy = w.crops[0]
    xs[0], ys[0] = cx, cy
    ref = oracle.correlate_at(w.image, w.templates[0], xs, ys, threads=threads)
    got = r.cpu().numpy()[ys, xs]
    np.testing.assert_allclose(got, ref, rtol=0, atol=TOL)
    assert abs(got[0] - 1.0) <= TOL
