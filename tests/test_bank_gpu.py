"""GPU parity of ncc_correlate_bank (the tensor-core bank path) against the
oracle.  SumIT/SumI/SumI2 bit-exact; coefficients within 1e-5 absolute.

Shapes cover: ragged image widths (not multiples of 128 or 16), banks whose
size is not a multiple of 16 (padded MMA N), templates wider than 16 (more
K chunks), and templates of more than 258 pixels (split into row groups with
separate exact accumulators)."""
import numpy as np
import pytest

import oracle
from gpu_util import moments, nan_map, to_dev
from normalized_cross_correlation_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = 1e-5


def gpu_bank(ncc, img, T):
    """Coefficients of a bank, written over a NaN-filled map."""
    dimg = to_dev(img)
    S, Q = ncc.ncc_sat_build(dimg)
    out = nan_map(T.shape[0], img.shape[0] - T.shape[1] + 1, img.shape[1] - T.shape[2] + 1)
    r = ncc.ncc_correlate_bank(dimg, to_dev(T), S, Q, out=out)
    assert ncc.ncc_sync_status() == 0
    return r.cpu().numpy()


BANKS = [  # (W, H, wT, hT, nT)
    (300, 200, 16, 16, 8), (257, 190, 16, 16, 5), (130, 70, 8, 8, 2), (400, 150, 13, 7, 20),
    (200, 100, 16, 16, 33), (300, 140, 32, 8, 16), (200, 200, 20, 20, 16), (170, 90, 64, 4, 4),
    (1000, 64, 16, 16, 64), (129, 40, 1, 1, 3), (520, 66, 17, 3, 96),
]


@pytest.mark.parametrize("W,H,wT,hT,nT", BANKS)
def test_bank_coefficients_match_oracle(ncc, threads, W, H, wT, hT, nT):
    w = inputs.random_case(W * 7 + H + nT, W, H, wT, hT, nT=nT, n_crops=min(nT, 3))
    r = gpu_bank(ncc, w.image, w.templates)
    ref = oracle.correlate(w.image, w.templates, threads=threads)
    assert r.shape == ref.shape
    np.testing.assert_allclose(r, ref, rtol=0, atol=TOL)
    if wT * hT > 1:
        for t, x, y in w.crops:
            assert abs(r[t, y, x] - 1.0) <= TOL


@pytest.mark.parametrize("W,H,wT,hT,nT", [BANKS[0], BANKS[1], BANKS[6], BANKS[7], BANKS[10]])
def test_bank_moments_bit_exact(ncc, threads, W, H, wT, hT, nT):
    w = inputs.random_case(W * 11 + H + nT, W, H, wT, hT, nT=nT, n_crops=1)
    dimg = to_dev(w.image)
    S, Q = ncc.ncc_sat_build(dimg)
    sI, sI2, sIT = moments(ncc, dimg, to_dev(w.templates), S, Q)
    _, oI, oI2, oIT = oracle.correlate(w.image, w.templates, with_sums=True, threads=threads)
    np.testing.assert_array_equal(sI.cpu().numpy(), oI[0])
    np.testing.assert_array_equal(sI2.cpu().numpy(), oI2[0])
    np.testing.assert_array_equal(sIT.cpu().numpy(), oIT)


def test_bank_agrees_with_single_template_path(ncc):
    import torch
    w = inputs.random_case(91, 640, 300, 16, 16, nT=12, n_crops=4)
    dimg = to_dev(w.image)
    S, Q = ncc.ncc_sat_build(dimg)
    bank = ncc.ncc_correlate_bank(dimg, to_dev(w.templates), S, Q,
                                  out=nan_map(12, w.Oy, w.Ox))
    for t in range(12):
        one = ncc.ncc_correlate(dimg, to_dev(w.templates[t]), S, Q, out=nan_map(w.Oy, w.Ox))
        assert torch.max(torch.abs(bank[t] - one)).item() <= 2 * TOL
    assert ncc.ncc_sync_status() == 0


def test_bank_zero_variance(ncc):
    rng = np.random.default_rng(17)
    img = rng.integers(0, 256, (150, 300), dtype=np.uint8)
    img[30:70, 40:120] = 200
    T = rng.integers(0, 256, (4, 16, 16), dtype=np.uint8)
    T[2] = 7                                              # constant template
    r = gpu_bank(ncc, img, T)
    assert np.all(r[2] == 0.0)
    assert np.all(r[:, 30:55, 40:105] == 0.0)             # constant windows
