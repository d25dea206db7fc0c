"""Pins for the CPU oracle: every check here compares the oracle with
something other than itself -- brute-force sums written with numpy slicing,
closed forms, library routines (scipy's 2-D correlation, numpy's Pearson
correlation) and exact identities of the Pearson coefficient.

The quantities follow The CUDA Handbook, chapter 15: the summed-area tables
and four-corner box sum of section 15.8 ("The Denominator: Summed Area
Tables", Figure 15-7) and the per-shift sums of Listing 15-5 ("Image in
shared memory").
"""
import json
import os

import numpy as np
import pytest

import oracle
from normalized_cross_correlation_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def brute_sat(img):
    """S and Q straight from the definition: sums of the (y+1) x (x+1)
    top-left block, one numpy slice per entry."""
    H, W = img.shape
    I = img.astype(np.int64)
    S = np.empty((H, W), np.int64)
    Q = np.empty((H, W), np.int64)
    for y in range(H):
        for x in range(W):
            blk = I[: y + 1, : x + 1]
            S[y, x] = blk.sum()
            Q[y, x] = (blk * blk).sum()
    return S, Q


@pytest.mark.parametrize("H,W", [(1, 1), (1, 7), (5, 1), (13, 9), (17, 31), (32, 32)])
def test_sat_equals_definition(H, W):
    rng = np.random.default_rng(H * 100 + W)
    img = rng.integers(0, 256, (H, W), dtype=np.uint8)
    S, Q = oracle.sat(img)
    bS, bQ = brute_sat(img)
    np.testing.assert_array_equal(S, bS)
    np.testing.assert_array_equal(Q, bQ)


def test_sat_bottom_right_is_whole_image_sum():
    w = inputs.tiny_ncc()
    S, Q = oracle.sat(w.image)
    I = w.image.astype(np.int64)
    assert S[-1, -1] == I.sum()
    assert Q[-1, -1] == (I * I).sum()


def test_sat_needs_int64_beyond_512_squared():
    # Section 15.8: the sum of squares of an 8-bit image passes 2^31 by
    # 512 x 512; all-255 pixels give 512*512*255^2 exactly.
    img = np.full((512, 512), 255, np.uint8)
    S, Q = oracle.sat(img)
    assert Q[-1, -1] == 512 * 512 * 255 * 255
    assert Q[-1, -1] > 2**31
    assert S[-1, -1] == 512 * 512 * 255


@pytest.mark.parametrize("c", [0, 1, 77, 255])
def test_sat_constant_image_closed_form(c):
    H, W = 23, 41
    img = np.full((H, W), c, np.uint8)
    S, Q = oracle.sat(img)
    ys, xs = np.mgrid[0:H, 0:W]
    area = (xs + 1).astype(np.int64) * (ys + 1)
    np.testing.assert_array_equal(S, c * area)
    np.testing.assert_array_equal(Q, c * c * area)


def test_sat_single_pixel_is_a_step():
    # One pixel of value v at (px, py): S is v exactly where x >= px and
    # y >= py, else 0 -- any transposed or shifted index breaks this.
    H, W, px, py, v = 9, 14, 11, 3, 200
    img = np.zeros((H, W), np.uint8)
    img[py, px] = v
    S, Q = oracle.sat(img)
    ys, xs = np.mgrid[0:H, 0:W]
    step = ((xs >= px) & (ys >= py)).astype(np.int64)
    np.testing.assert_array_equal(S, v * step)
    np.testing.assert_array_equal(Q, v * v * step)


def test_sat_box_four_corner_identity():
    rng = np.random.default_rng(7)
    H, W = 37, 53
    img = rng.integers(0, 256, (H, W), dtype=np.uint8)
    I = img.astype(np.int64)
    S, Q = oracle.sat(img)
    boxes = [(0, 0, W, H), (0, 0, 1, 1), (W - 1, H - 1, W, H), (0, 5, 9, 6),
             (4, 0, 5, H), (0, 0, W, 1), (0, 0, 1, H)]
    for _ in range(300):
        x0, x1 = sorted(rng.choice(W + 1, 2, replace=False))
        y0, y1 = sorted(rng.choice(H + 1, 2, replace=False))
        boxes.append((int(x0), int(y0), int(x1), int(y1)))
    for x0, y0, x1, y1 in boxes:
        blk = I[y0:y1, x0:x1]
        assert oracle.sat_box(S, x0, y0, x1, y1) == blk.sum()
        assert oracle.sat_box(Q, x0, y0, x1, y1) == (blk * blk).sum()


@pytest.mark.parametrize("H,W,hT,wT", [(40, 57, 7, 13), (33, 20, 16, 16), (19, 23, 1, 23),
                                       (21, 18, 21, 1), (12, 12, 12, 12)])
def test_window_sums_match_scipy_correlation(H, W, hT, wT):
    from scipy.signal import correlate2d
    rng = np.random.default_rng(H * W + hT)
    img = rng.integers(0, 256, (H, W), dtype=np.uint8)
    T = rng.integers(0, 256, (hT, wT), dtype=np.uint8)
    r, sI, sI2, sIT = oracle.correlate(img, T, with_sums=True)
    I = img.astype(np.int64)
    ones = np.ones((hT, wT), np.int64)
    np.testing.assert_array_equal(sIT, correlate2d(I, T.astype(np.int64), mode="valid"))
    np.testing.assert_array_equal(sI, correlate2d(I, ones, mode="valid"))
    np.testing.assert_array_equal(sI2, correlate2d(I * I, ones, mode="valid"))
    assert r.shape == (H - hT + 1, W - wT + 1)


def test_window_sums_agree_with_sat_box():
    rng = np.random.default_rng(11)
    img = rng.integers(0, 256, (30, 45), dtype=np.uint8)
    T = rng.integers(0, 256, (6, 9), dtype=np.uint8)
    S, Q = oracle.sat(img)
    _, sI, sI2, _ = oracle.correlate(img, T, with_sums=True)
    for y in range(sI.shape[0]):
        for x in range(sI.shape[1]):
            assert sI[y, x] == oracle.sat_box(S, x, y, x + 9, y + 6)
            assert sI2[y, x] == oracle.sat_box(Q, x, y, x + 9, y + 6)


def test_template_stats_closed_form():
    T = np.arange(12, dtype=np.uint8).reshape(3, 4) * 20
    sT, sT2 = oracle.template_stats(T)
    v = np.arange(12, dtype=np.int64) * 20
    assert sT == v.sum() and sT2 == (v * v).sum()


def test_coefficient_matches_numpy_pearson():
    rng = np.random.default_rng(5)
    img = rng.integers(0, 256, (48, 64), dtype=np.uint8)
    T = rng.integers(0, 256, (8, 11), dtype=np.uint8)
    r = oracle.correlate(img, T)
    for _ in range(200):
        y = int(rng.integers(0, r.shape[0]))
        x = int(rng.integers(0, r.shape[1]))
        win = img[y:y + 8, x:x + 11].astype(np.float64).ravel()
        ref = np.corrcoef(win, T.astype(np.float64).ravel())[0, 1]
        assert abs(r[y, x] - ref) < 1e-12


def test_coefficient_sign_and_scale():
    # Hand-evaluated: window (1,2,3), template (1,2,3) -> +1; template
    # (3,2,1) -> -1; template (1,3,2) -> num = 3*13 - 6*6 = 3,
    # vI = vT = 3*14 - 36 = 6, r = 3/6 = 0.5.
    img = np.array([[1, 2, 3]], np.uint8)
    for T, want in [((1, 2, 3), 1.0), ((3, 2, 1), -1.0), ((1, 3, 2), 0.5)]:
        r = oracle.correlate(img, np.array([T], np.uint8))
        assert r.shape == (1, 1)
        assert r[0, 0] == want


def test_exact_crop_gives_exactly_one():
    w = inputs.tiny_ncc()
    r = oracle.correlate(w.image, w.templates)
    assert r.shape == (1, 241, 241)
    assert r[0, 37, 100] == 1.0
    assert np.argmax(r[0]) == 37 * 241 + 100


def test_negated_crop_gives_exactly_minus_one():
    w = inputs.tiny_ncc()
    neg = (255 - w.templates).astype(np.uint8)
    r = oracle.correlate(w.image, neg)
    assert r[0, 37, 100] == -1.0
    assert np.argmin(r[0]) == 37 * 241 + 100


def test_zero_variance_gives_zero():
    rng = np.random.default_rng(3)
    img = rng.integers(0, 256, (40, 40), dtype=np.uint8)
    img[10:20, 5:15] = 42                      # a constant patch
    T = rng.integers(0, 256, (10, 10), dtype=np.uint8)
    r = oracle.correlate(img, T)
    assert r[10, 5] == 0.0
    flat = np.full((10, 10), 9, np.uint8)      # a constant template
    assert np.all(oracle.correlate(img, flat) == 0.0)


def test_range_is_minus_one_to_one():
    w = inputs.random_case(21, 90, 70, 9, 5, nT=3, n_crops=1)
    r = oracle.correlate(w.image, w.templates)
    assert np.all(r <= 1.0) and np.all(r >= -1.0)
    assert r[0, w.crops[0][2], w.crops[0][1]] == 1.0


def test_affine_invariance_of_template():
    rng = np.random.default_rng(8)
    img = rng.integers(0, 256, (30, 30), dtype=np.uint8)
    T = rng.integers(0, 100, (7, 7), dtype=np.uint8)
    T2 = (2 * T.astype(np.int64) + 17).astype(np.uint8)   # stays within [0, 255]
    np.testing.assert_allclose(oracle.correlate(img, T2), oracle.correlate(img, T),
                               rtol=0, atol=1e-12)


def test_correlate_at_matches_full_map():
    w = inputs.random_case(2, 64, 50, 12, 9, nT=3, n_crops=2)
    full, sI, sI2, sIT = oracle.correlate(w.image, w.templates, with_sums=True)
    rng = np.random.default_rng(0)
    ys = rng.integers(0, w.Oy, 40)
    xs = rng.integers(0, w.Ox, 40)
    r, a, b, c = oracle.correlate_at(w.image, w.templates, xs, ys, with_sums=True)
    np.testing.assert_array_equal(r, full[:, ys, xs])
    np.testing.assert_array_equal(a, sI[:, ys, xs])
    np.testing.assert_array_equal(b, sI2[:, ys, xs])
    np.testing.assert_array_equal(c, sIT[:, ys, xs])


def test_threads_do_not_change_results():
    w = inputs.random_case(4, 80, 60, 10, 6, nT=2)
    a = oracle.correlate(w.image, w.templates, threads=1)
    b = oracle.correlate(w.image, w.templates, threads=4)
    np.testing.assert_array_equal(a, b)


def test_bank_templates_are_independent():
    w = inputs.random_case(6, 50, 40, 8, 8, nT=4, n_crops=2)
    bank = oracle.correlate(w.image, w.templates)
    for t in range(4):
        np.testing.assert_array_equal(bank[t], oracle.correlate(w.image, w.templates[t]))


def test_golden_hand_worked_example():
    """tests/golden/hand_3x4.json: a 3x4 image with its tables and one
    coefficient worked by hand from the definitions (section 15.8 and the
    Pearson reading of Listing 15-5's coefficient)."""
    with open(os.path.join(GOLDEN, "hand_3x4.json")) as f:
        g = json.load(f)
    img = np.array(g["image"], np.uint8)
    S, Q = oracle.sat(img)
    np.testing.assert_array_equal(S, np.array(g["S"]))
    np.testing.assert_array_equal(Q, np.array(g["Q"]))
    T = np.array(g["template"], np.uint8)
    r, sI, sI2, sIT = oracle.correlate(img, T, with_sums=True)
    for (x, y), want in zip(g["shifts"], g["sums"]):
        assert [sI[y, x], sI2[y, x], sIT[y, x]] == want
    for (x, y), want in zip(g["shifts"], g["r"]):
        assert abs(r[y, x] - want) < 1e-15


def test_golden_regression_fixtures():
    """tests/golden/oracle_fixtures.json is written by make_golden.py, which
    calls only the oracle; this guards the oracle against drift."""
    with open(os.path.join(GOLDEN, "oracle_fixtures.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        w = inputs.NAMED[case["workload"]]() if case["workload"] in inputs.NAMED else \
            inputs.random_case(*case["random_args"])
        S, Q = oracle.sat(w.image)
        assert int(S[-1, -1]) == case["S_corner"] and int(Q[-1, -1]) == case["Q_corner"]
        assert int(S.sum() % (2**61 - 1)) == case["S_mod"]
        assert int(Q.sum() % (2**61 - 1)) == case["Q_mod"]
        xs = np.array(case["xs"]); ys = np.array(case["ys"])
        r, a, b, c = oracle.correlate_at(w.image, w.templates, xs, ys, with_sums=True)
        np.testing.assert_array_equal(a, np.array(case["sumI"]))
        np.testing.assert_array_equal(b, np.array(case["sumI2"]))
        np.testing.assert_array_equal(c, np.array(case["sumIT"]))
        np.testing.assert_allclose(r, np.array(case["r"]), rtol=0, atol=1e-15)
