"""The seeded synthetic workloads keep the shapes, value distributions and
structure the configurations describe (CPU only): exact crops where a
template is a crop, the stated noise on the smooth workload's template, the
saturated fraction of the large one, and the same arrays for the same seed."""
import numpy as np

from normalized_cross_correlation_gb300 import inputs


def test_tiny_workload():
    w = inputs.tiny_ncc()
    assert w.image.shape == (256, 256) and w.image.dtype == np.uint8
    assert w.templates.shape == (1, 16, 16)
    assert (w.Ox, w.Oy) == (241, 241)
    np.testing.assert_array_equal(w.templates[0], w.image[37:53, 100:116])
    assert w.crops == [(0, 100, 37)]
    # i.i.d. uniform over 0..255: every value appears, the mean is near 127.5
    assert np.unique(w.image).size == 256
    assert abs(float(w.image.mean()) - 127.5) < 2.0


def test_smooth_workload():
    w = inputs.smooth_1024()
    assert w.image.shape == (1024, 1024) and w.templates.shape == (1, 32, 32)
    # a 7x7 box blur of uniform noise: far smaller spread than uniform (std 73.9)
    assert float(w.image.std()) < 15.0
    diff = w.templates[0].astype(int) - w.image[300:332, 500:532].astype(int)
    assert diff.min() >= -8 and diff.max() <= 8 and np.any(diff != 0)


def test_headline_and_sat_workloads_share_the_image():
    h = inputs.headline_4096()
    s = inputs.sat_4096()
    np.testing.assert_array_equal(h.image, s.image)
    assert s.templates is None and h.templates.shape == (1, 16, 16)
    (t, x, y), = h.crops
    np.testing.assert_array_equal(h.templates[0], h.image[y:y + 16, x:x + 16])
    assert (h.Ox, h.Oy) == (4081, 4081)


def test_bank_workload():
    w = inputs.bank_2048()
    assert w.image.shape == (2048, 2048) and w.templates.shape == (64, 16, 16)
    assert len(w.crops) == 32
    for t, x, y in w.crops:
        np.testing.assert_array_equal(w.templates[t], w.image[y:y + 16, x:x + 16])
    # templates 32-63 are drawn noise: none repeats a crop template
    assert not any(np.array_equal(w.templates[32 + k], w.templates[k]) for k in range(32))


def test_large_workload():
    w = inputs.large_8192()
    assert w.image.shape == (8192, 8192) and w.templates.shape == (1, 64, 64)
    np.testing.assert_array_equal(w.templates[0], w.image[6000:6064, 4000:4064])
    # 20 % saturated to 0 or 255 with equal odds, on top of a 5x5 blur (which
    # itself almost never reaches 0 or 255)
    lo = float(np.mean(w.image == 0))
    hi = float(np.mean(w.image == 255))
    assert abs(lo - 0.1) < 0.005 and abs(hi - 0.1) < 0.005


def test_wide_workload():
    """The transform numerator's workload: a 3x3 box blur of uniform noise
    (values spread around 128, none saturated) with a 128x128 crop."""
    w = inputs.wide_4096()
    assert w.image.shape == (4096, 4096) and w.templates.shape == (1, 128, 128)
    np.testing.assert_array_equal(w.templates[0], w.image[2500:2628, 1500:1628])
    assert abs(float(w.image.mean()) - 127.5) < 0.5
    assert abs(float(w.image.std()) - 73.9 / 3) < 0.5   # a 3x3 mean of uniform bytes


def test_generators_are_deterministic():
    a, b = inputs.random_case(7, 300, 200, 9, 5, nT=3, n_crops=2), \
        inputs.random_case(7, 300, 200, 9, 5, nT=3, n_crops=2)
    np.testing.assert_array_equal(a.image, b.image)
    np.testing.assert_array_equal(a.templates, b.templates)
    assert a.crops == b.crops
    c = inputs.random_case(8, 300, 200, 9, 5, nT=3, n_crops=2)
    assert not np.array_equal(a.image, c.image)
