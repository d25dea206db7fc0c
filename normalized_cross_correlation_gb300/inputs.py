"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module only draws pixels: it holds none of the correlation arithmetic
(no prefix sums, no window sums, no coefficients), so the CUDA path and the
CPU oracle can both consume its arrays without sharing any of the method.

Every generator uses ``numpy.random.default_rng(seed)`` (PCG64) with a fixed
draw order.  Crop offsets are (x, y): column, then row.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass
class Workload:
    """One image, its templates and where exact crops of the image sit.

    ``templates`` is uint8 [nT][hT][wT]; ``crops`` lists (t, x, y) triples for
    templates that are exact copies of the image window at (x, y).
    """
    name: str
    image: np.ndarray
    templates: np.ndarray | None
    crops: list[tuple[int, int, int]] = field(default_factory=list)

    @property
    def W(self) -> int:
        return int(self.image.shape[1])

    @property
    def H(self) -> int:
        return int(self.image.shape[0])

    @property
    def nT(self) -> int:
        return 0 if self.templates is None else int(self.templates.shape[0])

    @property
    def wT(self) -> int:
        return int(self.templates.shape[2])

    @property
    def hT(self) -> int:
        return int(self.templates.shape[1])

    @property
    def Ox(self) -> int:
        return self.W - self.wT + 1

    @property
    def Oy(self) -> int:
        return self.H - self.hT + 1


def uniform_image(rng: np.random.Generator, H: int, W: int) -> np.ndarray:
    """i.i.d. uniform pixels in [0, 255]."""
    return rng.integers(0, 256, (H, W), dtype=np.uint8)


def box_blurred_image(rng: np.random.Generator, H: int, W: int, k: int) -> np.ndarray:
    """Uniform noise of size (H+k-1) x (W+k-1) averaged over k x k windows
    (valid windows only, so no border rule is needed), rounded half to even
    and clipped to [0, 255]."""
    noise = rng.integers(0, 256, (H + k - 1, W + k - 1), dtype=np.uint8)
    acc = np.zeros((H, W), np.int32)
    for dy in range(k):
        for dx in range(k):
            acc += noise[dy:dy + H, dx:dx + W]
    return np.clip(np.rint(acc / float(k * k)), 0, 255).astype(np.uint8)


def crop(img: np.ndarray, x: int, y: int, w: int, h: int) -> np.ndarray:
    return np.ascontiguousarray(img[y:y + h, x:x + w])


# --------------------------------------------------------------------------
# The five named workloads and the headline case.
# --------------------------------------------------------------------------

def tiny_ncc(seed: int = 0) -> Workload:
    """256x256 uniform image; template = 16x16 crop at (x=100, y=37)."""
    rng = np.random.default_rng(seed)
    img = uniform_image(rng, 256, 256)
    T = crop(img, 100, 37, 16, 16)[None]
    return Workload("tiny_ncc_256_t16", img, T, [(0, 100, 37)])


def smooth_1024(seed: int = 1) -> Workload:
    """1024x1024 7x7-box-blurred noise; template = 32x32 crop at (500, 300)
    plus i.i.d. integer noise in [-8, 8], clipped to [0, 255]."""
    rng = np.random.default_rng(seed)
    img = box_blurred_image(rng, 1024, 1024, 7)
    base = crop(img, 500, 300, 32, 32).astype(np.int16)
    noise = rng.integers(-8, 9, (32, 32)).astype(np.int16)
    T = np.clip(base + noise, 0, 255).astype(np.uint8)[None]
    return Workload("smooth_1024_t32", img, T, [])


def sat_4096(seed: int = 2) -> Workload:
    """4096x4096 uniform image, tables only (no template)."""
    rng = np.random.default_rng(seed)
    img = uniform_image(rng, 4096, 4096)
    return Workload("sat_4096", img, None, [])


def headline_4096(seed: int = 2) -> Workload:
    """The 4096x4096 uniform image of :func:`sat_4096` with one 16x16 template
    cropped at an offset drawn, after the image, from the same stream."""
    rng = np.random.default_rng(seed)
    img = uniform_image(rng, 4096, 4096)
    x, y = (int(v) for v in rng.integers(0, 4096 - 16 + 1, 2))
    T = crop(img, x, y, 16, 16)[None]
    return Workload("ncc_4096_t16", img, T, [(0, x, y)])


def bank_2048(seed: int = 3) -> Workload:
    """2048x2048 uniform image; 64 templates of 16x16: 0-31 are crops at
    seeded offsets, 32-63 are uniform noise."""
    rng = np.random.default_rng(seed)
    img = uniform_image(rng, 2048, 2048)
    offs = rng.integers(0, 2048 - 16 + 1, (32, 2))
    rand_t = rng.integers(0, 256, (32, 16, 16), dtype=np.uint8)
    crops = [crop(img, int(x), int(y), 16, 16) for x, y in offs]
    T = np.concatenate([np.stack(crops), rand_t], axis=0)
    return Workload("bank_2048_64x16", img, np.ascontiguousarray(T),
                    [(t, int(offs[t, 0]), int(offs[t, 1])) for t in range(32)])


def large_8192(seed: int = 4) -> Workload:
    """8192x8192 5x5-box-blurred noise with 20% of pixels saturated to 0 or
    255 (equal odds); template = 64x64 crop at (4000, 6000) after saturation."""
    rng = np.random.default_rng(seed)
    img = box_blurred_image(rng, 8192, 8192, 5)
    mask = rng.random((8192, 8192)) < 0.2
    sat = (rng.integers(0, 2, (8192, 8192), dtype=np.uint8) * np.uint8(255))
    img[mask] = sat[mask]
    T = crop(img, 4000, 6000, 64, 64)[None]
    return Workload("large_8192_t64", img, T, [(0, 4000, 6000)])


def wide_4096(seed: int = 5) -> Workload:
    """4096x4096 3x3-box-blurred noise; template = 128x128 crop at
    (1500, 2500): wider than the Toeplitz tensor-core kernel takes, so the
    transform numerator serves it (about 4096 dp4a per output otherwise)."""
    rng = np.random.default_rng(seed)
    img = box_blurred_image(rng, 4096, 4096, 3)
    T = crop(img, 1500, 2500, 128, 128)[None]
    return Workload("wide_4096_t128", img, T, [(0, 1500, 2500)])


def sat_8192(seed: int = 4) -> Workload:
    """The 8192x8192 image of :func:`large_8192`, tables only (no template)."""
    return Workload("sat_8192", large_8192(seed).image, None, [])


NAMED = {
    "tiny_ncc_256_t16": tiny_ncc,
    "smooth_1024_t32": smooth_1024,
    "sat_4096": sat_4096,
    "ncc_4096_t16": headline_4096,
    "bank_2048_64x16": bank_2048,
    "large_8192_t64": large_8192,
    "wide_4096_t128": wide_4096,
    "sat_8192": sat_8192,
}


def batch_shifts(n: int, W: int, H: int, seed: int = 77) -> np.ndarray:
    """Seeded circular shifts (dy, dx) that turn one workload image into a
    batch of n distinct images of the same pixel distribution (image 0 is
    unshifted).  Only offsets are drawn here; applying them is a copy."""
    rng = np.random.default_rng(seed)
    d = np.stack([rng.integers(1, max(2, H), n), rng.integers(1, max(2, W), n)], axis=1)
    d[0] = 0
    return d


def random_case(seed: int, W: int, H: int, wT: int, hT: int, nT: int = 1,
                n_crops: int = 1) -> Workload:
    """Uniform image of arbitrary (ragged) size with nT templates; the first
    ``n_crops`` templates are crops at seeded offsets, the rest noise."""
    rng = np.random.default_rng(seed)
    img = uniform_image(rng, H, W)
    n_crops = min(n_crops, nT)
    offs = rng.integers(0, [W - wT + 1, H - hT + 1], (n_crops, 2)) if n_crops else []
    Ts = [crop(img, int(x), int(y), wT, hT) for x, y in offs]
    if nT > n_crops:
        Ts.extend(rng.integers(0, 256, (nT - n_crops, hT, wT), dtype=np.uint8))
    T = np.ascontiguousarray(np.stack(Ts)) if Ts else None
    return Workload(f"random_{W}x{H}_t{wT}x{hT}x{nT}", img, T,
                    [(t, int(offs[t][0]), int(offs[t][1])) for t in range(n_crops)])
