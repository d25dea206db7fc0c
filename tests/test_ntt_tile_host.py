"""The transform numerator's tile arithmetic (ntt_tile.cuh), run on the host:
every pass of a 256 x 256 tile for all 512 thread indices, the in-place
combination of the two halves and the swizzled read-back, against a
brute-force correlation of the centered values, bit for bit.

The transforms are taken modulo the prime 998244353 with lazily reduced
residues; the correlation C of a window is recovered exactly because
|C| <= 2^14 * wT * hT < p / 2.  The cases reach that bound (constant blocks
at 0 and 255 against constant templates of 173 x 173 = 29929 pixels, where
|C| is 4.90e8 of the 4.99e8 allowed), cover 1 x 1 to 224-wide and 224-tall
templates, and every tile position the kernel keeps (257 - hT rows by
257 - wT columns of shifts).  Needs nvcc (a host-only build), no GPU.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def tile_exe(tmp_path_factory):
    nvcc = shutil.which("nvcc") or os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    out = str(tmp_path_factory.mktemp("ntt") / "ntt_tile_host")
    cmd = [nvcc, "-x", "cu", "-std=c++17", "-O2", "--expt-relaxed-constexpr", "-diag-suppress", "20013",
           "-o", out, os.path.join(HERE, "ntt_tile_host.cu")]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr[-3000:]
    return out


def brute_force(tile, T):
    """Sum over the window of (I - 128)(T - 128) for every non-wrapping shift,
    one template row at a time (int64, exact)."""
    hT, wT = T.shape
    Vy, Vx = 257 - hT, 257 - wT
    I = tile.astype(np.int64) - 128
    Tc = T.astype(np.int64) - 128
    C = np.zeros((Vy, Vx), np.int64)
    for j in range(hT):
        rows = np.lib.stride_tricks.sliding_window_view(I[j:j + Vy], wT, axis=1)  # (Vy, Vx, wT)
        C += rows @ Tc[j]
    return C


def run(exe, tmp_path, tile, T, order=0):
    hT, wT = T.shape
    src, dst = tmp_path / "in.bin", tmp_path / "out.bin"
    src.write_bytes(tile.astype(np.uint8).tobytes() + T.astype(np.uint8).tobytes())
    res = subprocess.run([exe, str(wT), str(hT), str(src), str(dst), str(order)],
                         capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    return np.fromfile(dst, dtype=np.int32).reshape(257 - hT, 257 - wT)


@pytest.mark.parametrize("wT,hT", [(64, 64), (1, 1), (17, 9), (100, 80), (224, 30), (20, 224), (128, 128)])
def test_tile_correlation_exact(tile_exe, tmp_path, wT, hT):
    rng = np.random.default_rng(wT * 1000 + hT)
    tile = rng.integers(0, 256, (256, 256), dtype=np.uint8)
    T = rng.integers(0, 256, (hT, wT), dtype=np.uint8)
    np.testing.assert_array_equal(run(tile_exe, tmp_path, tile, T), brute_force(tile, T))


@pytest.mark.parametrize("img_v,tmpl_v", [(0, 0), (255, 0), (0, 255), (255, 255)])
def test_tile_correlation_at_the_bound(tile_exe, tmp_path, img_v, tmpl_v):
    tile = np.full((256, 256), img_v, np.uint8)
    tile[200:, :] = np.random.default_rng(img_v + tmpl_v).integers(0, 256, (56, 256), dtype=np.uint8)
    T = np.full((173, 173), tmpl_v, np.uint8)
    got = run(tile_exe, tmp_path, tile, T)
    ref = brute_force(tile, T)
    np.testing.assert_array_equal(got, ref)
    assert np.abs(ref).max() >= 29929 * 16129       # 127 * 127 at (255, 255)
    assert np.abs(ref).max() < 998244353 // 2


@pytest.mark.parametrize("order", [1, 2])
@pytest.mark.parametrize("wT,hT", [(64, 64), (17, 9)])
def test_in_place_combination_in_any_item_order(tile_exe, tmp_path, wT, hT, order):
    """The halves are combined in place, each item rewriting only the words
    its own last pass read: visiting the items in another order (item-major,
    threads in reverse) gives the same correlations."""
    rng = np.random.default_rng(wT * 31 + hT + order)
    tile = rng.integers(0, 256, (256, 256), dtype=np.uint8)
    T = rng.integers(0, 256, (hT, wT), dtype=np.uint8)
    np.testing.assert_array_equal(run(tile_exe, tmp_path, tile, T, order), brute_force(tile, T))
