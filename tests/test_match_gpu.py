"""GPU parity of ncc_match, the combined call (SAT build, then the
correlation, whose single-template launch overlaps the build's tail).

Its tables and coefficients must equal, bit for bit, those of the separate
ncc_sat_build + ncc_correlate(_bank) calls (which the other GPU tests hold to
the oracle), and on small cases the oracle directly: tables bit-exact,
coefficients within 1e-5 absolute.
"""
import numpy as np
import pytest

import oracle
from gpu_util import nan_map, to_dev
from normalized_cross_correlation_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = 1e-5


def separate(ncc, dimg, dt):
    S, Q = ncc.ncc_sat_build(dimg)
    nT, hT, wT = dt.shape
    Oy, Ox = dimg.shape[0] - hT + 1, dimg.shape[1] - wT + 1
    if nT > 1:
        out = ncc.ncc_correlate_bank(dimg, dt, S, Q, out=nan_map(nT, Oy, Ox))
    else:
        out = ncc.ncc_correlate(dimg, dt[0], S, Q, out=nan_map(Oy, Ox)).unsqueeze(0)
    assert ncc.ncc_sync_status() == 0
    return S.cpu().numpy(), Q.cpu().numpy(), out.cpu().numpy()


# (W, H, wT, hT, nT): TMA paths with the fixed 16-row kernel, the plain-load
# paths (odd width), other heights, a bank, ragged last tiles
SHAPES = [
    (1024, 768, 16, 16, 1), (523, 300, 7, 5, 1), (2048, 1100, 8, 8, 1), (1000, 260, 13, 31, 1),
    (640, 480, 16, 16, 4), (272, 200, 16, 16, 1),
    # several templates where the bank kernel does not apply (odd width): one
    # single-template launch per template, the first one overlapped
    (523, 300, 7, 5, 3),
]


@pytest.mark.parametrize("W,H,wT,hT,nT", SHAPES)
def test_match_equals_separate_calls(ncc, W, H, wT, hT, nT):
    w = inputs.random_case(W * 7 + H * 3 + nT, W, H, wT, hT, nT=nT, n_crops=1)
    dimg, dt = to_dev(w.image), to_dev(w.templates)
    S0, Q0, r0 = separate(ncc, dimg, dt)
    S, Q, r = ncc.ncc_match(dimg, dt, out=nan_map(nT, w.Oy, w.Ox))
    assert ncc.ncc_sync_status() == 0
    np.testing.assert_array_equal(S.cpu().numpy(), S0)
    np.testing.assert_array_equal(Q.cpu().numpy(), Q0)
    np.testing.assert_array_equal(r.cpu().numpy(), r0)


def test_match_small_case_matches_oracle(ncc, threads):
    w = inputs.random_case(4242, 300, 200, 16, 16, nT=1, n_crops=1)
    S, Q, r = ncc.ncc_match(to_dev(w.image), to_dev(w.templates), out=nan_map(1, w.Oy, w.Ox))
    assert ncc.ncc_sync_status() == 0
    oS, oQ = oracle.sat(w.image)
    np.testing.assert_array_equal(S.cpu().numpy(), oS)
    np.testing.assert_array_equal(Q.cpu().numpy(), oQ)
    ref = oracle.correlate(w.image, w.templates[0], threads=threads)
    np.testing.assert_allclose(r.cpu().numpy()[0], ref, rtol=0, atol=TOL)


def test_headline_size_on_a_side_stream_repeatedly(ncc):
    """The bench's configuration (4096x4096, one 16x16 template), five calls
    in a row on a non-default stream, interleaved with the separate calls:
    every result is the same."""
    import torch
    w = inputs.headline_4096()
    dimg, dt = to_dev(w.image), to_dev(w.templates)
    _, _, r0 = separate(ncc, dimg, dt)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        S = torch.empty((w.H, w.W), dtype=torch.int64, device="cuda")
        Q = torch.empty_like(S)
        out = torch.empty((1, w.Oy, w.Ox), dtype=torch.float32, device="cuda")
        for _ in range(5):
            out.fill_(7.0)
            ncc.ncc_match(dimg, dt, S, Q, out, stream=s)
            assert ncc.ncc_sync_status(s) == 0
            np.testing.assert_array_equal(out.cpu().numpy(), r0)
            ncc.ncc_correlate(dimg, dt[0], S, Q, out[0], stream=s)
            assert ncc.ncc_sync_status(s) == 0
            np.testing.assert_array_equal(out.cpu().numpy(), r0)


@pytest.mark.parametrize("W,H,wT,hT,nT,pinned", [
    (1024, 600, 16, 16, 1, True), (1024, 600, 16, 16, 1, False),
    (523, 300, 7, 5, 1, True), (640, 480, 16, 16, 4, True), (640, 480, 16, 16, 4, False),
])
def test_host_entry_point_matches_device_path(ncc, W, H, wT, hT, nT, pinned):
    """ncc_match_host with page-locked output (the kernels store into it
    directly) and with pageable output (a device buffer and a copy back)."""
    import torch
    w = inputs.random_case(W + 5 * H + nT, W, H, wT, hT, nT=nT, n_crops=1)
    _, _, r0 = separate(ncc, to_dev(w.image), to_dev(w.templates))
    img, T = torch.from_numpy(w.image), torch.from_numpy(w.templates)
    out = torch.full((nT, w.Oy, w.Ox), 7.0, dtype=torch.float32)
    if pinned:
        img, T, out = img.pin_memory(), T.pin_memory(), out.pin_memory()
    for _ in range(2):                        # the second call reuses the pooled buffers
        out.fill_(7.0)
        ncc.ncc_match_host(img, T, out)
        np.testing.assert_array_equal(out.numpy(), r0)


# Single-template maps of at least 8 MB on the dp4a kernel: the host-buffer
# call correlates them in bands of whole tiles and copies each band back
# while the next one is computed.  (W, H, wT, hT): 1085 output rows in 6
# bands of 192 (the last ragged) on 128x32 tiles; 8 bands on 128x32 tiles;
# 128x64 tiles (a 20-wide template on a map with enough tiles); the
# plain-load path (a width that is not a multiple of 16).
BANDED = [(2048, 1100, 16, 16), (1536, 1500, 13, 7), (2560, 1100, 20, 20), (2051, 1100, 16, 16)]


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("W,H,wT,hT", BANDED)
def test_host_entry_point_in_bands(ncc, threads, W, H, wT, hT, pinned):
    import torch
    w = inputs.random_case(W * 3 + H + wT, W, H, wT, hT, nT=1, n_crops=1)
    assert w.Ox * w.Oy * 4 >= 8 << 20
    _, _, r0 = separate(ncc, to_dev(w.image), to_dev(w.templates))
    img, T = torch.from_numpy(w.image), torch.from_numpy(w.templates)
    out = torch.full((1, w.Oy, w.Ox), float("nan"), dtype=torch.float32)
    if pinned:
        img, T, out = img.pin_memory(), T.pin_memory(), out.pin_memory()
    for _ in range(2):                        # the second call reuses the pooled buffers
        out.fill_(float("nan"))
        ncc.ncc_match_host(img, T, out)
        assert ncc.lib().ncc_debug_last_path() == ncc.NCC_PATH_DP4A
        np.testing.assert_array_equal(out.numpy(), r0)
    if pinned and W == 2048:
        ref = oracle.correlate(w.image, w.templates[0], threads=threads)
        np.testing.assert_allclose(out.numpy()[0], ref, rtol=0, atol=TOL)


def test_match_on_two_streams_at_once(ncc):
    """Two images matched on two streams with their calls interleaved: the
    builds share the library's look-back workspace (ordered through an
    event) and each correlation overlaps its own stream's build."""
    import torch
    wa = inputs.random_case(501, 1536, 1100, 16, 16, nT=1, n_crops=1)
    wb = inputs.random_case(502, 1024, 1400, 12, 9, nT=1, n_crops=1)
    ref = []
    for w in (wa, wb):
        _, _, r0 = separate(ncc, to_dev(w.image), to_dev(w.templates))
        ref.append(r0)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    da, ta = to_dev(wa.image), to_dev(wa.templates)
    db, tb = to_dev(wb.image), to_dev(wb.templates)
    torch.cuda.synchronize()
    outs = []
    for _ in range(3):
        with torch.cuda.stream(sa):
            ra = ncc.ncc_match(da, ta, stream=sa)[2]
        with torch.cuda.stream(sb):
            rb = ncc.ncc_match(db, tb, stream=sb)[2]
        outs.append((ra, rb))
    torch.cuda.synchronize()
    assert ncc.ncc_sync_status() == 0
    for ra, rb in outs:
        np.testing.assert_array_equal(ra.cpu().numpy(), ref[0])
        np.testing.assert_array_equal(rb.cpu().numpy(), ref[1])
