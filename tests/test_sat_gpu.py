"""GPU parity of ncc_sat_build against the oracle's tables: S and Q must be
bit-exact (The CUDA Handbook, section 15.8)."""
import numpy as np
import pytest

import oracle
from normalized_cross_correlation_gb300 import inputs

pytestmark = pytest.mark.gpu

POISON = -0x5A5A5A5A5A5A5A5A


def run_sat(ncc, img_np, img_offset=0, table_offset=0):
    """Runs the builder through the C ABI.  Offsets (in elements) shift the
    image / table pointers inside larger buffers to exercise the unaligned
    load and store paths; the tables are poisoned first so an unwritten
    cell cannot pass."""
    import torch
    H, W = img_np.shape
    n = H * W
    ibuf = torch.zeros(n + 64, dtype=torch.uint8, device="cuda")
    ibuf[img_offset:img_offset + n] = torch.from_numpy(img_np.ravel()).cuda()
    sbuf = torch.full((n + 8,), POISON, dtype=torch.int64, device="cuda")
    qbuf = torch.full((n + 8,), POISON, dtype=torch.int64, device="cuda")
    rc = ncc.lib().ncc_sat_build(ibuf.data_ptr() + img_offset, W, H,
                                 sbuf.data_ptr() + 8 * table_offset,
                                 qbuf.data_ptr() + 8 * table_offset,
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == 0, ncc.ncc_status_string(rc)
    assert ncc.ncc_sync_status() == 0
    S = sbuf[table_offset:table_offset + n].view(H, W).cpu().numpy()
    Q = qbuf[table_offset:table_offset + n].view(H, W).cpu().numpy()
    return S, Q


def check_exact(ncc, img, **kw):
    S, Q = run_sat(ncc, img, **kw)
    oS, oQ = oracle.sat(img)
    np.testing.assert_array_equal(S, oS)
    np.testing.assert_array_equal(Q, oQ)


@pytest.mark.parametrize("H,W", [(1, 1), (1, 5), (7, 1), (3, 200), (129, 131), (128, 128),
                                 (256, 256), (333, 257), (777, 1000), (130, 127), (1025, 130),
                                 (64, 4100)])
def test_sat_bit_exact_shapes(ncc, H, W):
    rng = np.random.default_rng(H * 7919 + W)
    check_exact(ncc, rng.integers(0, 256, (H, W), dtype=np.uint8))


def test_sat_tiny_workload(ncc):
    check_exact(ncc, inputs.tiny_ncc().image)


def test_sat_saturated_image_extremes(ncc):
    # all-255 pixels: the largest row sums of squares and table values
    check_exact(ncc, np.full((300, 4104), 255, np.uint8))
    check_exact(ncc, np.zeros((200, 300), np.uint8))


def test_sat_widest_rows(ncc):
    # W = 66051 is the widest row whose running sum of squares fits uint32
    img = np.full((3, 66051), 255, np.uint8)
    img[1, ::7] = 0
    check_exact(ncc, img)


@pytest.mark.parametrize("img_offset,table_offset", [(1, 0), (0, 1), (3, 1)])
def test_sat_unaligned_pointers(ncc, img_offset, table_offset):
    rng = np.random.default_rng(99)
    check_exact(ncc, rng.integers(0, 256, (261, 388), dtype=np.uint8),
                img_offset=img_offset, table_offset=table_offset)


def test_sat_full_4096(ncc):
    check_exact(ncc, inputs.sat_4096().image)


def test_sat_full_8192(ncc):
    check_exact(ncc, inputs.large_8192().image)


def test_sat_repeated_calls_agree(ncc):
    import torch
    img = torch.from_numpy(inputs.tiny_ncc().image).cuda()
    S1, Q1 = ncc.ncc_sat_build(img)
    for _ in range(5):
        S2, Q2 = ncc.ncc_sat_build(img)
        assert torch.equal(S1, S2) and torch.equal(Q1, Q2)
    assert ncc.ncc_sync_status() == 0


def test_lookback_timeout_is_reported_and_recovers(ncc):
    """A tile that never publishes makes its successors' bounded waits run
    out: the status word reports NCC_ERR_TIMEOUT, the kernel returns, and the
    next call works normally."""
    import torch
    rng = np.random.default_rng(5)
    img_np = rng.integers(0, 256, (512, 512), dtype=np.uint8)
    img = torch.from_numpy(img_np).cuda()
    try:
        ncc.ncc_debug_set_fault(0, 20_000_000)      # tile 0 silent, 20 ms limit
        ncc.ncc_sat_build(img)
        assert ncc.ncc_sync_status() == ncc.NCC_ERR_TIMEOUT
        assert ncc.ncc_sync_status() == 0           # the word was cleared
    finally:
        ncc.ncc_debug_set_fault(-1, 0)
    # the calls after an aborted one must still write every cell (poisoned
    # buffers catch a call that silently does nothing)
    oS, oQ = oracle.sat(img_np)
    for _ in range(2):
        S, Q = run_sat(ncc, img_np)
        np.testing.assert_array_equal(S, oS)
        np.testing.assert_array_equal(Q, oQ)
    other = rng.integers(0, 256, (300, 700), dtype=np.uint8)
    check_exact(ncc, other)


def test_host_path_allocation_failure_reports_nomem_and_recovers(ncc):
    """A device allocation that fails (forced by the host-side hook) makes
    the call return NCC_ERR_NOMEM without launching anything; the next call
    allocates and computes normally."""
    w = inputs.random_case(404, 300, 200, 16, 16, nT=1, n_crops=1)
    out = np.full((1, w.Oy, w.Ox), np.nan, np.float32)
    ncc.ncc_debug_fail_alloc(1)
    try:
        with pytest.raises(ncc.NccError) as e:
            ncc.ncc_match_host(w.image, w.templates, out)
        assert e.value.code == ncc.NCC_ERR_NOMEM
        assert np.all(np.isnan(out))                 # nothing ran
    finally:
        ncc.ncc_debug_fail_alloc(0)
    assert ncc.ncc_sync_status() == 0
    ncc.ncc_match_host(w.image, w.templates, out)
    ref = oracle.correlate(w.image, w.templates[0])
    np.testing.assert_allclose(out[0], ref, rtol=0, atol=1e-5)


FRESH_PROCESS_NOMEM = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, {root!r})
import oracle
from normalized_cross_correlation_gb300 import ncc
img_np = np.random.default_rng(9).integers(0, 256, (300, 500), dtype=np.uint8)
img = torch.from_numpy(img_np).cuda()
ncc.ncc_debug_fail_alloc(1)            # the look-back workspace's first allocation fails
try:
    ncc.ncc_sat_build(img)
    sys.exit(3)
except ncc.NccError as e:
    if e.code != ncc.NCC_ERR_NOMEM:
        sys.exit(4)
if ncc.ncc_sync_status() != 0:
    sys.exit(5)
S, Q = ncc.ncc_sat_build(img)          # allocates now
if ncc.ncc_sync_status() != 0:
    sys.exit(6)
oS, oQ = oracle.sat(img_np)
sys.exit(0 if np.array_equal(S.cpu().numpy(), oS) and np.array_equal(Q.cpu().numpy(), oQ) else 7)
"""


def test_workspace_allocation_failure_in_a_fresh_process(ncc):
    """The SAT builder's look-back workspace is allocated on a device's first
    build: in a fresh process, a forced failure there gives NCC_ERR_NOMEM,
    and the following build allocates it and writes the oracle's tables."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    res = subprocess.run([sys.executable, "-c", FRESH_PROCESS_NOMEM.format(root=root)],
                         capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, (res.returncode, res.stdout[-2000:], res.stderr[-2000:])
