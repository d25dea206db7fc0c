"""ncc_sat_build_noalloc: the table builder for callers that cannot allocate
device memory (host callbacks and real-time loops, where cudaMalloc may
synchronize the device; frameworks that own every allocation).  It must give
exactly the tables of the allocating entry point -- and so the oracle's --
call after call, from its fixed scratch array.

This file is collected last on purpose: it also has to pass after every
other test has run in the same process (the scratch then holds an earlier
call's contents), and it passes when run alone in a fresh process (the first
call sets up the scratch address)."""
import numpy as np
import pytest

import oracle
from normalized_cross_correlation_gb300 import inputs

pytestmark = pytest.mark.gpu

POISON = -0x3C3C3C3C3C3C3C3C


def call_noalloc(ncc, img):
    """Calls the entry point through the C ABI into poisoned tables."""
    import torch
    H, W = img.shape
    S = torch.full((H, W), POISON, dtype=torch.int64, device="cuda")
    Q = torch.full((H, W), POISON, dtype=torch.int64, device="cuda")
    rc = ncc.lib().ncc_sat_build_noalloc(img.data_ptr(), W, H, S.data_ptr(), Q.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream)
    assert rc == ncc.NCC_OK, ncc.ncc_status_string(rc)
    assert ncc.ncc_sync_status() == ncc.NCC_OK
    return S, Q


def test_noalloc_tables_equal_the_allocating_builder_twice_in_a_row(ncc):
    import torch
    rng = np.random.default_rng(2024)
    images = [rng.integers(0, 256, (777, 1001), dtype=np.uint8),   # ragged, unaligned width
              inputs.sat_4096().image]                              # the 4096x4096 workload
    for img_np in images:                                           # two calls in a row
        img = torch.from_numpy(img_np).cuda()
        S_ref, Q_ref = ncc.ncc_sat_build(img)
        S, Q = call_noalloc(ncc, img)
        assert torch.equal(S, S_ref), "S differs from ncc_sat_build"
        assert torch.equal(Q, Q_ref), "Q differs from ncc_sat_build"
        oS, oQ = oracle.sat(img_np)
        np.testing.assert_array_equal(S.cpu().numpy(), oS)
        np.testing.assert_array_equal(Q.cpu().numpy(), oQ)
    # and once more on the first image, after the scratch held the larger one
    img = torch.from_numpy(images[0]).cuda()
    S_ref, Q_ref = ncc.ncc_sat_build(img)
    S, Q = call_noalloc(ncc, img)
    assert torch.equal(S, S_ref) and torch.equal(Q, Q_ref)


def test_noalloc_rejects_images_beyond_its_scratch(ncc):
    import torch
    img = torch.zeros((8192, 8192), dtype=torch.uint8, device="cuda")
    S = torch.empty((8192, 8192), dtype=torch.int64, device="cuda")
    Q = torch.empty((8192, 8192), dtype=torch.int64, device="cuda")
    rc = ncc.lib().ncc_sat_build_noalloc(img.data_ptr(), 8192, 8192, S.data_ptr(), Q.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream)
    assert rc == ncc.NCC_ERR_UNSUPPORTED
    assert ncc.ncc_sync_status() == ncc.NCC_OK
