"""GPU parity of the compared summed-area-table builders (The CUDA Handbook,
section 15.8, Figures 15-8 and 15-9): the naive one-thread-per-line build
and the two-pass build (uint32 row sums, column look-back) must give the
oracle's tables bit-exactly, like the fused single pass."""
import numpy as np
import pytest

import oracle
from normalized_cross_correlation_gb300 import inputs

pytestmark = pytest.mark.gpu

POISON = -0x5A5A5A5A5A5A5A5A
VARIANTS = [1, 2]  # NCC_SAT_NAIVE, NCC_SAT_TWO_PASS


def run_variant(ncc, img_np, variant):
    import torch
    H, W = img_np.shape
    img = torch.from_numpy(np.ascontiguousarray(img_np)).cuda()
    S = torch.full((H, W), POISON, dtype=torch.int64, device="cuda")
    Q = torch.full((H, W), POISON, dtype=torch.int64, device="cuda")
    ncc.ncc_sat_build_variant(img, variant, S, Q)
    assert ncc.ncc_sync_status() == 0
    return S.cpu().numpy(), Q.cpu().numpy()


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("H,W", [(1, 1), (1, 5), (7, 1), (3, 200), (129, 131), (128, 128),
                                 (333, 257), (1025, 130), (64, 4100), (300, 385)])
def test_variant_bit_exact_shapes(ncc, variant, H, W):
    rng = np.random.default_rng(H * 7919 + W + variant)
    img = rng.integers(0, 256, (H, W), dtype=np.uint8)
    S, Q = run_variant(ncc, img, variant)
    oS, oQ = oracle.sat(img)
    np.testing.assert_array_equal(S, oS)
    np.testing.assert_array_equal(Q, oQ)


@pytest.mark.parametrize("variant", VARIANTS)
def test_variant_saturated_extremes(ncc, variant):
    img = np.full((260, 1030), 255, np.uint8)
    S, Q = run_variant(ncc, img, variant)
    oS, oQ = oracle.sat(img)
    np.testing.assert_array_equal(S, oS)
    np.testing.assert_array_equal(Q, oQ)


@pytest.mark.parametrize("variant", VARIANTS)
def test_variant_full_4096_matches_fused(ncc, variant):
    # at the SAT workload's size, against the fused builder (itself checked
    # against the oracle in test_sat_gpu) and the oracle's last row
    import torch
    img_np = inputs.sat_4096().image
    S, Q = run_variant(ncc, img_np, variant)
    Sf, Qf = ncc.ncc_sat_build(torch.from_numpy(img_np).cuda())
    np.testing.assert_array_equal(S, Sf.cpu().numpy())
    np.testing.assert_array_equal(Q, Qf.cpu().numpy())
    assert S[-1, -1] == int(img_np.astype(np.int64).sum())
    assert Q[-1, -1] == int((img_np.astype(np.int64) ** 2).sum())


def test_unknown_variant_is_rejected(ncc):
    import torch
    img = torch.zeros((10, 10), dtype=torch.uint8, device="cuda")
    with pytest.raises(ncc.NccError) as e:
        ncc.ncc_sat_build_variant(img, 7)
    assert e.value.code == ncc.NCC_ERR_INVALID_ARG
