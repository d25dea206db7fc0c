"""The Python binding refuses caller tensors that do not fit the call --
wrong shape, dtype, layout or device -- before the library is called, so no
kernel is ever handed a table or an output it would read or write past."""
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture
def no_library_call(ncc, monkeypatch):
    """Makes any library call fail the test: the checks must answer first."""
    def refuse():
        raise AssertionError("the binding reached the library with bad arguments")
    monkeypatch.setattr(ncc, "lib", refuse)
    return ncc


def test_wrong_tables_outputs_and_devices_raise_before_the_library(no_library_call):
    import torch
    ncc = no_library_call
    dev = "cuda"
    img = torch.zeros((64, 80), dtype=torch.uint8, device=dev)
    T = torch.zeros((8, 6), dtype=torch.uint8, device=dev)
    Tb = torch.zeros((3, 8, 6), dtype=torch.uint8, device=dev)
    S = torch.zeros((64, 80), dtype=torch.int64, device=dev)
    Q = torch.zeros((64, 80), dtype=torch.int64, device=dev)
    small = torch.zeros((63, 80), dtype=torch.int64, device=dev)       # one row short
    wide = torch.zeros((64, 81), dtype=torch.int64, device=dev)
    cpuS = torch.zeros((64, 80), dtype=torch.int64)
    i32 = torch.zeros((64, 80), dtype=torch.int32, device=dev)
    strided = torch.zeros((64, 160), dtype=torch.int64, device=dev)[:, ::2]
    out1 = torch.zeros((57, 75), dtype=torch.float32, device=dev)       # the right map
    out_bad = torch.zeros((57, 74), dtype=torch.float32, device=dev)
    out3_bad = torch.zeros((2, 57, 75), dtype=torch.float32, device=dev)
    out_cpu = torch.zeros((57, 75), dtype=torch.float32)
    refused = [
        lambda: ncc.ncc_sat_build(img, small, Q),
        lambda: ncc.ncc_sat_build(img, S, wide),
        lambda: ncc.ncc_sat_build(img, cpuS, Q),
        lambda: ncc.ncc_sat_build(img, i32, Q),
        lambda: ncc.ncc_sat_build(img, strided, Q),
        lambda: ncc.ncc_sat_build_variant(img, ncc.NCC_SAT_NAIVE, S, small),
        lambda: ncc.ncc_sat_build_noalloc(img, small, Q),
        lambda: ncc.ncc_sat_build_noalloc(img, S, cpuS),
        lambda: ncc.ncc_correlate(img, T, small, Q),
        lambda: ncc.ncc_correlate(img, T, S, cpuS),
        lambda: ncc.ncc_correlate(img, T, S, Q, out=out_bad),
        lambda: ncc.ncc_correlate(img, T, S, Q, out=out_cpu),
        lambda: ncc.ncc_correlate(img, T.cpu(), S, Q, out=out1),
        lambda: ncc.ncc_correlate_bank(img, Tb, S, wide),
        lambda: ncc.ncc_correlate_bank(img, Tb, S, Q, out=out3_bad),
        lambda: ncc.ncc_correlate_bank(img, Tb, S, Q, out=out1),
        lambda: ncc.ncc_correlate_moments(img, Tb, small, Q),
        lambda: ncc.ncc_correlate_moments(img, Tb, S, i32),
        lambda: ncc.ncc_correlate_direct(img, Tb, out=out3_bad),
        lambda: ncc.ncc_match(img, Tb, S, small),
        lambda: ncc.ncc_match(img, Tb, S, Q, out=out3_bad),
        lambda: ncc.ncc_match(img, Tb, cpuS, Q),
    ]
    for call in refused:
        with pytest.raises((TypeError, ValueError)):
            call()
