"""Helpers shared by the GPU tests: device copies, and output buffers filled
with values no kernel writes, so that a cell a kernel skips can never pass a
comparison by holding an earlier result (a NaN fails every closeness test;
the int64 poison is no sum of 8-bit pixels)."""
import numpy as np

I64_POISON = -0x3C3C3C3C3C3C3C3C


def to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def nan_map(*shape):
    """A float32 CUDA buffer of the given shape, every cell NaN."""
    import torch
    return torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")


def poisoned_i64(*shape):
    import torch
    return torch.full(shape, I64_POISON, dtype=torch.int64, device="cuda")


def moments(ncc, dimg, dt, S=None, Q=None, direct=False):
    """(SumI, SumI2, SumIT) of templates dt [nT][hT][wT] against dimg through
    the C ABI, into poisoned int64 buffers: ncc_correlate_moments when S and
    Q are given, ncc_correlate_direct_moments when direct is set."""
    import torch
    if dt.dim() == 2:
        dt = dt.unsqueeze(0)
    H, W = dimg.shape
    nT, hT, wT = dt.shape
    Oy, Ox = H - hT + 1, W - wT + 1
    sI, sI2, sIT = poisoned_i64(Oy, Ox), poisoned_i64(Oy, Ox), poisoned_i64(nT, Oy, Ox)
    h = torch.cuda.current_stream().cuda_stream
    L = ncc.lib()
    if direct:
        rc = L.ncc_correlate_direct_moments(dimg.data_ptr(), W, H, dt.data_ptr(), wT, hT, nT,
                                            sI.data_ptr(), sI2.data_ptr(), sIT.data_ptr(), h)
    else:
        rc = L.ncc_correlate_moments(dimg.data_ptr(), W, H, dt.data_ptr(), wT, hT, nT,
                                     S.data_ptr(), Q.data_ptr(), sI.data_ptr(), sI2.data_ptr(),
                                     sIT.data_ptr(), h)
    assert rc == ncc.NCC_OK, ncc.ncc_status_string(rc)
    assert ncc.ncc_sync_status() == ncc.NCC_OK
    return sI, sI2, sIT
