"""Thin Python binding of the C ABI in include/ncc.h.

Argument marshalling only: every step of the path runs in the CUDA kernels
of libncc_gb300.so.  Tensors are torch tensors (PyTorch provides device
memory and streams); the functions keep the C names.  There is no CPU
fallback: if the library is missing, loading it raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import _build

NCC_OK = 0
NCC_ERR_INVALID_ARG = -1
NCC_ERR_UNSUPPORTED = -2
NCC_ERR_CUDA = -3
NCC_ERR_TIMEOUT = -4
NCC_ERR_NOMEM = -5
NCC_ERR_BOUNDS = -6

NCC_SAT_FUSED = 0      # the single-pass tiled look-back (ncc_sat_build)
NCC_SAT_NAIVE = 1      # one thread per row, then one thread per column
NCC_SAT_TWO_PASS = 2   # uint32 row sums, then a column look-back scan

EXPORTS = ("ncc_sat_build", "ncc_sat_build_noalloc", "ncc_sat_build_variant", "ncc_correlate", "ncc_correlate_bank", "ncc_correlate_moments",
           "ncc_correlate_direct", "ncc_correlate_direct_moments",
           "ncc_match", "ncc_match_host", "ncc_sync_status", "ncc_status_string", "ncc_version",
           "ncc_debug_set_fault", "ncc_debug_fail_alloc", "ncc_debug_set_path",
           "ncc_debug_last_path")

_lock = threading.Lock()
_lib = None


class NccError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {code} ({status_text(code)})")


def library_path() -> str:
    """The library to load: the regular build, or the build with device-side
    index checks when NCC_GB300_LIBRARY=debug is set in the environment."""
    return _build.DEBUG_LIB_PATH if os.environ.get("NCC_GB300_LIBRARY") == "debug" else _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library {path} is missing; build it with "
                    "normalized_cross_correlation_gb300._build.build()")
            L = ctypes.CDLL(path)
            vp, i, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64
            L.ncc_sat_build.argtypes = [vp, i, i, vp, vp, vp]
            L.ncc_sat_build_noalloc.argtypes = [vp, i, i, vp, vp, vp]
            L.ncc_sat_build_variant.argtypes = [vp, i, i, vp, vp, i, vp]
            L.ncc_correlate.argtypes = [vp, i, i, vp, i, i, vp, vp, vp, vp]
            L.ncc_correlate_bank.argtypes = [vp, i, i, vp, i, i, i, vp, vp, vp, vp]
            L.ncc_correlate_moments.argtypes = [vp, i, i, vp, i, i, i, vp, vp, vp, vp, vp, vp]
            L.ncc_correlate_direct.argtypes = [vp, i, i, vp, i, i, i, vp, vp]
            L.ncc_correlate_direct_moments.argtypes = [vp, i, i, vp, i, i, i, vp, vp, vp, vp]
            L.ncc_match.argtypes = [vp, i, i, vp, i, i, i, vp, vp, vp, vp]
            L.ncc_match_host.argtypes = [vp, i, i, vp, i, i, i, vp, vp]
            L.ncc_sync_status.argtypes = [vp]
            L.ncc_status_string.argtypes = [i]
            L.ncc_status_string.restype = ctypes.c_char_p
            L.ncc_version.argtypes = []
            L.ncc_debug_set_fault.argtypes = [i, u64]
            L.ncc_debug_fail_alloc.argtypes = [i]
            L.ncc_debug_set_path.argtypes = [i]
            L.ncc_debug_last_path.argtypes = []
            for name in EXPORTS:
                if name != "ncc_status_string":
                    getattr(L, name).restype = ctypes.c_int
            _lib = L
    return _lib


def status_text(code: int) -> str:
    try:
        return lib().ncc_status_string(int(code)).decode()
    except Exception:  # the text is only decoration for an error message
        return "?"


def _check(code: int, where: str) -> None:
    if code != NCC_OK:
        raise NccError(code, where)


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t, dtype, ndim: int, name: str, like=None, shape=None):
    """Checks that t is a contiguous CUDA tensor of the given dtype and rank,
    on the same device as `like` and of exactly `shape` when those are given,
    so that no kernel is handed a buffer it would read or write past."""
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype or t.dim() != ndim or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous {dtype} tensor with {ndim} dims")
    if like is not None and t.device != like.device:
        raise ValueError(f"{name} is on {t.device}, the image on {like.device}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


def _tables(img, S, Q):
    """Caller tables: int64 [H][W] on the image's device."""
    import torch
    _dev(S, torch.int64, 2, "S", img, img.shape)
    _dev(Q, torch.int64, 2, "Q", img, img.shape)


def _map_shape(img, nT, hT, wT):
    H, W = img.shape
    return (nT, max(H - hT + 1, 0), max(W - wT + 1, 0))


def _tmpl3(t):
    return t.unsqueeze(0) if t.dim() == 2 else t


# --------------------------------------------------------------------------
# Entry points (C names).
# --------------------------------------------------------------------------

def _new_tables(img):
    import torch
    return (torch.empty(tuple(img.shape), dtype=torch.int64, device=img.device),
            torch.empty(tuple(img.shape), dtype=torch.int64, device=img.device))


def ncc_sat_build(img, S=None, Q=None, stream=None):
    """S = SAT(I), Q = SAT(I^2): inclusive int64 tables of a uint8 [H][W] image."""
    import torch
    _dev(img, torch.uint8, 2, "img")
    H, W = img.shape
    nS, nQ = _new_tables(img) if S is None or Q is None else (S, Q)
    S = nS if S is None else S
    Q = nQ if Q is None else Q
    _tables(img, S, Q)
    _check(lib().ncc_sat_build(img.data_ptr(), W, H, S.data_ptr(), Q.data_ptr(),
                               _stream_handle(stream)), "ncc_sat_build")
    return S, Q


def ncc_sat_build_variant(img, variant, S=None, Q=None, stream=None):
    """The same tables by one of the compared builders (NCC_SAT_FUSED,
    NCC_SAT_NAIVE, NCC_SAT_TWO_PASS)."""
    import torch
    _dev(img, torch.uint8, 2, "img")
    H, W = img.shape
    nS, nQ = _new_tables(img) if S is None or Q is None else (S, Q)
    S = nS if S is None else S
    Q = nQ if Q is None else Q
    _tables(img, S, Q)
    _check(lib().ncc_sat_build_variant(img.data_ptr(), W, H, S.data_ptr(), Q.data_ptr(),
                                       int(variant), _stream_handle(stream)),
           "ncc_sat_build_variant")
    return S, Q


def ncc_sat_build_noalloc(img, S, Q, stream=None):
    """ncc_sat_build without any device allocation, into caller tables S, Q
    (int64 [H][W]); for callers that cannot allocate (see include/ncc.h)."""
    import torch
    _dev(img, torch.uint8, 2, "img")
    _tables(img, S, Q)
    H, W = img.shape
    _check(lib().ncc_sat_build_noalloc(img.data_ptr(), W, H, S.data_ptr(), Q.data_ptr(),
                                       _stream_handle(stream)), "ncc_sat_build_noalloc")
    return S, Q


def ncc_correlate(img, tmpl, S, Q, out=None, stream=None):
    """fp32 [Oy][Ox] coefficients of one uint8 [hT][wT] template."""
    import torch
    _dev(img, torch.uint8, 2, "img")
    _dev(tmpl, torch.uint8, 2, "tmpl", img)
    _tables(img, S, Q)
    H, W = img.shape
    hT, wT = tmpl.shape
    shape = _map_shape(img, 1, hT, wT)[1:]
    if out is None:
        out = torch.empty(shape, dtype=torch.float32, device=img.device)
    _dev(out, torch.float32, 2, "out", img, shape)
    _check(lib().ncc_correlate(img.data_ptr(), W, H, tmpl.data_ptr(), wT, hT, S.data_ptr(),
                               Q.data_ptr(), out.data_ptr(), _stream_handle(stream)),
           "ncc_correlate")
    return out


def ncc_correlate_bank(img, tmpls, S, Q, out=None, stream=None):
    """fp32 [nT][Oy][Ox] coefficients of a uint8 [nT][hT][wT] template bank."""
    import torch
    _dev(img, torch.uint8, 2, "img")
    tmpls = _tmpl3(tmpls)
    _dev(tmpls, torch.uint8, 3, "tmpls", img)
    _tables(img, S, Q)
    H, W = img.shape
    nT, hT, wT = tmpls.shape
    shape = _map_shape(img, nT, hT, wT)
    if out is None:
        out = torch.empty(shape, dtype=torch.float32, device=img.device)
    _dev(out, torch.float32, 3, "out", img, shape)
    _check(lib().ncc_correlate_bank(img.data_ptr(), W, H, tmpls.data_ptr(), wT, hT, nT,
                                    S.data_ptr(), Q.data_ptr(), out.data_ptr(),
                                    _stream_handle(stream)), "ncc_correlate_bank")
    return out


def _moment_buffers(img, nT, hT, wT):
    import torch
    shape = _map_shape(img, nT, hT, wT)
    return (torch.empty(shape[1:], dtype=torch.int64, device=img.device),
            torch.empty(shape[1:], dtype=torch.int64, device=img.device),
            torch.empty(shape, dtype=torch.int64, device=img.device))


def ncc_correlate_moments(img, tmpls, S, Q, stream=None):
    """(SumI [Oy][Ox], SumI2 [Oy][Ox], SumIT [nT][Oy][Ox]) as int64."""
    import torch
    _dev(img, torch.uint8, 2, "img")
    tmpls = _tmpl3(tmpls)
    _dev(tmpls, torch.uint8, 3, "tmpls", img)
    _tables(img, S, Q)
    H, W = img.shape
    nT, hT, wT = tmpls.shape
    sI, sI2, sIT = _moment_buffers(img, nT, hT, wT)
    _check(lib().ncc_correlate_moments(img.data_ptr(), W, H, tmpls.data_ptr(), wT, hT, nT,
                                       S.data_ptr(), Q.data_ptr(), sI.data_ptr(),
                                       sI2.data_ptr(), sIT.data_ptr(), _stream_handle(stream)),
           "ncc_correlate_moments")
    return sI, sI2, sIT


def ncc_correlate_direct(img, tmpls, out=None, stream=None):
    """fp32 [nT][Oy][Ox] coefficients with the window moments taken from the
    staged image tile (no summed-area tables)."""
    import torch
    _dev(img, torch.uint8, 2, "img")
    tmpls = _tmpl3(tmpls)
    _dev(tmpls, torch.uint8, 3, "tmpls", img)
    H, W = img.shape
    nT, hT, wT = tmpls.shape
    shape = _map_shape(img, nT, hT, wT)
    if out is None:
        out = torch.empty(shape, dtype=torch.float32, device=img.device)
    _dev(out, torch.float32, 3, "out", img, shape)
    _check(lib().ncc_correlate_direct(img.data_ptr(), W, H, tmpls.data_ptr(), wT, hT, nT,
                                      out.data_ptr(), _stream_handle(stream)),
           "ncc_correlate_direct")
    return out


def ncc_correlate_direct_moments(img, tmpls, stream=None):
    """(SumI [Oy][Ox], SumI2 [Oy][Ox], SumIT [nT][Oy][Ox]) as int64, the
    moments taken from the staged image tile."""
    import torch
    _dev(img, torch.uint8, 2, "img")
    tmpls = _tmpl3(tmpls)
    _dev(tmpls, torch.uint8, 3, "tmpls", img)
    H, W = img.shape
    nT, hT, wT = tmpls.shape
    sI, sI2, sIT = _moment_buffers(img, nT, hT, wT)
    _check(lib().ncc_correlate_direct_moments(img.data_ptr(), W, H, tmpls.data_ptr(), wT, hT, nT,
                                              sI.data_ptr(), sI2.data_ptr(), sIT.data_ptr(),
                                              _stream_handle(stream)),
           "ncc_correlate_direct_moments")
    return sI, sI2, sIT


def ncc_match(img, tmpls, S=None, Q=None, out=None, stream=None):
    """SAT build then correlation on device tensors, in one call: returns
    (S, Q, out), with out fp32 [nT][Oy][Ox] (the single-template correlation
    overlaps the build's tail)."""
    import torch
    _dev(img, torch.uint8, 2, "img")
    tmpls = _tmpl3(tmpls)
    _dev(tmpls, torch.uint8, 3, "tmpls", img)
    H, W = img.shape
    nT, hT, wT = tmpls.shape
    nS, nQ = _new_tables(img) if S is None or Q is None else (S, Q)
    S = nS if S is None else S
    Q = nQ if Q is None else Q
    _tables(img, S, Q)
    shape = _map_shape(img, nT, hT, wT)
    if out is None:
        out = torch.empty(shape, dtype=torch.float32, device=img.device)
    _dev(out, torch.float32, 3, "out", img, shape)
    _check(lib().ncc_match(img.data_ptr(), W, H, tmpls.data_ptr(), wT, hT, nT, S.data_ptr(),
                           Q.data_ptr(), out.data_ptr(), _stream_handle(stream)), "ncc_match")
    return S, Q, out


def ncc_match_host(img, tmpls, out=None, stream=None):
    """The whole path on HOST buffers (numpy arrays or CPU tensors; pinned
    tensors make the copies asynchronous).  Returns fp32 [nT][Oy][Ox] on the
    host; synchronizes the stream."""
    import torch
    kinds = {"uint8": (np.uint8, torch.uint8), "float32": (np.float32, torch.float32)}

    def host_ptr(a, kind, ndim, name, shape=None):
        np_t, torch_t = kinds[kind]
        if isinstance(a, np.ndarray):
            if not a.flags.c_contiguous or a.dtype != np_t or a.ndim != ndim:
                raise TypeError(f"{name} must be a C-contiguous {kind} array with {ndim} dims")
            dims = tuple(a.shape)
            ptr = a.ctypes.data
        elif isinstance(a, torch.Tensor):
            if a.is_cuda or not a.is_contiguous() or a.dtype != torch_t or a.dim() != ndim:
                raise TypeError(f"{name} must be a contiguous CPU {kind} tensor with {ndim} dims")
            dims = tuple(a.shape)
            ptr = a.data_ptr()
        else:
            raise TypeError(f"{name} must be a numpy array or a CPU tensor")
        if shape is not None and dims != tuple(shape):
            raise ValueError(f"{name} has shape {dims}, expected {tuple(shape)}")
        return ptr, dims

    ip, (H, W) = host_ptr(img, "uint8", 2, "img")
    if len(tmpls.shape) == 2:
        tmpls = tmpls.reshape((1,) + tuple(tmpls.shape))
    tp, (nT, hT, wT) = host_ptr(tmpls, "uint8", 3, "tmpls")
    shape = (nT, max(H - hT + 1, 0), max(W - wT + 1, 0))
    if out is None:
        out = np.empty(shape, np.float32)
    op, _ = host_ptr(out, "float32", 3, "out", shape)
    _check(lib().ncc_match_host(ip, W, H, tp, wT, hT, nT, op, _stream_handle(stream)),
           "ncc_match_host")
    return out


def ncc_sync_status(stream=None) -> int:
    return int(lib().ncc_sync_status(_stream_handle(stream)))


def ncc_status_string(code: int) -> str:
    return lib().ncc_status_string(int(code)).decode()


def ncc_version() -> int:
    return int(lib().ncc_version())


def ncc_debug_set_fault(suppress_tile: int, timeout_ns: int = 0) -> None:
    _check(lib().ncc_debug_set_fault(int(suppress_tile), int(timeout_ns)), "ncc_debug_set_fault")


def ncc_debug_fail_alloc(count: int) -> None:
    """The library's next `count` device allocations fail (NCC_ERR_NOMEM)."""
    _check(lib().ncc_debug_fail_alloc(int(count)), "ncc_debug_fail_alloc")


NCC_PATH_NONE, NCC_PATH_DP4A, NCC_PATH_BANK, NCC_PATH_TOEPLITZ, NCC_PATH_NTT = 0, 1, 3, 4, 5


def ncc_debug_set_path(path: int) -> None:
    """Restricts the single-template kernels (0 = automatic)."""
    _check(lib().ncc_debug_set_path(int(path)), "ncc_debug_set_path")


def ncc_debug_last_path() -> int:
    """Kernel launched by the most recent successful correlate call."""
    return int(lib().ncc_debug_last_path())
