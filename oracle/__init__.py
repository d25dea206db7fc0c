"""CPU oracle for normalized cross-correlation -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline and
reference legs of ``bench.py`` may import this package.  The product (the CUDA library and its
Python binding) never touches it, and it never touches the product.

The arithmetic lives in ``ncc_oracle.c`` (plain C, int64 sums, double
coefficients); this module compiles it with gcc on first use and wraps it
with ctypes.  What each function follows (The CUDA Handbook, chapter 15):

* :func:`sat` -- section 15.8, the summed-area tables S (of I) and Q (of I^2),
  inclusive, int64.
* :func:`sat_box` -- section 15.8, the four-corner box-sum equation
  (Figure 15-7), corners in row -1 / column -1 read as zero.
* :func:`template_stats`, :func:`window_sums` -- Listing 15-5 ("Image in
  shared memory"): SumT, and per shift SumI, SumI2 and SumIT.
* :func:`coefficient` -- the Pearson reading of the listing's coefficient
  routine (its body is not printed): r = num / sqrt(vI*vT) with exact-integer
  num, vI and vT; 0 for zero variance; clamped to [-1, 1].
* :func:`correlate`, :func:`correlate_at` -- the above for every valid shift
  (or a list of shifts) of every template.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ncc_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libncc_oracle.so")

_lock = threading.Lock()
_lib = None

_i64p = ctypes.POINTER(ctypes.c_int64)
_f64p = ctypes.POINTER(ctypes.c_double)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_i32p = ctypes.POINTER(ctypes.c_int32)


def build(force: bool = False) -> str:
    """Compile ncc_oracle.c into a shared library (OpenMP when gcc has it)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # NCC_ORACLE_LIB points the wrapper at another build of the same
            # source (the mutation tests use it to load planted mistakes).
            lib = ctypes.CDLL(os.environ.get("NCC_ORACLE_LIB") or build())
            lib.ncc_oracle_sat.argtypes = [_u8p, ctypes.c_int, ctypes.c_int, _i64p, _i64p]
            lib.ncc_oracle_sat.restype = ctypes.c_int
            lib.ncc_oracle_sat_box.argtypes = [_i64p, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int]
            lib.ncc_oracle_sat_box.restype = ctypes.c_int64
            lib.ncc_oracle_template_stats.argtypes = [_u8p, ctypes.c_int, ctypes.c_int,
                                                      _i64p, _i64p]
            lib.ncc_oracle_template_stats.restype = None
            lib.ncc_oracle_window_sums.argtypes = [_u8p, ctypes.c_int, _u8p, ctypes.c_int,
                                                   ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                   _i64p, _i64p, _i64p]
            lib.ncc_oracle_window_sums.restype = None
            lib.ncc_oracle_coefficient.argtypes = [ctypes.c_int64] * 6
            lib.ncc_oracle_coefficient.restype = ctypes.c_double
            lib.ncc_oracle_correlate.argtypes = [_u8p, ctypes.c_int, ctypes.c_int, _u8p,
                                                 ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                 _f64p, _i64p, _i64p, _i64p, ctypes.c_int]
            lib.ncc_oracle_correlate.restype = ctypes.c_int
            lib.ncc_oracle_correlate_at.argtypes = [_u8p, ctypes.c_int, ctypes.c_int, _u8p,
                                                    ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                    _i32p, _i32p, ctypes.c_int, _f64p,
                                                    _i64p, _i64p, _i64p, ctypes.c_int]
            lib.ncc_oracle_correlate_at.restype = ctypes.c_int
            lib.ncc_oracle_has_openmp.argtypes = []
            lib.ncc_oracle_has_openmp.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _u8_2d(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint8 or a.ndim != 2:
        raise ValueError("expected a 2-D uint8 array")
    return a


def _templates(t) -> np.ndarray:
    t = np.ascontiguousarray(t)
    if t.dtype != np.uint8 or t.ndim not in (2, 3):
        raise ValueError("templates must be uint8 [hT][wT] or [nT][hT][wT]")
    return t[None] if t.ndim == 2 else t


def has_openmp() -> bool:
    return bool(_load().ncc_oracle_has_openmp())


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def sat(img) -> tuple[np.ndarray, np.ndarray]:
    """Inclusive int64 summed-area tables (S of I, Q of I^2), each [H][W]."""
    img = _u8_2d(img)
    H, W = img.shape
    S = np.empty((H, W), np.int64)
    Q = np.empty((H, W), np.int64)
    rc = _load().ncc_oracle_sat(_ptr(img, ctypes.c_uint8), W, H,
                                _ptr(S, ctypes.c_int64), _ptr(Q, ctypes.c_int64))
    if rc != 0:
        raise ValueError("ncc_oracle_sat rejected its arguments")
    return S, Q


def sat_box(S, x0: int, y0: int, x1: int, y1: int) -> int:
    """Sum over [x0,x1) x [y0,y1) from an inclusive table by four corners."""
    S = np.ascontiguousarray(S, dtype=np.int64)
    H, W = S.shape
    if not (0 <= x0 < x1 <= W and 0 <= y0 < y1 <= H):
        raise ValueError("box outside the table")
    return int(_load().ncc_oracle_sat_box(_ptr(S, ctypes.c_int64), W, x0, y0, x1, y1))


def template_stats(T) -> tuple[int, int]:
    """(SumT, SumT2) of one template."""
    T = _u8_2d(T)
    hT, wT = T.shape
    a, b = ctypes.c_int64(), ctypes.c_int64()
    _load().ncc_oracle_template_stats(_ptr(T, ctypes.c_uint8), wT, hT,
                                      ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def window_sums(img, T, x: int, y: int) -> tuple[int, int, int]:
    """(SumI, SumI2, SumIT) of the window with top-left pixel (x, y)."""
    img = _u8_2d(img)
    T = _u8_2d(T)
    H, W = img.shape
    hT, wT = T.shape
    if not (0 <= x <= W - wT and 0 <= y <= H - hT):
        raise ValueError("shift outside the valid range")
    a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _load().ncc_oracle_window_sums(_ptr(img, ctypes.c_uint8), W, _ptr(T, ctypes.c_uint8),
                                   wT, hT, x, y, ctypes.byref(a), ctypes.byref(b),
                                   ctypes.byref(c))
    return a.value, b.value, c.value


def coefficient(N: int, sI: int, sI2: int, sIT: int, sT: int, sT2: int) -> float:
    """Pearson coefficient from the exact integer sums."""
    return float(_load().ncc_oracle_coefficient(N, sI, sI2, sIT, sT, sT2))


def correlate(img, templates, with_sums: bool = False, threads: int | None = None):
    """Coefficients of every valid shift for every template.

    Returns r as float64 [nT][Oy][Ox] (or [Oy][Ox] for a 2-D template), and
    with ``with_sums`` also SumI, SumI2 and SumIT as int64 of the same shape.
    """
    img = _u8_2d(img)
    squeeze = np.ndim(templates) == 2
    T = _templates(templates)
    nT, hT, wT = T.shape
    H, W = img.shape
    if not (1 <= wT <= W and 1 <= hT <= H):
        raise ValueError("template larger than the image")
    Oy, Ox = H - hT + 1, W - wT + 1
    out = np.empty((nT, Oy, Ox), np.float64)
    sums = [np.empty((nT, Oy, Ox), np.int64) for _ in range(3)] if with_sums else None
    null = ctypes.cast(None, _i64p)
    rc = _load().ncc_oracle_correlate(
        _ptr(img, ctypes.c_uint8), W, H, _ptr(T, ctypes.c_uint8), wT, hT, nT,
        _ptr(out, ctypes.c_double),
        *( [_ptr(s, ctypes.c_int64) for s in sums] if sums else [null, null, null]),
        threads or 1)
    if rc != 0:
        raise ValueError("ncc_oracle_correlate rejected its arguments")
    if squeeze:
        out = out[0]
        sums = [s[0] for s in sums] if sums else None
    return (out, *sums) if with_sums else out


def correlate_at(img, templates, xs, ys, with_sums: bool = False,
                 threads: int | None = None):
    """Coefficients at listed shifts; arrays are [nT][n] (or [n])."""
    img = _u8_2d(img)
    squeeze = np.ndim(templates) == 2
    T = _templates(templates)
    nT, hT, wT = T.shape
    H, W = img.shape
    xs = np.ascontiguousarray(xs, dtype=np.int32).ravel()
    ys = np.ascontiguousarray(ys, dtype=np.int32).ravel()
    if xs.shape != ys.shape:
        raise ValueError("xs and ys differ in length")
    n = xs.size
    out = np.empty((nT, n), np.float64)
    sums = [np.empty((nT, n), np.int64) for _ in range(3)] if with_sums else None
    null = ctypes.cast(None, _i64p)
    rc = _load().ncc_oracle_correlate_at(
        _ptr(img, ctypes.c_uint8), W, H, _ptr(T, ctypes.c_uint8), wT, hT, nT,
        _ptr(xs, ctypes.c_int32), _ptr(ys, ctypes.c_int32), n,
        _ptr(out, ctypes.c_double),
        *( [_ptr(s, ctypes.c_int64) for s in sums] if sums else [null, null, null]),
        threads or 1)
    if rc != 0:
        raise ValueError("ncc_oracle_correlate_at rejected its arguments")
    if squeeze:
        out = out[0]
        sums = [s[0] for s in sums] if sums else None
    return (out, *sums) if with_sums else out
