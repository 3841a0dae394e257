"""ctypes front end of the CPU GEMM oracle in ``gemm_oracle.c``.

TEST INFRASTRUCTURE ONLY: used by the tests, the package smoke check and the
benchmark's CPU baseline; never imported by the product path.

The arithmetic lives in C (fp32 running sum in ascending k, one hand-written
round-to-nearest-even narrowing to fp16). This module only hands numpy
buffers of fp16 bit patterns to it.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        lib.oracle_gemm_f16_rows.restype = ctypes.c_int
        lib.oracle_gemm_f16_rows.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_half_to_float.restype = ctypes.c_float
        lib.oracle_half_to_float.argtypes = [ctypes.c_uint16]
        lib.oracle_float_to_half_rne.restype = ctypes.c_uint16
        lib.oracle_float_to_half_rne.argtypes = [ctypes.c_float]
        for name in ("oracle_half_to_float_array", "oracle_float_to_half_rne_array"):
            fn = getattr(lib, name)
            fn.restype = None
            fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
        _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _bits(x) -> np.ndarray:
    """fp16 data (numpy float16/uint16 array or a CPU torch.float16 tensor) as
    a C-contiguous uint16 array of bit patterns."""
    if hasattr(x, "detach"):  # torch tensor
        import torch
        x = x.detach().cpu().contiguous().view(torch.int16).numpy()
    a = np.ascontiguousarray(x)
    if a.dtype == np.float16 or a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected fp16 bit patterns, got {a.dtype}")
    return a


def gemm_rows(A, B, rows=None, nthreads: int | None = None, want_c32: bool = False):
    """Rows ``rows`` of C = A B.

    A: [M,K] fp16, B: [K,N] fp16 (numpy float16/uint16 or CPU torch fp16).
    rows: iterable of row indices (default: all M rows).
    Returns C16 as a numpy float16 array [len(rows), N] and, if want_c32, the
    unrounded fp32 sums as well.
    """
    a = _bits(A)
    b = _bits(B)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[0]:
        raise ValueError(f"shape mismatch {a.shape} x {b.shape}")
    M, K = a.shape
    N = b.shape[1]
    r = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nr = int(r.shape[0])
    c16 = np.zeros((nr, N), dtype=np.uint16)
    c32 = np.zeros((nr, N), dtype=np.float32) if want_c32 else None
    if nthreads is None:
        nthreads = default_threads()
    rc = _load().oracle_gemm_f16_rows(
        a.ctypes.data, b.ctypes.data, M, N, K, r.ctypes.data, nr, int(nthreads),
        c16.ctypes.data, c32.ctypes.data if c32 is not None else None)
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_f16_rows failed with code {rc}")
    c16 = c16.view(np.float16)
    return (c16, c32) if want_c32 else c16


def half_to_float(bits: int) -> float:
    """The oracle's binary16 decoder on one bit pattern."""
    return float(_load().oracle_half_to_float(int(bits) & 0xFFFF))


def half_to_float_array(bits) -> np.ndarray:
    """The oracle's binary16 decoder over an array of bit patterns."""
    h = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    _load().oracle_half_to_float_array(h.ctypes.data, out.ctypes.data, h.size)
    return out


def float_to_half_bits_array(x) -> np.ndarray:
    """The oracle's fp32 -> fp16 narrowing over an array; returns uint16 bits."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(f.shape, dtype=np.uint16)
    _load().oracle_float_to_half_rne_array(f.ctypes.data, out.ctypes.data, f.size)
    return out


def float_to_half_bits(x: float) -> int:
    """The oracle's fp32 -> fp16 round-to-nearest-even on one fp32 value."""
    return int(_load().oracle_float_to_half_rne(float(x)))
