"""Helpers for the GPU parity tests: run the CUDA path and the CPU oracle on
the same seeded host bytes and compare element by element."""
import numpy as np
import torch

import dense_fp16_gemm_fp32_gb300 as g
from oracle import gemm as og

# Tolerance (fp16 outputs of the device path versus the oracle's fp16 C):
#   K <= 512: |d| <= 1e-2, rtol 0 (the tutorial's torch.allclose check);
#   K >  512: |d| <= 1e-2 + 1e-3 * |ref|, ref = the oracle's fp16 output.
# Both sides sum exact fp16 products in fp32, in different orders, and round
# once; a different order can move the fp32 sum by a few fp32 ulps and so
# flip the final fp16 rounding by one fp16 ulp, which is at most
# 2^-10 * |ref| < 1e-3 * |ref|, or 2^-24 below 2^-14.
ATOL = 1e-2
RTOL_LARGE_K = 1e-3


def tolerance(K: int, ref32: np.ndarray) -> np.ndarray:
    if K <= 512:
        return np.full(ref32.shape, ATOL, dtype=np.float64)
    return ATOL + RTOL_LARGE_K * np.abs(ref32.astype(np.float64))


def compare(got16: np.ndarray, ref16: np.ndarray, K: int):
    """Element-wise check; returns (max |d|, number of elements compared)."""
    got = got16.astype(np.float64)
    ref = ref16.astype(np.float64)
    assert got.shape == ref.shape
    assert not np.isnan(got).any(), "NaN in device output"
    assert np.array_equal(np.isinf(got), np.isinf(ref))
    fin = np.isfinite(ref)
    d = np.abs(got[fin] - ref[fin])
    tol = tolerance(K, ref16[fin])
    bad = np.nonzero(d > tol)[0]
    assert bad.size == 0, (f"{bad.size} elements beyond tolerance; worst |d|={d.max():.4g}", got[fin][bad[:8]],
                           ref[fin][bad[:8]])
    return (float(d.max()) if d.size else 0.0), int(d.size)


def device_gemm(A: torch.Tensor, B: torch.Tensor, **kw) -> torch.Tensor:
    return g.gemm(A.cuda(), B.cuda(), **kw)


def check_against_oracle(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor, rows=None):
    """C (device, [M,N]) against the oracle on `rows` (default: all rows)."""
    K = A.shape[1]
    if rows is None:
        got = C.cpu().numpy()
        ref = og.gemm_rows(A, B)
    else:
        rows_t = torch.as_tensor(rows, dtype=torch.long)
        got = C.index_select(0, rows_t.to(C.device)).cpu().numpy()
        ref = og.gemm_rows(A, B, rows=rows_t.numpy())
    return compare(got, ref, K)
