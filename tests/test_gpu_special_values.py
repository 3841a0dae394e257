"""IEEE special values through the device GEMM, against the oracle.

* fp16 overflow at the single narrowing: sums beyond 65504 become +/-inf
  (and exactly representable sums stay finite), bit for bit;
* NaN and infinities in A or B: the positions and signs of NaN/inf in C are
  independent of the summation order (inf + finite = inf, inf - inf = NaN,
  inf * 0 = NaN, NaN absorbs), so they must match the oracle exactly; the
  finite elements within the usual tolerance;
* fp16 subnormal inputs: products of integers times 2^-24 are exact in fp32
  and the narrowed results are exact subnormals, bit for bit.
Every tile configuration and the generic-load path.
"""
import numpy as np
import pytest
import torch

import dense_fp16_gemm_fp32_gb300 as g
from dense_fp16_gemm_fp32_gb300 import inputs
from oracle import gemm as og

from _gpu_util import tolerance

pytestmark = pytest.mark.gpu

CFGS = [g.TILE_AUTO, g.TILE_128x256x64, g.TILE_128x64x32, g.TILE_256x256x128_PAIR, g.TILE_128x128x64,
        g.TILE_128x128x64_SPLITK, g.TILE_128x64x64, g.TILE_64x64x64, "generic"]


def run(A: torch.Tensor, B: torch.Tensor, cfg) -> np.ndarray:
    a, b = A.cuda(), B.cuda()
    if cfg == "generic":   # A one element off a 16-byte boundary, no workspace: the plain-load kernel
        buf = torch.empty(a.numel() + 1, dtype=torch.float16, device="cuda")
        buf[1:] = a.reshape(-1)
        C = g.gemm(buf[1:].view(a.shape), b, repack=False)
    else:
        C = g.gemm(a, b, tile_cfg=cfg)
    assert g.query_status() == g.GEMM_OK
    return C.cpu().numpy()


@pytest.mark.parametrize("cfg", CFGS)
def test_overflow_at_the_narrowing(gemm_lib, cfg):
    M, N, K = 256, 256, 64
    A = torch.zeros((M, K), dtype=torch.float16)
    B = torch.zeros((K, N), dtype=torch.float16)
    A[:, :16] = 256.0
    B[:16, 0::5] = 256.0                  # 16 * 65536 = 1048576: +inf in fp16
    B[:16, 1::5] = -256.0                 # -inf
    B[0, 2::5] = 255.5                    # 256 * 255.5 = 65408: finite, exact
    B[0, 3::5] = 255.875                  # 65504: the largest finite fp16, exact
    B[0, 4::5] = 255.875                  # 65504 + 256 * 0.0625 = 65520: the midpoint to the next
    B[1, 4::5] = 0.0625                   # binade rounds (to even) past the largest finite: +inf
    got = run(A, B, cfg)
    want = og.gemm_rows(A, B)
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))
    assert np.isposinf(got[:, 0::5]).all() and np.isneginf(got[:, 1::5]).all()
    assert (got[:, 2::5] == 65408.0).all() and (got[:, 3::5] == 65504.0).all()
    assert np.isposinf(got[:, 4::5]).all()


@pytest.mark.parametrize("cfg", CFGS)
def test_nan_and_inf_positions(gemm_lib, cfg):
    M, N, K = 300, 264, 200
    A, B = inputs.gemm_inputs(M, N, K, seed=77)
    inf, nan = float("inf"), float("nan")
    A[3, 5] = nan                         # row 3: NaN everywhere
    A[7, 2] = inf                         # row 7: +/-inf by the sign of B[2, j]; NaN where B[2, j] == 0
    B[2, ::7] = 0.0
    B[9, 11] = -inf                       # column 11: -/+inf by the sign of A[i, 9]
    A[20, 9] = 0.0                        # ... except row 20: 0 * inf = NaN
    A[40, 9] = inf                        # row 40, column 11: +inf * -inf = -inf, plus row 40's own infinities
    B[9, 60] = inf
    A[50, 9] = -inf                       # row 50: -inf * (+inf at column 60) = -inf; column 11: +inf
    got = run(A, B, cfg).astype(np.float64)
    want = og.gemm_rows(A, B).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(want)), "NaN positions differ"
    assert np.array_equal(np.isposinf(got), np.isposinf(want)) and np.array_equal(np.isneginf(got), np.isneginf(want))
    fin = np.isfinite(want)
    assert np.isnan(want[3]).all() and np.isnan(want[20, 11])
    d = np.abs(got[fin] - want[fin])
    assert (d <= tolerance(K, want[fin])).all()


@pytest.mark.parametrize("cfg", CFGS)
def test_subnormal_inputs_exact(gemm_lib, cfg):
    M, N, K = 256, 128, 96
    gen = torch.Generator().manual_seed(5)
    ka = torch.randint(-6, 7, (M, K), generator=gen).double()
    kb = torch.randint(-3, 4, (K, N), generator=gen).double()
    A = (ka * 2.0 ** -24).half()          # fp16 subnormals (and zeros): k * 2^-24 is exact
    B = kb.half()
    assert torch.all(A.double() == ka * 2.0 ** -24)
    got = run(A, B, cfg)
    want = og.gemm_rows(A, B)
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))
    # the sums are integers times 2^-24, at most 96 * 18 = 1728 of them: exact subnormals or
    # small normals in fp16, so the device result is the exact product
    exact = (ka @ kb) * 2.0 ** -24
    assert np.array_equal(got.astype(np.float64), exact.numpy())
