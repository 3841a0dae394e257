"""The largest extents a single GB300 holds comfortably, against the CPU oracle on
sampled rows (the first and last rows always among them):

* an output of more than 2^31 elements (5.2 GB), so every store offset past
  the 32-bit range is exercised, with canaries behind C;
* a reduction over 2^20 k values into one 256 x 256 tile (small integers, so
  the comparison is bit for bit);
* 2^22 rows by 16 columns, and 16 rows by 2^22 columns: one tile band with
  tens of thousands of tiles, hundreds per CTA.

Tolerance as in every other parity test.
"""
import numpy as np
import pytest
import torch

import dense_fp16_gemm_fp32_gb300 as g
from dense_fp16_gemm_fp32_gb300 import inputs
from oracle import gemm as og

from _gpu_util import check_against_oracle

pytestmark = pytest.mark.gpu

CFGS = [g.TILE_AUTO, g.TILE_128x256x64, g.TILE_256x256x128_PAIR, g.TILE_128x64x64]


def _rows(M: int, seed: int, count: int = 64) -> torch.Tensor:
    r = set(inputs.sample_rows(M, seed, count).tolist()) | {0, M - 1}
    return torch.tensor(sorted(r))


@pytest.mark.parametrize("cfg", CFGS)
def test_output_beyond_2_31_elements(gemm_lib, cfg):
    M, N, K = 65536, 40000, 8                   # C: 2.62e9 elements
    A, B = inputs.gemm_inputs(M, N, K, seed=91)
    canary = 0x7E01
    buf = torch.full((M * N + 4096,), canary, dtype=torch.int16, device="cuda")
    C = buf[:M * N].view(torch.float16).view(M, N)
    g.gemm(A.cuda(), B.cuda(), out=C, tile_cfg=cfg)
    assert g.query_status() == g.GEMM_OK
    assert torch.all(buf[M * N:] == canary)
    check_against_oracle(A, B, C, _rows(M, 91))
    del buf, C
    torch.cuda.empty_cache()


def test_reduction_over_2_20_k(gemm_lib):
    # integers in [-2, 2]: every partial sum is an integer below 2^24 in magnitude, exact
    # in fp32 in any order, so the device result equals the oracle's bit for bit
    M, N, K = 256, 256, 1 << 20
    gen = torch.Generator().manual_seed(92)
    A = torch.randint(-2, 3, (M, K), generator=gen, dtype=torch.int8).half()
    B = torch.randint(-2, 3, (K, N), generator=gen, dtype=torch.int8).half()
    a, b = A.cuda(), B.cuda()
    rows = _rows(M, 92, 6)
    ref = og.gemm_rows(A, B, rows=rows.numpy())
    for cfg in CFGS:
        C = g.gemm(a, b, tile_cfg=cfg)
        assert g.query_status() == g.GEMM_OK
        got = C.index_select(0, rows.cuda()).cpu().numpy()
        assert np.array_equal(got.view(np.uint16), ref.view(np.uint16)), cfg
    del a, b
    torch.cuda.empty_cache()


@pytest.mark.parametrize("cfg", CFGS)
@pytest.mark.parametrize("M,N", [(1 << 22, 16), (16, 1 << 22)])
def test_one_band_of_many_tiles(gemm_lib, M, N, cfg):
    K = 16
    A, B = inputs.gemm_inputs(M, N, K, seed=93)
    C = g.gemm(A.cuda(), B.cuda(), tile_cfg=cfg)
    assert g.query_status() == g.GEMM_OK
    check_against_oracle(A, B, C, _rows(M, 93))
    del C
    torch.cuda.empty_cache()
