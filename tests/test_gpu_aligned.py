"""The aligned, mask-free configuration (GEMM_TILE_256x256x128_PAIR_ALIGNED):
the specialisation of "03: Matrix multiplication" that the @ph.aligned
decorator selects, where the caller promises whole tiles and the kernel
carries no edge tests.

On whole-tile shapes it must match the oracle element by element and give the
same bits as the general 256x256x128 pair configuration (same tiles, same
k-step order, same single rounding); on any other extents it must refuse the
call before launching anything.
"""
import pytest
import torch

import dense_fp16_gemm_fp32_gb300 as g
from dense_fp16_gemm_fp32_gb300 import inputs

from _gpu_util import check_against_oracle

pytestmark = pytest.mark.gpu

ALIGNED = g.TILE_256x256x128_PAIR_ALIGNED


@pytest.mark.parametrize("M,N,K", [
    (256, 256, 128),      # one tile, one k step: the tile is split into column halves
    (512, 768, 256),      # 6 tiles
    (2048, 2048, 2048),   # 64 tiles, below one wave of clusters
    (1024, 4096, 1024),   # 64 tiles, one band of groups clamped
    (768, 512, 4096),     # long K
    (8192, 2560, 384),    # 320 tiles: several per cluster, split tail
])
def test_aligned_matches_oracle_and_general_pair(gemm_lib, M, N, K):
    A, B = inputs.gemm_inputs(M, N, K, seed=M + 3 * N + 7 * K)
    a, b = A.cuda(), B.cuda()
    n0 = g.launch_count()
    C = g.gemm(a, b, tile_cfg=ALIGNED)
    assert g.query_status() == g.GEMM_OK
    assert g.launch_count() - n0 == 1
    rows = inputs.sample_rows(M, 7) if M * N * K > 1.3e10 else None
    check_against_oracle(A, B, C, rows)
    want = g.gemm(a, b, tile_cfg=g.TILE_256x256x128_PAIR)
    assert torch.equal(C.view(torch.int16), want.view(torch.int16))


def test_aligned_small_integers_exact(gemm_lib):
    M, N, K = 512, 512, 512
    gen = torch.Generator().manual_seed(3)
    A = torch.randint(-4, 5, (M, K), generator=gen).half()
    B = torch.randint(-4, 5, (K, N), generator=gen).half()
    C = g.gemm(A.cuda(), B.cuda(), tile_cfg=ALIGNED)
    assert g.query_status() == g.GEMM_OK
    assert torch.equal(C.cpu().float(), A.float() @ B.float())


def test_aligned_k_zero_writes_zeros(gemm_lib):
    a = torch.empty((256, 0), dtype=torch.float16, device="cuda")
    b = torch.empty((0, 512), dtype=torch.float16, device="cuda")
    C = torch.full((256, 512), float("nan"), dtype=torch.float16, device="cuda")
    g.gemm(a, b, out=C, tile_cfg=ALIGNED)
    assert g.query_status() == g.GEMM_OK
    assert torch.equal(C.view(torch.int16), torch.zeros_like(C).view(torch.int16))


@pytest.mark.parametrize("M,N,K", [(255, 256, 128), (256, 264, 128), (256, 256, 136), (4095, 3000, 1000),
                                   (256, 256, 64)])
def test_aligned_refuses_partial_tiles(gemm_lib, M, N, K):
    a = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    b = torch.zeros((K, N), dtype=torch.float16, device="cuda")
    n0 = g.launch_count()
    with pytest.raises(g.GemmError) as e:
        g.gemm(a, b, tile_cfg=ALIGNED)
    assert e.value.code == g.GEMM_ERR_UNSUPPORTED
    assert g.launch_count() == n0


def test_aligned_refuses_operands_tma_cannot_describe(gemm_lib):
    # whole tiles, but A one element off a 16-byte boundary and no workspace
    buf = torch.zeros(256 * 128 + 1, dtype=torch.float16, device="cuda")
    a = buf[1:].view(256, 128)
    b = torch.zeros((128, 256), dtype=torch.float16, device="cuda")
    with pytest.raises(g.GemmError) as e:
        g.gemm(a, b, tile_cfg=ALIGNED, repack=False)
    assert e.value.code == g.GEMM_ERR_UNSUPPORTED
    # with the workspace route the repacked copies are TMA-shaped: it runs
    A, B = inputs.gemm_inputs(256, 256, 128, seed=9)
    buf[1:] = A.cuda().reshape(-1)
    C = g.gemm(buf[1:].view(256, 128), B.cuda(), tile_cfg=ALIGNED)
    assert g.query_status() == g.GEMM_OK
    check_against_oracle(A, B, C)


def test_auto_never_picks_aligned(gemm_lib):
    for shape in ((8192, 8192, 8192), (4096, 4096, 4096), (1024, 1024, 1024), (256, 256, 128)):
        assert g.tile_config(g.TILE_AUTO, *shape) != ALIGNED
    assert g.tile_shape(ALIGNED) == (256, 256, 128)
