"""GPU parity: the CUDA path against the CPU oracle on the same seeded inputs.

Full-size workloads are compared on every row where the oracle is quick
(M*N*K <= 1.3e10) and on 256 seeded rows otherwise; small and ragged shapes
cover several tiles plus a partial tile in every dimension.
"""
import numpy as np
import pytest
import torch

import dense_fp16_gemm_fp32_gb300 as g
from dense_fp16_gemm_fp32_gb300 import inputs
from oracle import gemm as og

from _gpu_util import check_against_oracle

pytestmark = pytest.mark.gpu

ALL_CFGS = [g.TILE_128x256x64, g.TILE_128x64x32, g.TILE_256x256x64_PAIR, g.TILE_256x256x128_PAIR,
            g.TILE_128x128x64, g.TILE_128x128x64_SPLITK, g.TILE_128x64x64, g.TILE_64x64x64]


@pytest.mark.parametrize("w", inputs.WORKLOADS, ids=lambda w: w.name)
def test_workload_parity(gemm_lib, w):
    A, B = inputs.gemm_inputs(w.M, w.N, w.K, w.seed)
    C = g.gemm(A.cuda(), B.cuda(), group_size_m=w.group_size_m, tile_cfg=w.tile_cfg)
    assert g.query_status() == g.GEMM_OK
    rows = inputs.sample_rows(w.M, w.seed) if w.sampled else None
    maxd, n = check_against_oracle(A, B, C, rows)
    assert n == (256 if w.sampled else w.M) * w.N
    del C
    torch.cuda.empty_cache()


@pytest.mark.parametrize("w", [w for w in inputs.WORKLOADS if w.tile_cfg == 0], ids=lambda w: w.name)
@pytest.mark.parametrize("cfg", [g.TILE_128x256x64, g.TILE_256x256x64_PAIR, g.TILE_256x256x128_PAIR,
                                 g.TILE_128x128x64, g.TILE_128x128x64_SPLITK, g.TILE_128x64x64,
                                 g.TILE_64x64x64])
def test_workload_parity_each_large_tile(gemm_lib, w, cfg):
    A, B = inputs.gemm_inputs(w.M, w.N, w.K, w.seed)
    C = g.gemm(A.cuda(), B.cuda(), group_size_m=w.group_size_m, tile_cfg=cfg)
    assert g.query_status() == g.GEMM_OK
    rows = inputs.sample_rows(w.M, w.seed) if w.sampled else None
    check_against_oracle(A, B, C, rows)
    del C
    torch.cuda.empty_cache()


EDGE_SHAPES = [
    # (M, N, K): partial tiles in each dimension, single rows/columns of tiles
    (1, 8, 8), (7, 8, 16), (127, 64, 64), (128, 256, 64), (129, 264, 72), (255, 120, 1000),
    (300, 520, 136), (513, 72, 24), (64, 1000, 512), (1000, 56, 8), (3, 3000, 40),
    (256, 256, 64), (257, 264, 128), (129, 8, 64), (600, 600, 8),
]


@pytest.mark.parametrize("cfg", ALL_CFGS)
@pytest.mark.parametrize("M,N,K", EDGE_SHAPES)
def test_edge_shapes(gemm_lib, M, N, K, cfg):
    A, B = inputs.gemm_inputs(M, N, K, seed=M * 7 + N * 13 + K)
    C = g.gemm(A.cuda(), B.cuda(), group_size_m=3, tile_cfg=cfg)
    assert g.query_status() == g.GEMM_OK
    check_against_oracle(A, B, C)


@pytest.mark.parametrize("cfg", ALL_CFGS)
@pytest.mark.parametrize("M,N,K", [(4096, 4096, 8), (2000, 3000, 40), (8192, 1001, 8)])
def test_many_short_tiles(gemm_lib, M, N, K, cfg):
    # one k step per tile and many tiles per CTA: each tile's epilogue follows
    # the previous one at once, so a staging buffer is refilled while the
    # previous tile's store may still be reading it (N = 1001: the right-edge
    # blocks are stored directly, between TMA stores of other tiles)
    A, B = inputs.gemm_inputs(M, N, K, seed=M + N + K + 1)
    C = g.gemm(A.cuda(), B.cuda(), tile_cfg=cfg)
    assert g.query_status() == g.GEMM_OK
    check_against_oracle(A, B, C)


@pytest.mark.parametrize("cfg", ALL_CFGS)
def test_k_zero_writes_zeros(gemm_lib, cfg):
    M, N = 200, 264
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    A = torch.empty((M, 0), dtype=torch.float16, device="cuda")
    B = torch.empty((0, N), dtype=torch.float16, device="cuda")
    g.gemm(A, B, out=C, tile_cfg=cfg)
    assert g.query_status() == g.GEMM_OK
    assert torch.all(C.view(torch.int16) == 0)


def test_m_or_n_zero_is_noop(gemm_lib):
    A = torch.zeros((0, 64), dtype=torch.float16, device="cuda")
    B = torch.zeros((64, 32), dtype=torch.float16, device="cuda")
    assert g.gemm(A, B).shape == (0, 32)
    A = torch.zeros((16, 64), dtype=torch.float16, device="cuda")
    B = torch.zeros((64, 0), dtype=torch.float16, device="cuda")
    assert g.gemm(A, B).shape == (16, 0)


@pytest.mark.parametrize("cfg", ALL_CFGS)
def test_small_integers_exact(gemm_lib, cfg):
    # every partial sum is an integer below 2^11: any summation order is exact
    rng = np.random.default_rng(11)
    M, N, K = 300, 264, 128
    A = torch.from_numpy(rng.integers(-4, 5, size=(M, K)).astype(np.float16))
    B = torch.from_numpy(rng.integers(-4, 5, size=(K, N)).astype(np.float16))
    C = g.gemm(A.cuda(), B.cuda(), tile_cfg=cfg).cpu()
    ref = og.gemm_rows(A, B)
    assert np.array_equal(C.numpy().view(np.uint16), ref.view(np.uint16))
    assert np.array_equal(C.numpy().astype(np.int64), A.numpy().astype(np.int64) @ B.numpy().astype(np.int64))


def test_identity_exact(gemm_lib):
    rng = np.random.default_rng(12)
    K = 320
    B = torch.from_numpy(rng.uniform(-100, 100, size=(K, 200)).astype(np.float16))
    I = torch.eye(K, dtype=torch.float16)
    C = g.gemm(I.cuda(), B.cuda()).cpu()
    assert torch.equal(C.view(torch.int16), B.view(torch.int16))


def test_single_narrowing_on_device(gemm_lib):
    # 1024 + 8 * 0.25 over K = 16 (rest zeros): fp32 accumulation gives 1026,
    # an fp16 running sum would stay at 1024
    A = torch.zeros((128, 16), dtype=torch.float16)
    A[:, 0] = 1024.0
    A[:, 1:9] = 0.25
    B = torch.ones((16, 64), dtype=torch.float16)
    C = g.gemm(A.cuda(), B.cuda()).cpu()
    assert torch.all(C == 1026.0)


@pytest.mark.parametrize("cfg", ALL_CFGS)
def test_group_size_does_not_change_values(gemm_lib, cfg):
    # the grouped order only changes which CTA computes a tile, not how (every tile of
    # this shape is in the first wave, where the pair kernels sum k upwards)
    A, B = inputs.gemm_inputs(700, 1000, 520, seed=21)
    a, b = A.cuda(), B.cuda()
    ref = g.gemm(a, b, group_size_m=1, tile_cfg=cfg)
    for G in (2, 3, 8, 64, 10_000):
        assert torch.equal(g.gemm(a, b, group_size_m=G, tile_cfg=cfg).view(torch.int16), ref.view(torch.int16))
    check_against_oracle(A, B, ref)


def test_deterministic(gemm_lib):
    A, B = inputs.gemm_inputs(1024, 1024, 2048, seed=22)
    a, b = A.cuda(), B.cuda()
    c1 = g.gemm(a, b)
    c2 = g.gemm(a, b)
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))


def test_non_default_stream_and_out(gemm_lib):
    A, B = inputs.gemm_inputs(384, 512, 256, seed=23)
    a, b = A.cuda(), B.cuda()
    out = torch.empty((384, 512), dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        r = g.gemm(a, b, out=out)
    s.synchronize()
    assert r.data_ptr() == out.data_ptr()
    check_against_oracle(A, B, out)


STRIDED = [
    # (M, N, K, lda, ldb, ldc): odd extents inside padded rows, and views of wider arrays
    (300, 999, 1001, 1008, 1000, 1000),
    (257, 264, 72, 80, 272, 264),
    (1000, 100, 37, 64, 104, 128),
    (4095, 3000, 1000, 1024, 3072, 3008),
    (1, 7, 3, 8, 8, 8),
]


@pytest.mark.parametrize("cfg", [g.TILE_AUTO, g.TILE_128x256x64, g.TILE_256x256x64_PAIR])
@pytest.mark.parametrize("M,N,K,lda,ldb,ldc", STRIDED)
def test_strided_views(gemm_lib, M, N, K, lda, ldb, ldc, cfg):
    A, B = inputs.gemm_inputs(M, N, K, seed=M + 3 * N + 7 * K)
    a_buf = torch.full((M, lda), float("nan"), dtype=torch.float16)
    b_buf = torch.full((K, ldb), float("nan"), dtype=torch.float16)
    a_buf[:, :K] = A
    b_buf[:, :N] = B
    canary = 0x7E01
    c_buf = torch.full((M, ldc), canary, dtype=torch.int16, device="cuda")
    a_view = a_buf.cuda()[:, :K]
    b_view = b_buf.cuda()[:, :N]
    c_view = c_buf.view(torch.float16)[:, :N]
    g.gemm(a_view, b_view, out=c_view, tile_cfg=cfg)   # the NaN padding of A and B is never read
    assert g.query_status() == g.GEMM_OK
    check_against_oracle(A, B, c_view.contiguous())
    assert torch.all(c_buf[:, N:] == canary)          # padding columns of C untouched


def test_strided_k_zero_stops_at_n(gemm_lib):
    M, N, ldc = 300, 999, 1008
    c_buf = torch.full((M, ldc), 0x7E01, dtype=torch.int16, device="cuda")
    a = torch.empty((M, 0), dtype=torch.float16, device="cuda")
    b = torch.empty((0, N), dtype=torch.float16, device="cuda")
    g.gemm(a, b, out=c_buf.view(torch.float16)[:, :N])
    assert g.query_status() == g.GEMM_OK
    assert torch.all(c_buf[:, :N] == 0) and torch.all(c_buf[:, N:] == 0x7E01)


# ---- operands a tensor map cannot describe: the generic-load kernel
# (bases 2-byte aligned only, row pitches that are not multiples of 8)
GENERIC = [
    # M, N, K, lda, ldb, ldc, element offsets of the A, B, C bases
    (300, 999, 1001, 1001, 999, 999, 0, 0, 0),     # contiguous, odd N and K
    (129, 264, 72, 75, 270, 267, 0, 0, 0),        # odd pitches, aligned extents
    (300, 520, 264, 264, 520, 520, 1, 3, 5),      # TMA-shaped pitches, bases off by 2/6/10 bytes
    (257, 300, 77, 79, 301, 303, 7, 1, 1),        # everything odd
    (1, 8, 8, 8, 8, 8, 1, 1, 1),
    (1000, 37, 1000, 1003, 37, 41, 0, 0, 0),      # narrow N
    (2048, 2048, 2000, 2001, 2049, 2051, 1, 1, 1),  # several tiles per CTA, K > 512
]


@pytest.mark.parametrize("repack", [False, True])
@pytest.mark.parametrize("M,N,K,lda,ldb,ldc,oa,ob,oc", GENERIC)
def test_generic_load_path(gemm_lib, M, N, K, lda, ldb, ldc, oa, ob, oc, repack):
    """repack=False: the generic-load kernel; repack=True: operands copied into
    a workspace, the TMA kernels, C copied back."""
    A, B = inputs.gemm_inputs(M, N, K, seed=M + 5 * N + 11 * K)
    nan = float("nan")
    a_buf = torch.full((oa + M * lda,), nan, dtype=torch.float16)
    b_buf = torch.full((ob + K * ldb,), nan, dtype=torch.float16)
    a_buf[oa:].view(M, lda)[:, :K] = A
    b_buf[ob:].view(K, ldb)[:, :N] = B
    canary = 0x7E01
    pad = 64
    c_buf = torch.full((pad + oc + M * ldc + pad,), canary, dtype=torch.int16, device="cuda")
    a_view = a_buf.cuda()[oa:].view(M, lda)[:, :K]
    b_view = b_buf.cuda()[ob:].view(K, ldb)[:, :N]
    c_view = c_buf[pad + oc:pad + oc + M * ldc].view(torch.float16).view(M, ldc)[:, :N]
    n0 = g.launch_count()
    g.gemm(a_view, b_view, out=c_view, repack=repack)   # the NaN padding of A and B is never read
    assert g.query_status() == g.GEMM_OK
    copies = 0
    if repack:
        copies = sum(not (t.data_ptr() % 16 == 0 and (t.stride(0) % 8 == 0 or t.shape[0] == 1))
                     for t in (a_view, b_view, c_view))
        assert (g.workspace_bytes(a_view, b_view, c_view) > 0) == (copies > 0)
    assert g.launch_count() - n0 == 1 + copies
    check_against_oracle(A, B, c_view.contiguous())
    assert torch.all(c_buf[:pad + oc] == canary) and torch.all(c_buf[pad + oc + M * ldc:] == canary)
    if ldc > N:
        assert torch.all(c_buf[pad + oc:pad + oc + M * ldc].view(M, ldc)[:, N:] == canary)


def test_generic_path_small_integers_exact(gemm_lib):
    M, N, K = 200, 301, 517
    gen = torch.Generator().manual_seed(9)
    A = torch.randint(-4, 5, (M, K), generator=gen).half()
    B = torch.randint(-4, 5, (K, N), generator=gen).half()
    C = g.gemm(A.cuda(), B.cuda())         # K and N odd: contiguous pitches are not multiples of 8
    want = (A.double() @ B.double())
    assert torch.all(want.abs() <= 2048)
    assert torch.equal(C.cpu().double(), want)


def test_generic_path_k_zero_and_matches_tma_path(gemm_lib):
    # K == 0 through the generic kernel (odd ldc)
    M, N, ldc = 130, 99, 101
    c_buf = torch.full((M, ldc), 0x7E01, dtype=torch.int16, device="cuda")
    g.gemm(torch.empty((M, 0), dtype=torch.float16, device="cuda"),
           torch.empty((0, N), dtype=torch.float16, device="cuda"), out=c_buf.view(torch.float16)[:, :N])
    assert g.query_status() == g.GEMM_OK
    assert torch.all(c_buf[:, :N] == 0) and torch.all(c_buf[:, N:] == 0x7E01)
    # the same problem through the three routes: identical bits (the same
    # 128x256x64 tiles and MMA order over the same values)
    M, N, K = 384, 512, 640
    A, B = inputs.gemm_inputs(M, N, K, seed=77)
    a, b = A.cuda(), B.cuda()
    c_tma = g.gemm(a, b, tile_cfg=g.TILE_128x256x64)
    a_off = torch.empty(M * K + 1, dtype=torch.float16, device="cuda")
    a_off[1:] = a.reshape(-1)
    a_mis = a_off[1:].view(M, K)                     # A 2 bytes off a 16-byte boundary
    c_gen = g.gemm(a_mis, b, repack=False)
    c_rep = g.gemm(a_mis, b, tile_cfg=g.TILE_128x256x64, repack=True)
    assert torch.equal(c_tma, c_gen) and torch.equal(c_tma, c_rep)


def test_workspace_entry_point_rules(gemm_lib):
    lib = g.load()
    s = torch.cuda.current_stream().cuda_stream
    M, N, K = 200, 304, 100     # only A (pitch 100, base 2 bytes off) needs a copy; its pitch becomes 104
    A, B = inputs.gemm_inputs(M, N, K, seed=5)
    a_off = torch.empty(M * K + 1, dtype=torch.float16, device="cuda")
    a_off[1:] = A.cuda().reshape(-1)
    a = a_off[1:]
    b = B.cuda()
    c = torch.empty((M, N), dtype=torch.float16, device="cuda")
    need = g.workspace_bytes(a.view(M, K), b, c)
    assert need == -(-(M * 104 * 2) // 256) * 256
    args = (a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N, M, N, K, 8, 0, None)
    # too small or misaligned workspace: the generic kernel runs instead (same result)
    ws = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    n0 = g.launch_count()
    assert lib.gemm_f16_f32acc_strided_ws(*args, ws.data_ptr(), need - 1, s) == g.GEMM_OK
    assert lib.gemm_f16_f32acc_strided_ws(*args, ws.data_ptr() + 16, need, s) == g.GEMM_OK
    assert g.launch_count() - n0 == 2
    check_against_oracle(A, B, c)
    # a workspace over an operand (here C, whose 120 KB hold the 41 KB asked for) is an argument error
    assert c.data_ptr() % 256 == 0
    n0 = g.launch_count()
    assert lib.gemm_f16_f32acc_strided_ws(*args, c.data_ptr(), need, s) == g.GEMM_ERR_INVALID_ARG
    assert g.launch_count() == n0
    # the workspace route: one copy of A, one GEMM
    c.zero_()
    assert lib.gemm_f16_f32acc_strided_ws(*args, ws.data_ptr(), need, s) == g.GEMM_OK
    assert g.launch_count() - n0 == 2
    assert g.query_status() == g.GEMM_OK
    check_against_oracle(A, B, c)


def test_autotune_picks_fastest_and_auto_follows(gemm_lib):
    M, N, K = 1024, 768, 256
    A, B = inputs.gemm_inputs(M, N, K, seed=13)
    a, b = A.cuda(), B.cuda()
    default_shape = g.tile_shape(g.TILE_AUTO, M, N, K)
    try:
        r = g.autotune(a, b, reps=5)
        assert set(r["us"]) == set(range(1, g.TILE_COUNT))
        assert all(v > 0 for v in r["us"].values())
        assert r["best"] == min(r["us"], key=r["us"].get)
        # TILE_AUTO now resolves to the tuned configuration for this shape only
        assert g.tile_shape(g.TILE_AUTO, M, N, K) == g.tile_shape(r["best"])
        assert g.tile_shape(g.TILE_AUTO, 8192, 8192, 8192) == (256, 256, 64)    # other shapes: the default rule
        n0 = g.launch_count()
        C = g.gemm(a, b)
        assert g.launch_count() - n0 == 1 and g.query_status() == g.GEMM_OK
        check_against_oracle(A, B, C)
    finally:
        g.autotune_clear()
    assert g.tile_shape(g.TILE_AUTO, M, N, K) == default_shape


@pytest.mark.parametrize("M,N,K,S", [
    (512, 512, 512, 4),       # 16 tiles: eight-CTA clusters only up to 64 CTAs
    (1024, 768, 128, 2),      # 2 k steps: 2-way
    (300, 257, 320, 4),       # 5 k steps over a 4-CTA cluster: the last CTA has none (a zero partial)
    (129, 1000, 4000, 4),     # ragged M and N, long K, 16 tiles
    (300, 200, 4096, 8),      # 6 tiles: 48 CTAs in eight-CTA clusters
    (1, 8, 8, 1),
    (100, 100, 64, 1),        # a single k step: no split
])
def test_split_k_cluster(gemm_lib, M, N, K, S):
    A, B = inputs.gemm_inputs(M, N, K, seed=3 * M + N + K)
    plan = g.launch_plan(M, N, K, tile_cfg=g.TILE_128x128x64_SPLITK)
    tiles = -(-M // 128) * -(-N // 128)
    assert plan["num_tiles"] == tiles
    # one cluster of S CTAs per tile; S = 1 is the one-CTA 128 x 128 kernel
    assert plan["grid_ctas"] == S * tiles
    C = g.gemm(A.cuda(), B.cuda(), tile_cfg=g.TILE_128x128x64_SPLITK)
    assert g.query_status() == g.GEMM_OK
    check_against_oracle(A, B, C)
    C2 = g.gemm(A.cuda(), B.cuda(), tile_cfg=g.TILE_128x128x64_SPLITK)
    assert torch.equal(C, C2)   # the partials are summed in a fixed order


def test_autotune_checks_its_operands(gemm_lib):
    a = torch.zeros((256, 128), dtype=torch.float16, device="cuda")
    b = torch.zeros((128, 256), dtype=torch.float16, device="cuda")
    n0 = g.launch_count()
    with pytest.raises(ValueError):
        g.autotune(a, b[:64], reps=1)                                   # inner extents differ
    with pytest.raises(ValueError):
        g.autotune(a, b, out=torch.empty((256, 128), dtype=torch.float16, device="cuda"), reps=1)
    with pytest.raises(TypeError):
        g.autotune(a, b, out=torch.empty((256, 256), dtype=torch.float32, device="cuda"), reps=1)
    assert g.launch_count() == n0
