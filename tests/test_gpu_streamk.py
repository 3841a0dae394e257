"""The stream-K configuration (GEMM_TILE_256x256x64_PAIR_STREAMK).

Where the last partial wave of 256 x 256 tiles holds more than half of the
resident clusters, that wave and one full wave are split by k iterations into
one contiguous range per cluster (the stream-K decomposition of Osama et al.,
PPoPP 2023, in its hybrid form); where at most half of the clusters hold a
tile each and K is long, every tile is split into two k halves on two
clusters. A tile shared by two clusters has the fp32 partial sums of its
first k steps passed through a workspace and added before the single fp16
rounding. Elsewhere the configuration runs the plain pair schedule. Every
case is checked element by element against the CPU oracle.
"""

import pytest
import torch

import dense_fp16_gemm_fp32_gb300 as g
from dense_fp16_gemm_fp32_gb300 import inputs
from oracle import tile_map as tm

from _gpu_util import check_against_oracle

pytestmark = pytest.mark.gpu

SK = g.TILE_256x256x64_PAIR_STREAMK
CANARY = 0x7E01


def plan(M, N, K):
    p = g.launch_plan(M, N, K, tile_cfg=SK)
    clusters = p["grid_ctas"] // 2
    return clusters, p["num_tiles"], p["split_tiles"]


def resident_clusters():
    # the plain pair schedule of a problem with many tiles uses every resident cluster
    return g.launch_plan(8192, 8192, 64, tile_cfg=g.TILE_256x256x64_PAIR)["grid_ctas"] // 2


HALVES_MIN_K_STEPS = 160   # 64-deep k steps per tile from which the k-halves form applies


def expected_stream_k(tiles, k_tiles, clusters):
    """(stream-K tiles, clusters of the launch) on `clusters` resident clusters, (0, 0): plain."""
    if tiles == 0 or k_tiles == 0:
        return 0, 0
    if tiles < clusters:
        return (tiles, 2 * tiles) if 2 * tiles <= clusters and k_tiles >= HALVES_MIN_K_STEPS else (0, 0)
    rem = tiles % clusters
    return (rem + clusters, clusters) if 2 * rem > clusters else (0, 0)


SHAPES = [
    (4095, 3000, 1000),   # the ragged workload: 192 tiles, 16 k steps each
    (3072, 3072, 512),    # 144 tiles: every tile in the stream-K range
    (2048, 4608, 200),    # 4 k steps, the last one partial
    (4096, 3328, 72),     # 2 k steps
    (5120, 2816, 1000),   # 220 tiles: a wave of whole tiles first
    (4095, 3000, 64),     # one k step per tile: no tile is shared
    (2304, 4352, 64),     # 153 tiles: the split tail instead (plain schedule)
    (4095, 3000, 1001),   # K not a multiple of 8: the workspace route repacks, then stream-K
    (4096, 3072, 8192),   # long K: where GEMM_TILE_AUTO takes stream-K (256 sampled rows)
    (4000, 3072, 4100),   # ragged M and K, 65 k steps
    (256, 256, 10240),    # one tile in two k halves on two clusters
    (1000, 1100, 12200),  # 20 tiles, 191 k steps (odd, the last one partial): k halves
    (1536, 1536, 10240),  # 36 tiles on 72 clusters (256 sampled rows)
    (2048, 1024, 10176),  # 159 k steps: just short of the k-halves form (split tail)
]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_stream_k_matches_oracle(gemm_lib, M, N, K):
    clusters, tiles, split = plan(M, N, K)
    want_sk, want_clusters = expected_stream_k(tiles, -(-K // 64), resident_clusters())
    if want_sk:
        assert split == want_sk and clusters == want_clusters
    A, B = inputs.gemm_inputs(M, N, K, seed=M + N + K)
    a, b = A.cuda(), B.cuda()
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    g.gemm(a, b, out=C, tile_cfg=SK)
    assert g.query_status() == g.GEMM_OK
    check_against_oracle(A, B, C, inputs.sample_rows(M, 17) if M * N * K > 1.3e10 else None)
    # deterministic: the split points and the order of the two partial sums are fixed
    C2 = g.gemm(a, b, tile_cfg=SK)
    assert g.query_status() == g.GEMM_OK
    assert torch.equal(C.view(torch.int16), C2.view(torch.int16))


def test_stream_k_applies_to_the_ragged_workload(gemm_lib):
    clusters, tiles, split = plan(4095, 3000, 1000)
    assert tiles == 192
    if clusters == 76:
        assert split == 116  # 40 tiles in the last wave: that wave and one full wave, 116 x 16 iterations


def test_auto_runs_stream_k_for_long_k(gemm_lib):
    M, N, K = 4096, 3072, 8192
    assert g.tile_config(g.TILE_AUTO, M, N, K) == SK
    A, B = inputs.gemm_inputs(M, N, K, seed=5)
    a, b = A.cuda(), B.cuda()
    C = g.gemm(a, b)
    assert g.query_status() == g.GEMM_OK
    assert torch.equal(C, g.gemm(a, b, tile_cfg=SK))
    check_against_oracle(A, B, C, inputs.sample_rows(M, 19))


def test_auto_runs_k_halves_for_few_tiles_and_long_k(gemm_lib):
    M, N, K = 1536, 1536, 10240
    assert g.tile_config(g.TILE_AUTO, M, N, K) == SK
    clusters, tiles, split = plan(M, N, K)
    if resident_clusters() >= 72:
        assert (tiles, split, clusters) == (36, 36, 72)   # every tile in two halves
    A, B = inputs.gemm_inputs(M, N, K, seed=7)
    a, b = A.cuda(), B.cuda()
    C = g.gemm(a, b)
    assert g.query_status() == g.GEMM_OK
    assert torch.equal(C, g.gemm(a, b, tile_cfg=SK))
    check_against_oracle(A, B, C, inputs.sample_rows(M, 29))


def test_stream_k_small_integers_exact(gemm_lib):
    M, N, K = 4095, 3000, 1000
    gen = torch.Generator().manual_seed(11)
    A = torch.randint(-2, 3, (M, K), generator=gen).half()
    B = torch.randint(-2, 3, (K, N), generator=gen).half()
    C = g.gemm(A.cuda(), B.cuda(), tile_cfg=SK)
    assert g.query_status() == g.GEMM_OK
    # every partial sum is an integer of magnitude <= 4000 < 2^24: exact in fp32;
    # values above 2048 round to even in fp16 on both sides the same way
    assert torch.equal(C.cpu(), (A.float() @ B.float()).half())


@pytest.mark.parametrize("M,N,K", [(4095, 3000, 1000), (3072, 3072, 136), (1000, 1100, 12200)])
def test_stream_k_trace_and_schedule(gemm_lib, M, N, K):
    clusters, tiles, split = plan(M, N, K)
    G = 4
    trace = torch.full((3 * tiles,), -1, dtype=torch.int32, device="cuda")
    A, B = inputs.gemm_inputs(M, N, K, seed=3)
    C = g.gemm(A.cuda(), B.cuda(), group_size_m=G, tile_cfg=SK, trace=trace)
    assert g.query_status() == g.GEMM_OK
    tr = trace.view(tiles, 3).cpu()
    assert [(int(x), int(y)) for x, y in tr[:, :2].tolist()] == tm.tile_order(M, N, 256, 256, G)
    kt = -(-K // 64)
    first = tiles - split
    iters = split * kt
    for pid in range(tiles):
        if pid < first:
            want = pid % clusters  # whole tiles in turn
        else:
            # the cluster holding the tile's last k step finishes it
            i = (pid - first) * kt + kt - 1
            want = next(c for c in range(clusters) if c * iters // clusters <= i < (c + 1) * iters // clusters)
        assert int(tr[pid, 2]) == want, (pid, int(tr[pid, 2]), want)
    check_against_oracle(A, B, C, inputs.sample_rows(M, 23) if M * N * K > 1.3e10 else None)


def test_stream_k_no_store_outside_c(gemm_lib):
    M, N, K = 4095, 3000, 1000
    A, B = inputs.gemm_inputs(M, N, K, seed=21)
    pad = 4096
    buf = torch.full((pad + M * N + pad,), CANARY, dtype=torch.int16, device="cuda")
    C = buf[pad:pad + M * N].view(torch.float16).view(M, N)
    g.gemm(A.cuda(), B.cuda(), out=C, tile_cfg=SK)
    assert g.query_status() == g.GEMM_OK
    assert torch.all(buf[:pad] == CANARY) and torch.all(buf[pad + M * N:] == CANARY)
    check_against_oracle(A, B, C)


def test_stream_k_watchdog_reports_and_recovers(gemm_lib):
    M, N, K = 4095, 3000, 1000
    A, B = inputs.gemm_inputs(M, N, K, seed=23)
    a, b = A.cuda(), B.cuda()
    assert g.query_status() == g.GEMM_OK
    try:
        g.set_watchdog_ns(50_000_000)  # 50 ms
        g.set_fault_injection(1)       # no loads: the MMA warps' waits run out
        g.gemm(a, b, tile_cfg=SK)
        assert g.query_status() == g.GEMM_ERR_TIMEOUT   # also clears the stream-K flags
        assert g.query_status() == g.GEMM_OK
    finally:
        g.set_fault_injection(0)
        g.set_watchdog_ns(0)
    C = g.gemm(a, b, tile_cfg=SK)
    assert g.query_status() == g.GEMM_OK
    check_against_oracle(A, B, C)


def test_stream_k_on_two_streams_at_once(gemm_lib):
    # each stream has its own workspace: concurrent launches do not share partial tiles
    M, N, K = 4095, 3000, 1000
    A1, B1 = inputs.gemm_inputs(M, N, K, seed=31)
    A2, B2 = inputs.gemm_inputs(M, N, K, seed=32)
    a1, b1, a2, b2 = A1.cuda(), B1.cuda(), A2.cuda(), B2.cuda()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    c1 = torch.empty((M, N), dtype=torch.float16, device="cuda")
    c2 = torch.empty((M, N), dtype=torch.float16, device="cuda")
    for s in (s1, s2):
        s.wait_stream(torch.cuda.current_stream())
    for _ in range(3):
        with torch.cuda.stream(s1):
            g.gemm(a1, b1, out=c1, tile_cfg=SK)
        with torch.cuda.stream(s2):
            g.gemm(a2, b2, out=c2, tile_cfg=SK)
    torch.cuda.synchronize()
    assert g.query_status() == g.GEMM_OK
    check_against_oracle(A1, B1, c1)
    check_against_oracle(A2, B2, c2)
