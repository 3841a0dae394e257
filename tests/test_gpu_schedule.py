"""The device-side grouped tile map and the GEMM kernel's own tile order,
checked bit-exactly against the integer oracle (oracle/tile_map.py)."""
import pytest
import torch

import dense_fp16_gemm_fp32_gb300 as g
from dense_fp16_gemm_fp32_gb300 import inputs
from oracle import tile_map as tm

from _gpu_util import check_against_oracle

pytestmark = pytest.mark.gpu


SCHEDULE_CASES = [
    # (M, N, tile_m, tile_n, G)
    (1024, 768, 128, 64, 2),          # the notebook's worked example
    (8192, 8192, 128, 256, 8),
    (4095, 3000, 128, 256, 8),
    (7 * 128, 3 * 64, 128, 64, 2),    # clamped last band
    (7 * 128, 5 * 64, 128, 64, 4),
    (16384, 16384, 128, 256, 16),
    (1, 1, 128, 256, 1),
    (1000, 37, 16, 8, 3),
    (5000, 3000, 64, 48, 1000),
]


@pytest.mark.parametrize("M,N,TM,TN,G", SCHEDULE_CASES)
def test_device_tile_map_bit_exact(gemm_lib, M, N, TM, TN, G):
    pm, pn = g.tile_schedule(M, N, TM, TN, G)
    want = tm.tile_order(M, N, TM, TN, G)
    assert pm.numel() == len(want)
    got = list(zip(pm.cpu().tolist(), pn.cpu().tolist()))
    assert got == want


def test_worked_example_pid60_on_device(gemm_lib):
    pm, pn = g.tile_schedule(1024, 768, 128, 64, 2)
    assert pm.numel() == 96
    assert (int(pm[60]), int(pn[60])) == (4, 6)


def _kernel_trace(M, N, K, G, cfg, seed):
    tmm, tnn, _ = g.tile_shape(cfg)
    ntiles = -(-M // tmm) * -(-N // tnn)
    A, B = inputs.gemm_inputs(M, N, K, seed)
    trace = torch.full((3 * ntiles,), -1, dtype=torch.int32, device="cuda")
    C = g.gemm(A.cuda(), B.cuda(), group_size_m=G, tile_cfg=cfg, trace=trace)
    assert g.query_status() == g.GEMM_OK
    return A, B, C, trace.view(ntiles, 3).cpu(), tmm, tnn


@pytest.mark.parametrize("M,N,K,G,cfg", [
    (1024, 768, 128, 2, g.TILE_128x64x32),     # the worked example, 96 programs
    (8192, 8192, 256, 8, g.TILE_128x256x64),   # 2048 tiles: many per CTA
    (4095, 3000, 64, 5, g.TILE_128x256x64),    # ragged grid, clamped band
    (8192, 8192, 128, 8, g.TILE_256x256x64_PAIR),   # 1024 pair tiles, split tail on 76 clusters
    (4095, 3000, 64, 3, g.TILE_256x256x64_PAIR),
    (4095, 3000, 1000, 4, g.TILE_256x256x128_PAIR),
    (8192, 8192, 256, 8, g.TILE_256x256x128_PAIR),
    (512, 1024, 256, 2, g.TILE_256x256x128_PAIR),    # 8 tiles: every tile split
    (2048, 4096, 256, 3, g.TILE_256x256x128_PAIR),
    (2048, 4096, 256, 3, g.TILE_256x256x128_PAIR_ALIGNED),
    (8192, 8192, 256, 8, g.TILE_256x256x128_PAIR_ALIGNED),
    (896, 192, 64, 2, g.TILE_128x64x32),
    (4095, 3000, 200, 4, g.TILE_128x128x64),
    (512, 640, 512, 2, g.TILE_128x128x64_SPLITK),   # 20 tiles, one cluster each
    (1024, 768, 128, 2, g.TILE_128x64x64),     # the worked example's 96 tiles, 64-deep k steps
    (4095, 3000, 200, 3, g.TILE_128x64x64),    # 32 x 47 tiles: several per CTA
    (4095, 3000, 200, 3, g.TILE_128x64x32),    # the same with 32-deep k steps
    (512, 512, 512, 8, g.TILE_64x64x64),       # 64 tiles of 64 rows (tcgen05 M = 64)
    (4095, 3000, 200, 5, g.TILE_64x64x64),     # 64 x 47 tiles: several per CTA, clamped band
])
def test_kernel_walks_grouped_order(gemm_lib, M, N, K, G, cfg):
    A, B, C, tr, TM, TN = _kernel_trace(M, N, K, G, cfg, seed=31)
    want = tm.tile_order(M, N, TM, TN, G)
    got = [(int(a), int(b)) for a, b in tr[:, :2].tolist()]
    assert got == want                      # every pid processed once, with the oracle's tile
    ctas = tr[:, 2]
    plan = g.launch_plan(M, N, K, tile_cfg=cfg)
    assert plan["num_tiles"] == len(want)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if cfg in (g.TILE_256x256x64_PAIR, g.TILE_256x256x128_PAIR, g.TILE_256x256x128_PAIR_ALIGNED):
        clusters = plan["grid_ctas"] // 2
        assert 1 <= clusters <= sms // 2
        split = plan["split_tiles"]
        full = len(want) - split
        units = full + 2 * split
        if units > clusters:  # the grid is every resident cluster: the split rule applies
            rem = len(want) % clusters
            assert split == (rem if 0 < 2 * rem <= clusters else 0)
        # persistent schedule over units: the full tiles, then two halves per split pid
        pid = torch.arange(len(want))
        first_unit = torch.where(pid < full, pid, full + 2 * (pid - full))
        assert torch.equal(ctas.long(), first_unit % clusters)
    else:
        grid = int(ctas.max()) + 1
        # persistent schedule: CTA b processes pids b, b + grid, b + 2*grid, ...
        assert torch.equal(ctas, torch.arange(len(want), dtype=torch.int32) % grid)
        assert grid <= sms * 4
    if M * N * K <= 1.3e10:
        check_against_oracle(A, B, C)


@pytest.mark.parametrize("cfg", [g.TILE_256x256x64_PAIR, g.TILE_256x256x128_PAIR, g.TILE_256x256x128_PAIR_ALIGNED])
def test_pair_units_alternate_k_direction(gemm_lib, cfg):
    # A cluster's 2nd, 4th, ... unit sums its k steps downwards. Every entry of C is
    # 2048 + 1 (k = 0, 1) + 2^-13 (k = 128) + 2^-13 (k = 256), each term in its own k step.
    # Upwards, 2^-13 meets 2049, half an fp32 ulp there: both additions tie and keep 2049,
    # which narrows (a tie again) to 2048. Downwards the small terms first make 2^-12, and
    # 2049 + 2^-12 is exact in fp32 and narrows to 2050.
    M, N, K = 2048, 256 * 20, 384
    A = torch.zeros((M, K), dtype=torch.float16)
    B = torch.zeros((K, N), dtype=torch.float16)
    A[:, 0], A[:, 1], A[:, 128], A[:, 256] = 2048.0, 1.0, 2.0 ** -13, 2.0 ** -13
    B[[0, 1, 128, 256], :] = 1.0
    G = 8
    C = g.gemm(A.cuda(), B.cuda(), group_size_m=G, tile_cfg=cfg).cpu().float()
    assert g.query_status() == g.GEMM_OK
    plan = g.launch_plan(M, N, K, tile_cfg=cfg)
    clusters = plan["grid_ctas"] // 2
    tiles = plan["num_tiles"]
    split = plan["split_tiles"]
    full = tiles - split
    assert tiles > clusters                # some clusters take a second unit
    order = tm.tile_order(M, N, 256, 256, G)
    want = torch.empty_like(C)
    for u in range(full + 2 * split):
        pid, half = (u, -1) if u < full else (full + (u - full) // 2, (u - full) % 2)
        pm, pn = order[pid]
        c0 = pn * 256 + (0 if half < 0 else 128 * half)
        c1 = c0 + (256 if half < 0 else 128)
        want[pm * 256:(pm + 1) * 256, c0:c1] = 2050.0 if (u // clusters) % 2 == 1 else 2048.0
    assert torch.equal(C, want)
    assert (want == 2050.0).any() and (want == 2048.0).any()


def test_short_trace_is_refused_before_launch(gemm_lib):
    # the kernels write 3 entries per tile: a shorter trace would be written past its end
    A, B = inputs.gemm_inputs(512, 512, 64, seed=5)
    a, b = A.cuda(), B.cuda()
    n0 = g.launch_count()
    short = torch.zeros(3 * 4 - 1, dtype=torch.int32, device="cuda")     # 4 pair tiles
    with pytest.raises(ValueError):
        g.gemm(a, b, tile_cfg=g.TILE_256x256x64_PAIR, trace=short)
    # A one element off a 16-byte boundary without a workspace: the generic-load
    # kernel's 128 x 256 tiles (8 here) need more entries than the 4 pair tiles
    buf = torch.empty(a.numel() + 1, dtype=torch.float16, device="cuda")
    buf[1:] = a.reshape(-1)
    pair_sized = torch.zeros(3 * 4, dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        g.gemm(buf[1:].view(a.shape), b, tile_cfg=g.TILE_256x256x64_PAIR, trace=pair_sized, repack=False)
    assert g.launch_count() == n0
    full = torch.full((3 * 8,), -1, dtype=torch.int32, device="cuda")
    g.gemm(buf[1:].view(a.shape), b, tile_cfg=g.TILE_256x256x64_PAIR, trace=full, repack=False)
    assert g.query_status() == g.GEMM_OK
    assert sorted((int(full[3 * i]), int(full[3 * i + 1])) for i in range(8)) == [(m, n) for m in range(4) for n in range(2)]
