"""The kernels' grouped map, evaluated on the host through the C ABI
(gemm_tile_map_host: the same function the kernels call, with the group and
band divisions done as multiply-shift divisions), checked bit-exactly against
the integer oracle (oracle/tile_map.py). Needs no GPU."""
import random

import pytest

import dense_fp16_gemm_fp32_gb300 as g
from oracle import tile_map as tm


@pytest.fixture(scope="module")
def lib():
    g.build()
    return g.load()


CASES = [
    # (M, N, tile_m, tile_n, G)
    (1024, 768, 128, 64, 2),          # the notebook's worked example
    (8192, 8192, 256, 256, 8),        # the CTA-pair tiles at 8192^3
    (8192, 8192, 128, 256, 8),
    (4095, 3000, 256, 256, 8),
    (7 * 128, 3 * 64, 128, 64, 2),    # clamped last band of height 1
    (7 * 128, 5 * 64, 128, 64, 4),    # clamped last band of height 3
    (16384, 16384, 256, 256, 16),
    (1, 1, 128, 256, 1),
    (1000, 37, 16, 8, 3),
    (5000, 3000, 64, 48, 1000),       # G clamped to num_pid_m
    (999, 1001, 1, 1, 7),
]


@pytest.mark.parametrize("M,N,TM,TN,G", CASES)
def test_host_map_matches_oracle(lib, M, N, TM, TN, G):
    pm, pn = g.tile_map_host(M, N, TM, TN, G)
    assert list(zip(pm.tolist(), pn.tolist())) == tm.tile_order(M, N, TM, TN, G)


def test_worked_example_pid60(lib):
    pm, pn = g.tile_map_host(1024, 768, 128, 64, 2, pid0=60, count=1)
    assert (int(pm[0]), int(pn[0])) == (4, 6)


def test_random_grids_and_groups(lib):
    rng = random.Random(20261202)
    for _ in range(300):
        npm, npn = rng.randint(1, 90), rng.randint(1, 90)
        G = rng.choice([1, 2, 3, 5, 8, 13, 16, rng.randint(1, 100)])
        M, N = npm * 16 - rng.randint(0, 15), npn * 8 - rng.randint(0, 7)
        pm, pn = g.tile_map_host(M, N, 16, 8, G)
        assert list(zip(pm.tolist(), pn.tolist())) == tm.tile_order(M, N, 16, 8, G), (M, N, G)


@pytest.mark.parametrize("G", [1, 3, 7, 64, 1000, 46340])
def test_pids_near_the_int32_limit(lib, G):
    # 46340 x 46340 one-element tiles: 2,147,395,600 pids, so the divisions
    # see dividends up to 2^31 - 1 and group divisors up to ~2^31
    M = N = 46340
    n = M * N
    rng = random.Random(G)
    starts = [0, n - 64, n // 2, G * N - 32] + [rng.randrange(0, n - 64) for _ in range(20)]
    for p0 in starts:
        p0 = max(0, min(p0, n - 64))
        pm, pn = g.tile_map_host(M, N, 1, 1, G, pid0=p0, count=64)
        want = [tm.tile_of(p, M, N, 1, 1, G) for p in range(p0, p0 + 64)]
        assert list(zip(pm.tolist(), pn.tolist())) == want, (G, p0)


def test_host_map_validation(lib):
    import ctypes
    assert lib.gemm_tile_map_host(100, 100, 16, 16, 0, 0, 1, None, None) == g.GEMM_ERR_INVALID_ARG
    assert lib.gemm_tile_map_host(100, 100, 16, 16, 1, 0, -1, None, None) == g.GEMM_ERR_INVALID_ARG
    assert lib.gemm_tile_map_host(100, 100, 16, 16, 1, 0, 1, None, None) == g.GEMM_ERR_INVALID_ARG
    buf = (ctypes.c_int32 * 64)()
    assert lib.gemm_tile_map_host(100, 100, 16, 16, 1, 40, 10, buf, buf) == g.GEMM_ERR_INVALID_ARG  # past 49 tiles
    assert lib.gemm_tile_map_host(1 << 30, 1 << 30, 1, 1, 1, 0, 1, buf, buf) == g.GEMM_ERR_UNSUPPORTED
    assert lib.gemm_tile_map_host(100, 100, 16, 16, 1, 0, 0, None, None) == g.GEMM_OK
