"""Pins of the integer tile-map oracle (oracle/tile_map.py).

Each test ties the oracle to something other than its own formula: the values
the kernl notebook '2 - matmul offsets.ipynb' prints for its worked example,
its printed pointer matrices, closed forms of the map for special group sizes,
an independent nested-loop construction of the grouped order, and bijection.
"""
import itertools
import json
import os

import pytest

from oracle import tile_map as tm


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def test_worked_example_printed_values(golden_dir):
    g = _load(golden_dir, "tile_map_worked_example.json")
    i = g["inputs"]
    e = {k: v["value"] for k, v in g["expected"].items()}
    d = tm.grouped_pid(i["pid"], i["M"], i["N"], i["BLOCK_SIZE_M"], i["BLOCK_SIZE_N"], i["GROUP_SIZE_M"])
    assert d["num_pid_m"] == e["num_pid_m"]
    assert d["num_pid_n"] == e["num_pid_n"]
    assert d["num_pid_n"] * i["GROUP_SIZE_M"] == e["num_pid_n_times_group"]
    assert d["nb_programs"] == e["nb_programs"]
    assert tm.program_count(i["M"], i["N"], i["BLOCK_SIZE_M"], i["BLOCK_SIZE_N"]) == e["nb_programs"]
    assert d["num_pid_in_group"] == e["num_pid_in_group"]
    assert d["group_id"] == e["group_id"]
    assert d["first_pid_m"] == e["first_pid_m"]
    assert d["group_size_m"] == e["group_size_m"]
    assert (d["pid_m"], d["pid_n"]) == (e["pid_m"], e["pid_n"])


def test_cdiv_is_ceiling():
    for x in range(0, 300):
        for y in range(1, 40):
            q = tm.cdiv(x, y)
            assert (q - 1) * y < x <= q * y or (x == 0 and q == 0)


def test_pointer_matrices_pid60(golden_dir):
    """Relative element offsets of the printed a_ptrs / b_ptrs corners."""
    g = _load(golden_dir, "pointer_matrices_pid60.json")
    # contiguous operands of the worked example: A 1024x128, B 128x768
    pid_m, pid_n = tm.tile_of(60, 1024, 768, 128, 64, 2)
    a_offs, b_offs = tm.operand_offsets(pid_m, pid_n, 128, 64, 32,
                                        stride_am=128, stride_ak=1, stride_bk=768, stride_bn=1)
    assert (len(a_offs), len(a_offs[0])) == tuple(g["a_ptrs"]["shape"])
    assert (len(b_offs), len(b_offs[0])) == tuple(g["b_ptrs"]["shape"])
    for name, offs in (("a_ptrs", a_offs), ("b_ptrs", b_offs)):
        rows, cols, vals = g[name]["rows"], g[name]["cols"], g[name]["values"]
        base_printed = vals[0][0]
        base_oracle = offs[rows[0]][cols[0]]
        for ri, r in enumerate(rows):
            for ci, c in enumerate(cols):
                assert vals[ri][ci] - base_printed == offs[r][c] - base_oracle, (name, r, c)
    # absolute rows/columns the program touches: A rows 512..639, B cols 384..447
    assert a_offs[0][0] == 512 * 128 and a_offs[-1][-1] == 639 * 128 + 31
    assert b_offs[0][0] == 384 and b_offs[-1][-1] == 31 * 768 + 447


SHAPES = [
    # (M, N, BM, BN)
    (1024, 768, 128, 64),
    (8192, 8192, 128, 256),
    (4095, 3000, 128, 256),
    (512, 512, 64, 64),
    (7 * 128, 3 * 64, 128, 64),
    (1, 1, 128, 256),
    (129, 65, 128, 64),
    (1000, 37, 16, 8),
]


@pytest.mark.parametrize("M,N,BM,BN", SHAPES)
@pytest.mark.parametrize("G", [1, 2, 3, 4, 8, 16, 1000])
def test_bijection(M, N, BM, BN, G):
    order = tm.tile_order(M, N, BM, BN, G)
    npm, npn = tm.cdiv(M, BM), tm.cdiv(N, BN)
    assert len(order) == npm * npn
    assert set(order) == set(itertools.product(range(npm), range(npn)))


@pytest.mark.parametrize("M,N,BM,BN", SHAPES)
def test_group_one_is_row_major(M, N, BM, BN):
    # GROUP_SIZE_M = 1: every group is one tile row, walked along N.
    npn = tm.cdiv(N, BN)
    for pid, t in enumerate(tm.tile_order(M, N, BM, BN, 1)):
        assert t == (pid // npn, pid % npn)


@pytest.mark.parametrize("M,N,BM,BN", SHAPES)
def test_group_covering_grid_is_column_major(M, N, BM, BN):
    # GROUP_SIZE_M >= num_pid_m: one group, column-major over the whole grid.
    npm = tm.cdiv(M, BM)
    for G in (npm, npm + 1, 10 * npm):
        for pid, t in enumerate(tm.tile_order(M, N, BM, BN, G)):
            assert t == (pid % npm, pid // npm)


def _nested_loop_order(num_pid_m, num_pid_n, G):
    """The grouped order built from its description, not from the formula:
    bands of G tile rows, taken top to bottom; inside a band, columns left to
    right, and inside a column the band's rows top to bottom."""
    out = []
    for band_start in range(0, num_pid_m, G):
        rows = list(range(band_start, min(band_start + G, num_pid_m)))
        for pn in range(num_pid_n):
            for pm in rows:
                out.append((pm, pn))
    return out


@pytest.mark.parametrize("M,N,BM,BN", SHAPES)
@pytest.mark.parametrize("G", [1, 2, 3, 4, 8])
def test_matches_nested_loops(M, N, BM, BN, G):
    """Every full band follows the nested loops exactly. In a clamped last
    band the notebook's row index (full pid modulo the clamped height) may be
    a rotation of the nested-loop order; there the column and the set of rows
    per column must still agree."""
    npm, npn = tm.cdiv(M, BM), tm.cdiv(N, BN)
    order = tm.tile_order(M, N, BM, BN, G)
    want = _nested_loop_order(npm, npn, G)
    full = (npm // G) * G * npn
    assert order[:full] == want[:full]
    tail_got, tail_want = order[full:], want[full:]
    h = npm - (npm // G) * G
    for c in range(npn):
        got_c = tail_got[c * h:(c + 1) * h]
        want_c = tail_want[c * h:(c + 1) * h]
        assert all(t[1] == c for t in got_c)
        assert sorted(got_c) == sorted(want_c)


def test_clamped_band_example():
    # num_pid_m = 7, G = 2: last band is one row high; it ends (6,0),(6,1),(6,2)
    order = tm.tile_order(7 * 128, 3 * 64, 128, 64, 2)
    assert order[-3:] == [(6, 0), (6, 1), (6, 2)]
    assert order[:6] == [(0, 0), (1, 0), (0, 1), (1, 1), (0, 2), (1, 2)]


def test_rejects_bad_arguments():
    with pytest.raises(ValueError):
        tm.grouped_pid(96, 1024, 768, 128, 64, 2)
    with pytest.raises(ValueError):
        tm.grouped_pid(0, 1024, 768, 128, 64, 0)
