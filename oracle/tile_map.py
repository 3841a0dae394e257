"""Integer oracle of the grouped program-ID -> output-tile mapping.

TEST INFRASTRUCTURE ONLY: imported by the tests, the package smoke check and
the benchmark's CPU baseline, never by the product path. Pure Python ints; no
numpy, no torch, nothing shared with the CUDA library.

Source: "2 - matmul offsets.ipynb" (kernl tutorial notebook), the markdown
cell that restates the Triton matmul tutorial's program-ID code, and the code
cells that recompute it step by step for M=1024, N=768, K=128 with
BLOCK_SIZE_M=128, BLOCK_SIZE_N=64, BLOCK_SIZE_K=32, GROUP_SIZE_M=2.

Names follow the notebook (num_pid_m, num_pid_n, num_pid_in_group, group_id,
first_pid_m, group_size_m, pid_m, pid_n).

Reading: the notebook's row index is ``first_pid_m + pid % group_size_m``
(the full program id modulo the clamped group height). Later Triton releases
take ``(pid % num_pid_in_group) % group_size_m`` instead; the two agree on
every group except a clamped last group whose height does not divide the
group's first program id. This module follows the notebook.
"""
from __future__ import annotations


def cdiv(x: int, y: int) -> int:
    """Ceiling division, the notebook's ``cdiv`` (first code cell)."""
    return (x + y - 1) // y


def program_count(M: int, N: int, block_m: int, block_n: int) -> int:
    """Number of programs of the 1-D launch: tiles along M times tiles along N
    (the notebook's grid lambda and its ``nb_programs`` cell)."""
    return cdiv(M, block_m) * cdiv(N, block_n)


def grouped_pid(pid: int, M: int, N: int, block_m: int, block_n: int, group_size_m: int) -> dict:
    """All intermediate values of the grouped mapping for one program id.

    Follows the notebook's program-ID code in its order:
    tiles per axis, programs per group (GROUP_SIZE_M rows of tiles times every
    tile column), the group a program falls in, that group's first tile row,
    the group's real height (the last group is clamped by ``min``), and inside
    the group a column-major walk: the tile row cycles fastest.
    """
    GROUP_SIZE_M = group_size_m
    if not (block_m > 0 and block_n > 0 and GROUP_SIZE_M > 0):
        raise ValueError("block sizes and GROUP_SIZE_M must be positive")
    num_pid_m = cdiv(M, block_m)
    num_pid_n = cdiv(N, block_n)
    nb_programs = num_pid_m * num_pid_n
    if not (0 <= pid < nb_programs):
        raise ValueError(f"pid {pid} outside [0, {nb_programs})")
    num_pid_in_group = GROUP_SIZE_M * num_pid_n
    group_id = pid // num_pid_in_group
    first_pid_m = group_id * GROUP_SIZE_M
    gsm = min(num_pid_m - first_pid_m, GROUP_SIZE_M)
    assert gsm > 0  # the notebook asserts the same
    pid_m = first_pid_m + (pid % gsm)
    pid_n = (pid % num_pid_in_group) // gsm
    return {
        "num_pid_m": num_pid_m,
        "num_pid_n": num_pid_n,
        "nb_programs": nb_programs,
        "num_pid_in_group": num_pid_in_group,
        "group_id": group_id,
        "first_pid_m": first_pid_m,
        "group_size_m": gsm,
        "pid_m": pid_m,
        "pid_n": pid_n,
    }


def tile_of(pid: int, M: int, N: int, block_m: int, block_n: int, group_size_m: int) -> tuple[int, int]:
    """(pid_m, pid_n) of one program."""
    d = grouped_pid(pid, M, N, block_m, block_n, group_size_m)
    return d["pid_m"], d["pid_n"]


def tile_order(M: int, N: int, block_m: int, block_n: int, group_size_m: int) -> list[tuple[int, int]]:
    """(pid_m, pid_n) for every pid in launch order 0, 1, ..., nb_programs-1."""
    return [tile_of(p, M, N, block_m, block_n, group_size_m)
            for p in range(program_count(M, N, block_m, block_n))]


def operand_offsets(pid_m: int, pid_n: int, block_m: int, block_n: int, block_k: int,
                    stride_am: int, stride_ak: int, stride_bk: int, stride_bn: int):
    """Element offsets (from each operand's first element) that program
    (pid_m, pid_n) reads in its first k step, as the notebook's last code cell
    builds them by broadcasting: rows ``pid_m*BLOCK_SIZE_M + [0, BLOCK_SIZE_M)``
    of A against columns ``[0, BLOCK_SIZE_K)``, and rows ``[0, BLOCK_SIZE_K)``
    of B against columns ``pid_n*BLOCK_SIZE_N + [0, BLOCK_SIZE_N)``.

    Returns (a_offs, b_offs) as lists of lists: a_offs[i][k], b_offs[k][j].
    """
    offs_am = [pid_m * block_m + i for i in range(block_m)]
    offs_bn = [pid_n * block_n + j for j in range(block_n)]
    offs_k = list(range(block_k))
    a_offs = [[am * stride_am + k * stride_ak for k in offs_k] for am in offs_am]
    b_offs = [[k * stride_bk + bn * stride_bn for bn in offs_bn] for k in offs_k]
    return a_offs, b_offs
