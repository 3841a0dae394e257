"""Seeded synthetic inputs, shared by the tests and the benchmark.

This module holds no GEMM or softmax arithmetic: it only draws operands and
picks rows.

Recipe (the check of "03: Matrix multiplication", phobos-lang.dev tutorial,
seeds and shapes as listed in WORKLOADS): a host generator seeded with
`seed`, then A = rand([M,K], fp16) - 0.5 and B = rand([K,N], fp16) - 0.5 drawn
from it in that order, i.e. values in [-0.5, 0.5). Inputs are made on the host
and copied to the GPU, so the device path and the CPU oracle see the same
bytes (the CPU and CUDA generators of torch differ).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


def uniform_f16(shape, generator: torch.Generator) -> torch.Tensor:
    return torch.rand(tuple(shape), dtype=torch.float16, generator=generator) - 0.5


def gemm_inputs(M: int, N: int, K: int, seed: int):
    """(A [M,K], B [K,N]) fp16 on the host, uniform in [-0.5, 0.5)."""
    g = torch.Generator().manual_seed(seed)
    A = uniform_f16((M, K), g)
    B = uniform_f16((K, N), g)
    return A, B


def sample_rows(M: int, seed: int, count: int = 256) -> torch.Tensor:
    """`count` distinct rows of an M-row output, sorted (all rows if M <= count)."""
    if M <= count:
        return torch.arange(M)
    g = torch.Generator().manual_seed(seed + 1000)
    return torch.randperm(M, generator=g)[:count].sort().values


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    seed: int
    tile_cfg: int = 0          # 0 = library default
    group_size_m: int = 8
    sampled: bool = False      # verified on 256 seeded rows instead of every row


# The synthetic workloads: the tutorial's 512^3 check, the notebook's worked
# example shape with its 128x64x32 tile and GROUP_SIZE_M 2, a square sweep,
# a ragged shape with no extent a tile multiple, and a large square.
WORKLOADS = [
    Workload("square512", 512, 512, 512, 0),
    Workload("worked_example_1024x768x128", 1024, 768, 128, 1, tile_cfg=2, group_size_m=2),
    Workload("square1024", 1024, 1024, 1024, 2),
    Workload("square2048", 2048, 2048, 2048, 3),
    Workload("square4096", 4096, 4096, 4096, 4, sampled=True),
    Workload("square8192", 8192, 8192, 8192, 5, sampled=True),
    Workload("ragged_4095x3000x1000", 4095, 3000, 1000, 6),
    Workload("square16384", 16384, 16384, 16384, 7, sampled=True),
]

WORKLOADS_BY_NAME = {w.name: w for w in WORKLOADS}


def softmax_inputs(M: int, n: int, ld: int, seed: int, pad_value: float = 0.0) -> torch.Tensor:
    """X [M, ld] fp32 on the host: standard normal in the first n columns, `pad_value` after.

    Recipe (the check of "02: Fused softmax", phobos-lang.dev tutorial): a
    host generator seeded with `seed`, then randn([M, n]) in fp32, stored in
    rows `ld` wide (the tutorial stores its 781-column rows 784 wide).
    """
    if ld < n:
        raise ValueError("ld must be at least n")
    g = torch.Generator().manual_seed(seed)
    x = torch.full((M, ld), pad_value, dtype=torch.float32)
    x[:, :n] = torch.randn((M, n), generator=g, dtype=torch.float32)
    return x


@dataclass(frozen=True)
class SoftmaxWorkload:
    name: str
    M: int
    n: int
    ld: int
    seed: int
    sampled: bool = False      # verified on 256 seeded rows instead of every row


# The tutorial's 1823 x 781 input in 784-wide rows; the same row length over
# enough rows that the arrays exceed L2 (the bandwidth measurement); wider
# rows that one warp cannot hold (one CTA per row).
SOFTMAX_WORKLOADS = [
    SoftmaxWorkload("softmax_1823x781", 1823, 781, 784, 0),
    SoftmaxWorkload("softmax_262144x781", 262144, 781, 784, 8, sampled=True),
    SoftmaxWorkload("softmax_8192x8000", 8192, 8000, 8000, 9, sampled=True),
    SoftmaxWorkload("softmax_4096x32768", 4096, 32768, 32768, 10, sampled=True),
]

SOFTMAX_WORKLOADS_BY_NAME = {w.name: w for w in SOFTMAX_WORKLOADS}
