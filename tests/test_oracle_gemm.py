"""Pins of the CPU GEMM oracle (oracle/gemm_oracle.c).

The oracle is tied to things other than itself:
  * the fp16 decoder and the round-to-nearest-even narrowing, exhaustively
    against numpy's and torch's own fp16 conversions;
  * fp64 brute force on small random shapes, inside the standard bound for
    recursive fp32 summation, |c32 - c64| <= gamma_K * sum_k |a_ik||b_kj|
    with gamma_K = K u / (1 - K u), u = 2^-24;
  * identity and zero matrices, exact small-integer products;
  * sums whose fp32 ascending-k value is known in closed form and differs
    from the exact value and from other summation orders;
  * a sum whose single fp16 narrowing differs from narrowing at every step.
"""
import numpy as np
import pytest
import torch

from oracle import gemm as og

U = 2.0 ** -24


def _rand_f16(rng, shape, lo=-0.5, hi=0.5):
    return rng.uniform(lo, hi, size=shape).astype(np.float16)


# --------------------------------------------------------------------------
# fp16 conversions
# --------------------------------------------------------------------------
def test_decode_all_halves_matches_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = og.half_to_float_array(bits)
    want = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def _library_narrow(x32):
    """numpy's and torch's float32 -> float16 (both round to nearest even);
    returns uint16 bits after checking the two libraries agree."""
    with np.errstate(over="ignore"):
        a = x32.astype(np.float16).view(np.uint16)
    b = torch.from_numpy(x32).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    both_nan = np.isnan(a.view(np.float16)) & np.isnan(b.view(np.float16))
    assert np.array_equal(a[~both_nan], b[~both_nan])
    return a


def _check_narrow(x32):
    x32 = np.ascontiguousarray(x32, dtype=np.float32)
    got = og.float_to_half_bits_array(x32)
    want = _library_narrow(x32)
    nan = np.isnan(x32)
    assert np.all(np.isnan(got[nan].view(np.float16)))
    bad = np.nonzero(got[~nan] != want[~nan])[0]
    assert bad.size == 0, (x32[~nan][bad[:5]], got[~nan][bad[:5]], want[~nan][bad[:5]])


def test_narrow_every_half_roundtrips():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = bits.view(np.float16).astype(np.float32)
    _check_narrow(x)
    fin = np.isfinite(x)
    assert np.array_equal(og.float_to_half_bits_array(x[fin]), bits[fin])


def test_narrow_midpoints_and_neighbours():
    # every midpoint between consecutive positive finite halves (ties), and
    # the fp32 values just below and above each midpoint
    pos = np.arange(0, 0x7C00, dtype=np.uint32).astype(np.uint16)  # +0 .. 65504
    lo = pos[:-1].view(np.float16).astype(np.float64)
    hi = pos[1:].view(np.float16).astype(np.float64)
    mid = ((lo + hi) / 2).astype(np.float32)
    assert np.all(mid.astype(np.float64) == (lo + hi) / 2)  # midpoints exact in fp32
    below = np.nextafter(mid, np.float32(0))
    above = np.nextafter(mid, np.float32(np.inf))
    for arr in (mid, below, above, -mid, -below, -above):
        _check_narrow(arr)


def test_narrow_overflow_and_specials():
    x = np.array([65504.0, 65519.0, np.nextafter(np.float32(65520), np.float32(0)), 65520.0,
                  65536.0, 1e6, 3.0e38, np.inf, -65504.0, -65520.0, -np.inf, 0.0, -0.0,
                  2.0 ** -24, 2.0 ** -25, np.nextafter(np.float32(2.0 ** -25), np.float32(1)),
                  3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, 1e-30, np.nan],
                 dtype=np.float32)
    _check_narrow(x)
    bits = og.float_to_half_bits_array(x)
    assert bits[3] == 0x7C00 and bits[2] == 0x7BFF and bits[5] == 0x7C00
    assert bits[12] == 0x8000 and bits[11] == 0x0000
    assert bits[14] == 0x0000  # 2^-25 is half the smallest subnormal: ties to even (zero)
    assert bits[15] == 0x0001 and bits[16] == 0x0001


def test_narrow_random_bit_patterns():
    rng = np.random.default_rng(12345)
    x = rng.integers(0, 2 ** 32, size=2_000_000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    _check_narrow(x)
    # and a dense sample of the fp16 normal range
    y = rng.uniform(-70000, 70000, size=1_000_000).astype(np.float32)
    _check_narrow(y)
    z = (rng.uniform(-1, 1, size=1_000_000) * 2.0 ** -13).astype(np.float32)
    _check_narrow(z)


# --------------------------------------------------------------------------
# GEMM
# --------------------------------------------------------------------------
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (17, 33, 64), (64, 64, 64),
                                   (5, 8, 300), (2, 3, 1000), (40, 24, 513)])
def test_brute_force_fp64_bound(M, N, K):
    rng = np.random.default_rng(M * 1000003 + N * 1009 + K)
    A = _rand_f16(rng, (M, K), -2, 2)
    B = _rand_f16(rng, (K, N), -2, 2)
    c16, c32 = og.gemm_rows(A, B, want_c32=True)
    A64, B64 = A.astype(np.float64), B.astype(np.float64)
    c64 = A64 @ B64
    absprod = np.abs(A64) @ np.abs(B64)
    gamma = K * U / (1 - K * U)
    err = np.abs(c32.astype(np.float64) - c64)
    assert np.all(err <= gamma * absprod + 1e-300)
    # the single narrowing is numpy's round-to-nearest-even of the fp32 sum
    assert np.array_equal(c16.view(np.uint16), c32.astype(np.float16).view(np.uint16))


def test_brute_force_catches_transpose():
    # square case where A^T B differs from A B: the bound test would fail
    rng = np.random.default_rng(7)
    A = _rand_f16(rng, (16, 16))
    B = _rand_f16(rng, (16, 16))
    c16 = og.gemm_rows(A, B).astype(np.float64)
    assert np.max(np.abs(c16 - A.astype(np.float64) @ B.astype(np.float64))) < 2e-3
    assert np.max(np.abs(c16 - A.astype(np.float64).T @ B.astype(np.float64))) > 1e-2


def test_identity_left_and_right():
    rng = np.random.default_rng(3)
    K = 96
    B = _rand_f16(rng, (K, 40), -100, 100)
    I = np.eye(K, dtype=np.float16)
    assert np.array_equal(og.gemm_rows(I, B).view(np.uint16), B.view(np.uint16))
    A = _rand_f16(rng, (33, K), -100, 100)
    assert np.array_equal(og.gemm_rows(A, I).view(np.uint16), A.view(np.uint16))


def test_zero_matrices_give_positive_zero():
    rng = np.random.default_rng(4)
    A = np.zeros((9, 31), np.float16)
    B = _rand_f16(rng, (31, 12))
    assert np.all(og.gemm_rows(A, B).view(np.uint16) == 0)
    assert np.all(og.gemm_rows(B.T.copy(), np.zeros((31, 5), np.float16)).view(np.uint16) == 0)


def test_small_integers_exact():
    rng = np.random.default_rng(5)
    M, N, K = 37, 29, 128  # |c| <= 16 * 128 = 2048: every partial sum exact
    A = rng.integers(-4, 5, size=(M, K))
    B = rng.integers(-4, 5, size=(K, N))
    c = og.gemm_rows(A.astype(np.float16), B.astype(np.float16))
    assert np.array_equal(c.astype(np.int64), A @ B)


def test_ascending_k_fp32_order():
    # terms 2048, 2^-13, 2^-13: in fp32, 2048 + 2^-13 is a tie that rounds to
    # 2048 (even), twice. Exact sum 2048 + 2^-12; reversed order also gives
    # 2048 + 2^-12 (representable). Only ascending-k fp32 gives exactly 2048.
    A = np.array([[64.0, 2.0 ** -7, 2.0 ** -7]], np.float16)
    B = np.array([[32.0], [2.0 ** -6], [2.0 ** -6]], np.float16)
    c16, c32 = og.gemm_rows(A, B, want_c32=True)
    assert c32[0, 0] == np.float32(2048.0)
    assert np.float64(2048.0) + 2.0 ** -12 != c32[0, 0]
    # reversing k changes the fp32 result
    c16r, c32r = og.gemm_rows(A[:, ::-1].copy(), B[::-1].copy(), want_c32=True)
    assert c32r[0, 0] == np.float32(2048.0 + 2.0 ** -12)


def test_single_narrowing():
    # 1024 + 4 * 0.25: an fp16 running sum stays at 1024 (each +0.25 is below
    # half an fp16 ulp at 1024); the fp32 sum is 1025, narrowed once to 1025.
    A = np.array([[1024.0, 0.25, 0.25, 0.25, 0.25]], np.float16)
    B = np.ones((5, 1), np.float16)
    assert og.gemm_rows(A, B)[0, 0] == np.float16(1025.0)


def test_overflow_narrows_to_inf():
    A = np.array([[300.0], [-300.0]], np.float16)
    B = np.array([[300.0, 1.0]], np.float16)
    c = og.gemm_rows(A, B)
    assert c[0, 0] == np.inf and c[1, 0] == -np.inf
    assert c[0, 1] == np.float16(300.0)


def test_degenerate_shapes():
    rng = np.random.default_rng(6)
    c = og.gemm_rows(np.zeros((4, 0), np.float16), np.zeros((0, 3), np.float16))
    assert c.shape == (4, 3) and np.all(c.view(np.uint16) == 0)  # K = 0: empty sum
    assert og.gemm_rows(np.zeros((0, 5), np.float16), _rand_f16(rng, (5, 3))).shape == (0, 3)
    assert og.gemm_rows(_rand_f16(rng, (4, 5)), np.zeros((5, 0), np.float16)).shape == (4, 0)


def test_row_subset_and_threads_bitwise():
    rng = np.random.default_rng(8)
    A = _rand_f16(rng, (70, 100))
    B = _rand_f16(rng, (100, 48))
    full = og.gemm_rows(A, B, nthreads=1)
    rows = np.array([69, 0, 13, 13, 42])
    sub = og.gemm_rows(A, B, rows=rows, nthreads=3)
    assert np.array_equal(sub.view(np.uint16), full[rows].view(np.uint16))
    assert np.array_equal(og.gemm_rows(A, B, nthreads=8).view(np.uint16), full.view(np.uint16))


def test_accepts_torch_tensors():
    g = torch.Generator().manual_seed(0)
    A = torch.rand((8, 16), dtype=torch.float16, generator=g) - 0.5
    B = torch.rand((16, 4), dtype=torch.float16, generator=g) - 0.5
    c = og.gemm_rows(A, B)
    assert np.array_equal(c.view(np.uint16), og.gemm_rows(A.numpy(), B.numpy()).view(np.uint16))


def test_rejects_bad_rows():
    with pytest.raises(RuntimeError):
        og.gemm_rows(np.zeros((2, 2), np.float16), np.zeros((2, 2), np.float16), rows=[2])
