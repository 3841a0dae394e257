"""Parity of the CUDA row softmax with the CPU oracle (oracle/softmax.py),
through the C ABI (softmax_rows_f32), on seeded host inputs.

Tolerance: the fused-softmax tutorial's check, torch.allclose's defaults,
|got - want| <= 1e-8 + 1e-5·|want|, with want the oracle's fp64 value. The
device path computes in fp32 (sum of at most 65,536 positive terms in a
tree of four partial sums per thread and shuffles; exp through ex2.approx;
a reciprocal multiply), whose relative error stays near 1e-6 for the rows
that matter; NaN positions must agree exactly.
"""
import numpy as np
import pytest
import torch

import dense_fp16_gemm_fp32_gb300 as g
from dense_fp16_gemm_fp32_gb300 import inputs
from oracle import softmax as osm

pytestmark = pytest.mark.gpu

RTOL, ATOL = 1e-5, 1e-8
CANARY = -12345.5


def compare(got: np.ndarray, want: np.ndarray):
    got = got.astype(np.float64)
    assert got.shape == want.shape
    assert np.array_equal(np.isnan(got), np.isnan(want)), "NaN positions differ"
    fin = ~np.isnan(want)
    d = np.abs(got[fin] - want[fin])
    tol = ATOL + RTOL * np.abs(want[fin])
    bad = np.nonzero(d > tol)[0]
    assert bad.size == 0, (f"{bad.size} beyond tolerance; worst |d|={d.max():.3g}", got[fin][bad[:8]],
                           want[fin][bad[:8]])
    return float(d.max()) if d.size else 0.0


def run(x_host: torch.Tensor, n: int, ldy: int | None = None, y_offset: int = 0, x_offset: int = 0):
    """Copies x_host ([M, ld]) to the device (at an element offset), runs the
    softmax of its first n columns into a canary-filled [M, ldy] array and
    returns (y view, y buffer, pad) on the device."""
    M, ld = x_host.shape
    xbuf = torch.empty(x_offset + M * ld, dtype=torch.float32, device="cuda")
    xbuf[x_offset:] = x_host.reshape(-1).cuda()
    x = xbuf[x_offset:].view(M, ld)[:, :n]
    ldy = ldy or ld
    pad = 64
    ybuf = torch.full((pad + y_offset + M * ldy + pad,), CANARY, dtype=torch.float32, device="cuda")
    y = ybuf[pad + y_offset:pad + y_offset + M * ldy].view(M, ldy)[:, :n]
    out = g.softmax(x, out=y)
    assert out.data_ptr() == y.data_ptr()
    torch.cuda.synchronize()
    return y, ybuf, pad + y_offset


def check_canaries(y: torch.Tensor, ybuf: torch.Tensor, start: int, M: int, ldy: int, n: int):
    before = ybuf[:start]
    after = ybuf[start + M * ldy:]
    assert torch.all(before == CANARY) and torch.all(after == CANARY)
    if ldy > n:
        padcols = ybuf[start:start + M * ldy].view(M, ldy)[:, n:]
        assert torch.all(padcols == CANARY), "padding columns of Y written"


def test_tutorial_workload_1823x781(gemm_lib):
    w = inputs.SOFTMAX_WORKLOADS_BY_NAME["softmax_1823x781"]
    x = inputs.softmax_inputs(w.M, w.n, w.ld, w.seed)
    y, ybuf, start = run(x, w.n)
    check_canaries(y, ybuf, start, w.M, w.ld, w.n)
    compare(y.cpu().numpy(), osm.softmax_rows(x.numpy(), w.n))
    # the tutorial's own comparison, for context: torch's softmax on the same device
    ref = torch.softmax(x[:, :w.n].cuda(), dim=1)
    assert torch.allclose(y, ref)


NS = [1, 2, 3, 4, 5, 31, 64, 127, 128, 129, 255, 256, 257, 500, 511, 512, 513, 781, 1000, 1023, 1024,
      1025, 1500, 2048, 2049, 4095, 4096, 5000, 8191, 8192, 8193, 12000, 16384, 16385, 30000, 32768, 32769,
      50000, 65535, 65536]


@pytest.mark.parametrize("n", NS)
@pytest.mark.parametrize("aligned", [True, False])
def test_row_lengths_every_path(gemm_lib, n, aligned):
    M = 37 if n <= 8192 else 11
    # aligned: pitch a multiple of 4 and 16-byte bases (float4 path);
    # unaligned: an odd pitch and bases one float off (scalar path)
    ld = (-(-n // 4) * 4 + 4) if aligned else n + 1
    off = 0 if aligned else 1
    x = inputs.softmax_inputs(M, n, ld, seed=n, pad_value=float("nan"))
    y, ybuf, start = run(x, n, ldy=ld, y_offset=off, x_offset=off)
    check_canaries(y, ybuf, start, M, ld, n)
    compare(y.cpu().numpy(), osm.softmax_rows(x.numpy(), n))


@pytest.mark.parametrize("n,tpr,cl", [(1, 32, 1), (1024, 32, 1), (1025, 64, 1), (2048, 64, 1), (2049, 128, 1),
                                       (8192, 256, 1), (8193, 256, 2), (16385, 256, 4), (32769, 256, 8),
                                       (65536, 256, 8)])
def test_launch_plan(gemm_lib, n, tpr, cl):
    p = g.softmax_plan(100000, n)
    assert (p["threads_per_row"], p["cluster_ctas"]) == (tpr, cl)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert p["grid_ctas"] % cl == 0
    if tpr == 32:
        assert p["grid_ctas"] % sms == 0     # every resident CTA: a multiple of the SM count
    # a small row count gets no more CTAs than it can use
    q = g.softmax_plan(3, n)
    assert q["grid_ctas"] == (1 if tpr == 32 else 3 * cl)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["softmax_262144x781", "softmax_8192x8000", "softmax_4096x32768"])
def test_large_workloads_sampled_rows(gemm_lib, name):
    w = inputs.SOFTMAX_WORKLOADS_BY_NAME[name]
    x = inputs.softmax_inputs(w.M, w.n, w.ld, w.seed)
    xd = x.cuda()[:, :w.n]
    y = g.softmax(xd)
    rows = inputs.sample_rows(w.M, w.seed)
    got = y.index_select(0, rows.cuda()).cpu().numpy()
    compare(got, osm.softmax_rows(x.numpy(), w.n, rows=rows.numpy()))
    # properties at every row: each row sums to one, no NaN
    s = y.double().sum(dim=1)
    assert torch.all((s - 1).abs() < 1e-4)
    assert not torch.isnan(y).any()


def test_in_place(gemm_lib):
    x = inputs.softmax_inputs(300, 781, 784, seed=21)
    xd = x.cuda()
    v = xd[:, :781]
    out = g.softmax(v, out=v)
    assert out.data_ptr() == v.data_ptr()
    compare(v.cpu().numpy(), osm.softmax_rows(x.numpy(), 781))
    assert torch.all(xd[:, 781:] == 0)
    x = inputs.softmax_inputs(20, 20000, 20000, seed=22)
    xd = x.cuda()
    g.softmax(xd, out=xd)
    compare(xd.cpu().numpy(), osm.softmax_rows(x.numpy(), 20000))


@pytest.mark.parametrize("n", [4, 781, 5000, 20000])
def test_special_values_and_extremes(gemm_lib, n):
    inf, nan = float("inf"), float("nan")
    x = inputs.softmax_inputs(8, n, n, seed=31)
    x[0, n // 2] = -inf                          # one -inf: 0 there, the rest finite
    x[1, n - 1] = nan                            # NaN anywhere: the whole row NaN
    x[2, 0] = inf                                # +inf: the whole row NaN
    x[3, :] = -inf                               # all -inf: NaN
    x[4, :] += 1.0e4                             # a large common offset
    x[5, :] = -3.0e38                            # values near the fp32 limits:
    x[5, n // 3] = 3.0e38                        # one-hot, no overflow in x - m
    x[6, :] = 7.0                                # constant: uniform
    x[7, :] *= 60.0                              # wide spread: many exp(x - m) underflow
    y, _, _ = run(x, n)
    got = y.cpu().numpy()
    compare(got, osm.softmax_rows(x.numpy(), n))
    assert got[0, n // 2] == 0.0
    assert got[5, n // 3] == 1.0


def test_degenerate_and_errors(gemm_lib):
    lib = g.load()
    s = torch.cuda.current_stream().cuda_stream
    x = torch.zeros((16, 64), dtype=torch.float32, device="cuda")
    y = torch.zeros((16, 64), dtype=torch.float32, device="cuda")
    n0 = g.softmax_launch_count()
    assert lib.softmax_rows_f32(x.data_ptr(), 64, y.data_ptr(), 64, 0, 64, s) == g.GEMM_OK
    assert lib.softmax_rows_f32(x.data_ptr(), 64, y.data_ptr(), 64, 16, 0, s) == g.GEMM_OK
    assert g.softmax_launch_count() == n0                      # nothing launched
    assert lib.softmax_rows_f32(x.data_ptr() + 2, 64, y.data_ptr(), 64, 16, 64, s) == g.GEMM_ERR_UNSUPPORTED
    assert lib.softmax_rows_f32(x.data_ptr(), 64, x.data_ptr() + 4, 64, 16, 60, s) == g.GEMM_ERR_INVALID_ARG
    assert lib.softmax_rows_f32(x.data_ptr(), 64, x.data_ptr(), 32, 16, 32, s) == g.GEMM_ERR_INVALID_ARG
    with pytest.raises(g.GemmError):
        g.softmax(torch.zeros((2, 70000), dtype=torch.float32, device="cuda"))
    with pytest.raises(TypeError):
        g.softmax(x.half())
    g.softmax(x, out=y)
    assert g.softmax_launch_count() == n0 + 1
    torch.testing.assert_close(y, torch.full_like(y, 1 / 64), rtol=0, atol=0)


def test_deterministic_and_on_current_stream(gemm_lib):
    x = inputs.softmax_inputs(1000, 20000, 20000, seed=41).cuda()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        y1 = g.softmax(x)
        y2 = g.softmax(x)
    side.synchronize()
    assert torch.equal(y1, y2)
