"""Failure detection and memory safety on the GPU, without any fault:

* watchdog: a test hook makes the TMA producer issue nothing, so the MMA
  warp's bounded wait runs out; the kernel records GEMM_ERR_TIMEOUT, frees its
  tensor memory and returns; the context stays usable (a following GEMM is
  correct);
* canaries: C is placed inside a larger buffer filled with a NaN pattern; no
  store may land outside C, whatever the raggedness of the shape;
* argument errors on real device pointers come back as status codes.
"""
import pytest
import torch

import dense_fp16_gemm_fp32_gb300 as g
from dense_fp16_gemm_fp32_gb300 import inputs

from _gpu_util import check_against_oracle

pytestmark = pytest.mark.gpu

CANARY = 0x7E01  # a quiet-NaN fp16 bit pattern the kernel never produces from finite inputs


@pytest.mark.parametrize("cfg", [g.TILE_128x256x64, g.TILE_128x64x32, g.TILE_256x256x64_PAIR, g.TILE_256x256x128_PAIR,
                                 g.TILE_128x128x64, g.TILE_128x128x64_SPLITK, g.TILE_128x64x64, g.TILE_64x64x64, "generic"])
def test_watchdog_timeout_reports_and_recovers(gemm_lib, cfg):
    A, B = inputs.gemm_inputs(256, 512, 128, seed=41)
    a, b = A.cuda(), B.cuda()
    if cfg == "generic":  # A one element off a 16-byte boundary: the generic-load kernel
        buf = torch.empty(A.numel() + 1, dtype=torch.float16, device="cuda")
        buf[1:] = a.reshape(-1)
        a, cfg = buf[1:].view(A.shape), g.TILE_AUTO
    assert g.query_status() == g.GEMM_OK
    try:
        g.set_watchdog_ns(50_000_000)  # 50 ms
        g.set_fault_injection(1)
        g.gemm(a, b, tile_cfg=cfg, repack=False)
        assert g.query_status() == g.GEMM_ERR_TIMEOUT
        assert g.query_status() == g.GEMM_OK  # the query clears the word
    finally:
        g.set_fault_injection(0)
        g.set_watchdog_ns(0)
    C = g.gemm(a, b, tile_cfg=cfg, repack=False)
    assert g.query_status() == g.GEMM_OK
    check_against_oracle(A, B, C)


@pytest.mark.parametrize("cfg", [g.TILE_128x256x64, g.TILE_128x64x32, g.TILE_256x256x64_PAIR, g.TILE_256x256x128_PAIR,
                                 g.TILE_128x128x64, g.TILE_128x128x64_SPLITK, g.TILE_128x64x64, g.TILE_64x64x64])
@pytest.mark.parametrize("M,N,K", [(129, 264, 72), (4095, 3000, 1000), (1, 8, 8), (300, 8, 1000), (300, 999, 1001)])
def test_no_store_outside_c(gemm_lib, M, N, K, cfg):
    A, B = inputs.gemm_inputs(M, N, K, seed=M + N + K)
    pad = 4096  # elements before and after C (multiple of 8: C stays 16-byte aligned)
    buf = torch.full((pad + M * N + pad,), CANARY, dtype=torch.int16, device="cuda")
    C = buf[pad:pad + M * N].view(torch.float16).view(M, N)
    g.gemm(A.cuda(), B.cuda(), out=C, tile_cfg=cfg)
    assert g.query_status() == g.GEMM_OK
    assert torch.all(buf[:pad] == CANARY) and torch.all(buf[pad + M * N:] == CANARY)
    check_against_oracle(A, B, C)


def test_device_pointer_errors(gemm_lib):
    lib = g.load()
    a = torch.zeros((64, 64), dtype=torch.float16, device="cuda")
    b = torch.zeros((64, 64), dtype=torch.float16, device="cuda")
    c = torch.zeros((64 * 64 + 8,), dtype=torch.float16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    # C at a 1-byte offset: not an fp16 address
    rc = lib.gemm_f16_f32acc(a.data_ptr(), b.data_ptr(), c.data_ptr() + 1, 64, 64, 64, 8, s)
    assert rc == g.GEMM_ERR_UNSUPPORTED
    # C aliasing A
    rc = lib.gemm_f16_f32acc(a.data_ptr(), b.data_ptr(), a.data_ptr(), 64, 64, 64, 8, s)
    assert rc == g.GEMM_ERR_INVALID_ARG
    # C at a 2-byte offset: the generic-load kernel writes it; the elements
    # before and after C keep their values
    A, B = inputs.gemm_inputs(64, 64, 64, seed=43)
    a, b = A.cuda(), B.cuda()
    c.fill_(float("nan"))
    rc = lib.gemm_f16_f32acc(a.data_ptr(), b.data_ptr(), c.data_ptr() + 2, 64, 64, 64, 8, s)
    assert rc == g.GEMM_OK
    assert g.query_status() == g.GEMM_OK
    assert torch.isnan(c[0]) and torch.isnan(c[64 * 64 + 1:]).all()
    check_against_oracle(A, B, c[1:1 + 64 * 64].view(64, 64))
    # K = 60 (rows of 120 bytes): the generic-load kernel as well
    A, B = inputs.gemm_inputs(64, 64, 60, seed=44)
    check_against_oracle(A, B, g.gemm(A.cuda(), B.cuda()))
    assert g.query_status() == g.GEMM_OK


def test_launch_counter_counts_gemm_launches(gemm_lib):
    a = torch.zeros((128, 64), dtype=torch.float16, device="cuda")
    b = torch.zeros((64, 256), dtype=torch.float16, device="cuda")
    n0 = g.launch_count()
    for _ in range(3):
        g.gemm(a, b)
    assert g.launch_count() - n0 == 3
