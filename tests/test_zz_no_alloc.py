"""gemm_f16_f32acc_noalloc: the GEMM for callers that cannot allocate device
memory when they call it (runtime plugins whose enqueue step must not
allocate, hosts that reserve all device memory up front for their own
allocator, loops that cannot take a cudaMalloc's implicit synchronisation).
It keeps its only scratch, the watchdog status word, in a static device array
instead of the cudaMalloc'd word of the default entry point.

The tests call it through the C ABI: twice in a row on different shapes, each
output checked element by element against the CPU oracle and against the
default entry point's output, within the tolerance of the parity tests; and
with the watchdog test hook on, where the status word it hands back must show
the expired wait, after which the next call is complete and correct. This file
is collected last so that a failure here stops a `-x` run only after every
other test.
"""
import pytest
import torch

import dense_fp16_gemm_fp32_gb300 as g
from dense_fp16_gemm_fp32_gb300 import inputs

from _gpu_util import check_against_oracle, compare

pytestmark = pytest.mark.gpu

UNSET = 0x7FFFFFFF  # a value the status word never takes


def _noalloc(lib, a, b, c, status, group_size_m=8):
    M, K = a.shape
    N = b.shape[1]
    return lib.gemm_f16_f32acc_noalloc(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, group_size_m,
                                       status.data_ptr(), torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_oracle_two_calls(gemm_lib):
    lib = g.load()
    status = torch.full((1,), UNSET, dtype=torch.int32, device="cuda")
    for (M, N, K, seed) in ((1000, 1032, 520, 51), (4095, 3000, 1000, 52)):
        A, B = inputs.gemm_inputs(M, N, K, seed)
        a, b = A.cuda(), B.cuda()
        got = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        assert _noalloc(lib, a, b, got, status) == g.GEMM_OK
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        check_against_oracle(A, B, got)
        want = g.gemm(a, b)  # the default entry point on the same inputs
        compare(got.cpu().numpy(), want.cpu().numpy(), K)
        status.fill_(UNSET)


def test_noalloc_watchdog_reports_through_d_status(gemm_lib):
    lib = g.load()
    A, B = inputs.gemm_inputs(256, 512, 128, seed=53)
    a, b = A.cuda(), B.cuda()
    c = torch.zeros((256, 512), dtype=torch.float16, device="cuda")
    status = torch.full((1,), UNSET, dtype=torch.int32, device="cuda")
    try:
        g.set_watchdog_ns(50_000_000)  # 50 ms
        g.set_fault_injection(1)       # the TMA producer issues nothing: the MMA warp's wait runs out
        assert _noalloc(lib, a, b, c, status) == g.GEMM_OK
        torch.cuda.synchronize()
    finally:
        g.set_fault_injection(0)
        g.set_watchdog_ns(0)
    word = int(status.item())
    assert word & 1, f"status word {word:#x}: bit 0 (a bounded wait expired) not set"
    assert 1 <= (word >> 8) & 0xFF <= 4, f"status word {word:#x}: no role in bits 8..15"
    # the default entry point's status word is untouched by this call
    assert g.query_status() == g.GEMM_OK
    # the next call starts from a cleared word and completes
    status.fill_(UNSET)
    got = torch.full((256, 512), float("nan"), dtype=torch.float16, device="cuda")
    assert _noalloc(lib, a, b, got, status) == g.GEMM_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    check_against_oracle(A, B, got)


def test_noalloc_validates_like_default(gemm_lib):
    lib = g.load()
    a = torch.zeros((64, 64), dtype=torch.float16, device="cuda")
    b = torch.zeros((64, 64), dtype=torch.float16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert lib.gemm_f16_f32acc_noalloc(a.data_ptr(), b.data_ptr(), a.data_ptr(), 64, 64, 64, 8, None, s) \
        == g.GEMM_ERR_INVALID_ARG
    assert lib.gemm_f16_f32acc_noalloc(a.data_ptr(), b.data_ptr(), 0, 64, 64, 64, 8, None, s) \
        == g.GEMM_ERR_INVALID_ARG
    c = torch.empty((64 * 64 + 8,), dtype=torch.float16, device="cuda")
    assert lib.gemm_f16_f32acc_noalloc(a.data_ptr(), b.data_ptr(), c.data_ptr() + 2, 64, 64, 64, 8, None, s) \
        == g.GEMM_ERR_UNSUPPORTED
