"""gemm_f16_f32acc_noalloc: the GEMM for callers that cannot allocate device
memory when they call it (code under CUDA-graph capture, runtime plugins whose
enqueue must not allocate, hosts with their own allocator). It keeps its only
scratch, the watchdog status word, in a static device array instead of the
cudaMalloc'd word of the default entry point.

The test calls it through the C ABI twice in a row, on different shapes, and
compares each output with the default entry point's output on the same
inputs, within the tolerance of the parity tests. This file is collected
last so that a failure here stops a `-x` run only after every other test.
"""
import numpy as np
import pytest
import torch

import dense_fp16_gemm_fp32_gb300 as g
from dense_fp16_gemm_fp32_gb300 import inputs

from _gpu_util import compare

pytestmark = pytest.mark.gpu


def _noalloc(lib, a, b, c, status, group_size_m=8):
    M, K = a.shape
    N = b.shape[1]
    return lib.gemm_f16_f32acc_noalloc(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, group_size_m,
                                       status.data_ptr(), torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_default_entry_point_two_calls(gemm_lib):
    lib = g.load()
    status = torch.full((1,), 0x7FFFFFFF, dtype=torch.int32, device="cuda")
    for (M, N, K, seed) in ((1000, 1032, 520, 51), (4095, 3000, 1000, 52)):
        A, B = inputs.gemm_inputs(M, N, K, seed)
        a, b = A.cuda(), B.cuda()
        want = g.gemm(a, b)  # the default entry point
        got = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        assert _noalloc(lib, a, b, got, status) == g.GEMM_OK
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        compare(got.cpu().numpy(), want.cpu().numpy(), K)
        status.fill_(0x7FFFFFFF)


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
