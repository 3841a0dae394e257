"""The boundary's primary call, gemm_f16_f32acc(A, B, C, M, N, K,
group_size_m, stream), called directly through the C ABI with device buffers
from torch and the current stream, its output checked element by element
against the CPU oracle (the binding's gemm() goes through the strided entry
point; this covers the signature of the tutorial's matmul launch itself:
"03: Matrix multiplication", the launch inside check).
"""
import ctypes

import pytest
import torch

import dense_fp16_gemm_fp32_gb300 as g
from dense_fp16_gemm_fp32_gb300 import inputs

from _gpu_util import check_against_oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K,G,seed", [
    (512, 512, 512, 8, 0),        # the tutorial's check: M = N = K = 512, seed 0
    (1024, 768, 128, 2, 1),       # the notebook's worked example, GROUP_SIZE_M = 2
    (4095, 3000, 1000, 8, 6),     # ragged: no extent a whole number of tiles
])
def test_primary_entry_point_matches_oracle(gemm_lib, M, N, K, G, seed):
    lib = g.load()
    A, B = inputs.gemm_inputs(M, N, K, seed)
    a, b = A.cuda(), B.cuda()
    c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    n0 = g.launch_count()
    rc = lib.gemm_f16_f32acc(ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(b.data_ptr()),
                             ctypes.c_void_p(c.data_ptr()), M, N, K, G, ctypes.c_void_p(stream))
    assert rc == g.GEMM_OK
    assert g.launch_count() - n0 >= 1
    assert g.query_status() == g.GEMM_OK
    check_against_oracle(A, B, c)


def test_primary_entry_point_on_a_side_stream(gemm_lib):
    lib = g.load()
    M, N, K = 640, 520, 264
    A, B = inputs.gemm_inputs(M, N, K, 61)
    a, b = A.cuda(), B.cuda()
    c = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        assert lib.gemm_f16_f32acc(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, 8, s.cuda_stream) == g.GEMM_OK
        assert g.query_status() == g.GEMM_OK
    check_against_oracle(A, B, c)
