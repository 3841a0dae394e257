"""The library's launches inside CUDA graphs (stream capture).

The C entry points enqueue kernels on the caller's stream and allocate
nothing per call, so after one eager call (which sets up the per-device
state: status word, shared-memory attributes) they can be captured. Graph
replays must give the same bits as eager calls, for the TMA kernels, the
split-K cluster kernel, the workspace route and the softmax.
"""
import pytest
import torch

import dense_fp16_gemm_fp32_gb300 as g
from dense_fp16_gemm_fp32_gb300 import inputs

from _gpu_util import check_against_oracle

pytestmark = pytest.mark.gpu


def capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()                          # eager call on the capture stream: per-device set-up
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        fn()
    return graph


@pytest.mark.parametrize("M,N,K,cfg", [
    (4096, 2048, 1024, g.TILE_AUTO),                   # the pair kernel (64-deep stages)
    (300, 520, 264, g.TILE_128x128x64),
    (512, 512, 512, g.TILE_128x128x64_SPLITK),         # cluster split-K
    (1024, 768, 128, g.TILE_AUTO),                     # 128 x 64 x 64 tiles
    (1000, 37, 1000, g.TILE_AUTO),                     # N not a multiple of 8: the workspace route
    (4095, 3000, 1000, g.TILE_256x256x64_PAIR_STREAMK),  # stream-K: the capture stream's workspace
])
def test_gemm_graph_replay_matches_eager(gemm_lib, M, N, K, cfg):
    A, B = inputs.gemm_inputs(M, N, K, seed=M + N + K)
    a, b = A.cuda(), B.cuda()
    eager = g.gemm(a, b, tile_cfg=cfg)
    out = torch.empty_like(eager)
    graph = capture(lambda: g.gemm(a, b, out=out, tile_cfg=cfg))
    out.zero_()
    n0 = g.launch_count()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert g.launch_count() == n0          # replays go through no host code of the library
    assert g.query_status() == g.GEMM_OK
    assert torch.equal(out, eager)
    check_against_oracle(A, B, out)


def test_softmax_graph_replay_matches_eager(gemm_lib):
    x = inputs.softmax_inputs(1823, 781, 784, seed=0).cuda()[:, :781]
    eager = g.softmax(x)              # rows padded to 784: the float4 kernel
    out = torch.empty((1823, 784), dtype=torch.float32, device="cuda")[:, :781]   # the same layout
    graph = capture(lambda: g.softmax(x, out=out))
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)


def test_graph_sees_new_operand_values(gemm_lib):
    # a graph replays the captured pointers: new values written into the same
    # buffers give the new product
    M = N = K = 1024
    A1, B1 = inputs.gemm_inputs(M, N, K, seed=1)
    A2, B2 = inputs.gemm_inputs(M, N, K, seed=2)
    a, b = A1.cuda(), B1.cuda()
    out = torch.empty((M, N), dtype=torch.float16, device="cuda")
    graph = capture(lambda: g.gemm(a, b, out=out))
    a.copy_(A2.cuda())
    b.copy_(B2.cuda())
    graph.replay()
    torch.cuda.synchronize()
    check_against_oracle(A2, B2, out)
