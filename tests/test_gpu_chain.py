"""Dependent GEMMs issued back to back on one stream, with no host
synchronisation between them: each output feeds the next call (read after
write) and a later call overwrites an earlier call's input (write after
read). The GEMM kernels are launched with programmatic stream serialisation,
so a call may start while the previous one still runs; their results must be
bit-identical to the same chain run with a synchronisation after every call.
The shapes make consecutive calls run different kernels (one-CTA tiles of
three widths, CTA-pair, split-K)."""
import pytest
import torch

import dense_fp16_gemm_fp32_gb300 as g
from dense_fp16_gemm_fp32_gb300 import inputs

pytestmark = pytest.mark.gpu

# (K_in, N_out, tile configuration) of each link; M is the chain's row count
LINKS = [
    (512, 2048, g.TILE_AUTO),                  # 1024 x 2048 x 512: one-CTA tiles (few k steps)
    (2048, 1024, g.TILE_256x256x64_PAIR),      # the CTA-pair kernel
    (1024, 128, g.TILE_128x128x64_SPLITK),     # few tiles: split-K across a cluster
    (128, 512, g.TILE_128x256x64),
    (512, 256, g.TILE_AUTO),                   # 1024 x 256 x 512: 32 tiles of 128 x 64
]
M = 1024


def _weights():
    ws = []
    for i, (k, n, _) in enumerate(LINKS):
        _, b = inputs.gemm_inputs(1, n, k, seed=900 + i)
        ws.append((b / 4).cuda())  # keep the chain's values well inside fp16
    return ws


def _chain(x, ws, sync):
    outs = []
    h = x
    for w, (_, _, cfg) in zip(ws, LINKS):
        h = g.gemm(h, w, tile_cfg=cfg)
        if sync:
            torch.cuda.synchronize()
        outs.append(h)
    return outs


def test_dependent_chain_matches_serialised(gemm_lib):
    A, _ = inputs.gemm_inputs(M, 1, LINKS[0][0], seed=901)
    x = A.cuda()
    ws = _weights()
    want = _chain(x, ws, sync=True)
    for _ in range(3):
        got = _chain(x, ws, sync=False)
        torch.cuda.synchronize()
        assert g.query_status() == g.GEMM_OK
        for i, (a, b) in enumerate(zip(got, want)):
            assert torch.equal(a, b), f"link {i} differs from the serialised chain"


def test_write_after_read_on_the_stream(gemm_lib):
    # call 1 reads x; call 2, queued right behind it, overwrites x
    A, B = inputs.gemm_inputs(M, 2048, 512, seed=902)
    P, Q = inputs.gemm_inputs(M, 512, 256, seed=903)
    x, w, p, q = A.cuda(), B.cuda(), P.cuda(), Q.cuda()
    for _ in range(3):
        x.copy_(A.cuda())
        torch.cuda.synchronize()
        h = g.gemm(x, w, tile_cfg=g.TILE_256x256x64_PAIR)
        g.gemm(p, q, out=x)  # x: M x 512, the first call's A operand
        torch.cuda.synchronize()
        assert g.query_status() == g.GEMM_OK
        assert torch.equal(h, g.gemm(A.cuda(), w, tile_cfg=g.TILE_256x256x64_PAIR))
        assert torch.equal(x, g.gemm(p, q))
