"""The seeded input recipe: shapes, dtype, range, determinism, row sampling."""
import torch

from dense_fp16_gemm_fp32_gb300 import inputs


def test_recipe_shape_dtype_range():
    A, B = inputs.gemm_inputs(64, 48, 32, seed=0)
    assert A.shape == (64, 32) and B.shape == (32, 48)
    assert A.dtype == B.dtype == torch.float16
    for t in (A, B):
        assert t.device.type == "cpu"
        assert float(t.min()) >= -0.5 and float(t.max()) < 0.5


def test_recipe_deterministic_and_seed_dependent():
    A1, B1 = inputs.gemm_inputs(32, 16, 24, seed=3)
    A2, B2 = inputs.gemm_inputs(32, 16, 24, seed=3)
    A3, _ = inputs.gemm_inputs(32, 16, 24, seed=4)
    assert torch.equal(A1, A2) and torch.equal(B1, B2)
    assert not torch.equal(A1, A3)


def test_sample_rows():
    r = inputs.sample_rows(8192, seed=5)
    assert r.numel() == 256 and torch.all(r[1:] > r[:-1])
    assert int(r.min()) >= 0 and int(r.max()) < 8192
    assert torch.equal(r, inputs.sample_rows(8192, seed=5))
    assert torch.equal(inputs.sample_rows(100, seed=1), torch.arange(100))


def test_workload_table():
    names = [w.name for w in inputs.WORKLOADS]
    assert len(names) == len(set(names))
    w = inputs.WORKLOADS_BY_NAME["square8192"]
    assert (w.M, w.N, w.K, w.seed) == (8192, 8192, 8192, 5)
    we = inputs.WORKLOADS_BY_NAME["worked_example_1024x768x128"]
    assert (we.M, we.N, we.K, we.tile_cfg, we.group_size_m) == (1024, 768, 128, 2, 2)
