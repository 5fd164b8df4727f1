"""The seeded input generators: determinism, shapes, dtypes and moments."""
import math

import torch

from sm_rmsnorm_matmul_gb300 import inputs


def test_deterministic():
    a = inputs.random_problem(7, 64, 24, seed=3)
    b = inputs.random_problem(7, 64, 24, seed=3)
    c = inputs.random_problem(7, 64, 24, seed=4)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert not torch.equal(a[0], c[0])


def test_shapes_and_dtypes():
    X, g, W = inputs.random_problem(5, 72, 40, seed=0)
    assert X.shape == (5, 72) and g.shape == (72,) and W.shape == (72, 40)
    for t in (X, g, W):
        assert t.dtype == torch.bfloat16 and t.is_contiguous() and t.device.type == "cpu"


def test_moments():
    X, g, W = inputs.generate(64, 4096, 256, seed=9, w_std=1.0 / 64)
    assert abs(X.float().mean().item()) < 0.01
    assert abs(X.float().std().item() - 1.0) < 0.01
    assert 0.5 <= g.float().min().item() and g.float().max().item() <= 1.5
    assert abs(g.float().mean().item() - 1.0) < 0.02
    assert abs(W.float().std().item() - 1.0 / 64) < 2e-4


def test_outlier_entries():
    X, _, _ = inputs.generate(16, 4096, 8, seed=1, w_std=1.0 / 64, x_kind="outlier_entries")
    frac = (X.float().abs() > 6.0).float().mean().item()
    # ~1% of entries are x20; |20 z| > 6 unless |z| < 0.3 (prob ~0.24)
    assert 0.005 < frac < 0.012


def test_row_scaled():
    X, _, _ = inputs.generate(512, 1024, 8, seed=3, w_std=1.0 / 64, x_kind="row_scaled")
    rms = X.float().pow(2).mean(dim=1).sqrt()
    assert rms.min().item() > 0.08 and rms.max().item() < 12.0
    logs = rms.log()
    assert abs(logs.mean().item()) < 0.3  # log-uniform on [ln 0.1, ln 10] has mean 0
    assert abs(logs.std().item() - (2 * math.log(10)) / math.sqrt(12)) < 0.15


def test_workload_table():
    names = inputs.WORKLOAD_ORDER
    assert len(names) == 5
    w = inputs.WORKLOADS["decode_qkv_16x4096x6144"]
    assert (w.M, w.K, w.N, w.eps, w.seed) == (16, 4096, 6144, 1e-6, 1)
    assert w.bytes_xwy == 50_659_328
    big = inputs.WORKLOADS["large_prefill_16384x8192x8192"]
    assert big.flops == 2 * 16384 * 8192 * 8192


def test_sample_rows():
    rows = inputs.sample_rows(16384)
    assert len(rows) == 256 and rows[0] == 0 and rows[-1] == 16383
    assert len({r % 64 for r in rows}) == 64
    small = inputs.sample_rows(100)
    assert small[0] == 0 and small[-1] == 99 and all(0 <= r < 100 for r in small)
