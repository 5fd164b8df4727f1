"""The bounded in-kernel waits, run out on purpose without any fault.

A test hook makes the row-tile kernel's K-split reduction skip the stores of
its partials, so that every owning CTA's wait for them runs out (after a
shortened limit); for the attention kernel it makes the loader leave out its
first key/value stage.  The kernel must then record RMM_ERR_DEVICE_TIMEOUT, skip
its remaining work, free its tensor memory and exit; rmm_device_status()
reports it; and the next call on the same context runs normally.
"""
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rmm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sm_rmsnorm_matmul_gb300 as m
    from sm_rmsnorm_matmul_gb300 import build
    build.build()
    m.lib()
    return m


def test_timeout_is_reported_and_the_context_recovers(rmm):
    # the row-tile kernel's cluster K split (the small-M path has no waits)
    from sm_rmsnorm_matmul_gb300 import inputs
    M, K, N = 16, 4096, 6144
    prev = rmm.force_path(rmm.PATH_ROWS)
    l = rmm.lib()
    try:
        plan = rmm.describe_plan(M, K, N)
        assert plan["splits"] > 1 and plan["cluster"] == 1   # the K-split reduction runs
        X, g, W = (t.cuda() for t in inputs.random_problem(M, K, N, seed=31))
        assert rmm.device_status() == 0
        assert l.rmm_test_hooks(1, 50_000_000) == 0          # skip the sends; 50 ms per wait
        try:
            rmm.rmsnorm_matmul(X, g, W, 1e-6)
            assert rmm.device_status() == 5                  # RMM_ERR_DEVICE_TIMEOUT
        finally:
            assert l.rmm_test_hooks(0, 0) == 0               # normal operation, 2 s limit
        Y = rmm.rmsnorm_matmul(X, g, W, 1e-6)
        torch.cuda.synchronize()
        assert rmm.device_status() == 0
    finally:
        rmm.force_path(prev)
    bad, max_abs, _ = oracle.tolerance_violations(Y.cpu(), oracle.rmsnorm_matmul(X.cpu(), g.cpu(), W.cpu(), 1e-6))
    assert bad == 0, max_abs


def test_paired_timeout_is_reported_and_the_context_recovers(rmm):
    # the paired prefill kernel (one pair MMA per 256-row unit, two CTAs of a
    # cluster): the second CTA leaves out its first "stage ready" signal, the
    # first CTA's MMA issuer waits for it until the limit, and every role of
    # both CTAs leaves its loop through its own bounded waits
    from sm_rmsnorm_matmul_gb300 import inputs
    M, K, N = 2048, 512, 3840
    plan = rmm.describe_plan(M, K, N)
    assert plan["splits"] == 1 and plan["grid"] % 2 == 0
    X, g, W = inputs.random_problem(M, K, N, seed=37, x_kind="row_scaled")
    Xd, gd, Wd = X.cuda(), g.cuda(), W.cuda()
    l = rmm.lib()
    assert rmm.device_status() == 0
    assert l.rmm_test_hooks(1, 50_000_000) == 0
    try:
        rmm.rmsnorm_matmul(Xd, gd, Wd, 1e-6)
        assert rmm.device_status() == 5                  # RMM_ERR_DEVICE_TIMEOUT
    finally:
        assert l.rmm_test_hooks(0, 0) == 0
    Y = rmm.rmsnorm_matmul(Xd, gd, Wd, 1e-6)
    torch.cuda.synchronize()
    assert rmm.device_status() == 0
    rows = list(range(0, M, 16))
    bad, max_abs, _ = oracle.tolerance_violations(Y.cpu()[rows], oracle.rmsnorm_matmul(X[rows], g, W, 1e-6))
    assert bad == 0, max_abs


def test_hook_rejects_negative_limit(rmm):
    assert rmm.lib().rmm_test_hooks(0, -1) == 1


@pytest.mark.parametrize("D", [128, 64])
def test_attention_timeout_is_reported_and_the_context_recovers(rmm, D):
    # the same hook makes the attention loader leave out its first key/value
    # stage: both MMA issuers' waits for it run out, every role leaves its
    # loop, and the CTA frees its tensor memory and exits (both head
    # dimensions: each has its own kernel instantiation)
    from sm_rmsnorm_matmul_gb300 import inputs
    B, S, Hq, Hkv = 1, 512, 4, 2
    qkv, gq, gk = inputs.attention_inputs(B, S, Hq, Hkv, D, seed=7)
    Qd, Kd, Vd = inputs.split_qkv(qkv.cuda(), B, S, Hq, Hkv, D)
    l = rmm.lib()
    assert rmm.device_status() == 0
    assert l.rmm_test_hooks(1, 50_000_000) == 0
    try:
        rmm.qknorm_attention(Qd, Kd, Vd, gq.cuda(), gk.cuda(), 1e-6, causal=True)
        assert rmm.device_status() == 5                  # RMM_ERR_DEVICE_TIMEOUT
    finally:
        assert l.rmm_test_hooks(0, 0) == 0
    O = rmm.qknorm_attention(Qd, Kd, Vd, gq.cuda(), gk.cuda(), 1e-6, causal=True)
    torch.cuda.synchronize()
    assert rmm.device_status() == 0
    Q, K, V = inputs.split_qkv(qkv, B, S, Hq, Hkv, D)
    ref = oracle.qknorm_attention(Q, K, V, gq, gk, 1e-6, causal=True)
    bad, max_abs, _ = oracle.tolerance_violations(O.cpu(), ref, atol=3e-2, rtol=3e-2)
    assert bad == 0, max_abs
