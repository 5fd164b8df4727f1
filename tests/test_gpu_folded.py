"""GPU parity of the folded-gain form: fold_gain() once, then
rmsnorm_matmul_folded(), against the fp64 oracle of RMSNorm + MatMul on the
same seeded inputs (the identity (X * g * r) @ W = r * (X @ (diag(g) W))).

Acceptance as for the fused path: |y - y_ref| <= 1e-2 + 1e-2 * |y_ref|."""
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2


@pytest.fixture(scope="module")
def rmm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sm_rmsnorm_matmul_gb300 as m
    from sm_rmsnorm_matmul_gb300 import build
    build.build()
    m.lib()
    return m


def folded(rmm, X, g, W, eps):
    Wg = rmm.fold_gain(g.cuda(), W.cuda())
    Y = rmm.rmsnorm_matmul_folded(X.cuda(), Wg, eps)
    torch.cuda.synchronize()
    assert rmm.device_status() == 0
    return Y.cpu()


def assert_close(Y, ref, what):
    bad, max_abs, _ = oracle.tolerance_violations(Y, ref, ATOL, RTOL)
    assert bad == 0, f"{what}: {bad} of {ref.size} elements out of tolerance (max abs err {max_abs:.3e})"


@pytest.mark.parametrize("K,N", [(8, 8), (520, 264), (4096, 6144)])
def test_fold_gain_is_one_rounding_of_the_product(rmm, K, N):
    """Wg = bf16(g[k] * W[k,n]): the bf16 product is exact in fp32, so torch's
    fp32 product rounded once to bf16 must match bit for bit."""
    from sm_rmsnorm_matmul_gb300 import inputs
    _, g, W = inputs.random_problem(4, K, N, seed=K + N)
    Wg = rmm.fold_gain(g.cuda(), W.cuda()).cpu()
    ref = (g.float()[:, None] * W.float()).to(torch.bfloat16)
    assert torch.equal(Wg.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("name", ["tiny_8x1024x1024", "decode_qkv_16x4096x6144",
                                  "decode_gatedmlp_64x4096x28672"])
def test_folded_workload_all_rows(rmm, name):
    from sm_rmsnorm_matmul_gb300 import inputs
    w = inputs.WORKLOADS[name]
    X, g, W = inputs.generate_workload(w)
    Y = folded(rmm, X, g, W, w.eps)
    assert_close(Y, oracle.rmsnorm_matmul(X, g, W, w.eps), name)


@pytest.mark.parametrize("name", ["prefill_qkv_4096x4096x6144", "large_prefill_16384x8192x8192"])
def test_folded_workload_sampled_rows(rmm, name):
    """Full size, in the launch configuration the benchmark times (the large
    shape's last tiles are cut along K); a 256-row sample against the oracle."""
    from sm_rmsnorm_matmul_gb300 import inputs
    w = inputs.WORKLOADS[name]
    X, g, W = inputs.generate_workload(w)
    Y = folded(rmm, X, g, W, w.eps)
    rows = inputs.sample_rows(w.M, 256)
    assert_close(Y[rows], oracle.rmsnorm_matmul(X[rows], g, W, w.eps), name)
    assert torch.isfinite(Y.float()).all()


RAGGED = [
    (1, 64, 8), (7, 72, 136), (16, 1024, 1000), (33, 520, 264), (64, 4096, 1032),
    (129, 1032, 520), (255, 328, 392), (256, 512, 256), (257, 136, 264), (300, 2048, 2056),
    (48, 8192, 264), (600, 4104, 776),
]


@pytest.mark.parametrize("M,K,N", RAGGED)
def test_folded_ragged(rmm, M, K, N):
    """Partial row and column tiles, a K past the last whole k-block, and
    shapes whose every tile is cut into K pieces (few tiles for the SMs)."""
    from sm_rmsnorm_matmul_gb300 import inputs
    X, g, W = inputs.random_problem(M, K, N, seed=M * 5 + K + N, x_kind="row_scaled")
    Y = folded(rmm, X, g, W, 1e-5)
    assert_close(Y, oracle.rmsnorm_matmul(X, g, W, 1e-5), f"{M}x{K}x{N}")


def test_folded_rows_of_zeros(rmm):
    """A row of zeros gives r = 1/sqrt(eps) times a zero row: zeros."""
    from sm_rmsnorm_matmul_gb300 import inputs
    X, g, W = inputs.random_problem(300, 512, 264, seed=11)
    X[5] = 0
    X[290] = 0
    Y = folded(rmm, X, g, W, 1e-6)
    assert torch.count_nonzero(Y[5]) == 0 and torch.count_nonzero(Y[290]) == 0
    assert_close(Y, oracle.rmsnorm_matmul(X, g, W, 1e-6), "zero rows")


def test_folded_beside_another_stream_holding_sms(rmm):
    """Tiles wait for their row block's published r, so the folded launch is
    cooperative: all its CTAs are resident together even while kernels on
    another stream hold SMs; the call completes with a clean status and the
    right result, and calls on two streams (each with its own workspace)
    both do."""
    from sm_rmsnorm_matmul_gb300 import inputs
    M, K, N = 2048, 1024, 4096
    X, g, W = inputs.random_problem(M, K, N, seed=31, x_kind="row_scaled")
    Xd, Wg = X.cuda(), rmm.fold_gain(g.cuda(), W.cuda())
    a = torch.randn(8192, 8192, device="cuda", dtype=torch.bfloat16)
    other = torch.cuda.Stream()
    second = torch.cuda.Stream()
    main = torch.cuda.current_stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(other):
        for _ in range(8):      # a few milliseconds of full-device GEMMs
            a = (a @ a).clamp_(-1, 1)
    Y = rmm.rmsnorm_matmul_folded(Xd, Wg, 1e-6, stream=main)
    Y2 = rmm.rmsnorm_matmul_folded(Xd, Wg, 1e-6, stream=second)
    other.synchronize()
    second.synchronize()
    main.synchronize()
    assert rmm.device_status() == 0
    ref = oracle.rmsnorm_matmul(X, g, W, 1e-6)
    assert_close(Y.cpu(), ref, "folded beside another stream")
    assert torch.equal(Y, Y2)
