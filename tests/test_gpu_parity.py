"""GPU parity: the CUDA library, called through its C ABI, against the fp64
oracle on the same seeded inputs.

Acceptance for every checked element (bf16 in/out, fp32 accumulation):
    |y - y_ref| <= 1e-2 + 1e-2 * |y_ref|,   NaN/Inf fail.
"""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2
SMALL_M = 16   # rows the small-M path (path 2) takes


@pytest.fixture(scope="module")
def rmm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sm_rmsnorm_matmul_gb300 as m
    from sm_rmsnorm_matmul_gb300 import build
    build.build()
    m.lib()
    return m


@pytest.fixture
def forced(rmm):
    prev = []

    def set_path(p):
        prev.append(rmm.force_path(p))

    yield set_path
    if prev:
        rmm.force_path(prev[0])


def run_fused(rmm, X, g, W, eps):
    Y = rmm.rmsnorm_matmul(X.cuda(), g.cuda(), W.cuda(), eps)
    torch.cuda.synchronize()
    assert rmm.device_status() == 0
    return Y.cpu()


def assert_close(Y, ref, what):
    bad, max_abs, max_rel = oracle.tolerance_violations(Y, ref, ATOL, RTOL)
    assert bad == 0, f"{what}: {bad} of {ref.size} elements out of tolerance (max abs err {max_abs:.3e})"


# --------------------------------------------------------------- workloads
SMALL_WORKLOADS = ["tiny_8x1024x1024", "decode_qkv_16x4096x6144",
                   "decode_gatedmlp_64x4096x28672"]
LARGE_WORKLOADS = ["prefill_qkv_4096x4096x6144", "large_prefill_16384x8192x8192"]


@pytest.mark.parametrize("name", SMALL_WORKLOADS)
@pytest.mark.parametrize("path", [0, 1, 2])
def test_workload_all_rows(rmm, forced, name, path):
    from sm_rmsnorm_matmul_gb300 import inputs
    w = inputs.WORKLOADS[name]
    if path == 2 and w.M > SMALL_M:
        pytest.skip("the small-M path holds at most 16 rows")
    X, g, W = inputs.generate_workload(w)
    forced(path)
    Y = run_fused(rmm, X, g, W, w.eps)
    ref = oracle.rmsnorm_matmul(X, g, W, w.eps)
    assert_close(Y, ref, f"{name} path {path}")


@pytest.mark.parametrize("name", LARGE_WORKLOADS)
def test_workload_sampled_rows(rmm, name):
    """Full-size launch (the configuration the benchmark times); the oracle
    checks a 256-row sample of every output column."""
    from sm_rmsnorm_matmul_gb300 import inputs
    w = inputs.WORKLOADS[name]
    X, g, W = inputs.generate_workload(w)
    Y = run_fused(rmm, X, g, W, w.eps)
    rows = inputs.sample_rows(w.M, 256)
    ref = oracle.rmsnorm_matmul(X[rows], g, W, w.eps)
    assert_close(Y[rows], ref, name)
    assert torch.isfinite(Y.float()).all()


# -------------------------------------------------------- ragged and edges
RAGGED = [
    (1, 64, 8), (7, 72, 136), (16, 1024, 1000), (33, 520, 264), (64, 4096, 1032),
    (65, 256, 256), (129, 1032, 520), (255, 328, 392), (300, 2048, 2056),
    # few column tiles and long K: many K pieces (small-M path) or splits
    (16, 16384, 128), (48, 8192, 264),
    # small-M path: one partial k-step, a k-step half past K, one row, ragged units
    (3, 8, 8), (12, 4104, 72), (1, 2056, 6152), (9, 520, 4096),
]


@pytest.mark.parametrize("M,K,N", RAGGED)
@pytest.mark.parametrize("path", [1, 2])
def test_ragged(rmm, forced, M, K, N, path):
    from sm_rmsnorm_matmul_gb300 import inputs
    if path == 2 and M > SMALL_M:
        pytest.skip("the small-M path holds at most 16 rows")
    X, g, W = inputs.random_problem(M, K, N, seed=M * 7 + K + N, x_kind="row_scaled")
    forced(path)
    Y = run_fused(rmm, X, g, W, 1e-5)
    ref = oracle.rmsnorm_matmul(X, g, W, 1e-5)
    assert_close(Y, ref, f"{M}x{K}x{N} path {path}")
    # the K pieces are added in a fixed order: a second call gives the same bits
    assert torch.equal(Y, run_fused(rmm, X, g, W, 1e-5))


# Several row tiles whose last wave of CTAs would be at most half full: those
# last tiles are cut along K, one piece per CTA, and the pieces are combined
# through the workspace (here 160 tiles on 152 SMs leave 8; 170 leave 18, with
# a partial row tile, a partial column tile and a partial K block).
TAIL = [(1280, 1024, 4096), (1200, 1000, 4104)]


@pytest.mark.parametrize("M,K,N", TAIL)
def test_tail_tiles_cut_along_k(rmm, M, K, N):
    from sm_rmsnorm_matmul_gb300 import inputs
    X, g, W = inputs.random_problem(M, K, N, seed=M + K + N, x_kind="row_scaled")
    Y = run_fused(rmm, X, g, W, 1e-6)
    assert_close(Y, oracle.rmsnorm_matmul(X, g, W, 1e-6), f"{M}x{K}x{N}")
    # the pieces are added in a fixed order: a second call gives the same bits
    assert torch.equal(Y, run_fused(rmm, X, g, W, 1e-6))


def test_tail_tiles_with_another_stream_holding_sms(rmm):
    # The pieces of a tail tile wait for one another; the launch is
    # cooperative, so all its CTAs are resident together even while kernels
    # on another stream hold SMs: the call completes with a clean status and
    # the right result.
    from sm_rmsnorm_matmul_gb300 import inputs
    M, K, N = 1280, 1024, 4096
    assert rmm.describe_plan(M, K, N)["splits"] > 1   # tail tiles cut along K
    X, g, W = inputs.random_problem(M, K, N, seed=77, x_kind="row_scaled")
    Xd, gd, Wd = X.cuda(), g.cuda(), W.cuda()
    a = torch.randn(8192, 8192, device="cuda", dtype=torch.bfloat16)
    other = torch.cuda.Stream()
    main = torch.cuda.current_stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(other):
        for _ in range(8):      # a few milliseconds of full-device GEMMs
            a = (a @ a).clamp_(-1, 1)
    Y = rmm.rmsnorm_matmul(Xd, gd, Wd, 1e-6, stream=main)
    other.synchronize()
    main.synchronize()
    assert rmm.device_status() == 0
    assert_close(Y.cpu(), oracle.rmsnorm_matmul(X, g, W, 1e-6), f"{M}x{K}x{N} beside another stream")


# The paired kernel (two CTAs, one pair MMA per 256-row unit) on ragged units:
# the last unit's second row block past M, and a last column tile whose
# second half (rank 1's W columns) lies wholly past N.
@pytest.mark.parametrize("M,K,N", [(2432, 520, 3840), (3840, 1024, 1152)])
def test_paired_ragged_units(rmm, M, K, N):
    from sm_rmsnorm_matmul_gb300 import inputs
    p = rmm.describe_plan(M, K, N)
    assert p["splits"] == 1 and p["cluster"] == 0 and p["grid"] % 2 == 0
    X, g, W = inputs.random_problem(M, K, N, seed=M + K + N, x_kind="row_scaled")
    Y = run_fused(rmm, X, g, W, 1e-5)
    assert_close(Y, oracle.rmsnorm_matmul(X, g, W, 1e-5), f"{M}x{K}x{N} paired")
    assert torch.equal(Y, run_fused(rmm, X, g, W, 1e-5))


@pytest.mark.parametrize("M,K,N", [(2048, 512, 3840),    # paired CTAs, whole tiles
                                   (1280, 1024, 4096)])   # tail tiles cut along K (cooperative)
def test_prefill_calls_replayed_from_a_cuda_graph(rmm, M, K, N):
    # the benchmark's way of calling: captured once, replayed; the same bits
    # as an eager call, and the oracle's result
    from sm_rmsnorm_matmul_gb300 import inputs
    X, g, W = inputs.random_problem(M, K, N, seed=M + N, x_kind="row_scaled")
    Xd, gd, Wd = X.cuda(), g.cuda(), W.cuda()
    eager = run_fused(rmm, X, g, W, 1e-6)
    s = torch.cuda.Stream()
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(s):
        rmm.rmsnorm_matmul(Xd, gd, Wd, 1e-6, out=Y, stream=s)   # workspace, if any, before capture
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        rmm.rmsnorm_matmul(Xd, gd, Wd, 1e-6, out=Y, stream=s)
    for _ in range(2):
        Y.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert rmm.device_status() == 0
        assert torch.equal(Y.cpu(), eager)
    assert_close(eager, oracle.rmsnorm_matmul(X, g, W, 1e-6), f"{M}x{K}x{N}")


# One row tile of 65..128 rows: the K-split receive blocks are too large to
# sit beside the pipeline, so they reuse the pipeline buffers once every
# split has finished its last MMA (handshake between the CTAs of a cluster).
WIDE_DECODE = [(128, 4096, 6144), (100, 2048, 2056), (80, 1024, 512)]


@pytest.mark.parametrize("M,K,N", WIDE_DECODE)
def test_wide_decode_split_over_pipeline_buffers(rmm, M, K, N):
    from sm_rmsnorm_matmul_gb300 import inputs
    X, g, W = inputs.random_problem(M, K, N, seed=M * 5 + N, x_kind="outlier_entries")
    Y = run_fused(rmm, X, g, W, 1e-5)
    assert_close(Y, oracle.rmsnorm_matmul(X, g, W, 1e-5), f"{M}x{K}x{N}")
    assert torch.equal(Y, run_fused(rmm, X, g, W, 1e-5))


# ------------------------------------------------------- gated MLP on top
# rmsnorm_matmul_swiglu: W [K, 2F] = [gate | up], Y [M, F] = silu(Z_gate) * Z_up.
GATED = [
    (64, 4096, 28672),   # decode gate|up, the benchmark shape
    (16, 1032, 2000),    # F = 1000: a partial output tile, K split over a cluster
    (1, 64, 16),         # one row, one k-block, F = 8
    (100, 2048, 2064),   # 100 rows: receive blocks over the pipeline buffers
    (300, 520, 528),     # several row tiles (prefill kernel), ragged everywhere
    (1280, 1024, 8192),  # 320 tiles: the last 16 cut along K (prefill kernel's tail)
]


def assert_gated_close(Y, X, g, W, eps, what):
    """Y = silu(Z_gate) * Z_up against the oracle, with the tolerance of the
    ungated output Z (|dz| <= 1e-2 + 1e-2 |z|) carried through silu(a) * b to
    first order, plus the second-order term and Y's own bf16 rounding:
      |dy| <= |silu'(zg)| e_g |zu| + |silu(zg)| e_u + e_g e_u + 2^-8 |y|.
    The gate multiplies Z's errors (chiefly the bf16 rounding of X*g before
    the tensor cores) by |z_up|, so the ungated bound does not hold for Y."""
    F = W.shape[1] // 2
    ref = oracle.rmsnorm_matmul_swiglu(X, g, W, eps)
    Z = oracle.rmsnorm_matmul(X, g, W, eps)
    zg, zu = Z[:, :F], Z[:, F:]
    eg, eu = ATOL + RTOL * np.abs(zg), ATOL + RTOL * np.abs(zu)
    sig = 1.0 / (1.0 + np.exp(-zg))
    dsilu = sig * (1.0 + zg * (1.0 - sig))
    tol = np.abs(dsilu) * eg * np.abs(zu) + np.abs(zg * sig) * eu + eg * eu + 2.0 ** -8 * np.abs(ref)
    y = oracle.to_f64(Y)
    bad = ~(np.abs(y - ref) <= tol)   # NaN fails
    assert not bad.any(), f"{what}: {int(bad.sum())} of {ref.size} outside the propagated tolerance"


@pytest.mark.parametrize("M,K,N", GATED)
def test_gated(rmm, M, K, N):
    from sm_rmsnorm_matmul_gb300 import inputs
    X, g, W = inputs.random_problem(M, K, N, seed=M + 3 * K + N, x_kind="row_scaled")
    Y = rmm.rmsnorm_matmul_swiglu(X.cuda(), g.cuda(), W.cuda(), 1e-5)
    torch.cuda.synchronize()
    assert rmm.device_status() == 0
    assert Y.shape == (M, N // 2)
    assert_gated_close(Y.cpu(), X, g, W, 1e-5, f"gated {M}x{K}x{N}")
    assert torch.equal(Y, rmm.rmsnorm_matmul_swiglu(X.cuda(), g.cuda(), W.cuda(), 1e-5))


def test_gated_prefill_sampled_rows(rmm):
    from sm_rmsnorm_matmul_gb300 import inputs
    M, K, N = 4096, 4096, 12288
    X, g, W = inputs.random_problem(M, K, N, seed=99, x_kind="row_scaled")
    Y = rmm.rmsnorm_matmul_swiglu(X.cuda(), g.cuda(), W.cuda(), 1e-6)
    torch.cuda.synchronize()
    assert rmm.device_status() == 0
    rows = inputs.sample_rows(M, 256)
    assert_gated_close(Y.cpu()[rows], X[rows], g, W, 1e-6, "gated prefill")


# ------------------------------------------- weights stored [N, K] (K-major)
# rmsnorm_matmul_ex(weight_nk=True): W as a linear layer stores it, Y = RMSNorm(X) @ W^T.
WEIGHT_NK = [
    (16, 4096, 6144, False),   # decode QKV: K split over a cluster
    (64, 4096, 28672, False),  # decode gate|up: one CTA per column tile
    (7, 72, 136, False),       # ragged rows, K and N
    (1280, 1024, 4096, False), # prefill kernel with the K-split tail
    (300, 520, 264, False),    # several row tiles, ragged
    (16, 1032, 2000, True),    # gated, K split
    (300, 520, 528, True),     # gated, prefill kernel
]


@pytest.mark.parametrize("M,K,N,gated", WEIGHT_NK)
def test_weight_nk(rmm, M, K, N, gated):
    from sm_rmsnorm_matmul_gb300 import inputs
    X, g, W = inputs.random_problem(M, K, N, seed=2 * M + K + 5 * N, x_kind="outlier_entries")
    Wt = W.t().contiguous()   # [N, K]
    Y = rmm.rmsnorm_matmul_ex(X.cuda(), g.cuda(), Wt.cuda(), 1e-6, weight_nk=True, gated=gated)
    torch.cuda.synchronize()
    assert rmm.device_status() == 0
    if gated:
        assert_gated_close(Y.cpu(), X, g, W, 1e-6, f"[N,K] gated {M}x{K}x{N}")
    else:
        assert_close(Y.cpu(), oracle.rmsnorm_matmul(X, g, W, 1e-6), f"[N,K] {M}x{K}x{N}")


# The paired prefill kernel with weights stored [N, K] (each CTA loads boxes
# of 128 weight rows; gated: the gate rows in one CTA, the up rows in the
# other): the same bits as the [K, N] layout, and the oracle at the plain
# bound on unit-RMS outputs (millions of outputs: reading S25).
@pytest.mark.parametrize("gated", [False, True])
def test_weight_nk_paired(rmm, gated):
    from sm_rmsnorm_matmul_gb300 import inputs
    M, K, N = 2048, 520, 3840
    X, g, W = inputs.random_problem(M, K, N, seed=11 + gated, x_kind="row_scaled")
    Xd, gd = X.cuda(), g.cuda()
    Y_nk = rmm.rmsnorm_matmul_ex(Xd, gd, W.t().contiguous().cuda(), 1e-6, weight_nk=True, gated=gated)
    Y_kn = rmm.rmsnorm_matmul_ex(Xd, gd, W.cuda(), 1e-6, weight_nk=False, gated=gated)
    torch.cuda.synchronize()
    assert rmm.device_status() == 0
    assert torch.equal(Y_nk, Y_kn)
    if gated:
        assert_gated_close(Y_nk.cpu(), X, g, W, 1e-6, f"[N,K] paired gated {M}x{K}x{N}")
    else:
        assert_close(Y_nk.cpu(), oracle.rmsnorm_matmul(X, g, W, 1e-6), f"[N,K] paired {M}x{K}x{N}")


# ------------------------------------------------------- low-rank adapter
# rmsnorm_matmul_lora: Y = RMSNorm(X) @ (W + A @ B), A [K,R], B [R,N].
LORA = [
    (16, 4096, 6144, 16),    # decode QKV shape: K split, the adapter stages in split 0
    (64, 4096, 28672, 64),   # one CTA per column tile
    (7, 72, 136, 8),         # ragged rows, K and N; a single k-block plus the adapter
    (1280, 1024, 4096, 32),  # prefill kernel: whole tiles and K pieces (piece 0 adds it)
    (300, 520, 264, 24),     # several row tiles, ragged
    (4096, 4096, 6144, 64),  # prefill QKV shape (the benchmark's adapter line): T's launch cut along K
    (20000, 1024, 512, 56),  # 157 row tiles for T's launch: whole tiles (TMA stores) and a K-cut tail
    (2432, 520, 3840, 40),   # paired main kernel: 19 row blocks (the last unit's second past M), ragged K
]


def bf16_round(a):
    """fp64 -> fp32 -> bf16 (nearest even) -> fp64."""
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.float32).to(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("M,K,N,R", LORA)
def test_lora(rmm, M, K, N, R):
    """Against the oracle at the plain bound, on inputs with unit-RMS outputs
    like every workload (W and the adapter each carry half of the weight
    variance).  Then, with an adapter as large as W (outputs of RMS ~1.4),
    against the oracle's definition with one change, the reading that every
    form shares: the products X*g rounded to bf16 before the tensor cores.
    What the device may add to that is fp32 accumulation and Y's one bf16
    rounding, |dy| <= 2^-8 |y| + 1e-4; an adapter intermediate T rounded to a
    single bf16 (relative 2^-9 per element) would add r * sum_j dT_j B[j,n],
    about 1e-3 per output, and fail it."""
    from sm_rmsnorm_matmul_gb300 import inputs
    X, g, W, A, B = inputs.lora_problem(M, K, N, R, seed=M + K + N + R)
    Xd, gd, Wd = X.cuda(), g.cuda(), W.cuda()
    Y = rmm.rmsnorm_matmul_lora(Xd, gd, Wd, A.cuda(), B.cuda(), 1e-5)
    torch.cuda.synchronize()
    assert rmm.device_status() == 0
    rows = inputs.sample_rows(M, 512) if M > 4096 else list(range(M))
    assert_close(Y.cpu()[rows], oracle.rmsnorm_matmul_lora(X[rows], g, W, A, B, 1e-5),
                 f"lora {M}x{K}x{N} R={R}")
    # an adapter as large as W
    A2, B2 = inputs.lora_adapter(K, N, R, seed=R + 1)
    Y2 = rmm.rmsnorm_matmul_lora(Xd, gd, Wd, A2.cuda(), B2.cuda(), 1e-5)
    torch.cuda.synchronize()
    assert rmm.device_status() == 0
    Xf, gf, Wf, Af, Bf = (oracle.to_f64(t) for t in (X[rows], g, W, A2, B2))
    r = 1.0 / np.sqrt((Xf * Xf).mean(axis=1) + 1e-5)
    xg = bf16_round(Xf * gf[None, :])
    emu = r[:, None] * (xg @ Wf + (xg @ Af) @ Bf)
    err = np.abs(oracle.to_f64(Y2.cpu()[rows]) - emu)
    bad = ~(err <= 2.0 ** -8 * np.abs(emu) + 1e-4)   # NaN fails
    assert not bad.any(), f"lora {M}x{K}x{N} R={R}: {int(bad.sum())} beyond the rounding of X*g (max {err.max():.3e})"
    # a zero adapter gives the plain result
    Y0 = rmm.rmsnorm_matmul_lora(Xd, gd, Wd, torch.zeros_like(A).cuda(), B.cuda(), 1e-5)
    torch.cuda.synchronize()
    assert rmm.device_status() == 0
    assert_close(Y0.cpu()[rows], oracle.rmsnorm_matmul(X[rows], g, W, 1e-5), f"lora zero adapter {M}x{K}x{N}")


def test_small_m_rejects_large_m_when_forced(rmm, forced):
    forced(2)
    X = torch.zeros(SMALL_M + 1, 64, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rmm.RmmError):
        rmm.rmsnorm_matmul(X, g, W)


def test_empty_output_is_noop(rmm):
    X = torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    Y = rmm.rmsnorm_matmul(X, g, W)
    assert Y.shape == (0, 64)


def test_zero_row_gives_zero(rmm):
    from sm_rmsnorm_matmul_gb300 import inputs
    X, g, W = inputs.random_problem(16, 256, 128, seed=3)
    X[5] = 0
    for path in (1, 2):
        prev = rmm.force_path(path)
        try:
            Y = run_fused(rmm, X, g, W, 1e-6)
        finally:
            rmm.force_path(prev)
        assert torch.all(Y[5] == 0)
        assert_close(Y, oracle.rmsnorm_matmul(X, g, W, 1e-6), f"zero row, path {path}")


def test_deterministic(rmm):
    from sm_rmsnorm_matmul_gb300 import inputs
    X, g, W = inputs.random_problem(16, 4096, 6144, seed=21)
    a = run_fused(rmm, X, g, W, 1e-6)
    b = run_fused(rmm, X, g, W, 1e-6)
    assert torch.equal(a, b)


def test_scale_invariance_on_gpu(rmm):
    # Scaling X by a power of two leaves the rounded products and the
    # statistic's ratio unchanged; with eps = 0 the outputs stay in tolerance
    # of each other and of the oracle.
    from sm_rmsnorm_matmul_gb300 import inputs
    X, g, W = inputs.random_problem(16, 2048, 1024, seed=8)
    for path in (1, 2):
        prev = rmm.force_path(path)
        try:
            a = run_fused(rmm, X, g, W, 0.0)
            b = run_fused(rmm, (X.float() * 4).to(torch.bfloat16), g, W, 0.0)
        finally:
            rmm.force_path(prev)
        assert_close(b, a.double().numpy(), f"scale invariance path {path}")


def test_identity_weight_is_rmsnorm(rmm):
    from sm_rmsnorm_matmul_gb300 import inputs
    X, g, _ = inputs.random_problem(48, 256, 8, seed=4, x_kind="row_scaled")
    W = torch.eye(256, dtype=torch.bfloat16)
    Y = run_fused(rmm, X, g, W, 1e-6)
    ref = oracle.rmsnorm(X, g, 1e-6)
    assert_close(Y, ref, "W = I")


# ------------------------------------------------------------ unfused pair
@pytest.mark.parametrize("M,K", [(1, 8), (16, 4096), (300, 1032), (4096, 4096)])
def test_unfused_rmsnorm(rmm, M, K):
    from sm_rmsnorm_matmul_gb300 import inputs
    X, g, _ = inputs.random_problem(M, K, 8, seed=M + K, x_kind="outlier_entries")
    Xn = rmm.rmsnorm(X.cuda(), g.cuda(), 1e-6)
    torch.cuda.synchronize()
    assert_close(Xn.cpu(), oracle.rmsnorm(X, g, 1e-6), f"rmsnorm {M}x{K}")


@pytest.mark.parametrize("M,K,N", [(16, 4096, 6144), (5, 1032, 1000), (100, 520, 264), (512, 1024, 2048)])
@pytest.mark.parametrize("path", [0, 1, 2])
def test_unfused_matmul(rmm, forced, M, K, N, path):
    from sm_rmsnorm_matmul_gb300 import inputs
    if path == 2 and M > SMALL_M:
        pytest.skip("the small-M path holds at most 16 rows")
    A, _, B = inputs.random_problem(M, K, N, seed=M * 3 + N)
    forced(path)
    C = rmm.matmul(A.cuda(), B.cuda())
    torch.cuda.synchronize()
    assert rmm.device_status() == 0
    assert_close(C.cpu(), oracle.matmul(A, B), f"matmul {M}x{K}x{N} path {path}")


def test_unfused_pair_matches_fused(rmm):
    from sm_rmsnorm_matmul_gb300 import inputs
    w = inputs.WORKLOADS["decode_qkv_16x4096x6144"]
    X, g, W = inputs.generate_workload(w)
    Xd, gd, Wd = X.cuda(), g.cuda(), W.cuda()
    Y2 = rmm.matmul(rmm.rmsnorm(Xd, gd, w.eps), Wd)
    torch.cuda.synchronize()
    assert_close(Y2.cpu(), oracle.rmsnorm_matmul(X, g, W, w.eps), "unfused pair")


def test_streams_are_honoured(rmm):
    from sm_rmsnorm_matmul_gb300 import inputs
    X, g, W = inputs.random_problem(16, 1024, 2048, seed=6)
    Xd, gd, Wd = X.cuda(), g.cuda(), W.cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        Y = rmm.rmsnorm_matmul(Xd, gd, Wd, 1e-6)
    s.synchronize()
    assert_close(Y.cpu(), oracle.rmsnorm_matmul(X, g, W, 1e-6), "side stream")


def test_device_status_clean(rmm):
    assert rmm.device_status() == 0


# ---------------------------------- paired, a last round of a few units
# 2048 x 520 x 2560: 8 row-block pairs x 10 column tiles = 80 paired units on
# 76 clusters of two: a second round of 4 units, in every paired form.
@pytest.mark.parametrize("form", ["plain", "gated", "weight_nk", "lora"])
def test_paired_small_last_round(rmm, form):
    from sm_rmsnorm_matmul_gb300 import inputs
    M, K, N = 2048, 520, 2560
    if form == "lora":
        X, g, W, A, B = inputs.lora_problem(M, K, N, 40, seed=7)
        Y = rmm.rmsnorm_matmul_lora(X.cuda(), g.cuda(), W.cuda(), A.cuda(), B.cuda(), 1e-5)
        torch.cuda.synchronize()
        assert rmm.device_status() == 0
        assert_close(Y.cpu(), oracle.rmsnorm_matmul_lora(X, g, W, A, B, 1e-5), "lora, small last round")
        return
    X, g, W = inputs.random_problem(M, K, N, seed=5, x_kind="row_scaled")
    Xd, gd = X.cuda(), g.cuda()
    if form == "gated":
        Y = rmm.rmsnorm_matmul_swiglu(Xd, gd, W.cuda(), 1e-5)
        torch.cuda.synchronize()
        assert rmm.device_status() == 0
        assert_gated_close(Y.cpu(), X, g, W, 1e-5, "gated, small last round")
        return
    Wd = W.t().contiguous().cuda() if form == "weight_nk" else W.cuda()
    Y = rmm.rmsnorm_matmul_ex(Xd, gd, Wd, 1e-5, weight_nk=form == "weight_nk")
    torch.cuda.synchronize()
    assert rmm.device_status() == 0
    assert_close(Y.cpu(), oracle.rmsnorm_matmul(X, g, W, 1e-5), f"{form}, small last round")
    # deterministic: the same bits again
    assert torch.equal(Y, rmm.rmsnorm_matmul_ex(Xd, gd, Wd, 1e-5, weight_nk=form == "weight_nk"))
