"""rmsnorm_matmul_noalloc() through the C ABI.

Some callers cannot let a library allocate device memory during a call:
inference runtimes and plugin hosts that own all device memory through their
own pool and forbid allocation inside their enqueue step, processes whose
device-memory budget is fixed at start-up, and latency-critical paths where
cudaMalloc (which may synchronise the device) is not acceptable.  For them
this entry point runs rmsnorm_matmul()'s launch plan with its K-split partial
sums in one fixed 20 MiB array inside the library, shared by all calls.

Every case makes two calls in a row and checks each against the fp64 oracle at
the tolerance of the other GPU tests (the second call starts from whatever the
first left in the shared array), and against rmsnorm_matmul() bit for bit
(the same plan, so the same additions in the same order).  The plan query
shows which cases really put partial sums in the array.

This file is named so that pytest collects it last.
"""
import ctypes

import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2
SCRATCH_LIMIT = 7                    # RMM_ERR_SCRATCH_LIMIT
AREA_BYTES = (20 << 20) - (64 << 10)  # the array's room for partial sums


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sm_rmsnorm_matmul_gb300 as rmm
    from sm_rmsnorm_matmul_gb300 import build
    build.build()
    l = rmm.lib()
    prev = l.rmm_force_path(0)
    yield l
    l.rmm_force_path(prev)


def _call(lib, fn, X, g, W, Y, eps):
    M, K = X.shape
    N = W.shape[1]
    stream = torch.cuda.current_stream().cuda_stream
    return getattr(lib, fn)(X.data_ptr(), g.data_ptr(), W.data_ptr(), Y.data_ptr(),
                            M, K, N, eps, stream)


def _plan(lib, M, K, N):
    info = (ctypes.c_int * 8)()
    assert lib.rmm_describe_plan(M, K, N, 1, info) == 0
    return dict(zip(("path", "splits", "cluster", "grid", "stages", "MP", "tiles", "kbps"), info))


def _uses_scratch(plan):
    # a K split whose partials go through memory, not a cluster's shared memory
    return plan["splits"] > 1 and plan["cluster"] == 0


# (name or (M, K, N), forced path, whether the plan puts partials in the array)
CASES = [
    ("tiny_8x1024x1024", 0, False),                # row-tile kernel, K split inside a cluster
    ("decode_qkv_16x4096x6144", 0, False),
    ((16, 8192, 1024), 0, True),                   # small-M path, K cut into pieces
    ("decode_gatedmlp_64x4096x28672", 0, False),   # row-tile kernel, whole tiles
    ("prefill_qkv_4096x4096x6144", 0, False),     # paired CTAs, whole units
    ((1280, 1024, 4096), 0, True),                 # 8 tail tiles
    ((1200, 1000, 4104), 0, True),                 # 18 tail tiles, partial row, column and K blocks
    ("tiny_8x1024x1024", 1, False),                # row-tile kernel, K split inside a cluster
    ("decode_qkv_16x4096x6144", 2, True),          # small-M path, K cut into pieces
    ((16, 16384, 128), 2, True),                   # long K: many pieces per unit
    ((12, 8192, 264), 2, True),                    # ragged last unit
]


def _problem(spec):
    from sm_rmsnorm_matmul_gb300 import inputs
    if isinstance(spec, str):
        w = inputs.WORKLOADS[spec]
        X, g, W = inputs.generate_workload(w)
        return spec, X, g, W, w.eps
    M, K, N = spec
    X, g, W = inputs.random_problem(M, K, N, seed=M + 3 * K + N, x_kind="row_scaled")
    return f"{M}x{K}x{N}", X, g, W, 1e-5


@pytest.mark.parametrize("spec,path,scratch", CASES)
def test_noalloc_matches_oracle_on_two_calls(lib, spec, path, scratch):
    from sm_rmsnorm_matmul_gb300 import inputs
    name, X, g, W, eps = _problem(spec)
    M, K = X.shape
    N = W.shape[1]
    rows = inputs.sample_rows(M, 256) if M > 1024 else list(range(M))
    ref = oracle.rmsnorm_matmul(X[rows], g, W, eps)
    Xd, gd, Wd = X.cuda(), g.cuda(), W.cuda()
    prev = lib.rmm_force_path(path)
    try:
        plan = _plan(lib, M, K, N)
        if scratch is not None:
            assert _uses_scratch(plan) == scratch, f"{name}: plan {plan}"
        fused = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        assert _call(lib, "rmsnorm_matmul", Xd, gd, Wd, fused, eps) == 0
        for call in range(2):
            Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
            assert _call(lib, "rmsnorm_matmul_noalloc", Xd, gd, Wd, Y, eps) == 0
            torch.cuda.synchronize()
            assert lib.rmm_device_status(torch.cuda.current_stream().cuda_stream) == 0
            Yc = Y.cpu()
            bad, max_abs, _ = oracle.tolerance_violations(Yc[rows], ref, ATOL, RTOL)
            assert bad == 0, f"{name} path {path} call {call}: {bad} outside tolerance (max {max_abs:.3e})"
            assert torch.equal(Yc, fused.cpu()), f"{name} path {path} call {call}: differs from rmsnorm_matmul"
    finally:
        lib.rmm_force_path(prev)


def test_noalloc_back_to_back_different_inputs(lib):
    # Two different problems queued in a row share the array; neither may see
    # the other's partial sums.  (Prefill kernel with tail pieces in the array.)
    from sm_rmsnorm_matmul_gb300 import inputs
    M, K, N = 1280, 1024, 4096
    assert _uses_scratch(_plan(lib, M, K, N))
    runs = []
    for seed in (11, 12):
        X, g, W = inputs.random_problem(M, K, N, seed=seed, x_kind="row_scaled")
        Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        assert _call(lib, "rmsnorm_matmul_noalloc", X.cuda(), g.cuda(), W.cuda(), Y, 1e-6) == 0
        runs.append((X, g, W, Y))
    torch.cuda.synchronize()
    assert lib.rmm_device_status(torch.cuda.current_stream().cuda_stream) == 0
    for X, g, W, Y in runs:
        bad, max_abs, _ = oracle.tolerance_violations(Y.cpu(), oracle.rmsnorm_matmul(X, g, W, 1e-6),
                                                      ATOL, RTOL)
        assert bad == 0, max_abs


def test_noalloc_rejects_plans_beyond_its_scratch(lib):
    # A small-M launch whose K pieces (16 x 64 fp32 and 16 row sums per piece)
    # exceed the array: refused before any launch, the output left untouched.
    prev = lib.rmm_force_path(2)
    try:
        for M, K, N in [(16, 2048, 65536), (16, 4096, 65536), (16, 2048, 131072)]:
            p = _plan(lib, M, K, N)
            need = p["splits"] * p["tiles"] * (16 * 64 + 16) * 4
            if _uses_scratch(p) and need > AREA_BYTES:
                break
        else:
            pytest.skip("no candidate shape needs more than the array on this device")
        X = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
        g = torch.ones(K, dtype=torch.bfloat16, device="cuda")
        W = torch.zeros(K, N, dtype=torch.bfloat16, device="cuda")
        Y = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
        rc = _call(lib, "rmsnorm_matmul_noalloc", X, g, W, Y, 1e-6)
    finally:
        lib.rmm_force_path(prev)
    torch.cuda.synchronize()
    assert rc == SCRATCH_LIMIT
    assert lib.rmm_status_string(SCRATCH_LIMIT) == b"RMM_ERR_SCRATCH_LIMIT"
    assert bool((Y == 3.0).all())
