"""rmsnorm_matmul_noalloc() through the C ABI.

This entry point serves callers that cannot let a library allocate device
memory: code being captured into a CUDA graph (cudaMalloc is refused there),
runtimes and plugin hosts that own every byte of device memory, and processes
with a fixed budget.  Instead of a workspace allocated on first use, its
split-K partial sums live in one fixed array inside the library, shared by
all calls.  Its output must agree with rmsnorm_matmul() within the tolerance
the other GPU tests use, on two calls in a row (the second call starts from
whatever the first one left in the shared array).

This file is named so that pytest collects it last.
"""
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2


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


@pytest.mark.parametrize("name", ["decode_qkv_16x4096x6144", "decode_gatedmlp_64x4096x28672",
                                  "tiny_8x1024x1024", "prefill_qkv_4096x4096x6144"])
@pytest.mark.parametrize("path", [0, 2])
def test_noalloc_matches_fused_on_two_calls(lib, name, path):
    # path 2 forces the small-M path, whose K split keeps its partial sums in
    # the fixed scratch array; path 0 is the default (row-tile) dispatch.
    from sm_rmsnorm_matmul_gb300 import inputs
    w = inputs.WORKLOADS[name]
    if path == 2 and w.M > 128:
        pytest.skip("small-M path holds at most 128 rows")
    X, g, W = (t.cuda() for t in inputs.generate_workload(w))
    prev = lib.rmm_force_path(path)
    try:
        ref = torch.empty((w.M, w.N), dtype=torch.bfloat16, device="cuda")
        assert _call(lib, "rmsnorm_matmul", X, g, W, ref, w.eps) == 0
        torch.cuda.synchronize()
        ref_np = oracle.to_f64(ref.cpu())
        for _ in range(2):
            Y = torch.full((w.M, w.N), float("nan"), dtype=torch.bfloat16, device="cuda")
            assert _call(lib, "rmsnorm_matmul_noalloc", X, g, W, Y, w.eps) == 0
            torch.cuda.synchronize()
            assert lib.rmm_device_status(torch.cuda.current_stream().cuda_stream) == 0
            bad, max_abs, _ = oracle.tolerance_violations(Y.cpu(), ref_np, ATOL, RTOL)
            assert bad == 0, f"{name}: {bad} elements differ from rmsnorm_matmul (max {max_abs:.3e})"
    finally:
        lib.rmm_force_path(prev)


def test_noalloc_back_to_back_different_inputs(lib):
    # Two different problems in a row share the scratch array; neither may see
    # the other's partial sums.  (Small-M path forced, so the array is used.)
    from sm_rmsnorm_matmul_gb300 import inputs
    outs = []
    prev = lib.rmm_force_path(2)
    for seed in (11, 12):
        X, g, W = (t.cuda() for t in inputs.random_problem(16, 4096, 6144, seed=seed))
        Y = torch.empty((16, 6144), dtype=torch.bfloat16, device="cuda")
        assert _call(lib, "rmsnorm_matmul_noalloc", X, g, W, Y, 1e-6) == 0
        outs.append((X, g, W, Y))
    torch.cuda.synchronize()
    lib.rmm_force_path(prev)
    for X, g, W, Y in outs:
        ref = torch.empty_like(Y)
        assert _call(lib, "rmsnorm_matmul", X, g, W, ref, 1e-6) == 0
        torch.cuda.synchronize()
        bad, max_abs, _ = oracle.tolerance_violations(Y.cpu(), oracle.to_f64(ref.cpu()), ATOL, RTOL)
        assert bad == 0, max_abs


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    # M = 128 on the small-M path with N = 12288, K = 8192 splits K three ways
    # on 152 SMs: 3 x 128 x 12288 x 4 bytes = 18.9 MB of partials > 15 MiB.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    X = torch.zeros(128, 8192, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(8192, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(8192, 12288, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(128, 12288, dtype=torch.bfloat16, device="cuda")
    prev = lib.rmm_force_path(2)
    try:
        rc = _call(lib, "rmsnorm_matmul_noalloc", X, g, W, Y, 1e-6)
    finally:
        lib.rmm_force_path(prev)
    torch.cuda.synchronize()
    if sms == 152:
        assert rc == 7  # RMM_ERR_SCRATCH_LIMIT
    else:
        assert rc in (0, 7)
    assert lib.rmm_status_string(7) == b"RMM_ERR_SCRATCH_LIMIT"
