"""The C ABI on the CPU: the library loads, exports every declared symbol, and
rejects bad arguments before making any CUDA call."""
import ctypes
import os
import re

import pytest

import sm_rmsnorm_matmul_gb300 as rmm
from sm_rmsnorm_matmul_gb300 import build as rbuild

HEADERS = [os.path.join(rbuild.INCLUDE, h) for h in ("rmsnorm_matmul.h", "qknorm_attention.h")]


@pytest.fixture(scope="module")
def lib():
    rbuild.build()
    return rmm.lib()


def declared_functions():
    src = ""
    for h in HEADERS:
        with open(h) as f:
            src += f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"^\s*(?:int|const char\*)\s+(\w+)\s*\(", src, flags=re.M))


def test_header_declares_binding_functions():
    assert declared_functions() == set(rmm.ABI_FUNCTIONS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for code, name in rmm.STATUS.items():
        assert rmm.status_string(code) == name
    assert rmm.status_string(99) == "RMM_UNKNOWN_STATUS"


def test_force_path_roundtrip(lib):
    assert rmm.force_path(rmm.PATH_ROWS) == rmm.PATH_AUTO
    assert rmm.dispatch_path(8, 1024, 1024) == rmm.PATH_ROWS   # forced
    assert rmm.force_path(rmm.PATH_SMALL_M) == rmm.PATH_ROWS
    assert rmm.dispatch_path(4096, 4096, 4096) == rmm.PATH_SMALL_M
    assert rmm.force_path(rmm.PATH_AUTO) == rmm.PATH_SMALL_M
    assert lib.rmm_force_path(7) == -1
    assert rmm.force_path(rmm.PATH_AUTO) == rmm.PATH_AUTO


def test_default_dispatch_crossover(lib):
    # Up to 16 rows: the small-M path where it streams W faster than the
    # row-tile kernel (long K over a narrow N), on the measured shapes; more
    # rows always the row-tile kernels.  Without a GPU the dispatch assumes a
    # 152-SM GB300.
    small = [(16, 8192, 1024), (16, 14336, 2048), (4, 2048, 512), (16, 4096, 1024), (8, 4096, 2048)]
    rows = [(16, 2048, 2048), (8, 1024, 1024), (1, 1024, 1024), (16, 4096, 6144), (16, 4096, 28672),
            (16, 4096, 2560), (64, 4096, 28672)]
    for M, K, N in small:
        assert rmm.dispatch_path(M, K, N) == rmm.PATH_SMALL_M, (M, K, N)
    for M, K, N in rows:
        assert rmm.dispatch_path(M, K, N) == rmm.PATH_ROWS, (M, K, N)
    for M in (17, 64, 65, 128, 4096):
        assert rmm.dispatch_path(M, 8192, 1024) == rmm.PATH_ROWS


A16 = 0x10000          # a 16-byte aligned fake address; never dereferenced
B16 = 0x20000000
C16 = 0x40000000
D16 = 0x60000000


@pytest.mark.parametrize("args,expect", [
    # (X, g, W, Y, M, K, N, eps)
    ((0, B16, C16, D16, 8, 64, 64, 1e-6), 1),                  # NULL X
    ((A16, B16, C16, 0, 8, 64, 64, 1e-6), 1),                  # NULL Y
    ((A16, B16, C16, D16, -1, 64, 64, 1e-6), 1),               # M < 0
    ((A16, B16, C16, D16, 8, 0, 64, 1e-6), 1),                 # K = 0
    ((A16, B16, C16, D16, 8, 64, -8, 1e-6), 1),                # N < 0
    ((A16, B16, C16, D16, 8, 64, 64, -1.0), 1),                # eps < 0
    ((A16, B16, C16, D16, 8, 64, 64, float("nan")), 1),        # eps NaN
    ((A16, B16, C16, D16, 8, 64, 64, float("inf")), 1),        # eps inf
    ((A16, B16, C16, D16, 8, 60, 64, 1e-6), 2),                # K % 8
    ((A16, B16, C16, D16, 8, 64, 68, 1e-6), 2),                # N % 8
    ((A16 + 2, B16, C16, D16, 8, 64, 64, 1e-6), 2),            # X misaligned
    ((A16, B16, C16, D16 + 8, 8, 64, 64, 1e-6), 2),            # Y misaligned
    ((A16, B16, C16, A16 + 512, 8, 64, 64, 1e-6), 1),          # Y overlaps X
    ((A16, B16, C16, C16, 8, 64, 64, 1e-6), 1),                # Y aliases W
    ((A16, B16, C16, D16, 2**31, 64, 64, 1e-6), 1),            # M too large
    ((0, 0, 0, 0, 0, 64, 64, 1e-6), 0),                        # M = 0: no-op
    ((0, 0, 0, 0, 8, 64, 0, 1e-6), 0),                         # N = 0: no-op
])
def test_fused_validation(lib, args, expect):
    X, g, W, Y, M, K, N, eps = args
    assert lib.rmsnorm_matmul(X, g, W, Y, M, K, N, eps, None) == expect


def test_gated_validation(lib):
    f = lib.rmsnorm_matmul_swiglu
    assert f(A16, B16, C16, D16, 8, 64, 24, 1e-6, None) == 2      # N % 16 (F = 12)
    assert f(A16, B16, C16, D16, 8, 64, 20, 1e-6, None) == 2      # N % 8
    assert f(A16, B16, C16, 0, 8, 64, 32, 1e-6, None) == 1        # NULL Y
    assert f(A16, B16, C16, A16 + 64, 8, 64, 32, 1e-6, None) == 1 # Y overlaps X
    assert f(A16, B16, C16, D16, 8, 64, 32, -1.0, None) == 1      # eps < 0
    assert f(0, 0, 0, 0, 0, 64, 32, 1e-6, None) == 0              # M = 0: no-op


def test_ex_validation(lib):
    f = lib.rmsnorm_matmul_ex
    assert f(A16, B16, C16, D16, 8, 64, 64, 1e-6, 4, None) == 1      # unknown flag bit
    assert f(A16, B16, C16, D16, 8, 64, 24, 1e-6, 2, None) == 2      # gated: N % 16
    assert f(A16, B16, C16, D16, 8, 60, 64, 1e-6, 1, None) == 2      # K % 8
    assert f(A16, B16, C16, C16, 8, 64, 64, 1e-6, 1, None) == 1      # Y aliases W
    assert f(0, 0, 0, 0, 8, 64, 0, 1e-6, 3, None) == 0               # N = 0: no-op


def test_lora_validation(lib):
    f = lib.rmsnorm_matmul_lora
    E16 = 0x70000000
    assert f(A16, B16, C16, D16, E16, D16 + 0x100000, 8, 64, 64, 0, 1e-6, None) == 1    # R = 0
    assert f(A16, B16, C16, D16, E16, D16 + 0x100000, 8, 64, 64, 72, 1e-6, None) == 1   # R > 64
    assert f(A16, B16, C16, D16, E16, D16 + 0x100000, 8, 64, 64, 12, 1e-6, None) == 2   # R % 8
    assert f(A16, B16, C16, D16, 0, D16 + 0x100000, 8, 64, 64, 16, 1e-6, None) == 1     # NULL B
    assert f(A16, B16, C16, D16, E16, D16, 8, 64, 64, 16, 1e-6, None) == 1              # Y aliases A
    assert f(0, 0, 0, 0, 0, 0, 0, 64, 64, 16, 1e-6, None) == 0                          # M = 0: no-op


def test_attention_validation(lib):
    f = lib.qknorm_attention
    E16, F16 = 0x70000000, 0x7000_0000_0
    # (Q, ldq, K, ldk, V, ldv, gq, gk, O, ldo, B, S, Hq, Hkv, D, eps, scale, causal)
    ok = [A16, 6144, A16 + 8192, 6144, A16 + 10240, 6144, B16, B16 + 256, F16, 4096,
          1, 256, 32, 8, 128, 1e-6, 0.0, 1]

    def call(**kw):
        a = list(ok)
        names = ["Q", "ldq", "K", "ldk", "V", "ldv", "gq", "gk", "O", "ldo", "B", "S", "Hq",
                 "Hkv", "D", "eps", "scale", "causal"]
        for k, v in kw.items():
            a[names.index(k)] = v
        return f(*a, None)

    assert call(D=96) == 1                 # head dimension other than 64 or 128
    assert call(Hq=12) == 1                # Hq not a multiple of Hkv
    assert call(ldq=4000) == 1             # row stride narrower than the heads
    assert call(ldo=4100) == 2             # row stride not a multiple of 8
    assert call(Q=A16 + 4) == 2            # misaligned pointer
    assert call(O=0) == 1                  # NULL output
    assert call(O=A16 + 4096) == 1         # output overlaps the inputs
    assert call(eps=-1.0) == 1
    assert call(scale=float("nan")) == 1
    assert call(S=0) == 0 and call(B=0) == 0   # no-ops
    h = lib.rmsnorm_heads
    assert h(A16, 1024, B16, D16, 1024, 4, 8, 128, 1e-6, None) != 1   # valid (fails later without a GPU)
    assert h(A16, 1024, B16, D16, 1024, 4, 8, 100, 1e-6, None) == 1   # D % 8
    assert h(A16, 1024, B16, D16, 1024, 4, 2, 512, 1e-6, None) == 1   # D > 256
    assert h(A16, 1000, B16, D16, 1024, 4, 8, 128, 1e-6, None) == 1   # ldx < H * D
    assert h(A16, 1028, B16, D16, 1028, 4, 8, 128, 1e-6, None) == 2   # ld % 8
    assert h(A16, 1024, B16, A16, 1024, 4, 8, 128, 1e-6, None) == 1   # Y aliases X
    assert h(0, 1024, 0, 0, 1024, 0, 8, 128, 1e-6, None) == 0         # T = 0: no-op


def test_unfused_validation(lib):
    assert lib.rmsnorm(0, B16, D16, 8, 64, 1e-6, None) == 1
    assert lib.rmsnorm(A16, B16, D16, 8, 63, 1e-6, None) == 2
    assert lib.rmsnorm(A16, B16, A16, 8, 64, 1e-6, None) == 1
    assert lib.rmsnorm(0, 0, 0, 0, 64, 1e-6, None) == 0
    assert lib.matmul(A16, C16, 0, 8, 64, 64, None) == 1
    assert lib.matmul(A16, C16, D16 + 4, 8, 64, 64, None) == 2
    assert lib.matmul(A16, C16, D16, 8, 0, 64, None) == 1
    assert lib.matmul(0, 0, 0, 8, 64, 0, None) == 0


def test_binding_rejects_cpu_tensors(lib):
    torch = pytest.importorskip("torch")
    X = torch.zeros(8, 64, dtype=torch.bfloat16)
    g = torch.ones(64, dtype=torch.bfloat16)
    W = torch.zeros(64, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        rmm.rmsnorm_matmul(X, g, W)
    with pytest.raises(TypeError, match="bfloat16"):
        rmm.rmsnorm_matmul(X.float(), g, W)


def test_no_oracle_in_product_path():
    # The library package must not import the test oracle.
    pkg = os.path.dirname(rmm.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                with open(os.path.join(root, f)) as fh:
                    src = fh.read()
                assert not re.search(r"^\s*(import|from)\s+oracle", src, flags=re.M), f
                assert "rmm_oracle" not in src, f


def test_attention_binding_checks_tensors(lib):
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 8, 4, 128, dtype=torch.bfloat16)
    k = torch.zeros(1, 8, 2, 128, dtype=torch.bfloat16)
    g = torch.ones(128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        rmm.qknorm_attention(q, k, k, g, g)                       # CPU tensors
    with pytest.raises(TypeError, match="bfloat16"):
        rmm.qknorm_attention(q.float(), k, k, g, g)
    with pytest.raises(ValueError, match="CUDA"):
        rmm.rmsnorm_heads(q[0], g)                                 # CPU tensor
    with pytest.raises(TypeError, match="torch.Tensor"):
        rmm.qknorm_attention([0], k, k, g, g)


def test_attention_abi_rejects_grouping_and_head_dim(lib):
    f = lib.qknorm_attention
    # (Q, ldq, K, ldk, V, ldv, gq, gk, O, ldo, B, S, Hq, Hkv, D, eps, scale, causal)
    assert f(A16, 768, A16 + 512, 768, A16 + 768, 768, B16, B16 + 256, C16, 512,
             1, 16, 5, 2, 128, 1e-6, 0.0, 1, None) == 1               # 5 query heads over 2
    assert f(A16, 480, A16 + 320, 480, A16 + 400, 480, B16, B16 + 256, C16, 320,
             1, 16, 4, 1, 80, 1e-6, 0.0, 1, None) == 1                # D = 80 is not built
