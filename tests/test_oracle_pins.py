"""The fp64 oracle against its pins, and planted mistakes against the pins.

CPU only.  The mutation tests copy the oracle's C source to a temporary
directory, plant one plausible mistake in the copy, compile it, and check
that at least one pin fails; the committed oracle is never modified.
"""
import subprocess

import numpy as np
import pytest

import oracle
from oracle_pins import ALL_PINS, load_p5_cases, zp_rewrite_holds


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("name", sorted(ALL_PINS))
def test_pin(lib, name):
    ok, detail = ALL_PINS[name](lib)
    assert ok, detail


@pytest.mark.parametrize("K", [1, 3, 64, 1000])
def test_zp_identity_holds(K):
    for seed in range(5):
        assert zp_rewrite_holds(K, seed)


def test_zp_identity_catches_k_dependent_divisor():
    # A divisor that varies with k cannot move past the sum; the finite-field
    # test must see the difference (with overwhelming probability).
    assert not any(zp_rewrite_holds(16, s, k_dependent_divisor=True) for s in range(5))


def test_golden_fixture_parses():
    cases = load_p5_cases()
    assert [c["name"] for c in cases] == ["A", "B", "C"]
    for c in cases:
        assert c["X"].shape == (2, 3) and c["W"].shape == (3, 2) and c["Y"].shape == (2, 2)


def test_bf16_decode_exact():
    bits = np.array([0x0000, 0x3F80, 0xBF80, 0x4049, 0x7F7F, 0x0001, 0x8000], dtype=np.uint16)
    vals = oracle.bf16_bits_to_f64(bits)
    assert vals[0] == 0.0 and vals[1] == 1.0 and vals[2] == -1.0
    assert vals[3] == 3.140625
    assert vals[4] == float(np.float32(3.3895313892515355e38))
    assert vals[5] == 2.0 ** -133  # smallest bf16 subnormal
    assert vals[6] == 0.0 and np.signbit(vals[6])


def test_bf16_decode_matches_torch():
    torch = pytest.importorskip("torch")
    t = torch.randn(1000, dtype=torch.float32).to(torch.bfloat16)
    assert np.array_equal(oracle.to_f64(t), t.double().numpy())


def test_zero_row_gives_zero():
    y = oracle.rmsnorm_matmul(np.zeros((1, 8)), np.ones(8), np.ones((8, 3)), 1e-6)
    assert np.array_equal(y, np.zeros((1, 3)))


def test_gated_rejects_odd_width():
    with pytest.raises(RuntimeError):
        oracle.rmsnorm_matmul_swiglu(np.ones((1, 4)), np.ones(4), np.ones((4, 3)), 1e-6)


def test_empty_rows():
    y = oracle.rmsnorm_matmul(np.zeros((0, 8)), np.ones(8), np.ones((8, 3)), 1e-6)
    assert y.shape == (0, 3)


def test_threads_do_not_change_result(lib):
    rng = np.random.default_rng(5)
    X, g, W = rng.standard_normal((33, 50)), rng.uniform(0.5, 1.5, 50), rng.standard_normal((50, 21))
    a = oracle.rmsnorm_matmul(X, g, W, 1e-5, nthreads=1, lib=lib)
    b = oracle.rmsnorm_matmul(X, g, W, 1e-5, nthreads=4, lib=lib)
    assert np.array_equal(a, b)


# Each mutant: (description, original snippet, replacement).  Every occurrence
# of the snippet is replaced.
MUTANTS = [
    ("eps outside the square root", "1.0 / sqrt(ms + eps)", "1.0 / (sqrt(ms) + eps)"),
    ("mean over K-1", "ss / (double)K", "ss / (double)(K - 1)"),
    ("no square root", "1.0 / sqrt(ms + eps)", "1.0 / (ms + eps)"),
    ("gain dropped", "x[k] * g[k] * r", "x[k] * r"),
    ("gain read as 1+g", "x[k] * g[k] * r", "x[k] * (1.0 + g[k]) * r"),
    ("W read transposed", "const double *w = W + k * N;",
     "const double *w = W + k; /* mutant */"),
    ("sign flipped", "y[n] += a * w[n];", "y[n] -= a * w[n];"),
    ("last k dropped from the statistic", "for (long k = 0; k < K; ++k)\n        ss +=",
     "for (long k = 0; k < K - 1; ++k)\n        ss +="),
    ("statistic scaled by a constant", "ss += x[k] * x[k];", "ss += x[k] * x[k] * 1.25;"),
    # the gated form
    ("gate and up swapped", "silu(Z[m * N + f]) * Z[m * N + F + f]",
     "silu(Z[m * N + F + f]) * Z[m * N + f]"),
    ("sigmoid instead of silu", "return z / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(-z));"),
    ("exponent sign flipped in silu", "return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    ("up column off by one", "* Z[m * N + F + f];", "* Z[m * N + F + f - (f > 0)];"),
    ("gate not activated", "silu(Z[m * N + f]) * Z[m * N + F + f]", "Z[m * N + f] * Z[m * N + F + f]"),
    # the LoRA form
    ("adapter subtracted", "wk[n] += akj * bj[n];", "wk[n] -= akj * bj[n];"),
    ("adapter doubled", "wk[n] += akj * bj[n];", "wk[n] += 2.0 * akj * bj[n];"),
    ("adapter B read transposed", "const double *bj = B + j * N;", "const double *bj = B + j; /* mutant */"),
    ("adapter A row and column swapped", "const double akj = A[k * R + j];",
     "const double akj = A[(j * K + k) % (K * R)];"),
    ("last adapter rank dropped", "for (long j = 0; j < R; ++j) {\n            const double akj",
     "for (long j = 0; j < R - 1; ++j) {\n            const double akj"),
    # QKNorm + Attention
    ("attention scale dropped", "sc[j] = scale * dot;", "sc[j] = dot;"),
    ("causal mask hides the diagonal", "const long nkeys = causal ? i + 1 : S;",
     "const long nkeys = causal ? i : S;"),
    ("causal mask shows one key too many", "const long nkeys = causal ? i + 1 : S;",
     "const long nkeys = causal ? (i + 2 < S ? i + 2 : S) : S;"),
    ("key/value head taken modulo Hkv", "const long c = h / group;", "const long c = h % Hkv;"),
    ("keys not normalised", "rc = oracle_rmsnorm(K, gk, Kn, B * S * Hkv, D, eps, nthreads);",
     "memcpy(Kn, K, nke * sizeof(double));"),
    ("query and key gains swapped", "oracle_rmsnorm(Q, gq, Qn,", "oracle_rmsnorm(Q, gk, Qn,"),
    ("softmax not normalised", "const double pj = sc[j] / denom;", "const double pj = sc[j];"),
    ("values read in reverse order", "const double *v = V + ((b * S + j) * Hkv + c) * D;",
     "const double *v = V + ((b * S + nkeys - 1 - j) * Hkv + c) * D;"),
]


@pytest.mark.parametrize("desc,orig,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, desc, orig, repl):
    with open(oracle.SOURCE) as f:
        src = f.read()
    assert orig in src, f"mutation site for {desc!r} not found"
    mutated = src.replace(orig, repl)
    if desc == "W read transposed":
        # read W as if stored [N,K]: element (k,n) at n*K + k (stays in bounds)
        mutated = mutated.replace("y[n] += a * w[n];", "y[n] += a * w[n * K];")
    if desc == "adapter B read transposed":
        # read B as if stored [N,R]: element (j,n) at n*R + j (stays in bounds)
        mutated = mutated.replace("wk[n] += akj * bj[n];", "wk[n] += akj * bj[n * R];")
    path = tmp_path / "mutant.c"
    path.write_text(mutated)
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", str(so), str(path), "-lm"], check=True)
    mlib = oracle.load(str(so))
    failed = []
    for name, pin in ALL_PINS.items():
        try:
            ok, _ = pin(mlib)
        except Exception:  # noqa: BLE001 - a crash also counts as caught
            ok = False
        if not ok:
            failed.append(name)
    assert failed, f"no pin caught the mutant: {desc}"


def test_attention_rejects_bad_arguments():
    Q = np.zeros((1, 4, 3, 8))
    K = np.zeros((1, 4, 2, 8))
    with pytest.raises(RuntimeError):          # 3 query heads over 2 key/value heads
        oracle.attention(Q, K, K, 1.0)
    Q = np.zeros((1, 4, 2, 8))
    with pytest.raises(RuntimeError):          # query position outside the sequence
        oracle.attention(Q, K, K, 1.0, qpos=[4])


def test_attention_positions_select_rows(lib):
    rng = np.random.default_rng(7)
    Q, K, V = (rng.standard_normal((2, 9, h, 8)) for h in (4, 2, 2))
    full = oracle.attention(Q, K, V, 0.3, causal=True, lib=lib)
    part = oracle.attention(Q, K, V, 0.3, causal=True, qpos=[8, 0, 3], lib=lib)
    assert np.array_equal(part, full[:, [8, 0, 3]])


# Random shapes against torch's float64 library routines (an implementation
# the oracle does not call): every form, several sizes, causal and full.
def _torch():
    return pytest.importorskip("torch")


@pytest.mark.parametrize("seed", range(6))
def test_forms_match_torch_on_random_shapes(lib, seed):
    torch = _torch()
    F = torch.nn.functional
    rng = np.random.default_rng(100 + seed)
    M, K, N, R = (int(v) for v in rng.integers(1, 40, 4))
    N += N % 2   # the gated form needs an even width
    eps = float(10.0 ** rng.uniform(-6, 0))
    X = rng.standard_normal((M, K)) * np.exp(rng.standard_normal((M, 1)))
    g = rng.uniform(0.5, 1.5, K)
    W = rng.standard_normal((K, N))
    A, B = rng.standard_normal((K, R)), rng.standard_normal((R, N))
    Xn = F.rms_norm(torch.tensor(X), (K,), torch.tensor(g), eps)
    Z = Xn @ torch.tensor(W)
    ref = Z.numpy()
    assert np.abs(oracle.rmsnorm_matmul(X, g, W, eps, lib=lib) - ref).max() <= 1e-12 * (1 + np.abs(ref).max())
    half = N // 2
    gated = (F.silu(Z[:, :half]) * Z[:, half:]).numpy()
    got = oracle.rmsnorm_matmul_swiglu(X, g, W, eps, lib=lib)
    assert np.abs(got - gated).max() <= 1e-12 * (1 + np.abs(gated).max())
    lora = (Xn @ (torch.tensor(W) + torch.tensor(A) @ torch.tensor(B))).numpy()
    got = oracle.rmsnorm_matmul_lora(X, g, W, A, B, eps, lib=lib)
    assert np.abs(got - lora).max() <= 1e-12 * (1 + np.abs(lora).max())


@pytest.mark.parametrize("seed", range(6))
def test_attention_matches_torch_on_random_shapes(lib, seed):
    torch = _torch()
    F = torch.nn.functional
    rng = np.random.default_rng(200 + seed)
    Hkv = int(rng.integers(1, 4))
    Hq = Hkv * int(rng.integers(1, 4))
    B, S, D = int(rng.integers(1, 3)), int(rng.integers(1, 40)), int(rng.integers(2, 24))
    causal = bool(seed % 2)
    eps = float(10.0 ** rng.uniform(-6, -1))
    scale = float(rng.uniform(0.05, 1.0))
    Q = rng.standard_normal((B, S, Hq, D)) * np.exp(rng.standard_normal((B, S, Hq, 1)))
    K = rng.standard_normal((B, S, Hkv, D)) * np.exp(rng.standard_normal((B, S, Hkv, 1)))
    V = rng.standard_normal((B, S, Hkv, D))
    gq, gk = rng.uniform(0.5, 1.5, D), rng.uniform(0.5, 1.5, D)
    o = oracle.qknorm_attention(Q, K, V, gq, gk, eps, scale=scale, causal=causal, lib=lib)
    qn = F.rms_norm(torch.tensor(Q), (D,), torch.tensor(gq), eps)
    kn = F.rms_norm(torch.tensor(K), (D,), torch.tensor(gk), eps)
    rep = Hq // Hkv
    ref = F.scaled_dot_product_attention(qn.transpose(1, 2), kn.repeat_interleave(rep, dim=2).transpose(1, 2),
                                         torch.tensor(V).repeat_interleave(rep, dim=2).transpose(1, 2),
                                         is_causal=causal, scale=scale).transpose(1, 2).numpy()
    assert np.abs(o - ref).max() <= 1e-12 * (1 + np.abs(ref).max())
