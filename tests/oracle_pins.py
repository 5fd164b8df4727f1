"""Pins that tie the fp64 oracle to facts other than its own code.

Each ``pin_*`` function takes a loaded oracle library (so the mutation tests
can run the same pins against a deliberately broken copy) and returns
``(ok, detail)``.  None of them re-types the oracle's formula: each checks a
property that the operation must have, a closed form, a library routine, or
values worked out by hand.

Operation (Mirage review page, section 3, "muGraph example" and "core
formula"): Y = RMSNorm(X; g, eps) @ W with
r[m] = 1/sqrt(mean_k X[m,k]^2 + eps) and Y[m,n] = sum_k X[m,k] g[k] r[m] W[k,n].
"""
from __future__ import annotations

import math
import os
import random
from fractions import Fraction

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _rel_normwise(a, b):
    scale = max(float(np.abs(b).max()), 1e-300)
    return float(np.abs(a - b).max()) / scale


# ---------------------------------------------------------------------------
# P1: the identity behind the fusion, checked exactly in a finite field (the
# review page's equivalence verifier tests programs on random inputs in Z_p;
# section 3 "equivalence verification").  sum_k (a_k * c) == (sum_k a_k) * c
# when c does not depend on k; a k-dependent divisor breaks it.
# ---------------------------------------------------------------------------
P_PRIME = 2_147_483_647  # 2^31 - 1


def zp_rewrite_holds(K: int, seed: int, k_dependent_divisor: bool = False) -> bool:
    rnd = random.Random(seed)
    p = P_PRIME
    x = [rnd.randrange(p) for _ in range(K)]
    g = [rnd.randrange(p) for _ in range(K)]
    w = [rnd.randrange(p) for _ in range(K)]
    r = rnd.randrange(1, p)
    rk = [rnd.randrange(1, p) for _ in range(K)]
    divisor = [rk[k] if k_dependent_divisor else r for k in range(K)]
    inv = [pow(d, p - 2, p) for d in divisor]  # division = multiplication by inverse
    lhs = sum(x[k] * g[k] % p * w[k] % p * inv[k] for k in range(K)) % p
    rhs = sum(x[k] * g[k] % p * w[k] for k in range(K)) % p * pow(r, p - 2, p) % p
    return lhs == rhs


def pin_rewrite_agrees(lib, seed=11):
    """The oracle's unfused and rewritten forms agree to fp64 rounding."""
    rng = _rng(seed)
    X = rng.standard_normal((7, 96))
    g = rng.uniform(0.5, 1.5, 96)
    W = rng.standard_normal((96, 40)) / math.sqrt(96)
    a = oracle.rmsnorm_matmul(X, g, W, 1e-6, lib=lib)
    b = oracle.rmsnorm_matmul_rewritten(X, g, W, 1e-6, lib=lib)
    err = _rel_normwise(a, b)
    return err <= 1e-12, f"normwise rel diff {err:.3e}"


# ---------------------------------------------------------------------------
# P2: scale invariance.  RMSNorm(c X) = RMSNorm(X) when eps = 0; for a power
# of two c every fp64 rounding scales exactly, so the outputs are bitwise equal.
# ---------------------------------------------------------------------------
def pin_scale_invariance(lib, seed=12):
    rng = _rng(seed)
    X = rng.standard_normal((5, 64))
    g = rng.uniform(0.5, 1.5, 64)
    W = rng.standard_normal((64, 24)) / 8.0
    y = oracle.rmsnorm_matmul(X, g, W, 0.0, lib=lib)
    for c in (2.0 ** -4, 2.0, 2.0 ** 8):
        yc = oracle.rmsnorm_matmul(c * X, g, W, 0.0, lib=lib)
        if not np.array_equal(y, yc):
            return False, f"Y(cX) != Y(X) bitwise for c={c}"
    y3 = oracle.rmsnorm_matmul(3.0 * X, g, W, 1e-12, lib=lib)
    err = _rel_normwise(y3, y)
    if err > 1e-11:
        return False, f"c=3, eps=1e-12: normwise rel diff {err:.3e}"
    return True, "ok"


# ---------------------------------------------------------------------------
# P3: W = identity reduces the operation to RMSNorm alone; torch's
# functional rms_norm (a library routine) computes x * rsqrt(mean(x^2)+eps) * g.
# ---------------------------------------------------------------------------
def pin_identity_is_rmsnorm(lib, seed=13):
    import torch
    rng = _rng(seed)
    K = 48
    X = rng.standard_normal((6, K)) * rng.uniform(0.1, 10.0, (6, 1))
    g = rng.uniform(0.5, 1.5, K)
    for eps in (1e-6, 0.5):
        y = oracle.rmsnorm_matmul(X, g, np.eye(K), eps, lib=lib)
        ref = torch.nn.functional.rms_norm(torch.from_numpy(X), (K,),
                                           weight=torch.from_numpy(g), eps=eps).numpy()
        err = _rel_normwise(y, ref)
        if err > 1e-13:
            return False, f"eps={eps}: normwise rel diff {err:.3e}"
        xn = oracle.rmsnorm(X, g, eps, lib=lib)
        err = _rel_normwise(xn, ref)
        if err > 1e-13:
            return False, f"rmsnorm alone, eps={eps}: normwise rel diff {err:.3e}"
    return True, "ok"


# ---------------------------------------------------------------------------
# P4: constant rows.  X[m,:] = c gives mean square c^2, so
# Y[m,n] = c / sqrt(c^2 + eps) * sum_k g[k] W[k,n]  (numpy's g @ W).
# ---------------------------------------------------------------------------
def pin_constant_rows(lib, seed=14):
    rng = _rng(seed)
    K, N = 40, 12
    g = rng.uniform(0.5, 1.5, K)
    W = rng.standard_normal((K, N))
    cs = np.array([1.0, -2.5, 0.125, 7.0])
    X = np.repeat(cs[:, None], K, axis=1)
    gw = g @ W
    for eps in (0.0, 1e-6, 3.0):
        y = oracle.rmsnorm_matmul(X, g, W, eps, lib=lib)
        ref = (cs / np.sqrt(cs * cs + eps))[:, None] * gw[None, :]
        err = _rel_normwise(y, ref)
        if err > 1e-13:
            return False, f"eps={eps}: normwise rel diff {err:.3e}"
    return True, "ok"


# ---------------------------------------------------------------------------
# P5: hand-worked 2x3x2 examples (tests/golden/p5_bruteforce.txt).
# ---------------------------------------------------------------------------
def _parse_rows(s, conv):
    return [[conv(v) for v in row.split()] for row in s.split(";")]


def _parse_value(tok):
    if "@" in tok:
        num, d = tok.split("@")
        return float(Fraction(num)) / math.sqrt(int(d))
    return float(Fraction(tok))


def load_p5_cases():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "p5_bruteforce.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                cur = {"name": rest}
                cases.append(cur)
            elif key == "eps":
                cur["eps"] = float(Fraction(rest))
            elif key in ("X", "W"):
                cur[key] = np.array(_parse_rows(rest, lambda v: float(Fraction(v))))
            elif key == "g":
                cur["g"] = np.array([float(Fraction(v)) for v in rest.split()])
            elif key == "Y":
                cur["Y"] = np.array(_parse_rows(rest, _parse_value))
    return cases


def pin_hand_worked(lib):
    for c in load_p5_cases():
        y = oracle.rmsnorm_matmul(c["X"], c["g"], c["W"], c["eps"], lib=lib)
        if not np.allclose(y, c["Y"], rtol=1e-15, atol=1e-15):
            return False, f"case {c['name']}: got {y.tolist()} want {c['Y'].tolist()}"
    return True, "ok"


# ---------------------------------------------------------------------------
# P6: the matmul part.  g = 1 and rows of +-1 with eps = 0 give r = 1, so
# Y = X @ W, which numpy computes independently.
# ---------------------------------------------------------------------------
def pin_matmul_part(lib, seed=16):
    rng = _rng(seed)
    M, K, N = 9, 33, 17
    X = rng.choice([-1.0, 1.0], size=(M, K))
    W = rng.standard_normal((K, N))
    y = oracle.rmsnorm_matmul(X, np.ones(K), W, 0.0, lib=lib)
    err = _rel_normwise(y, X @ W)
    if err > 1e-13:
        return False, f"fused vs numpy: normwise rel diff {err:.3e}"
    c = oracle.matmul(X, W, lib=lib)
    err = _rel_normwise(c, X @ W)
    if err > 1e-13:
        return False, f"matmul vs numpy: normwise rel diff {err:.3e}"
    return True, "ok"


# ---------------------------------------------------------------------------
# P7: structure.  Rows are independent (a row permutation of X permutes Y's
# rows bitwise), columns are independent (a column permutation of W permutes
# Y's columns bitwise), and g travels with the k index (permuting k in X, g
# and W together changes only the summation order).
# ---------------------------------------------------------------------------
def pin_permutations(lib, seed=17):
    rng = _rng(seed)
    M, K, N = 6, 20, 10
    X = rng.standard_normal((M, K))
    g = rng.uniform(0.5, 1.5, K)
    W = rng.standard_normal((K, N))
    y = oracle.rmsnorm_matmul(X, g, W, 1e-6, lib=lib)
    pm, pn, pk = rng.permutation(M), rng.permutation(N), rng.permutation(K)
    if not np.array_equal(oracle.rmsnorm_matmul(X[pm], g, W, 1e-6, lib=lib), y[pm]):
        return False, "row permutation"
    if not np.array_equal(oracle.rmsnorm_matmul(X, g, W[:, pn], 1e-6, lib=lib), y[:, pn]):
        return False, "column permutation"
    yk = oracle.rmsnorm_matmul(X[:, pk], g[pk], W[pk], 1e-6, lib=lib)
    err = _rel_normwise(yk, y)
    if err > 1e-13:
        return False, f"k permutation: normwise rel diff {err:.3e}"
    return True, "ok"


# ---------------------------------------------------------------------------
# G: the gated MLP on top (review page, section 5, benchmark table: GatedMLP;
# read as Y = silu(Z_gate) * Z_up with Z = RMSNorm(X) @ [W_gate | W_up]).
# Z itself is the main oracle, pinned above; these pins tie the gate to facts
# about silu(z) = z * sigmoid(z):
#   G1 a zero gate gives exactly zero;
#   G2 the odd part is exact: silu(z) - silu(-z) = z (sigmoid(z) + sigmoid(-z)
#      = 1), so Y(W_gate) - Y(-W_gate) = Z_gate * Z_up;
#   G3 silu(z) -> z for large z, G4 silu(z) -> 0 for large negative z;
#   G5 with W_gate = W_up, Y = Z^2 sigmoid(Z) >= 0.
# ---------------------------------------------------------------------------
def _gated_problem(rng, M=5, K=24, F=7):
    X = rng.standard_normal((M, K))
    g = rng.uniform(0.5, 1.5, K)
    Wg = rng.standard_normal((K, F))
    Wu = rng.standard_normal((K, F))
    return X, g, Wg, Wu


def pin_gated_zero_gate(lib, seed=21):
    X, g, _, Wu = _gated_problem(_rng(seed))
    y = oracle.rmsnorm_matmul_swiglu(X, g, np.hstack([np.zeros_like(Wu), Wu]), 1e-6, lib=lib)
    return (bool(np.all(y == 0.0)), "zero gate gives zero")


def pin_gated_odd_part(lib, seed=22):
    X, g, Wg, Wu = _gated_problem(_rng(seed))
    yp = oracle.rmsnorm_matmul_swiglu(X, g, np.hstack([Wg, Wu]), 1e-6, lib=lib)
    yn = oracle.rmsnorm_matmul_swiglu(X, g, np.hstack([-Wg, Wu]), 1e-6, lib=lib)
    F = Wg.shape[1]
    z = oracle.rmsnorm_matmul(X, g, np.hstack([Wg, Wu]), 1e-6, lib=lib)
    ref = z[:, :F] * z[:, F:]
    err = _rel_normwise(yp - yn, ref)
    return (err <= 1e-12, f"odd part: normwise rel diff {err:.3e}")


def pin_gated_limits(lib, seed=23):
    rng = _rng(seed)
    K, F = 16, 5
    # constant rows: Z = sign(c) * (g @ W) / sqrt(1 + eps/c^2), here with a
    # positive gate of at least 40 or a negative one of at most -40
    X = np.full((2, K), 3.0)
    g = rng.uniform(0.5, 1.5, K)
    Wu = rng.standard_normal((K, F))
    for sign in (1.0, -1.0):
        Wg = sign * rng.uniform(5.0, 6.0, (K, F))
        y = oracle.rmsnorm_matmul_swiglu(X, g, np.hstack([Wg, Wu]), 0.0, lib=lib)
        zg, zu = g @ Wg, g @ Wu
        if sign > 0:
            err = _rel_normwise(y, np.broadcast_to(zg * zu, y.shape))
            if not (zg.min() >= 40.0 and err <= 1e-14):
                return False, f"large positive gate: rel diff {err:.3e}"
        else:
            bound = float(np.abs(zg * zu).max() * np.exp(-40.0))
            if not (zg.max() <= -40.0 and float(np.abs(y).max()) <= bound):
                return False, "large negative gate is not ~0"
    return True, "ok"


def pin_gated_equal_projections(lib, seed=24):
    X, g, Wg, _ = _gated_problem(_rng(seed))
    y = oracle.rmsnorm_matmul_swiglu(X, g, np.hstack([Wg, Wg]), 1e-6, lib=lib)
    return (bool(np.all(y >= 0.0)) and bool(np.any(y > 0.0)), "gate = up gives y >= 0")


# ---------------------------------------------------------------------------
# L: LoRA (review page, section 5, benchmark table; read as
# Y = RMSNorm(X) @ (W + A @ B)).  Pinned by
#   L1 a zero adapter (A = 0, or B = 0) gives the plain oracle bitwise;
#   L2 W = 0: Y = (RMSNorm(X) @ A) @ B, numpy's matmuls on the pinned RMSNorm;
#   L3 a rank-one adapter a b^T with W = 0 has the closed form
#      Y[m,n] = (sum_k Xn[m,k] a[k]) * b[n].
# ---------------------------------------------------------------------------
def _lora_problem(rng, M=6, K=20, N=9, R=4):
    X = rng.standard_normal((M, K))
    g = rng.uniform(0.5, 1.5, K)
    W = rng.standard_normal((K, N))
    A = rng.standard_normal((K, R))
    B = rng.standard_normal((R, N))
    return X, g, W, A, B


def pin_lora_zero_adapter(lib, seed=31):
    X, g, W, A, B = _lora_problem(_rng(seed))
    y = oracle.rmsnorm_matmul(X, g, W, 1e-6, lib=lib)
    ya = oracle.rmsnorm_matmul_lora(X, g, W, np.zeros_like(A), B, 1e-6, lib=lib)
    yb = oracle.rmsnorm_matmul_lora(X, g, W, A, np.zeros_like(B), 1e-6, lib=lib)
    return (bool(np.array_equal(ya, y) and np.array_equal(yb, y)), "zero adapter")


def pin_lora_adapter_alone(lib, seed=32):
    X, g, W, A, B = _lora_problem(_rng(seed))
    y = oracle.rmsnorm_matmul_lora(X, g, np.zeros_like(W), A, B, 1e-6, lib=lib)
    ref = (oracle.rmsnorm(X, g, 1e-6, lib=lib) @ A) @ B
    err = _rel_normwise(y, ref)
    return (err <= 1e-13, f"W = 0: normwise rel diff {err:.3e}")


def pin_lora_rank_one(lib, seed=33):
    X, g, W, A, B = _lora_problem(_rng(seed), R=1)
    y = oracle.rmsnorm_matmul_lora(X, g, np.zeros_like(W), A, B, 0.0, lib=lib)
    ms = (X * X).mean(axis=1)
    xn = X * g[None, :] / np.sqrt(ms)[:, None]
    ref = np.outer(xn @ A[:, 0], B[0])
    err = _rel_normwise(y, ref)
    return (err <= 1e-13, f"rank one: normwise rel diff {err:.3e}")


# ---------------------------------------------------------------------------
# A: QKNorm + Attention (review page, section 5, benchmark table; read as
# per-head RMSNorm with gains on queries and keys, then softmax attention with
# grouped key/value heads).  Pinned by
#   A1 torch's rms_norm and scaled_dot_product_attention (library routines,
#      float64 on the CPU), causal and not, grouped heads expanded with
#      repeat_interleave, a small and a large eps;
#   A2 the first query of a causal row sees one key: O = V[0] of its group, bitwise;
#   A3 equal keys give uniform weights: O[i] = mean of V over the visible keys;
#   A4 with eps = 0, scaling query rows by 2^3 and key rows by 2^-5 changes
#      nothing (bitwise: the normalisation removes any row scale);
#   A5 values constant along the sequence come back unchanged (weights sum to 1);
#   A6 grouped heads equal full multi-head attention with repeated key/value heads;
#   A7 a 2-token, D = 2 case worked out by hand.
# ---------------------------------------------------------------------------
def _attn_problem(rng, B=2, S=23, Hq=4, Hkv=2, D=8):
    Q = rng.standard_normal((B, S, Hq, D)) * rng.uniform(0.1, 10, (B, S, Hq, 1))
    K = rng.standard_normal((B, S, Hkv, D)) * rng.uniform(0.1, 10, (B, S, Hkv, 1))
    V = rng.standard_normal((B, S, Hkv, D))
    gq = rng.uniform(0.5, 1.5, D)
    gk = rng.uniform(0.5, 1.5, D)
    return Q, K, V, gq, gk


def pin_attn_library(lib, seed=41):
    import torch
    F = torch.nn.functional
    Q, K, V, gq, gk = _attn_problem(_rng(seed))
    B, S, Hq, D = Q.shape
    rep = Hq // K.shape[2]
    worst = 0.0
    for causal in (True, False):
        for eps in (1e-6, 0.5):
            o = oracle.qknorm_attention(Q, K, V, gq, gk, eps, causal=causal, lib=lib)
            qn = F.rms_norm(torch.tensor(Q), (D,), torch.tensor(gq), eps)
            kn = F.rms_norm(torch.tensor(K), (D,), torch.tensor(gk), eps)
            kr = kn.repeat_interleave(rep, dim=2)
            vr = torch.tensor(V).repeat_interleave(rep, dim=2)
            ref = F.scaled_dot_product_attention(qn.transpose(1, 2), kr.transpose(1, 2),
                                                 vr.transpose(1, 2), is_causal=causal)
            ref = ref.transpose(1, 2).numpy()
            worst = max(worst, float(np.abs(o - ref).max()))
    return (worst <= 1e-12, f"vs torch rms_norm + sdpa: max abs diff {worst:.3e}")


def pin_attn_single_key(lib, seed=42):
    Q, K, V, gq, gk = _attn_problem(_rng(seed))
    B, S, Hq, D = Q.shape
    rep = Hq // K.shape[2]
    o = oracle.qknorm_attention(Q, K, V, gq, gk, 1e-6, causal=True, qpos=[0], lib=lib)
    ref = np.repeat(V[:, 0:1], rep, axis=2)
    return (bool(np.array_equal(o, ref)), "first causal query = V[0] of its group")


def pin_attn_equal_keys(lib, seed=43):
    Q, K, V, gq, gk = _attn_problem(_rng(seed))
    B, S, Hq, D = Q.shape
    rep = Hq // K.shape[2]
    K = np.repeat(K[:, :1], S, axis=1)   # every key equal to the first
    o = oracle.qknorm_attention(Q, K, V, gq, gk, 1e-6, causal=True, lib=lib)
    prefix_mean = np.cumsum(V, axis=1) / np.arange(1, S + 1)[None, :, None, None]
    ref = np.repeat(prefix_mean, rep, axis=2)
    err = float(np.abs(o - ref).max())
    o2 = oracle.qknorm_attention(Q, K, V, gq, gk, 1e-6, causal=False, lib=lib)
    ref2 = np.repeat(np.repeat(V.mean(axis=1, keepdims=True), S, axis=1), rep, axis=2)
    err = max(err, float(np.abs(o2 - ref2).max()))
    return (err <= 1e-13, f"equal keys: max abs diff from the mean {err:.3e}")


def pin_attn_scale_invariance(lib, seed=44):
    Q, K, V, gq, gk = _attn_problem(_rng(seed))
    a = oracle.qknorm_attention(Q, K, V, gq, gk, 0.0, causal=True, lib=lib)
    b = oracle.qknorm_attention(Q * 8.0, K / 32.0, V, gq, gk, 0.0, causal=True, lib=lib)
    return (bool(np.array_equal(a, b)), "row scale removed by the normalisation (bitwise)")


def pin_attn_constant_values(lib, seed=45):
    rng = _rng(seed)
    Q, K, V, gq, gk = _attn_problem(rng)
    c = rng.standard_normal((V.shape[0], 1, V.shape[2], V.shape[3]))
    V = np.repeat(c, V.shape[1], axis=1)
    rep = Q.shape[2] // K.shape[2]
    worst = 0.0
    for causal in (True, False):
        o = oracle.qknorm_attention(Q, K, V, gq, gk, 1e-6, causal=causal, lib=lib)
        ref = np.repeat(V, rep, axis=2)
        worst = max(worst, float(np.abs(o - ref).max()))
    return (worst <= 1e-14, f"constant values: max abs diff {worst:.3e}")


def pin_attn_gqa_is_repeated_mha(lib, seed=46):
    Q, K, V, gq, gk = _attn_problem(_rng(seed))
    rep = Q.shape[2] // K.shape[2]
    g = oracle.qknorm_attention(Q, K, V, gq, gk, 1e-6, causal=True, lib=lib)
    m = oracle.qknorm_attention(Q, np.repeat(K, rep, axis=2), np.repeat(V, rep, axis=2), gq, gk,
                                1e-6, causal=True, lib=lib)
    return (bool(np.array_equal(g, m)), "grouped heads = repeated key/value heads (bitwise)")


def pin_attn_hand_worked(lib):
    # D = 2, unit gains, eps = 0, scale 1/sqrt(2).  Queries (1, -1) and (3, 3)
    # normalise to (1, -1) and (1, 1); keys (2, 2) and (1, -1) to (1, 1) and
    # (1, -1).  Scores: position 0 against keys 0, 1: 0 and sqrt(2); position 1:
    # sqrt(2) and 0.  With V = (1, 0), (0, 4) and e = exp(sqrt(2)):
    #   causal:     O0 = (1, 0),                O1 = (e, 4) / (e + 1)
    #   not causal: O0 = (1, 4e) / (1 + e),     O1 = (e, 4) / (e + 1)
    Q = np.array([[1.0, -1.0], [3.0, 3.0]]).reshape(1, 2, 1, 2)
    K = np.array([[2.0, 2.0], [1.0, -1.0]]).reshape(1, 2, 1, 2)
    V = np.array([[1.0, 0.0], [0.0, 4.0]]).reshape(1, 2, 1, 2)
    one = np.ones(2)
    e = math.exp(math.sqrt(2.0))
    o1 = np.array([e / (e + 1.0), 4.0 / (e + 1.0)])
    want = {True: np.array([[1.0, 0.0], o1]),
            False: np.array([[1.0 / (1.0 + e), 4.0 * e / (1.0 + e)], o1])}
    worst = 0.0
    for causal in (True, False):
        o = oracle.qknorm_attention(Q, K, V, one, one, 0.0, causal=causal, lib=lib)
        worst = max(worst, float(np.abs(o.reshape(2, 2) - want[causal]).max()))
    return (worst <= 1e-15, f"hand-worked case: max abs diff {worst:.3e}")


ALL_PINS = {
    "rewrite_agrees": pin_rewrite_agrees,
    "scale_invariance": pin_scale_invariance,
    "identity_is_rmsnorm": pin_identity_is_rmsnorm,
    "constant_rows": pin_constant_rows,
    "hand_worked": pin_hand_worked,
    "matmul_part": pin_matmul_part,
    "permutations": pin_permutations,
    "gated_zero_gate": pin_gated_zero_gate,
    "gated_odd_part": pin_gated_odd_part,
    "gated_limits": pin_gated_limits,
    "gated_equal_projections": pin_gated_equal_projections,
    "lora_zero_adapter": pin_lora_zero_adapter,
    "lora_adapter_alone": pin_lora_adapter_alone,
    "lora_rank_one": pin_lora_rank_one,
    "attn_library": pin_attn_library,
    "attn_single_key": pin_attn_single_key,
    "attn_equal_keys": pin_attn_equal_keys,
    "attn_scale_invariance": pin_attn_scale_invariance,
    "attn_constant_values": pin_attn_constant_values,
    "attn_gqa_is_repeated_mha": pin_attn_gqa_is_repeated_mha,
    "attn_hand_worked": pin_attn_hand_worked,
}
