"""fp64 CPU oracle for RMSNorm followed by MatMul.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` leg / ``--impl reference`` arm of ``bench.py`` may import
or run anything in this package.  The CUDA library (``sm_rmsnorm_matmul_gb300``)
never imports it, and this package imports nothing from the CUDA library.

The arithmetic lives in ``rmm_oracle.c`` (plain C, fp64, OpenMP over rows),
compiled with ``-ffp-contract=off`` so that no multiply-add is fused and x86
and Arm hosts round identically.  This module only builds it, decodes bf16
bit patterns exactly to float64, and marshals numpy arrays.

Pins (tests/test_oracle_pins.py): the finite-field identity behind the
rewrite, the rewritten and unfused forms agreeing, scale invariance,
W = identity against torch's RMSNorm, constant rows against a closed form, a
hand-worked 2x3x2 example, and the matmul part against numpy.  The gated
form is pinned by a zero gate giving zero, the exact odd part of SiLU
(Y(W_gate) - Y(-W_gate) = Z_gate * Z_up), its two limits, and Y >= 0 when the
gate and up projections coincide.  The LoRA form is pinned by a zero adapter
giving the plain result bitwise, a zero W against the associativity of
(RMSNorm(X) @ A) @ B in numpy, and a rank-one adapter against its closed form.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "rmm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

CFLAGS = ["-O3", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off", "-std=c11"]

_lock = threading.Lock()
_lib = None


def build(source: str = SOURCE, out: str = LIB_PATH, force: bool = False) -> str:
    """Compile the oracle with gcc; returns the path of the shared object."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(source)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, source, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    dp = ctypes.POINTER(ctypes.c_double)
    L, D, I = ctypes.c_long, ctypes.c_double, ctypes.c_int
    lib.oracle_rmsnorm.argtypes = [dp, dp, dp, L, L, D, I]
    lib.oracle_matmul.argtypes = [dp, dp, dp, L, L, L, I]
    lib.oracle_rmsnorm_matmul.argtypes = [dp, dp, dp, dp, L, L, L, D, I]
    lib.oracle_rmsnorm_matmul_rewritten.argtypes = [dp, dp, dp, dp, L, L, L, D, I]
    lib.oracle_rmsnorm_matmul_swiglu.argtypes = [dp, dp, dp, dp, L, L, L, D, I]
    lib.oracle_rmsnorm_matmul_lora.argtypes = [dp, dp, dp, dp, dp, dp, L, L, L, L, D, I]
    lp = ctypes.POINTER(ctypes.c_long)
    lib.oracle_attention.argtypes = [dp, dp, dp, dp, L, L, L, L, L, D, I, lp, L, I]
    lib.oracle_qknorm_attention.argtypes = [dp, dp, dp, dp, dp, dp, L, L, L, L, L, D, D, I,
                                            lp, L, I]
    for f in (lib.oracle_rmsnorm, lib.oracle_matmul, lib.oracle_rmsnorm_matmul,
              lib.oracle_rmsnorm_matmul_rewritten, lib.oracle_rmsnorm_matmul_swiglu,
              lib.oracle_rmsnorm_matmul_lora, lib.oracle_attention, lib.oracle_qknorm_attention,
              lib.oracle_max_threads):
        f.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = []
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Decode bf16 bit patterns (uint16/int16 array) exactly to float64."""
    b = np.ascontiguousarray(np.asarray(bits).view(np.uint16))
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_f64(t) -> np.ndarray:
    """A bf16 torch tensor, or any numeric array, as a contiguous float64 array.

    bf16 tensors are decoded from their bit patterns, not through torch's
    dtype conversion.
    """
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu()
            if t.dtype == torch.bfloat16:
                return bf16_bits_to_f64(t.contiguous().view(torch.int16).numpy())
            return np.ascontiguousarray(t.numpy(), dtype=np.float64)
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(t, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def rmsnorm_matmul(X, g, W, eps: float, nthreads: int = 0, lib=None) -> np.ndarray:
    """Y = RMSNorm(X; g, eps) @ W in fp64 (unfused definition)."""
    lib = lib or load()
    X, g, W = to_f64(X), to_f64(g), to_f64(W)
    M, K = X.shape
    K2, N = W.shape
    assert K == K2 and g.shape == (K,)
    Y = np.empty((M, N), dtype=np.float64)
    _check(lib.oracle_rmsnorm_matmul(_ptr(X), _ptr(g), _ptr(W), _ptr(Y), M, K, N,
                                     float(eps), nthreads), "rmsnorm_matmul")
    return Y


def rmsnorm_matmul_rewritten(X, g, W, eps: float, nthreads: int = 0, lib=None) -> np.ndarray:
    """Y = ((X*g) @ W) * r in fp64: the division moved past the K-sum."""
    lib = lib or load()
    X, g, W = to_f64(X), to_f64(g), to_f64(W)
    M, K = X.shape
    N = W.shape[1]
    Y = np.empty((M, N), dtype=np.float64)
    _check(lib.oracle_rmsnorm_matmul_rewritten(_ptr(X), _ptr(g), _ptr(W), _ptr(Y),
                                               M, K, N, float(eps), nthreads),
           "rmsnorm_matmul_rewritten")
    return Y


def rmsnorm_matmul_swiglu(X, g, W, eps: float, nthreads: int = 0, lib=None) -> np.ndarray:
    """Y = silu(Z[:, :F]) * Z[:, F:] with Z = RMSNorm(X; g, eps) @ W, W [K, 2F], in fp64."""
    lib = lib or load()
    X, g, W = to_f64(X), to_f64(g), to_f64(W)
    M, K = X.shape
    N = W.shape[1]
    Y = np.empty((M, N // 2), dtype=np.float64)
    _check(lib.oracle_rmsnorm_matmul_swiglu(_ptr(X), _ptr(g), _ptr(W), _ptr(Y), M, K, N,
                                            float(eps), nthreads), "rmsnorm_matmul_swiglu")
    return Y


def rmsnorm_matmul_lora(X, g, W, A, B, eps: float, nthreads: int = 0, lib=None) -> np.ndarray:
    """Y = RMSNorm(X; g, eps) @ (W + A @ B) in fp64; A [K, R], B [R, N]."""
    lib = lib or load()
    X, g, W, A, B = to_f64(X), to_f64(g), to_f64(W), to_f64(A), to_f64(B)
    M, K = X.shape
    N = W.shape[1]
    R = A.shape[1]
    assert A.shape == (K, R) and B.shape == (R, N)
    Y = np.empty((M, N), dtype=np.float64)
    _check(lib.oracle_rmsnorm_matmul_lora(_ptr(X), _ptr(g), _ptr(W), _ptr(A), _ptr(B), _ptr(Y),
                                          M, K, N, R, float(eps), nthreads), "rmsnorm_matmul_lora")
    return Y


def rmsnorm(X, g, eps: float, nthreads: int = 0, lib=None) -> np.ndarray:
    """Xn = X * g * r in fp64."""
    lib = lib or load()
    X, g = to_f64(X), to_f64(g)
    M, K = X.shape
    Xn = np.empty((M, K), dtype=np.float64)
    _check(lib.oracle_rmsnorm(_ptr(X), _ptr(g), _ptr(Xn), M, K, float(eps), nthreads),
           "rmsnorm")
    return Xn


def matmul(A, B, nthreads: int = 0, lib=None) -> np.ndarray:
    """C = A @ B in fp64 (triple loop)."""
    lib = lib or load()
    A, B = to_f64(A), to_f64(B)
    M, K = A.shape
    N = B.shape[1]
    C = np.empty((M, N), dtype=np.float64)
    _check(lib.oracle_matmul(_ptr(A), _ptr(B), _ptr(C), M, K, N, nthreads), "matmul")
    return C


def _heads(t, name):
    a = to_f64(t)
    if a.ndim != 4:
        raise ValueError(f"{name} must be [B, S, heads, D]")
    return np.ascontiguousarray(a)


def _positions(qpos, S):
    if qpos is None:
        return None, S
    q = np.ascontiguousarray(np.asarray(qpos, dtype=np.int64)).astype(ctypes.c_long)
    return q, len(q)


def attention(Q, K, V, scale: float, causal: bool = True, qpos=None, nthreads: int = 0,
              lib=None) -> np.ndarray:
    """Scaled dot-product attention in fp64.  Q [B,S,Hq,D], K and V [B,S,Hkv,D];
    returns O [B, len(qpos) or S, Hq, D] for the query positions qpos."""
    lib = lib or load()
    Q, K, V = _heads(Q, "Q"), _heads(K, "K"), _heads(V, "V")
    B, S, Hq, D = Q.shape
    Hkv = K.shape[2]
    assert K.shape == (B, S, Hkv, D) and V.shape == K.shape
    q, nq = _positions(qpos, S)
    O = np.empty((B, nq, Hq, D), dtype=np.float64)
    qp = q.ctypes.data_as(ctypes.POINTER(ctypes.c_long)) if q is not None else None
    _check(lib.oracle_attention(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), B, S, Hq, Hkv, D,
                                float(scale), int(bool(causal)), qp, nq, nthreads), "attention")
    return O


def qknorm_attention(Q, K, V, gq, gk, eps: float, scale: float | None = None,
                     causal: bool = True, qpos=None, nthreads: int = 0, lib=None) -> np.ndarray:
    """RMSNorm(Q; gq) and RMSNorm(K; gk) over the head dimension, then
    attention with scale 1/sqrt(D) unless given; fp64."""
    lib = lib or load()
    Q, K, V = _heads(Q, "Q"), _heads(K, "K"), _heads(V, "V")
    gq, gk = to_f64(gq), to_f64(gk)
    B, S, Hq, D = Q.shape
    Hkv = K.shape[2]
    assert K.shape == (B, S, Hkv, D) and V.shape == K.shape
    assert gq.shape == (D,) and gk.shape == (D,)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    q, nq = _positions(qpos, S)
    O = np.empty((B, nq, Hq, D), dtype=np.float64)
    qp = q.ctypes.data_as(ctypes.POINTER(ctypes.c_long)) if q is not None else None
    _check(lib.oracle_qknorm_attention(_ptr(Q), _ptr(K), _ptr(V), _ptr(gq), _ptr(gk), _ptr(O),
                                       B, S, Hq, Hkv, D, float(eps), float(scale),
                                       int(bool(causal)), qp, nq, nthreads), "qknorm_attention")
    return O


def max_threads(lib=None) -> int:
    return int((lib or load()).oracle_max_threads())


def tolerance_violations(y, y_ref, atol: float = 1e-2, rtol: float = 1e-2):
    """Element-wise check |y - y_ref| <= atol + rtol*|y_ref|; NaN/Inf fail.

    Returns (violations, max_abs_err, max_rel_err).
    """
    y = to_f64(y)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    err = np.abs(y - y_ref)
    bad = ~np.isfinite(y) | (err > atol + rtol * np.abs(y_ref))
    rel = err / np.maximum(np.abs(y_ref), 1e-30)
    finite = np.isfinite(err)
    max_abs = float(err[finite].max()) if finite.any() else float("nan")
    max_rel = float(rel[finite].max()) if finite.any() else float("nan")
    return int(bad.sum()), max_abs, max_rel
