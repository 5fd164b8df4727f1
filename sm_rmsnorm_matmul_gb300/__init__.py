"""Python binding of libsm_rmsnorm_matmul.so (GB300 / sm_103a).

Argument marshalling only: tensors are checked (bf16, contiguous, on the
current CUDA device), their data pointers and the current CUDA stream are
passed to the C ABI declared in ``include/rmsnorm_matmul.h``, and a non-zero
status is raised as :class:`RmmError`.  Every step of the computation runs in
the library's kernels; there is no CPU or PyTorch fallback.  If the library
has not been built, the first call raises.

    Y = rmsnorm_matmul(X, g, W, eps)   # RMSNorm(X; g, eps) @ W, fused
    Xn = rmsnorm(X, g, eps)            # unfused pair, for comparison
    C = matmul(A, B)

PyTorch provides device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB_PATH

__all__ = [
    "RmmError", "lib", "rmsnorm_matmul", "rmsnorm_matmul_noalloc", "rmsnorm_matmul_swiglu",
    "rmsnorm_matmul_ex", "rmsnorm_matmul_lora", "WEIGHT_NK", "GATED_SILU", "rmsnorm", "matmul",
    "force_path",
    "dispatch_path", "describe_plan", "device_status", "status_string", "STATUS", "PATH_AUTO",
    "PATH_ROWS", "PATH_SMALL_M", "ABI_FUNCTIONS", "rmsnorm_heads", "qknorm_attention",
    "fold_gain", "rmsnorm_matmul_folded",
]

STATUS = {
    0: "RMM_OK", 1: "RMM_ERR_INVALID_ARG", 2: "RMM_ERR_ALIGNMENT",
    3: "RMM_ERR_UNSUPPORTED_DEVICE", 4: "RMM_ERR_LAUNCH",
    5: "RMM_ERR_DEVICE_TIMEOUT", 6: "RMM_ERR_INTERNAL", 7: "RMM_ERR_SCRATCH_LIMIT",
}
PATH_AUTO, PATH_ROWS, PATH_SMALL_M = 0, 1, 2
WEIGHT_NK, GATED_SILU = 1, 2   # flags of rmsnorm_matmul_ex

# Every function declared in include/rmsnorm_matmul.h and include/qknorm_attention.h.
ABI_FUNCTIONS = ("rmsnorm_matmul", "rmsnorm", "matmul", "rmm_force_path",
                 "rmm_device_status", "rmm_status_string", "rmm_dispatch_path",
                 "rmsnorm_matmul_noalloc", "rmm_describe_plan", "rmsnorm_matmul_swiglu",
                 "rmsnorm_matmul_ex", "rmm_test_hooks", "rmsnorm_matmul_lora",
                 "rmsnorm_heads", "qknorm_attention", "fold_gain", "rmsnorm_matmul_folded")


class RmmError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)}")


_lock = threading.Lock()
_lib = None


def _bind(l: ctypes.CDLL) -> ctypes.CDLL:
    vp, i64, f32, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
    l.rmsnorm_matmul.argtypes = [vp, vp, vp, vp, i64, i64, i64, f32, vp]
    l.rmsnorm_matmul_noalloc.argtypes = [vp, vp, vp, vp, i64, i64, i64, f32, vp]
    l.rmsnorm_matmul_swiglu.argtypes = [vp, vp, vp, vp, i64, i64, i64, f32, vp]
    l.rmsnorm_matmul_ex.argtypes = [vp, vp, vp, vp, i64, i64, i64, f32, ctypes.c_uint, vp]
    l.rmsnorm.argtypes = [vp, vp, vp, i64, i64, f32, vp]
    l.matmul.argtypes = [vp, vp, vp, i64, i64, i64, vp]
    l.fold_gain.argtypes = [vp, vp, vp, i64, i64, vp]
    l.rmsnorm_matmul_folded.argtypes = [vp, vp, vp, i64, i64, i64, f32, vp]
    l.rmm_force_path.argtypes = [i32]
    l.rmm_device_status.argtypes = [vp]
    l.rmm_status_string.argtypes = [i32]
    l.rmm_status_string.restype = ctypes.c_char_p
    l.rmm_dispatch_path.argtypes = [i64, i64, i64]
    l.rmm_describe_plan.argtypes = [i64, i64, i64, i32, ctypes.POINTER(ctypes.c_int)]
    l.rmm_test_hooks.argtypes = [i32, i64]
    l.rmsnorm_matmul_lora.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, f32, vp]
    l.rmsnorm_heads.argtypes = [vp, i64, vp, vp, i64, i64, i64, i64, f32, vp]
    l.qknorm_attention.argtypes = [vp, i64, vp, i64, vp, i64, vp, vp, vp, i64,
                                   i64, i64, i64, i64, i64, f32, f32, i32, vp]
    for name in ("rmsnorm_matmul", "rmsnorm_matmul_noalloc", "rmsnorm_matmul_swiglu", "rmsnorm_matmul_ex",
                 "rmsnorm",
                 "matmul", "rmm_force_path", "rmm_device_status", "rmm_dispatch_path",
                 "rmm_describe_plan", "rmm_test_hooks", "rmsnorm_matmul_lora",
                 "rmsnorm_heads", "qknorm_attention", "fold_gain", "rmsnorm_matmul_folded"):
        getattr(l, name).restype = i32
    return l


def lib(path: str | None = None) -> ctypes.CDLL:
    """The loaded C library.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(
                    f"CUDA library not built ({p} missing): run "
                    "`python -m sm_rmsnorm_matmul_gb300.build` or __graft_entry__.build()")
            _lib = _bind(ctypes.CDLL(p))
        return _lib


def _stream_ptr(stream) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _check_bf16(name, t, ndim):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _raise(code: int, what: str):
    if code != 0:
        raise RmmError(code, what)


def rmsnorm_matmul(X, g, W, eps: float = 1e-6, out=None, stream=None):
    """Y[M,N] = RMSNorm(X[M,K]; g[K], eps) @ W[K,N] in one fused launch (bf16)."""
    import torch
    _check_bf16("X", X, 2)
    _check_bf16("g", g, 1)
    _check_bf16("W", W, 2)
    M, K = X.shape
    if g.shape[0] != K or W.shape[0] != K:
        raise ValueError(f"shape mismatch: X {tuple(X.shape)}, g {tuple(g.shape)}, W {tuple(W.shape)}")
    N = W.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    else:
        _check_bf16("out", out, 2)
        if tuple(out.shape) != (M, N):
            raise ValueError(f"out must have shape {(M, N)}")
    _raise(lib().rmsnorm_matmul(X.data_ptr(), g.data_ptr(), W.data_ptr(), out.data_ptr(),
                                M, K, N, float(eps), _stream_ptr(stream)), "rmsnorm_matmul")
    return out


def rmsnorm_matmul_swiglu(X, g, W, eps: float = 1e-6, out=None, stream=None):
    """Y[M,F] = silu(Z[:, :F]) * Z[:, F:] with Z = RMSNorm(X; g, eps) @ W, W [K, 2F]:
    the gated MLP over the concatenated gate and up projections, one fused launch."""
    import torch
    _check_bf16("X", X, 2)
    _check_bf16("g", g, 1)
    _check_bf16("W", W, 2)
    M, K = X.shape
    if g.shape[0] != K or W.shape[0] != K or W.shape[1] % 2:
        raise ValueError(f"shape mismatch: X {tuple(X.shape)}, g {tuple(g.shape)}, W {tuple(W.shape)}")
    N = W.shape[1]
    F = N // 2
    if out is None:
        out = torch.empty((M, F), dtype=torch.bfloat16, device=X.device)
    else:
        _check_bf16("out", out, 2)
        if tuple(out.shape) != (M, F):
            raise ValueError(f"out must have shape {(M, F)}")
    _raise(lib().rmsnorm_matmul_swiglu(X.data_ptr(), g.data_ptr(), W.data_ptr(), out.data_ptr(),
                                       M, K, N, float(eps), _stream_ptr(stream)),
           "rmsnorm_matmul_swiglu")
    return out


def rmsnorm_matmul_ex(X, g, W, eps: float = 1e-6, weight_nk: bool = False, gated: bool = False,
                      out=None, stream=None):
    """rmsnorm_matmul() with options.  weight_nk: W is [N, K] (a linear layer's
    weight, K contiguous) and Y = RMSNorm(X) @ W.T; gated: Y = silu(Z[:, :F]) *
    Z[:, F:] with F = N / 2, as rmsnorm_matmul_swiglu()."""
    import torch
    _check_bf16("X", X, 2)
    _check_bf16("g", g, 1)
    _check_bf16("W", W, 2)
    M, K = X.shape
    N = W.shape[0] if weight_nk else W.shape[1]
    if g.shape[0] != K or W.shape[1 if weight_nk else 0] != K or (gated and N % 2):
        raise ValueError(f"shape mismatch: X {tuple(X.shape)}, g {tuple(g.shape)}, W {tuple(W.shape)}")
    cols = N // 2 if gated else N
    if out is None:
        out = torch.empty((M, cols), dtype=torch.bfloat16, device=X.device)
    else:
        _check_bf16("out", out, 2)
        if tuple(out.shape) != (M, cols):
            raise ValueError(f"out must have shape {(M, cols)}")
    flags = (WEIGHT_NK if weight_nk else 0) | (GATED_SILU if gated else 0)
    _raise(lib().rmsnorm_matmul_ex(X.data_ptr(), g.data_ptr(), W.data_ptr(), out.data_ptr(),
                                   M, K, N, float(eps), flags, _stream_ptr(stream)), "rmsnorm_matmul_ex")
    return out


def rmsnorm_matmul_lora(X, g, W, A, B, eps: float = 1e-6, out=None, stream=None):
    """Y[M,N] = RMSNorm(X; g, eps) @ (W + A @ B) with a low-rank adapter A [K,R],
    B [R,N] (R <= 64, a multiple of 8)."""
    import torch
    for name, t in (("X", X), ("g", g), ("W", W), ("A", A), ("B", B)):
        _check_bf16(name, t, 1 if name == "g" else 2)
    M, K = X.shape
    N = W.shape[1]
    R = A.shape[1]
    if g.shape[0] != K or W.shape[0] != K or A.shape[0] != K or tuple(B.shape) != (R, N):
        raise ValueError(f"shape mismatch: X {tuple(X.shape)}, W {tuple(W.shape)}, A {tuple(A.shape)}, "
                         f"B {tuple(B.shape)}")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    else:
        _check_bf16("out", out, 2)
        if tuple(out.shape) != (M, N):
            raise ValueError(f"out must have shape {(M, N)}")
    _raise(lib().rmsnorm_matmul_lora(X.data_ptr(), g.data_ptr(), W.data_ptr(), A.data_ptr(), B.data_ptr(),
                                     out.data_ptr(), M, K, N, R, float(eps), _stream_ptr(stream)),
           "rmsnorm_matmul_lora")
    return out


def _check_heads(name, t):
    """A bf16 CUDA tensor [B, S, H, D] whose heads are contiguous and whose
    tokens are a constant stride apart (a column block of a [B*S, width]
    matrix qualifies).  Returns that token stride in elements."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dim() != 4:
        raise ValueError(f"{name} must be [B, S, heads, D], got shape {tuple(t.shape)}")
    B, S, H, D = t.shape
    st = t.stride()
    if st[3] != 1 or (H > 1 and st[2] != D) or (B > 1 and st[0] != S * st[1]):
        raise ValueError(f"{name}: heads must be contiguous and tokens evenly spaced, "
                         f"got strides {st}")
    return st[1] if S > 1 else H * D


def rmsnorm_heads(X, g, eps: float = 1e-6, out=None, stream=None):
    """Y[t,h,:] = RMSNorm(X[t,h,:]; g, eps) over the last dimension for X [T, H, D]
    (heads contiguous, rows evenly spaced)."""
    import torch
    _check_bf16("g", g, 1)
    ldx = _check_heads("X", X.unsqueeze(0))
    T, H, D = X.shape
    if g.shape[0] != D:
        raise ValueError(f"g must have {D} elements")
    if out is None:
        out = torch.empty((T, H, D), dtype=torch.bfloat16, device=X.device)
    ldy = _check_heads("out", out.unsqueeze(0))
    _raise(lib().rmsnorm_heads(X.data_ptr(), ldx, g.data_ptr(), out.data_ptr(), ldy, T, H, D,
                               float(eps), _stream_ptr(stream)), "rmsnorm_heads")
    return out


def qknorm_attention(Q, K, V, gq, gk, eps: float = 1e-6, scale: float | None = None,
                     causal: bool = True, out=None, stream=None):
    """O = softmax(scale * RMSNorm(Q; gq) RMSNorm(K; gk)^T) V per head (causal by
    default), grouped key/value heads.  Q [B,S,Hq,D], K and V [B,S,Hkv,D]; views
    of a fused QKV projection output are accepted as they are.  O [B,S,Hq,D]."""
    import torch
    ldq, ldk, ldv = _check_heads("Q", Q), _check_heads("K", K), _check_heads("V", V)
    _check_bf16("gq", gq, 1)
    _check_bf16("gk", gk, 1)
    B, S, Hq, D = Q.shape
    Hkv = K.shape[2]
    if tuple(K.shape) != (B, S, Hkv, D) or tuple(V.shape) != (B, S, Hkv, D):
        raise ValueError(f"shape mismatch: Q {tuple(Q.shape)}, K {tuple(K.shape)}, V {tuple(V.shape)}")
    if out is None:
        out = torch.empty((B, S, Hq, D), dtype=torch.bfloat16, device=Q.device)
    if tuple(out.shape) != (B, S, Hq, D):
        raise ValueError(f"out must have shape {(B, S, Hq, D)}")
    ldo = _check_heads("out", out)
    _raise(lib().qknorm_attention(Q.data_ptr(), ldq, K.data_ptr(), ldk, V.data_ptr(), ldv,
                                  gq.data_ptr(), gk.data_ptr(), out.data_ptr(), ldo, B, S, Hq, Hkv, D,
                                  float(eps), float(scale or 0.0), int(bool(causal)),
                                  _stream_ptr(stream)), "qknorm_attention")
    return out


def rmsnorm_matmul_noalloc(X, g, W, eps: float = 1e-6, out=None, stream=None):
    """rmsnorm_matmul() for callers that cannot let the library allocate device
    memory during a call (runtimes that own all device memory, fixed budgets,
    latency-critical paths).

    The library allocates nothing: it runs rmsnorm_matmul()'s plan with the
    K-split partial sums in a fixed 20 MiB array inside the library.  `out`
    must be given, since allocating it here would defeat the purpose.  Calls
    that overlap on the GPU share that array and race; a plan whose partials do
    not fit raises RmmError(RMM_ERR_SCRATCH_LIMIT).
    """
    _check_bf16("X", X, 2)
    _check_bf16("g", g, 1)
    _check_bf16("W", W, 2)
    _check_bf16("out", out, 2)
    M, K = X.shape
    N = W.shape[1]
    if g.shape[0] != K or W.shape[0] != K or tuple(out.shape) != (M, N):
        raise ValueError("shape mismatch")
    _raise(lib().rmsnorm_matmul_noalloc(X.data_ptr(), g.data_ptr(), W.data_ptr(), out.data_ptr(),
                                        M, K, N, float(eps), _stream_ptr(stream)),
           "rmsnorm_matmul_noalloc")
    return out


def fold_gain(g, W, out=None, stream=None):
    """Wg[K,N] = bf16(g[k] * W[k,n]): the gain folded into the weights, once,
    for rmsnorm_matmul_folded()."""
    import torch
    _check_bf16("g", g, 1)
    _check_bf16("W", W, 2)
    K, N = W.shape
    if g.shape[0] != K:
        raise ValueError("g must have K elements")
    if out is None:
        out = torch.empty_like(W)
    else:
        _check_bf16("out", out, 2)
        if tuple(out.shape) != (K, N):
            raise ValueError(f"out must have shape {(K, N)}")
    _raise(lib().fold_gain(g.data_ptr(), W.data_ptr(), out.data_ptr(), K, N, _stream_ptr(stream)),
           "fold_gain")
    return out


def rmsnorm_matmul_folded(X, Wg, eps: float = 1e-6, out=None, stream=None):
    """Y[M,N] = bf16(r[m] * (X @ Wg)) with r[m] = rsqrt(mean(X[m]^2) + eps):
    rmsnorm_matmul(X, g, W) for Wg = fold_gain(g, W)."""
    import torch
    _check_bf16("X", X, 2)
    _check_bf16("Wg", Wg, 2)
    M, K = X.shape
    if Wg.shape[0] != K:
        raise ValueError("inner dimensions differ")
    N = Wg.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    else:
        _check_bf16("out", out, 2)
        if tuple(out.shape) != (M, N):
            raise ValueError(f"out must have shape {(M, N)}")
    _raise(lib().rmsnorm_matmul_folded(X.data_ptr(), Wg.data_ptr(), out.data_ptr(), M, K, N, float(eps),
                                       _stream_ptr(stream)), "rmsnorm_matmul_folded")
    return out


def rmsnorm(X, g, eps: float = 1e-6, out=None, stream=None):
    """Xn[M,K] = bf16(X * g * r) (unfused RMSNorm)."""
    import torch
    _check_bf16("X", X, 2)
    _check_bf16("g", g, 1)
    M, K = X.shape
    if g.shape[0] != K:
        raise ValueError("g must have K elements")
    if out is None:
        out = torch.empty_like(X)
    else:
        _check_bf16("out", out, 2)
        if out.shape != X.shape:
            raise ValueError("out must have the shape of X")
    _raise(lib().rmsnorm(X.data_ptr(), g.data_ptr(), out.data_ptr(), M, K, float(eps),
                         _stream_ptr(stream)), "rmsnorm")
    return out


def matmul(A, B, out=None, stream=None):
    """C[M,N] = bf16(A[M,K] @ B[K,N]) with fp32 accumulation (unfused MatMul)."""
    import torch
    _check_bf16("A", A, 2)
    _check_bf16("B", B, 2)
    M, K = A.shape
    if B.shape[0] != K:
        raise ValueError("inner dimensions differ")
    N = B.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    else:
        _check_bf16("out", out, 2)
        if tuple(out.shape) != (M, N):
            raise ValueError(f"out must have shape {(M, N)}")
    _raise(lib().matmul(A.data_ptr(), B.data_ptr(), out.data_ptr(), M, K, N,
                        _stream_ptr(stream)), "matmul")
    return out


def force_path(path: int) -> int:
    """0 auto, 1 row-tile path, 2 small-M path (M <= 16).  Returns the previous value."""
    prev = lib().rmm_force_path(int(path))
    if prev < 0:
        raise ValueError(f"unknown path {path}")
    return prev


PLAN_FIELDS = ("path", "splits", "cluster", "grid", "stages", "MP", "tiles", "kb_per_split")


def describe_plan(M: int, K: int, N: int, fused: bool = True, gated: bool = False) -> dict:
    """The launch plan for this shape on the current device (no launch).
    gated: the plan of rmsnorm_matmul_swiglu (N is then the width of W)."""
    info = (ctypes.c_int * 8)()
    _raise(lib().rmm_describe_plan(M, K, N, 2 if gated else int(fused), info), "rmm_describe_plan")
    return dict(zip(PLAN_FIELDS, list(info)))


def dispatch_path(M: int, K: int, N: int) -> int:
    return int(lib().rmm_dispatch_path(M, K, N))


def device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the in-kernel status."""
    return int(lib().rmm_device_status(_stream_ptr(stream)))


def status_string(code: int) -> str:
    return lib().rmm_status_string(int(code)).decode()
