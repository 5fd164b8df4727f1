"""QK-normalised attention on the GPU against the fp64 oracle, through the C ABI.

The device multiplies the raw bf16 queries with keys normalised once and
multiplied by the query gain, Kg = bf16(RMSNorm(K; gk) * gq) (the only
operand rounding), and scales each query row's scores by its 1/RMS times
scale * log2(e) in fp32.  The reference applies the same rounding to the
oracle's own RMSNorm (fp64), takes the queries as Q * r * scale * log2(e)
unrounded, and runs the oracle's fp64 attention with base-2 exponentials
(scale ln 2), so that what is left to compare is the device's softmax and
products.  What remains on the device side, per output element, and the
bound used here:

  * P rounded to bf16 (relative 2^-9 per weight), ex2.approx (relative ~2^-22),
    fp32 scores and sums, and the rare key element whose fp32 statistic put
    it on the other side of a rounding boundary: together below
    2^-8 * sum_j p_j |v_jd|;
  * O rounded to bf16 once: 2^-9 |o|, taken as 2^-8 |o|.

  |O - O_ref| <= 2^-8 * sum_j p_j |v_jd| + 2^-8 |O_ref| + 1e-5

sum_j p_j |v_jd| is the oracle's attention with |V| as the values.  A second
check compares with the fully exact oracle (no rounding anywhere) under the
first-order bound of the key rounding.
"""
import math

import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

LN2 = math.log(2.0)
LOG2E = 1.0 / LN2


@pytest.fixture(scope="module")
def rmm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sm_rmsnorm_matmul_gb300 as m
    m.lib()
    return m


def bf16_round(x):
    """fp64 -> fp32 -> bf16 (nearest even) -> fp64: the device computes its
    operands in fp32 and rounds them once."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.float32).to(torch.bfloat16).double().numpy()


def references(Q, K, V, gq, gk, eps, causal, qpos=None, scale=None):
    B, S, Hq, D = Q.shape
    Hkv = K.shape[2]
    c = (1.0 / math.sqrt(D) if scale is None else scale) * LOG2E
    qr = oracle.rmsnorm(Q.reshape(-1, D), np.ones(D), eps).reshape(B, S, Hq, D)   # Q * r
    kn = oracle.rmsnorm(K.reshape(-1, D), gk, eps).reshape(B, S, Hkv, D)
    qd = qr * c
    kd = bf16_round(kn * oracle.to_f64(gq))
    Vf = oracle.to_f64(V)
    ref = oracle.attention(qd, kd, Vf, LN2, causal=causal, qpos=qpos)
    wabs = oracle.attention(qd, kd, np.abs(Vf), LN2, causal=causal, qpos=qpos)
    qn = qr * oracle.to_f64(gq)
    return ref, wabs, qn, kn


def assert_attention_close(O, Q, K, V, gq, gk, eps, causal, what, qpos=None, scale=None):
    ref, wabs, qn, kn = references(Q, K, V, gq, gk, eps, causal, qpos, scale=scale)
    o = oracle.to_f64(O)
    if qpos is not None:
        o = o[:, qpos]
    tol = 2.0 ** -8 * wabs + 2.0 ** -8 * np.abs(ref) + 1e-5
    err = np.abs(o - ref)
    bad = ~(err <= tol)   # NaN fails
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {ref.size} outside the bound, "
                           f"max err {float(np.nanmax(err)):.3e}")
    # The exact oracle (no rounding anywhere).  The reference differs from it
    # only in the keys: kd = bf16(fp32(kn * gq)) is within (2^-9 + 2^-23) of
    # kn * gq relatively (one fp32 and one bf16 rounding to nearest), so every
    # score moves by |delta_j| <= Delta = (2^-9 + 2^-23) * scale *
    # sum_d |qn_d| max_j |kn_jd|.  Each softmax weight then changes by the
    # factor e^delta_j / sum_i p_i e^delta_i, within [e^-2Delta, e^2Delta], so
    # |p'_j - p_j| <= (e^2Delta - 1) p_j <= (e^2Delta - 1) e^2Delta p'_j and
    # |O_ref - O_exact| <= (e^2Delta - 1) e^2Delta sum_j p'_j |v_jd|, where
    # sum_j p'_j |v_jd| is wabs (the reference's weights).  No first-order
    # step: the bound holds for any Delta.
    exact = oracle.qknorm_attention(Q, K, V, gq, gk, eps, scale=scale, causal=causal, qpos=qpos)
    rep = Q.shape[2] // K.shape[2]
    qs = np.abs(qn if qpos is None else qn[:, qpos])
    ks = np.repeat(np.abs(kn), rep, axis=2).max(axis=1, keepdims=True)
    c = (1.0 / math.sqrt(Q.shape[3]) if scale is None else scale)
    delta = (2.0 ** -9 + 2.0 ** -23) * c * (qs * ks).sum(axis=3, keepdims=True)
    tol_e = tol + np.expm1(2 * delta) * np.exp(2 * delta) * wabs
    bad = ~(np.abs(o - exact) <= tol_e)
    assert not bad.any(), f"{what}: {int(bad.sum())} outside the bound of the exact oracle"


def run(rmm, B, S, Hq, Hkv, causal, seed, eps=1e-6, D=128, qkv=None):
    from sm_rmsnorm_matmul_gb300 import inputs
    if qkv is None:
        qkv, gq, gk = inputs.attention_inputs(B, S, Hq, Hkv, D, seed)
    else:
        _, gq, gk = inputs.attention_inputs(B, 1, Hq, Hkv, D, seed)
    Q, K, V = inputs.split_qkv(qkv, B, S, Hq, Hkv, D)
    Qd, Kd, Vd = inputs.split_qkv(qkv.cuda(), B, S, Hq, Hkv, D)
    O = rmm.qknorm_attention(Qd, Kd, Vd, gq.cuda(), gk.cuda(), eps, causal=causal)
    torch.cuda.synchronize()
    assert rmm.device_status() == 0
    return O.cpu(), Q, K, V, gq, gk


ATTN = [
    # (B, S, Hq, Hkv, causal)
    (1, 256, 4, 2, True),      # two query tiles, two key tiles, diagonal masks
    (2, 300, 4, 1, True),      # ragged sequence, two sequences, four query heads per key head
    (1, 200, 2, 2, False),     # full attention over a ragged last key tile
    (1, 1, 2, 1, True),        # one token
    (1, 1100, 2, 1, True),     # nine key tiles
    (3, 130, 8, 8, False),     # multi-head, full, two tiles with a 2-key tail
]


@pytest.mark.parametrize("B,S,Hq,Hkv,causal", ATTN)
def test_qknorm_attention(rmm, B, S, Hq, Hkv, causal):
    O, Q, K, V, gq, gk = run(rmm, B, S, Hq, Hkv, causal, seed=B * 1000 + S + Hq)
    assert_attention_close(O, Q, K, V, gq, gk, 1e-6, causal, f"attention {B}x{S} {Hq}/{Hkv}")


ATTN_D64 = [
    # (B, S, Hq, Hkv, causal), head dimension 64
    (1, 256, 4, 2, True),
    (2, 300, 4, 1, True),      # ragged, two sequences, 4:1 grouping
    (1, 200, 2, 2, False),     # full attention, ragged last key tile
    (1, 1100, 2, 1, True),     # nine key tiles
]


@pytest.mark.parametrize("B,S,Hq,Hkv,causal", ATTN_D64)
def test_qknorm_attention_head_dim_64(rmm, B, S, Hq, Hkv, causal):
    O, Q, K, V, gq, gk = run(rmm, B, S, Hq, Hkv, causal, seed=B * 977 + S + Hq, D=64)
    assert_attention_close(O, Q, K, V, gq, gk, 1e-6, causal, f"D=64 attention {B}x{S} {Hq}/{Hkv}")


@pytest.mark.parametrize("gain_scale", [1.0, 2.5])
def test_first_causal_row_is_first_value(rmm, gain_scale):
    """One visible key: softmax weight 1, O = V[0].  With the scores' bound as
    the reference (gains U(0.5, 1.5)) the weight is 2^(s - bound), rounded to
    bf16 for P V but summed unrounded, so O is V[0] within one bf16 unit in
    the last place; with a running maximum (gains 2.5 times larger) the
    weight is 2^0 = 1 and O = V[0] exactly."""
    from sm_rmsnorm_matmul_gb300 import inputs
    B, S, Hq, Hkv, D = 1, 64, 4, 2, 128
    qkv, gq, gk = inputs.attention_inputs(B, S, Hq, Hkv, D, 9)
    gq = (gq.float() * gain_scale).to(torch.bfloat16)
    gk = (gk.float() * gain_scale).to(torch.bfloat16)
    _, _, V = inputs.split_qkv(qkv, B, S, Hq, Hkv, D)
    Qd, Kd, Vd = inputs.split_qkv(qkv.cuda(), B, S, Hq, Hkv, D)
    O = rmm.qknorm_attention(Qd, Kd, Vd, gq.cuda(), gk.cuda(), 1e-6, causal=True).cpu()
    torch.cuda.synchronize()
    assert rmm.device_status() == 0
    want = V[:, 0].repeat_interleave(Hq // Hkv, dim=1)
    if gain_scale == 1.0:
        assert torch.allclose(O[:, 0].float(), want.float(), rtol=2.0 ** -7, atol=0.0)
    else:
        assert torch.equal(O[:, 0], want)


@pytest.mark.parametrize("D,gain", [(128, 1.5), (64, 1.5), (128, 1.7265625), (64, 2.046875),
                                    (128, 2.5), (64, 2.5)])
def test_rescaled_rows(rmm, D, gain):
    # every query of a head equals one direction u and so does one late key:
    # that key's score dwarfs the first tile's by far more than 2^8.  With
    # gains of 1.5 the scores' bound (scale * log2(e) * D * gain^2, times
    # 1 + 1/64) is at most 50 and serves as the softmax reference: the
    # weights span ~2^-70 .. 1.  Gains of 1.7265625 (D = 128) and 2.046875
    # (D = 64) put the bound just below 50 (49.4, 49.1): rows that see only
    # the opposite keys have every weight near 2^-98, the smallest the
    # bound allows.  With gains of 2.5 the bound is too loose, the kernel
    # keeps a running maximum and the accumulator is rescaled (for D = 64
    # after the previous tile's P V, which P apart from S lets run late,
    # completes)
    bound = (1.0 / D ** 0.5) * 1.4426950408889634 * D * gain * gain * (1 + 1 / 64)
    assert (bound <= 50.0) == (gain < 2.1)
    from sm_rmsnorm_matmul_gb300 import inputs
    B, S, Hq, Hkv = 1, 700, 2, 1
    qkv, gq, gk = inputs.attention_inputs(B, S, Hq, Hkv, D, 21)
    gq = torch.full((D,), gain, dtype=torch.bfloat16)
    gk = torch.full((D,), gain, dtype=torch.bfloat16)
    t = qkv.view(B * S, Hq + 2 * Hkv, D)
    u = torch.randn(D, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    t[:, 0] = u
    t[:, 1] = -u
    t[:, Hq] = -u                   # every key points away ...
    t[450, Hq] = u                  # ... except one, late in the sequence
    t[451:, Hq] = torch.randn(S - 451, D, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    Q, K, V = inputs.split_qkv(qkv, B, S, Hq, Hkv, D)
    Qd, Kd, Vd = inputs.split_qkv(qkv.cuda(), B, S, Hq, Hkv, D)
    O = rmm.qknorm_attention(Qd, Kd, Vd, gq.cuda(), gk.cuda(), 1e-6, causal=True)
    torch.cuda.synchronize()
    assert rmm.device_status() == 0
    assert_attention_close(O.cpu(), Q, K, V, gq, gk, 1e-6, True, "rescaled rows")


def test_explicit_scale_and_eps(rmm):
    from sm_rmsnorm_matmul_gb300 import inputs
    B, S, Hq, Hkv, D = 1, 150, 2, 1, 128
    qkv, gq, gk = inputs.attention_inputs(B, S, Hq, Hkv, D, 33)
    Q, K, V = inputs.split_qkv(qkv, B, S, Hq, Hkv, D)
    Qd, Kd, Vd = inputs.split_qkv(qkv.cuda(), B, S, Hq, Hkv, D)
    O = rmm.qknorm_attention(Qd, Kd, Vd, gq.cuda(), gk.cuda(), 0.25, scale=1.0 / 16, causal=False)
    torch.cuda.synchronize()
    assert rmm.device_status() == 0
    assert_attention_close(O.cpu(), Q, K, V, gq, gk, 0.25, False, "explicit scale and eps", scale=1.0 / 16)


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("B,S,Hq,Hkv,causal", [
    (2, 2048, 16, 4, False),   # full attention, two sequences
    (1, 3000, 32, 8, True),    # ragged length: the last block half past the end, a partial last band
])
def test_large_sampled_rows(rmm, B, S, Hq, Hkv, causal, D):
    """Several blocks per CTA: the key stream, the score buffer and (D = 64)
    the P columns carry over from one block to the next."""
    from sm_rmsnorm_matmul_gb300 import inputs
    qkv, gq, gk = inputs.attention_inputs(B, S, Hq, Hkv, D, seed=S + Hq)
    Q, K, V = inputs.split_qkv(qkv, B, S, Hq, Hkv, D)
    Qd, Kd, Vd = inputs.split_qkv(qkv.cuda(), B, S, Hq, Hkv, D)
    O = rmm.qknorm_attention(Qd, Kd, Vd, gq.cuda(), gk.cuda(), 1e-6, causal=causal)
    torch.cuda.synchronize()
    assert rmm.device_status() == 0
    qpos = sorted({0, 127, 128, 255, 256, S - 129, S - 128, S - 1} | set(inputs.sample_rows(S, 24)))
    assert_attention_close(O.cpu(), Q, K, V, gq, gk, 1e-6, causal, f"{B}x{S} {Hq}/{Hkv}", qpos=qpos)


@pytest.mark.parametrize("D", [128, 64])
def test_running_maximum_sampled_rows(rmm, D):
    """Gains of 1.25 .. 3.75 make the scores' bound too loose to serve as the
    softmax reference: the running maximum across several blocks per CTA."""
    from sm_rmsnorm_matmul_gb300 import inputs
    B, S, Hq, Hkv, causal = 1, 3000, 32, 8, True
    qkv, gq, gk = inputs.attention_inputs(B, S, Hq, Hkv, D, seed=S + D)
    gq = (gq.float() * 2.5).to(torch.bfloat16)
    gk = (gk.float() * 2.5).to(torch.bfloat16)
    Q, K, V = inputs.split_qkv(qkv, B, S, Hq, Hkv, D)
    Qd, Kd, Vd = inputs.split_qkv(qkv.cuda(), B, S, Hq, Hkv, D)
    O = rmm.qknorm_attention(Qd, Kd, Vd, gq.cuda(), gk.cuda(), 1e-6, causal=causal)
    torch.cuda.synchronize()
    assert rmm.device_status() == 0
    qpos = sorted({0, 127, 128, 255, 256, S - 129, S - 128, S - 1} | set(inputs.sample_rows(S, 24)))
    assert_attention_close(O.cpu(), Q, K, V, gq, gk, 1e-6, causal, f"running maximum D={D}", qpos=qpos)


def test_output_row_stride(rmm):
    # O written into the first Hq * D columns of a wider buffer (row stride
    # Hq * D + 64): the same values as a dense output, the padding untouched
    from sm_rmsnorm_matmul_gb300 import inputs
    B, S, Hq, Hkv, D = 2, 300, 4, 2, 128
    qkv, gq, gk = inputs.attention_inputs(B, S, Hq, Hkv, D, 61)
    Qd, Kd, Vd = inputs.split_qkv(qkv.cuda(), B, S, Hq, Hkv, D)
    dense = rmm.qknorm_attention(Qd, Kd, Vd, gq.cuda(), gk.cuda(), 1e-6, causal=True)
    wide = torch.full((B * S, Hq * D + 64), 7.0, dtype=torch.bfloat16, device="cuda")
    view = wide[:, :Hq * D].view(B, S, Hq, D)
    rmm.qknorm_attention(Qd, Kd, Vd, gq.cuda(), gk.cuda(), 1e-6, causal=True, out=view)
    torch.cuda.synchronize()
    assert rmm.device_status() == 0
    assert torch.equal(view.cpu(), dense.cpu())
    assert bool((wide[:, Hq * D:] == 7.0).all())


@pytest.mark.parametrize("name", ["prefill_attention_1x4096_h32_kv8_d128_causal",
                                  "prefill_attention_1x4096_h32_kv8_d64_causal"])
def test_full_size_sampled_rows(rmm, name):
    # the benchmark's workloads (one 4096-token sequence, 32 query heads over
    # 8 key/value heads, causal), sampled query positions checked one by one
    from sm_rmsnorm_matmul_gb300 import inputs
    w = inputs.ATTENTION_WORKLOADS[name]
    qkv, gq, gk = inputs.attention_inputs(w.B, w.S, w.Hq, w.Hkv, w.D, w.seed)
    Q, K, V = inputs.split_qkv(qkv, w.B, w.S, w.Hq, w.Hkv, w.D)
    Qd, Kd, Vd = inputs.split_qkv(qkv.cuda(), w.B, w.S, w.Hq, w.Hkv, w.D)
    O = rmm.qknorm_attention(Qd, Kd, Vd, gq.cuda(), gk.cuda(), w.eps, causal=w.causal)
    torch.cuda.synchronize()
    assert rmm.device_status() == 0
    qpos = sorted({0, 1, 127, 128, 129, 2047, 2048, 4094, 4095} |
                  set(inputs.sample_rows(w.S, 24)))
    assert_attention_close(O.cpu(), Q, K, V, gq, gk, w.eps, w.causal, "full size", qpos=qpos)


@pytest.mark.parametrize("T,H,D,pad", [
    (333, 2, 128, 0),     # one warp per row (two heads of 128)
    (130, 8, 128, 16),    # eight heads, row stride wider than the heads
    (64, 8, 256, 0),      # the widest row the one-warp kernel takes (8 chunks per lane)
    (77, 5, 64, 8),
    (50, 3, 96, 0),       # D not a power of two: one warp per head
    (20, 40, 64, 0),      # a row too wide for one warp: one warp per head
])
def test_rmsnorm_heads_matches_oracle(rmm, T, H, D, pad):
    g = torch.Generator().manual_seed(T + H + D)
    X = (torch.randn(T, H * D + pad, generator=g) * torch.exp(torch.randn(T, 1, generator=g))).to(torch.bfloat16)
    gain = (0.5 + torch.rand(D, generator=g)).to(torch.bfloat16)
    Xv = X[:, :H * D].view(T, H, D)
    Y = rmm.rmsnorm_heads(X.cuda()[:, :H * D].view(T, H, D), gain.cuda(), 1e-6).cpu()
    assert rmm.device_status() == 0
    ref = oracle.rmsnorm(Xv.reshape(-1, D), gain, 1e-6).reshape(T, H, D)
    y = oracle.to_f64(Y)
    # one rounding of an fp32 value: the nearest bf16 or, at a boundary, its neighbour
    assert (np.abs(y - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-30).all()
    same = (y == bf16_round(ref)).mean()
    assert same > 0.99, same
