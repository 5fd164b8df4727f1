/*
 * qknorm_attention.h -- C ABI of the QK-normalised attention path on GB300
 * (sm_103a): per-head RMSNorm of queries and keys fused with causal or full
 * softmax attention over grouped key/value heads.
 *
 * The operation is the "QKNorm + Attention" workload of the Mirage review
 * page's benchmark table (section 5, "experimental results"); the pages give
 * it no formula.  Read here as the query/key normalisation of recent decoder
 * models: for batch b, position i, query head h and its key/value head
 * c = h / (Hq / Hkv),
 *
 *   Qn[b,i,h,:] = Q[b,i,h,:] * gq[:] / sqrt(mean_d Q[b,i,h,d]^2 + eps)
 *   Kn[b,j,c,:] = K[b,j,c,:] * gk[:] / sqrt(mean_d K[b,j,c,d]^2 + eps)
 *   s_j         = scale * <Qn[b,i,h,:], Kn[b,j,c,:]>      j < S (j <= i if causal)
 *   O[b,i,h,:]  = sum_j softmax(s)_j * V[b,j,c,:]
 *
 * Tensors are bf16 on the current device.  A tensor "[B, S, H, D] with row
 * stride ld" holds element (b, s, h, d) at index (b*S + s)*ld + h*D + d: the
 * heads of one token are contiguous, tokens are ld elements apart.  The
 * query, key and value column blocks of a fused QKV projection output
 * [B*S, (Hq + 2*Hkv)*D] are such tensors (ld = (Hq + 2*Hkv)*D, offsets 0,
 * Hq*D and (Hq + Hkv)*D).  The library never takes ownership of a pointer.
 *
 * Return values are the rmm_status codes of rmsnorm_matmul.h; in-kernel
 * timeouts are reported by rmm_device_status().
 */
#ifndef SM_RMSNORM_MATMUL_QKNORM_ATTENTION_H
#define SM_RMSNORM_MATMUL_QKNORM_ATTENTION_H

#include <stdint.h>

#include "rmsnorm_matmul.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Per-head RMSNorm over the last dimension:
 *   Y[t,h,:] = bf16( X[t,h,:] * g[:] / sqrt(mean_d X[t,h,d]^2 + eps) )
 * for T rows t of H heads of D elements; X row stride ldx, Y row stride ldy
 * (elements).  Statistic and products in fp32, one rounding to bf16.
 * D a multiple of 8, 8 <= D <= 256; ldx, ldy >= H*D and multiples of 8;
 * X, g, Y 16-byte aligned (RMM_ERR_ALIGNMENT otherwise); Y may not overlap X
 * or g; eps finite and >= 0.  T = 0 is a no-op.  Asynchronous on `stream`.
 */
int rmsnorm_heads(const void* X, int64_t ldx, const void* g, void* Y, int64_t ldy,
                  int64_t T, int64_t H, int64_t D, float eps, cudaStream_t stream);

/*
 * QK-normalised attention (formula above).  Q and O are [B, S, Hq, D] with
 * row strides ldq and ldo, K and V [B, S, Hkv, D] with ldk and ldv; gq and gk
 * are [D].  scale <= 0 selects 1/sqrt(D).  causal != 0 restricts query i to
 * keys j <= i.
 *
 * Requirements: D = 64 or 128; Hq a multiple of Hkv; every ld a multiple of 8 and
 * at least the width of its tensor's heads; all pointers 16-byte aligned;
 * O may not overlap any input.  B = 0 or S = 0 is a no-op.
 *
 * Device arithmetic: the keys are normalised once, with both gains, into a
 * library workspace, Kg = bf16(RMSNorm(K; gk) * gq) (per device and stream,
 * grown on demand; a growing call synchronises the stream and may not run
 * under stream capture).  The raw bf16 queries enter the tensor cores, and
 * each query row's scores are multiplied by its 1/RMS times scale * log2(e)
 * in fp32 (the query normalisation is a row scale of the scores), so Kg is
 * the only rounded operand.  Scores accumulate in fp32 in tensor memory, the
 * softmax weights are rounded to bf16 for the second product, the output
 * accumulates in fp32 and is rounded once.  The softmax subtracts, per query
 * row, a reference no smaller than (about) its largest score: the row's
 * Cauchy-Schwarz bound on its scores when the gains keep every such bound at
 * most 50 (log2 units, scale * log2(e) * D * max_i |gq_i gk_i|), so that no
 * weight falls below 2^-100, else a running maximum.  Two kernel launches on `stream`:
 * the key pass and a persistent attention kernel (one CTA per SM).
 */
int qknorm_attention(const void* Q, int64_t ldq, const void* K, int64_t ldk, const void* V,
                     int64_t ldv, const void* gq, const void* gk, void* O, int64_t ldo,
                     int64_t B, int64_t S, int64_t Hq, int64_t Hkv, int64_t D, float eps,
                     float scale, int causal, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SM_RMSNORM_MATMUL_QKNORM_ATTENTION_H */
