/*
 * rmsnorm_matmul.h -- C ABI of libsm_rmsnorm_matmul.so, a GB300 (sm_103a)
 * library for RMSNorm followed by MatMul, fused into one pass.
 *
 * Operation (Mirage review page, "Mirage: A Multi-Level Superoptimizer for
 * Tensor Programs", section 3 "muGraph example": existing systems run RMSNorm
 * and MatMul as two kernels, Mirage fuses them and never materialises the
 * normalised tensor; section 3 "core formula": E(O) = sum(k, div(mul(E(I1),
 * E(I2)), E(I3))), i.e. a divisor that does not depend on k moves past the
 * k-sum):
 *
 *     r[m]   = 1 / sqrt( (1/K) * sum_k X[m,k]^2 + eps )
 *     Y[m,n] = r[m] * sum_k (X[m,k] * g[k]) * W[k,n]
 *
 * Conventions shared by every entry point:
 *  - Tensors are dense, row-major (last index contiguous) bf16 arrays in
 *    device memory of the CURRENT device: X [M,K], g [K], W [K,N], Y [M,N].
 *    W is stored K-by-N (N contiguous), as the product X.W is written.
 *  - Pointers are owned by the caller.  The library never frees them and
 *    keeps none of them after the call returns.
 *  - Every call is stream-ordered and asynchronous on `stream` (a
 *    cudaStream_t; NULL means the legacy default stream).  RMM_OK means the
 *    work was enqueued.  Faults inside a kernel surface at the caller's next
 *    synchronisation with that stream; a bounded wait that ran out inside a
 *    kernel is reported by rmm_device_status().
 *  - Arguments are validated before any CUDA call.  Rules:
 *      M >= 0, N >= 0, K >= 1 (an empty row has no mean square);
 *      M == 0 or N == 0 is a no-op that returns RMM_OK (pointers unused);
 *      K and N multiples of 8 (16-byte row strides) -> else RMM_ERR_ALIGNMENT;
 *      every pointer non-NULL and 16-byte aligned -> else RMM_ERR_INVALID_ARG
 *        (NULL) or RMM_ERR_ALIGNMENT (misaligned);
 *      eps finite and >= 0 -> else RMM_ERR_INVALID_ARG;
 *      the output may not overlap any input -> else RMM_ERR_INVALID_ARG;
 *      the current device must have compute capability 10.3
 *        -> else RMM_ERR_UNSUPPORTED_DEVICE.
 *  - Rounding: products X*g are rounded to bf16 before the tensor-core
 *    contraction; accumulation is fp32; Y is rounded once to bf16 (nearest
 *    even).  eps = 0 on an all-zero row gives NaN, as the formula does.
 *  - Thread safety: calls from several host threads are safe.  The
 *    library's lazily created per-(device, stream) state is guarded by a
 *    mutex; rmm_force_path() is a process-wide test and benchmark switch.
 */
#ifndef SM_RMSNORM_MATMUL_H
#define SM_RMSNORM_MATMUL_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    RMM_OK = 0,
    RMM_ERR_INVALID_ARG = 1,        /* NULL pointer, bad size, bad eps, aliasing */
    RMM_ERR_ALIGNMENT = 2,          /* pointer not 16-byte aligned, K or N % 8 != 0 */
    RMM_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not compute capability 10.3 */
    RMM_ERR_LAUNCH = 4,             /* a CUDA launch or API call failed */
    RMM_ERR_DEVICE_TIMEOUT = 5,     /* a bounded in-kernel wait ran out (rmm_device_status) */
    RMM_ERR_INTERNAL = 6,           /* workspace allocation or tensor-map encoding failed */
    RMM_ERR_SCRATCH_LIMIT = 7       /* rmsnorm_matmul_noalloc: problem needs more than its fixed scratch */
} rmm_status;

/*
 * Fused RMSNorm + MatMul (the operation above), one launch.
 *   X  [M,K] bf16 input rows           g [K] bf16 gain
 *   W  [K,N] bf16 weights (N contiguous) Y [M,N] bf16 output (written)
 *   eps added to the mean square inside the square root.
 * Shape-based dispatch between two kernels:
 *  - M <= 16 and a W that the row-tile kernel, whose 256-column tiles take
 *    at most 8 K splits, would stream more slowly (a long K over a narrow N:
 *    a model of both kernels' streaming rates decides): the small-M path, a
 *    split-K GEMV-style kernel: W, X and g streamed by TMA through a
 *    shared-memory ring into mma.sync, X*g and the row sums of squares formed
 *    on the fly, 64-column units whose K range may be cut into pieces; the
 *    pieces meet in a library-owned fp32 workspace per (device, stream) and
 *    the last CTA of a unit adds them in a fixed order (no CTA waits for
 *    another).
 *  - otherwise: the tcgen05 row-tile kernels: 128-row x 256-column tiles, X*g
 *    and the row sum of squares computed in the same pass as the contraction,
 *    r[m] applied in the epilogue.  For M <= 128 the K range may be split over
 *    up to 8 CTAs of a thread-block cluster whose partial sums are combined in
 *    shared memory, in a fixed order; with a K split over at most 32 rows the
 *    plain form may use 128-column tiles instead (twice the CTAs, half the
 *    partial sums each exchanges).  For more row tiles, when the tiles
 *    leave a last wave of CTAs at most half full, those last tiles are cut
 *    along K, one piece per CTA, and the pieces are combined, in a fixed
 *    order, through the same workspace; the pieces of a tile wait for one
 *    another, so such a launch is cooperative: all its CTAs (at most one per
 *    SM) are resident at once, or the launch fails with RMM_ERR_LAUNCH (for
 *    example on a device partition with fewer SMs than the device reports).
 *    Where clusters of two fit and the 256-row units of a tile pair need no
 *    such cut (or leave at most a fifth of their rounds idle), the two CTAs
 *    of a cluster instead compute each 256 x 256 unit together as one MMA of
 *    M = 256 (tcgen05 cta_group::2), each loading half of every W stage;
 *    units are never cut along K there.
 * The workspace is allocated on first use of a shape that needs it (make that
 * first call outside any CUDA-graph capture).
 * Returns an rmm_status.
 */
int rmsnorm_matmul(const void* X, const void* g, const void* W, void* Y,
                   int64_t M, int64_t K, int64_t N, float eps, cudaStream_t stream);

/*
 * Fused RMSNorm + MatMul + gated MLP, one launch (GatedMLP: one of the review
 * page's benchmark workloads, section 5, "experimental results"; the pages
 * give no formula, read here as the gated MLP of the LLaMA family):
 *   W [K,N] holds the gate projection in columns [0, F) and the up projection
 *   in columns [F, 2F), N = 2F;  Z = RMSNorm(X; g, eps) @ W as above (fp32
 *   accumulation, never rounded to bf16);
 *   Y [M,F] bf16:  Y[m,f] = silu(Z[m,f]) * Z[m,F+f],  silu(z) = z / (1 + e^-z).
 * N must be a multiple of 16 (F a multiple of 8); the other rules are those of
 * rmsnorm_matmul().  Always the row-tile kernels (rmm_force_path(2) does not
 * apply); each 128 x 256 tile multiplies the gate columns f0..f0+127 and the
 * matching up columns F+f0.., so the gate and up values of one output meet in
 * the same accumulator row.  May use the per-(device, stream) workspace like
 * rmsnorm_matmul().  Returns an rmm_status.
 */
int rmsnorm_matmul_swiglu(const void* X, const void* g, const void* W, void* Y,
                          int64_t M, int64_t K, int64_t N, float eps, cudaStream_t stream);

/* Flags of rmsnorm_matmul_ex(). */
enum {
    RMM_WEIGHT_NK = 1u,   /* W is stored [N, K] (K contiguous: a linear layer's weight),
                             not [K, N]; Y = RMSNorm(X) @ W^T */
    RMM_GATED_SILU = 2u   /* the gated form of rmsnorm_matmul_swiglu(): the N rows (or
                             columns) of W are gate then up, Y is [M, N/2] */
};

/*
 * rmsnorm_matmul() with options: any combination of the flags above (0 is
 * rmsnorm_matmul() itself, RMM_GATED_SILU is rmsnorm_matmul_swiglu()).  With
 * RMM_WEIGHT_NK, W [N, K] is row-major with K contiguous and the tensor cores
 * read it K-major; every other rule (sizes, alignment, no overlap, results)
 * is that of the flagless form.  Always the row-tile kernels.  Unknown flag
 * bits return RMM_ERR_INVALID_ARG.  Returns an rmm_status.
 */
int rmsnorm_matmul_ex(const void* X, const void* g, const void* W, void* Y,
                      int64_t M, int64_t K, int64_t N, float eps, unsigned flags,
                      cudaStream_t stream);

/*
 * RMSNorm + MatMul with a low-rank adapter (LoRA: another of the review page's
 * benchmark workloads, section 5 table; no formula given, read as the standard
 * adapter with its scaling folded into B):
 *   Y [M,N] = RMSNorm(X; g, eps) @ (W + A @ B),  A [K,R], B [R,N] bf16,
 *   1 <= R <= 64, R a multiple of 8; the other rules are those of
 *   rmsnorm_matmul().
 * Two launches of the row-tile kernels.  The first computes T = (X*g) @ A
 * (fp32 accumulation, no division by the RMS) and stores it as a pair of bf16
 * matrices, T_hi = bf16(T) and T_lo = bf16(T - T_hi), [M, 2 x 64] in a
 * library-owned buffer per (device, stream) (allocated on first use; make
 * that first call outside any CUDA-graph capture).  The second is the main
 * contraction with two more 64-deep stages per tile, T_hi @ B and T_lo @ B,
 * so that Y = r * ((X*g) @ W + T @ B) with one division by the row RMS and T
 * carried to about 2^-16 relative (no rounding beyond that of the plain
 * form's operands).  Returns an rmm_status.
 */
int rmsnorm_matmul_lora(const void* X, const void* g, const void* W, const void* A,
                        const void* B, void* Y, int64_t M, int64_t K, int64_t N, int64_t R,
                        float eps, cudaStream_t stream);

/*
 * Unfused RMSNorm alone (the first of the two kernels that the review page's
 * muGraph example says existing systems launch):
 *   Xn[m,k] = bf16( X[m,k] * g[k] * r[m] ),  X, Xn [M,K] bf16, g [K] bf16.
 * Kept for comparison with the fused path.  Xn may not overlap X or g.
 */
int rmsnorm(const void* X, const void* g, void* Xn,
            int64_t M, int64_t K, float eps, cudaStream_t stream);

/*
 * Unfused MatMul alone (the second kernel of that pair):
 *   C[m,n] = bf16( sum_k A[m,k] * B[k,n] ),  A [M,K], B [K,N], C [M,N] bf16,
 * fp32 accumulation on the tensor cores.  Same validation rules.  From 512
 * rows of A up it runs tiles of 256 rows (two M = 128 MMAs sharing each B
 * stage), the last tiles cut along K as above.
 */
int matmul(const void* A, const void* B, void* C,
           int64_t M, int64_t K, int64_t N, cudaStream_t stream);

/*
 * RMSNorm + MatMul with the gain folded into the weights.  RMSNorm's gain
 * scales the columns of the row vector that meets W, so
 *   (X[m,:] * g * r[m]) @ W = r[m] * (X[m,:] @ W'),  W'[k,n] = g[k] * W[k,n]
 * (the review page's RMSNorm, eq. (1), with its MatMul).  Where g and W stay
 * fixed across calls (inference weights), W' is formed once by fold_gain()
 * and every call then reads raw X as the MMA's A operand:
 *
 * fold_gain:  Wg[k,n] = bf16( g[k] * W[k,n] ),  g [K], W and Wg [K,N] bf16
 *   (the product of two bf16 values is exact in fp32: one rounding).  N must
 *   be a multiple of 8; Wg may not overlap g or W.  Asynchronous on `stream`.
 *
 * rmsnorm_matmul_folded:  Y[m,n] = bf16( r[m] * sum_k X[m,k] * Wg[k,n] ),
 *   r[m] = 1 / sqrt( mean_k X[m,k]^2 + eps ),  X [M,K], Wg [K,N], Y [M,N] bf16,
 *   fp32 accumulation.  The same rules on sizes, alignment and overlap as
 *   rmsnorm_matmul().  From 129 rows up it runs the 256-row kernel: two
 *   M = 128 MMAs per W stage read X as the copy wrote it, two more warps read
 *   each X stage for the row sums of squares, and the epilogue scales row m
 *   by r[m]; the last tiles are cut along K as for matmul() (partial products
 *   and partial row sums combined in piece order through a library-owned
 *   workspace, so the call may allocate device memory like rmsnorm_matmul()).
 *   Up to 128 rows it runs rmsnorm_matmul()'s kernels with a library-owned
 *   gain of ones (allocated on the first call with a longer K and kept, like
 *   the workspaces, for the life of the process: that call may not be made
 *   during stream capture, which returns RMM_ERR_INTERNAL, and the device may
 *   not be reset while the library is in use).
 *   The result differs from rmsnorm_matmul(X, g, W)'s only in where the bf16
 *   rounding of the gain product falls (g*W instead of X*g).
 */
int fold_gain(const void* g, const void* W, void* Wg, int64_t K, int64_t N, cudaStream_t stream);
int rmsnorm_matmul_folded(const void* X, const void* Wg, void* Y, int64_t M, int64_t K, int64_t N,
                          float eps, cudaStream_t stream);

/*
 * Test and benchmark switch for the dispatcher of rmsnorm_matmul() and
 * matmul(): 0 = shape-based choice (default), 1 = always the row-tile path,
 * 2 = always the small-M path (requires M <= 16; larger M returns
 * RMM_ERR_INVALID_ARG while forced).  Returns the previous setting, or -1 for
 * an unknown value (the setting is then unchanged).
 */
int rmm_force_path(int path);

/*
 * Synchronises `stream`, then returns and clears the current device's
 * in-kernel status word: RMM_OK, or RMM_ERR_DEVICE_TIMEOUT if a bounded wait
 * inside a kernel gave up (that kernel then skipped its remaining work and
 * released its tensor memory), or RMM_ERR_INTERNAL if a kernel was launched
 * with a configuration it does not support.  On either, the arrival counters
 * of every workspace of the current device are cleared (synchronously), since
 * a kernel that gave up may have left them set.  RMM_ERR_LAUNCH if the
 * synchronisation itself failed.
 */
int rmm_device_status(cudaStream_t stream);

/*
 * Test hook, not for production use (the timeout path, exercised without any
 * fault).  wait_limit_ns > 0 sets the limit of every bounded in-kernel wait
 * (microsecond resolution, at most the 2 s default; 0 restores the default).
 * skip_sends != 0 makes the row-tile kernels' K-split reduction skip the
 * stores of its partials, the paired prefill kernel's second CTA leave out
 * its first "stage ready" signal (and qknorm_attention's loader leave out its
 * first key/value stage), so that each waiting CTA's wait runs out:
 * the kernel then records RMM_ERR_DEVICE_TIMEOUT, skips its remaining work,
 * frees its tensor memory and exits normally, and rmm_device_status() reports
 * it.  Both settings are process-wide host state, passed to every later
 * launch as kernel parameters (no device memory is written; launches already
 * enqueued keep their values).  Returns RMM_ERR_INVALID_ARG for a negative
 * limit.
 */
int rmm_test_hooks(int skip_sends, int64_t wait_limit_ns);

/* Static, NUL-terminated name of a status code ("RMM_OK", ...). */
const char* rmm_status_string(int code);

/*
 * rmsnorm_matmul_noalloc -- the same computation, arguments and results as
 * rmsnorm_matmul(), for callers that cannot let a library allocate device
 * memory during a call: inference runtimes and plugin hosts that own all
 * device memory through their own pool and forbid allocation inside their
 * enqueue step, processes that fix their device-memory budget at start-up,
 * and latency-critical paths where cudaMalloc (which may synchronise the
 * device) is not acceptable.  It calls no cudaMalloc, cudaFree or allocating
 * library routine.  The paper has no counterpart to this entry point.
 *
 * It runs the same kernels with the same launch plan as rmsnorm_matmul()
 * (results agree bit for bit), but the K-split partial sums that
 * rmsnorm_matmul() keeps in a workspace allocated on first use -- the K
 * pieces of the small-M path and the tail pieces of the prefill kernel --
 * live in one fixed 20 MiB device array inside this
 * library (a file-scope __device__ array), held on every device where the
 * library's device code is loaded until the process exits.  Limit: the plan's
 * partials (fp32 sums plus row sums of squares) must fit in 20 MiB - 64 KiB
 * and its arrival counters in 64 KiB; the tail pieces of any shape fit on a
 * device of up to 152 SMs (at most one 128 x 256 fp32 piece per SM), and a
 * plan that needs more returns RMM_ERR_SCRATCH_LIMIT before any launch.
 * Plans without a K split through memory (whole tiles, or a K split inside a
 * cluster) use no scratch.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current) and keeps it for the life of the process;
 * make that first call before any stream capture, and do not reset the device
 * while the library is in use.  Every call shares the one array, which keeps
 * the previous call's contents; each call that uses it clears its arrival
 * counters on `stream` before its kernel.  Calls whose kernels overlap on the
 * GPU (for example on two streams at once) race on the array: order them on
 * one stream or with events.
 */
int rmsnorm_matmul_noalloc(const void* X, const void* g, const void* W, void* Y,
                           int64_t M, int64_t K, int64_t N, float eps, cudaStream_t stream);

/*
 * Launch plan the library would use for this shape on the current device
 * (introspection for tests and benchmarks; `fused` = 1 for rmsnorm_matmul,
 * 0 for matmul, 2 for rmsnorm_matmul_swiglu, whose N is the width of W; the
 * plan does not depend on RMM_WEIGHT_NK).
 * Fills info[0..7] with: path (1 row-tile, 2 small-M),
 * K splits, 1 if the splits reduce through a cluster's shared memory, grid
 * size, pipeline stages, padded rows MP, column tiles, k-blocks per split.
 * For the fused kernel over several row tiles, the K splits and k-blocks per
 * split are those of its tail tiles (1 split: every tile whole), and splits
 * without a cluster mean partial sums in the workspace (the grid counts CTAs:
 * twice the clusters when the tile pairs run as pair MMAs).  For matmul()
 * from 512 rows up (fused = 0), padded rows 256 and 3 stages mark the 256-row
 * kernel, whose column tiles count 256-row tiles; with a K split over at
 * most 32 rows the column tiles may be 128 columns wide (then N / 128 of
 * them, rounded up).  The plan described is
 * rmsnorm_matmul()'s, which rmsnorm_matmul_noalloc() runs too.
 * Queries device attributes; launches nothing.
 */
int rmm_describe_plan(int64_t M, int64_t K, int64_t N, int fused, int* info);

/* Which path the dispatcher would take for this shape right now on the
 * current device (a 152-SM GB300 if there is none): 1 = row-tile path,
 * 2 = small-M path; RMM_ERR_INVALID_ARG for a size < 1.  Queries device
 * attributes; launches nothing. */
int rmm_dispatch_path(int64_t M, int64_t K, int64_t N);

#ifdef __cplusplus
}
#endif

#endif /* SM_RMSNORM_MATMUL_H */
