/*
 * fp64 CPU oracle for RMSNorm followed by MatMul.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline leg may load or run this file.  The CUDA
 * library never links, includes or calls it, and this file includes nothing
 * from the CUDA library.
 *
 * What it computes (plain definition, no blocking, no fusion, no reordering):
 *
 *   ms[m]   = (1/K) * sum_k X[m,k]^2                      (row mean square)
 *   r[m]    = 1 / sqrt(ms[m] + eps)                       (reciprocal RMS)
 *   Xn[m,k] = X[m,k] * g[k] * r[m]                        (RMSNorm with gain g)
 *   Y[m,n]  = sum_k Xn[m,k] * W[k,n]                      (MatMul)
 *
 * This is the unfused pair that the Mirage review page ("Mirage: A
 * Multi-Level Superoptimizer for Tensor Programs" review, section 3,
 * "muGraph example") describes existing systems running as two kernels:
 * RMSNorm, then MatMul.  The MatMul is the broadcast-multiply-then-sum
 * definition (Luminal talk page, "12 primitive ops": matmul is a multiply
 * followed by a sum reduction).  The pages do not write the RMSNorm formula;
 * the placement of eps inside the square root, the mean over K (not K-1) and
 * the per-k multiplicative gain applied to X while the statistic uses the
 * unscaled X are the plain reading of RMSNorm.
 *
 * oracle_rmsnorm_matmul_rewritten() evaluates the form that the fusion rests
 * on (review page, section 3, "core formula": E(O) = sum(k, div(mul(E(I1),
 * E(I2)), E(I3))) with a divisor I3 that does not depend on k, so the division
 * may move outside the sum):
 *
 *   Y[m,n] = ( sum_k (X[m,k]*g[k]) * W[k,n] ) * r[m]
 *
 * oracle_rmsnorm_matmul_swiglu() adds the gated MLP on top (GatedMLP is one
 * of the review page's benchmark workloads, section 5 "experimental results",
 * table of the six benchmarks; the pages give no formula for it).  Read as
 * the gated MLP of the LLaMA family: W holds the gate projection in columns
 * [0, F) and the up projection in columns [F, 2F), N = 2F, and
 *
 *   Z[m,n]  = RMSNorm(X)[m,:] . W[:,n]                    (as above)
 *   Y[m,f]  = silu(Z[m,f]) * Z[m,F+f],  silu(z) = z / (1 + exp(-z)),  f < F.
 *
 * oracle_rmsnorm_matmul_lora() is the LoRA variant (LoRA is another of the
 * review page's benchmark workloads, section 5 table; no formula is given).
 * Read as the standard low-rank adapter: A [K,R], B [R,N] with the scaling
 * folded into B, and the effective weight W + A.B:
 *
 *   Weff[k,n] = W[k,n] + sum_j A[k,j] * B[j,n]
 *   Y[m,n]    = RMSNorm(X)[m,:] . Weff[:,n]
 *
 * oracle_attention() and oracle_qknorm_attention() are the QKNorm + Attention
 * workload (another row of the review page's section 5 benchmark table; the
 * pages give only its name).  Read as the query/key normalisation of recent
 * decoder models: RMSNorm with a gain over the head dimension D, applied to
 * every query head and every key head, then scaled dot-product attention,
 * causal or not, with grouped key/value heads (query head h reads key/value
 * head h / (Hq / Hkv)):
 *
 *   Qn[b,i,h,:] = RMSNorm(Q[b,i,h,:]; gq, eps)            (over d < D)
 *   Kn[b,j,c,:] = RMSNorm(K[b,j,c,:]; gk, eps)
 *   s_j         = scale * sum_d Qn[b,i,h,d] * Kn[b,j,c,d]  (c = h / (Hq/Hkv);
 *                                                          j < S, j <= i if causal)
 *   O[b,i,h,:]  = sum_j softmax(s)_j * V[b,j,c,:]
 *
 * Everything is double precision; nothing is rounded to bf16.  Row-major
 * layouts: X [M,K], g [K], W [K,N], Y [M,N] (Y [M,F] for the gated form);
 * Q and O [B,S,Hq,D], K and V [B,S,Hkv,D].
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ALLOC 1
#define ORACLE_ERR_ARG 2

/* Mean square of one row: (1/K) * sum_k x_k^2, summed in k order. */
static double row_mean_square(const double *x, long K)
{
    double ss = 0.0;
    for (long k = 0; k < K; ++k)
        ss += x[k] * x[k];
    return ss / (double)K;
}

/* Reciprocal RMS: 1 / sqrt(ms + eps).  libm sqrt is correctly rounded. */
static double reciprocal_rms(double ms, double eps)
{
    return 1.0 / sqrt(ms + eps);
}

static int resolve_threads(int nthreads)
{
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* RMSNorm: Xn[m,k] = X[m,k] * g[k] * r[m]. */
int oracle_rmsnorm(const double *X, const double *g, double *Xn,
                   long M, long K, double eps, int nthreads)
{
    int nt = resolve_threads(nthreads);
    (void)nt;
#pragma omp parallel for num_threads(nt) schedule(static)
    for (long m = 0; m < M; ++m) {
        const double *x = X + m * K;
        double r = reciprocal_rms(row_mean_square(x, K), eps);
        for (long k = 0; k < K; ++k)
            Xn[m * K + k] = x[k] * g[k] * r;
    }
    return ORACLE_OK;
}

/* MatMul: C[m,n] = sum_k A[m,k] * B[k,n], loop order m, k, n. */
int oracle_matmul(const double *A, const double *B, double *C,
                  long M, long K, long N, int nthreads)
{
    int nt = resolve_threads(nthreads);
    (void)nt;
#pragma omp parallel for num_threads(nt) schedule(static)
    for (long m = 0; m < M; ++m) {
        double *c = C + m * N;
        for (long n = 0; n < N; ++n)
            c[n] = 0.0;
        for (long k = 0; k < K; ++k) {
            const double a = A[m * K + k];
            const double *b = B + k * N;
            for (long n = 0; n < N; ++n)
                c[n] += a * b[n];
        }
    }
    return ORACLE_OK;
}

/* Unfused RMSNorm then MatMul, one row at a time (the rows are independent). */
int oracle_rmsnorm_matmul(const double *X, const double *g, const double *W,
                          double *Y, long M, long K, long N, double eps,
                          int nthreads)
{
    int nt = resolve_threads(nthreads);
    int failed = 0;
    (void)nt;
#pragma omp parallel num_threads(nt) reduction(| : failed)
    {
        double *xn = (double *)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
        if (!xn) {
            failed = 1;
        } else {
#pragma omp for schedule(static)
            for (long m = 0; m < M; ++m) {
                const double *x = X + m * K;
                /* step 1-3: the normalised row, kept in fp64 */
                double r = reciprocal_rms(row_mean_square(x, K), eps);
                for (long k = 0; k < K; ++k)
                    xn[k] = x[k] * g[k] * r;
                /* step 4: y = xn . W */
                double *y = Y + m * N;
                for (long n = 0; n < N; ++n)
                    y[n] = 0.0;
                for (long k = 0; k < K; ++k) {
                    const double a = xn[k];
                    const double *w = W + k * N;
                    for (long n = 0; n < N; ++n)
                        y[n] += a * w[n];
                }
            }
            free(xn);
        }
    }
    return failed ? ORACLE_ERR_ALLOC : ORACLE_OK;
}

/* The rewritten form: contract (X*g) with W first, divide by the RMS after. */
int oracle_rmsnorm_matmul_rewritten(const double *X, const double *g,
                                    const double *W, double *Y, long M, long K,
                                    long N, double eps, int nthreads)
{
    int nt = resolve_threads(nthreads);
    (void)nt;
#pragma omp parallel for num_threads(nt) schedule(static)
    for (long m = 0; m < M; ++m) {
        const double *x = X + m * K;
        double *y = Y + m * N;
        for (long n = 0; n < N; ++n)
            y[n] = 0.0;
        for (long k = 0; k < K; ++k) {
            const double a = x[k] * g[k];
            const double *w = W + k * N;
            for (long n = 0; n < N; ++n)
                y[n] += a * w[n];
        }
        double r = reciprocal_rms(row_mean_square(x, K), eps);
        for (long n = 0; n < N; ++n)
            y[n] *= r;
    }
    return ORACLE_OK;
}

/* Swish gate: silu(z) = z * sigmoid(z) = z / (1 + exp(-z)). */
static double silu(double z)
{
    return z / (1.0 + exp(-z));
}

/* Gated MLP: Z = RMSNorm(X) @ W over N = 2F columns, then
 * Y[m,f] = silu(Z[m,f]) * Z[m,F+f].  Y is [M, F]. */
int oracle_rmsnorm_matmul_swiglu(const double *X, const double *g, const double *W,
                                 double *Y, long M, long K, long N, double eps,
                                 int nthreads)
{
    if (N % 2 != 0)
        return ORACLE_ERR_ARG;
    const long F = N / 2;
    double *Z = (double *)malloc((size_t)(M * N > 0 ? M * N : 1) * sizeof(double));
    if (!Z)
        return ORACLE_ERR_ALLOC;
    int rc = oracle_rmsnorm_matmul(X, g, W, Z, M, K, N, eps, nthreads);
    if (rc == ORACLE_OK) {
        for (long m = 0; m < M; ++m)
            for (long f = 0; f < F; ++f)
                Y[m * F + f] = silu(Z[m * N + f]) * Z[m * N + F + f];
    }
    free(Z);
    return rc;
}

/* LoRA: Y = RMSNorm(X) @ (W + A @ B).  A [K,R], B [R,N]. */
int oracle_rmsnorm_matmul_lora(const double *X, const double *g, const double *W,
                               const double *A, const double *B, double *Y, long M,
                               long K, long N, long R, double eps, int nthreads)
{
    double *Weff = (double *)malloc((size_t)(K * N > 0 ? K * N : 1) * sizeof(double));
    if (!Weff)
        return ORACLE_ERR_ALLOC;
    /* the effective weight, W + A @ B, loop order k, j, n */
    for (long k = 0; k < K; ++k) {
        double *wk = Weff + k * N;
        for (long n = 0; n < N; ++n)
            wk[n] = W[k * N + n];
        for (long j = 0; j < R; ++j) {
            const double akj = A[k * R + j];
            const double *bj = B + j * N;
            for (long n = 0; n < N; ++n)
                wk[n] += akj * bj[n];
        }
    }
    int rc = oracle_rmsnorm_matmul(X, g, Weff, Y, M, K, N, eps, nthreads);
    free(Weff);
    return rc;
}

/* Attention for the query positions qpos[0..nq) of every sequence (all S
 * positions, in order, when qpos is NULL; nq must then be S).  O is
 * [B, nq, Hq, D].  The softmax subtracts the row maximum before exp, which
 * changes nothing in exact arithmetic and keeps exp in range. */
int oracle_attention(const double *Q, const double *K, const double *V, double *O,
                     long B, long S, long Hq, long Hkv, long D, double scale, int causal,
                     const long *qpos, long nq, int nthreads)
{
    if (B < 0 || S < 0 || Hq < 1 || Hkv < 1 || D < 1 || Hq % Hkv != 0)
        return ORACLE_ERR_ARG;
    if (!qpos && nq != S)
        return ORACLE_ERR_ARG;
    for (long t = 0; qpos && t < nq; ++t)
        if (qpos[t] < 0 || qpos[t] >= S)
            return ORACLE_ERR_ARG;
    const long group = Hq / Hkv;
    int nt = resolve_threads(nthreads);
    (void)nt;
    int rc = ORACLE_OK;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 4)
    for (long row = 0; row < B * nq * Hq; ++row) {
        const long b = row / (nq * Hq);
        const long t = (row / Hq) % nq;
        const long h = row % Hq;
        const long c = h / group;                 /* key/value head of query head h */
        const long i = qpos ? qpos[t] : t;        /* query position */
        const long nkeys = causal ? i + 1 : S;    /* keys j < nkeys take part */
        const double *q = Q + ((b * S + i) * Hq + h) * D;
        double *o = O + ((b * nq + t) * Hq + h) * D;
        double *sc = (double *)malloc((size_t)(nkeys > 0 ? nkeys : 1) * sizeof(double));
        if (!sc) {
#pragma omp atomic write
            rc = ORACLE_ERR_ALLOC;
            continue;
        }
        double smax = -INFINITY;
        for (long j = 0; j < nkeys; ++j) {
            const double *k = K + ((b * S + j) * Hkv + c) * D;
            double dot = 0.0;
            for (long d = 0; d < D; ++d)
                dot += q[d] * k[d];
            sc[j] = scale * dot;
            if (sc[j] > smax)
                smax = sc[j];
        }
        double denom = 0.0;
        for (long j = 0; j < nkeys; ++j) {
            sc[j] = exp(sc[j] - smax);
            denom += sc[j];
        }
        for (long d = 0; d < D; ++d)
            o[d] = 0.0;
        for (long j = 0; j < nkeys; ++j) {
            const double *v = V + ((b * S + j) * Hkv + c) * D;
            const double pj = sc[j] / denom;
            for (long d = 0; d < D; ++d)
                o[d] += pj * v[d];
        }
        free(sc);
    }
    return rc;
}

/* QK-normalised attention: the RMSNorm above over every query and key head
 * (rows of length D), then oracle_attention().  scale is taken as given
 * (callers pass 1/sqrt(D) for the usual scaled dot product). */
int oracle_qknorm_attention(const double *Q, const double *K, const double *V,
                            const double *gq, const double *gk, double *O, long B, long S,
                            long Hq, long Hkv, long D, double eps, double scale, int causal,
                            const long *qpos, long nq, int nthreads)
{
    if (B < 0 || S < 0 || Hq < 1 || Hkv < 1 || D < 1)
        return ORACLE_ERR_ARG;
    const size_t nqe = (size_t)(B * S * Hq * D), nke = (size_t)(B * S * Hkv * D);
    double *Qn = (double *)malloc((nqe > 0 ? nqe : 1) * sizeof(double));
    double *Kn = (double *)malloc((nke > 0 ? nke : 1) * sizeof(double));
    int rc = (Qn && Kn) ? ORACLE_OK : ORACLE_ERR_ALLOC;
    if (rc == ORACLE_OK)
        rc = oracle_rmsnorm(Q, gq, Qn, B * S * Hq, D, eps, nthreads);
    if (rc == ORACLE_OK)
        rc = oracle_rmsnorm(K, gk, Kn, B * S * Hkv, D, eps, nthreads);
    if (rc == ORACLE_OK)
        rc = oracle_attention(Qn, Kn, V, O, B, S, Hq, Hkv, D, scale, causal, qpos, nq, nthreads);
    free(Qn);
    free(Kn);
    return rc;
}

int oracle_max_threads(void)
{
    return resolve_threads(0);
}
