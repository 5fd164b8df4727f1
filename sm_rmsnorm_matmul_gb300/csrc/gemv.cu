// gemv.cu -- the small-M path: Y = RMSNorm(X) @ W (or X @ W) for at most 16
// rows of X, a split-K GEMV-style kernel.
//
// The fusion is the one of the Mirage review page ("Mirage: A Multi-Level
// Superoptimizer for Tensor Programs" review, section 3, "core formula"): the
// per-row divisor does not depend on k, so it is applied after the k-sum, and
// X*g is formed on the fly, never written to memory.
//
// With 16 rows or fewer the work is W bytes, not FLOPs: every element of W is
// read once and used for at most 16 multiply-adds.  So the kernel has no
// set-up to speak of (no tensor-memory allocation, no cluster, no barrier
// ring, no tensor maps): each thread streams W with 128-bit loads straight
// into the B fragments of mma.sync.m16n8k16 (bf16 x bf16 -> fp32), whose
// throughput is far above what the HBM stream needs at this size.
//
// Index mapping.  A warp step covers 16 k x 64 n of W.  Thread (gi = lane/4,
// q = lane%4) loads 16 bytes (8 consecutive columns n0 + 8 gi .. + 7) from
// each of the rows k0 + 2q, +1, +8, +9: one warp-wide load touches four whole
// 128-byte row segments.  Byte permutes pair rows (k, k+1) per column, which
// is the B fragment of column gi for MMA i when MMA i's column j stands for
// W column n0 + 8 j + i.  The accumulator fragment of MMA i then holds, for
// thread (gi, q), Y columns n0 + 16 q + {0, 8} + i: over the 8 MMAs, two runs
// of 8 consecutive columns per row, stored with 16-byte stores.  The A
// fragment is bf16(X*g) (the exact product rounded once, as in the row-tile
// kernels) built from 32-bit loads of X and g, beside the row sums of squares
// of the unscaled X.
//
// Work split: units of 64 columns; the K range of a unit may be cut into
// `splits` pieces, one CTA each.  The 8 warps of a CTA take interleaved
// 16-deep k-steps of its piece and combine their accumulators in shared
// memory in warp order.  With more than one piece, each CTA publishes its
// partial tile (16 x 64 fp32 and the 16 partial row sums) to the workspace
// and the last CTA to arrive on the unit's counter adds all pieces in piece
// order (deterministic), scales by 1/rms and writes Y; no CTA ever waits for
// another.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "launch.h"

namespace rmm {
namespace {

constexpr int kGvWarps = 8;
constexpr int kGvThreads = kGvWarps * 32;
constexpr int kGvGroup = 3;                    // k-steps whose loads a warp issues together
constexpr int kGvPiece = kGvPieceFloats;

__device__ __forceinline__ uint4 ldg_stream128(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg32(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t word(const uint4& v, int j) {
    return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
// bf16x2 product rounded once to bf16 (nearest even).
__device__ __forceinline__ uint32_t mul_bf16x2_rn(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}
// D (16 x 8 fp32) += A (16 x 16 bf16, row-major) * B (16 x 8 bf16, column-major).
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void grid_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Row m (< M), columns n..n+7 (< N, n a multiple of 8) of Y from fp32 sums.
__device__ __forceinline__ void store8(__nv_bfloat16* Y, int N, int m, int n, const float (&v)[8], float r) {
    uint4 o;
    o.x = pack2(v[0] * r, v[1] * r);
    o.y = pack2(v[2] * r, v[3] * r);
    o.z = pack2(v[4] * r, v[5] * r);
    o.w = pack2(v[6] * r, v[7] * r);
    *reinterpret_cast<uint4*>(Y + static_cast<size_t>(m) * N + n) = o;
}

template <bool kFused>
__global__ void __launch_bounds__(kGvThreads, 2)
    gemv_kernel(const __nv_bfloat16* __restrict__ X, const __nv_bfloat16* __restrict__ g,
                const __nv_bfloat16* __restrict__ W, __nv_bfloat16* __restrict__ Y, GemvLaunch a) {
    __shared__ float red[kGvWarps * 8 * 4 * 32];   // [warp][mma][fragment][lane]
    __shared__ float red_ss[kGvWarps * kGvMaxM];    // [warp][row]
    __shared__ int is_last;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int gi = lane >> 2, q = lane & 3;
    const int unit = blockIdx.x / a.splits, piece = blockIdx.x - unit * a.splits;
    const int n0 = unit * kGvBN;
    const int s0 = piece * a.steps_per_piece, s1 = min(a.ksteps, s0 + a.steps_per_piece);
    const int K = a.K, N = a.N;
    const int ncol = n0 + 8 * gi;            // this thread's 8 columns of W
    const bool col_ok = ncol < N;
    const bool row0 = gi < a.M, row1 = gi + 8 < a.M;
    const __nv_bfloat16* wcol = W + ncol;
    const __nv_bfloat16* xr0 = X + static_cast<size_t>(gi) * K;
    const __nv_bfloat16* xr1 = X + static_cast<size_t>(gi + 8) * K;

    // X, g and W may be the previous kernel's output: wait for it; the next
    // kernel on the stream may be scheduled at once (it waits for this one).
    grid_wait();
    grid_launch();

    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    float ss0 = 0.f, ss1 = 0.f;   // rows gi and gi + 8

    for (int base = s0 + w; base < s1; base += kGvWarps * kGvGroup) {
        uint4 wv[kGvGroup][4];
        uint32_t xa[kGvGroup][4], ga[kGvGroup][2];
        // all loads of the group first, so that they are in flight together
#pragma unroll
        for (int u = 0; u < kGvGroup; ++u) {
            const int step = base + u * kGvWarps;
            const bool st = step < s1;          // warp-uniform
            const int k0 = step * kGvBK;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int kr = k0 + 2 * q + (j & 1) + 8 * (j >> 1);
                wv[u][j] = st && col_ok && kr < K ? ldg_stream128(wcol + static_cast<size_t>(kr) * N)
                                                  : make_uint4(0u, 0u, 0u, 0u);
            }
            const int ka = k0 + 2 * q, kb = ka + 8;   // K is a multiple of 8: ka < K covers ka + 1
            const bool oka = st && ka < K, okb = st && kb < K;
            xa[u][0] = oka && row0 ? ldg32(xr0 + ka) : 0u;
            xa[u][1] = oka && row1 ? ldg32(xr1 + ka) : 0u;
            xa[u][2] = okb && row0 ? ldg32(xr0 + kb) : 0u;
            xa[u][3] = okb && row1 ? ldg32(xr1 + kb) : 0u;
            if (kFused) {
                ga[u][0] = oka ? ldg32(g + ka) : 0u;
                ga[u][1] = okb ? ldg32(g + kb) : 0u;
            }
        }
#pragma unroll
        for (int u = 0; u < kGvGroup; ++u) {
            if (base + u * kGvWarps >= s1) break;   // warp-uniform
            uint32_t af[4];
            if (kFused) {
                ss0 = fmaf(bf_lo(xa[u][0]), bf_lo(xa[u][0]), ss0);
                ss0 = fmaf(bf_hi(xa[u][0]), bf_hi(xa[u][0]), ss0);
                ss0 = fmaf(bf_lo(xa[u][2]), bf_lo(xa[u][2]), ss0);
                ss0 = fmaf(bf_hi(xa[u][2]), bf_hi(xa[u][2]), ss0);
                ss1 = fmaf(bf_lo(xa[u][1]), bf_lo(xa[u][1]), ss1);
                ss1 = fmaf(bf_hi(xa[u][1]), bf_hi(xa[u][1]), ss1);
                ss1 = fmaf(bf_lo(xa[u][3]), bf_lo(xa[u][3]), ss1);
                ss1 = fmaf(bf_hi(xa[u][3]), bf_hi(xa[u][3]), ss1);
                af[0] = mul_bf16x2_rn(xa[u][0], ga[u][0]);
                af[1] = mul_bf16x2_rn(xa[u][1], ga[u][0]);
                af[2] = mul_bf16x2_rn(xa[u][2], ga[u][1]);
                af[3] = mul_bf16x2_rn(xa[u][3], ga[u][1]);
            } else {
                af[0] = xa[u][0];
                af[1] = xa[u][1];
                af[2] = xa[u][2];
                af[3] = xa[u][3];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                // column n0 + 8 gi + i: rows (2q, 2q + 1) and (2q + 8, 2q + 9)
                const uint32_t sel = (i & 1) ? 0x7632u : 0x5410u;
                const uint32_t b0 = __byte_perm(word(wv[u][0], i >> 1), word(wv[u][1], i >> 1), sel);
                const uint32_t b1 = __byte_perm(word(wv[u][2], i >> 1), word(wv[u][3], i >> 1), sel);
                mma_16816(acc[i], af, b0, b1);
            }
        }
    }

    // ---- combine the warps in warp order
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) red[((w * 8 + i) * 4 + j) * 32 + lane] = acc[i][j];
    if (kFused) {
        ss0 += __shfl_xor_sync(0xffffffffu, ss0, 1);
        ss0 += __shfl_xor_sync(0xffffffffu, ss0, 2);
        ss1 += __shfl_xor_sync(0xffffffffu, ss1, 1);
        ss1 += __shfl_xor_sync(0xffffffffu, ss1, 2);
        if (q == 0) {
            red_ss[w * kGvMaxM + gi] = ss0;
            red_ss[w * kGvMaxM + gi + 8] = ss1;
        }
    }
    __syncthreads();
    // thread (j, l) of the first 128: fragment j of lane l over the 8 MMAs,
    // i.e. row m, columns n0 + nl .. + 7
    const int tj = threadIdx.x >> 5, tl = threadIdx.x & 31;
    const int m = (tl >> 2) + 8 * (tj >> 1);
    const int nl = 16 * (tl & 3) + 8 * (tj & 1);
    const bool worker = threadIdx.x < 128;
    float v[8];
    float ssm = 0.f;
    if (worker) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float t = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < kGvWarps; ++w2) t += red[((w2 * 8 + i) * 4 + tj) * 32 + tl];
            v[i] = t;
        }
        if (kFused)
#pragma unroll
            for (int w2 = 0; w2 < kGvWarps; ++w2) ssm += red_ss[w2 * kGvMaxM + m];
    }
    const float inv_k = 1.f / static_cast<float>(K);
    if (a.splits == 1) {
        if (worker && m < a.M && n0 + nl < N)
            store8(Y, N, m, n0 + nl, v, kFused ? rsqrtf(ssm * inv_k + a.eps) : 1.f);
        return;
    }

    // ---- K pieces: publish, and the last CTA of the unit adds them in order
    float* mine = a.ws + static_cast<size_t>(blockIdx.x) * kGvPiece;
    if (worker) {
        __stcg(reinterpret_cast<float4*>(mine + m * kGvBN + nl), make_float4(v[0], v[1], v[2], v[3]));
        __stcg(reinterpret_cast<float4*>(mine + m * kGvBN + nl + 4), make_float4(v[4], v[5], v[6], v[7]));
        if ((tl & 3) == 0 && (tj & 1) == 0) __stcg(mine + kGvMaxM * kGvBN + m, ssm);
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        is_last = atomicAdd(a.counters + unit, 1) == a.splits - 1;
        __threadfence();
    }
    __syncthreads();
    if (!is_last) return;
    if (worker) {
        const float* first = a.ws + static_cast<size_t>(unit) * a.splits * kGvPiece;
        float t[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        float tss = 0.f;
        // eight pieces' loads in flight at a time, added in piece order
        constexpr int kBatch = 8;
        for (int p0 = 0; p0 < a.splits; p0 += kBatch) {
            float4 lo[kBatch], hi[kBatch];
            float sv[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                if (p0 + j < a.splits) {
                    const float* src = first + static_cast<size_t>(p0 + j) * kGvPiece;
                    lo[j] = __ldcg(reinterpret_cast<const float4*>(src + m * kGvBN + nl));
                    hi[j] = __ldcg(reinterpret_cast<const float4*>(src + m * kGvBN + nl + 4));
                    sv[j] = kFused ? __ldcg(src + kGvMaxM * kGvBN + m) : 0.f;
                }
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                if (p0 + j < a.splits) {
                    t[0] += lo[j].x; t[1] += lo[j].y; t[2] += lo[j].z; t[3] += lo[j].w;
                    t[4] += hi[j].x; t[5] += hi[j].y; t[6] += hi[j].z; t[7] += hi[j].w;
                    tss += sv[j];
                }
            }
        }
        if (m < a.M && n0 + nl < N) store8(Y, N, m, n0 + nl, t, kFused ? rsqrtf(tss * inv_k + a.eps) : 1.f);
    }
    // every piece of this unit has arrived: reset its counter for the next launch
    if (threadIdx.x == 0) a.counters[unit] = 0;
}

}  // namespace

cudaError_t launch_gemv(bool fused, const void* X, const void* g, const void* W, void* Y, const GemvLaunch& a,
                        cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.units * a.splits);
    cfg.blockDim = dim3(kGvThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    const auto* x = static_cast<const __nv_bfloat16*>(X);
    const auto* gg = static_cast<const __nv_bfloat16*>(g);
    const auto* w = static_cast<const __nv_bfloat16*>(W);
    auto* y = static_cast<__nv_bfloat16*>(Y);
    cudaError_t e = fused ? cudaLaunchKernelEx(&cfg, gemv_kernel<true>, x, gg, w, y, a)
                          : cudaLaunchKernelEx(&cfg, gemv_kernel<false>, x, gg, w, y, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

int gemv_ctas_per_sm(bool fused) {
    int n = 0;
    const cudaError_t e = fused ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gemv_kernel<true>, kGvThreads, 0)
                                : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gemv_kernel<false>, kGvThreads, 0);
    return e == cudaSuccess ? n : 0;
}

}  // namespace rmm
