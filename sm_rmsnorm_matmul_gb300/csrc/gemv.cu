// gemv.cu -- the small-M path: Y = RMSNorm(X) @ W (or X @ W) for at most 16
// rows of X, a split-K GEMV-style kernel.
//
// The fusion is the one of the Mirage review page ("Mirage: A Multi-Level
// Superoptimizer for Tensor Programs" review, section 3, "core formula"): the
// per-row divisor does not depend on k, so it is applied after the k-sum, and
// X*g is formed on the fly, never written to memory.
//
// With 16 rows or fewer the work is W bytes, not FLOPs: every element of W is
// read once and used for at most 16 multiply-adds.  So the kernel keeps its
// set-up small (no tensor-memory allocation, no cluster): one producer thread
// streams W, X and g through a ring of shared-memory stages with TMA (128-byte
// swizzle, mbarrier-tracked, five stages of 20 KB in flight per CTA, two CTAs
// per SM), and eight consumer warps feed mma.sync.m16n8k16 (bf16 x bf16 ->
// fp32) from it with ldmatrix; the tensor-core rate needed at this size is a
// small fraction of what mma.sync gives.
//
// Stage s of a CTA covers 128 k: W [128 k][64 n] (two [64 k][64 n] boxes),
// X [16 rows][128 k] (two [16][64] boxes, rows past M read as zero) and
// g [128].  Consumer warp w takes k-step w (16 deep) of every stage: its A
// fragment is one ldmatrix.x4 of X, multiplied by g in bf16x2 (the exact
// product rounded once, as in the row-tile kernels) after the row sums of
// squares of the unscaled values are taken; its B fragments are four
// ldmatrix.x4.trans of W (eight 16 x 8 blocks: MMA i covers columns
// n0 + 8 i .. + 7).
//
// Work split: units of 64 columns; the K range of a unit may be cut into
// `splits` pieces of whole stages, one CTA each.  The warps of a CTA combine
// their accumulators in shared memory (over the idle ring) in warp order.
// With more than one piece, each CTA publishes its partial tile (16 x 64 fp32
// and the 16 partial row sums) to the workspace, and the last CTA to arrive on
// the unit's counter adds all pieces in piece order (deterministic), scales by
// 1/rms and writes Y; no CTA ever waits for another.  Every mbarrier wait is
// bounded; a wait that runs out records RMM_ERR_DEVICE_TIMEOUT in this file's
// status word and the CTA leaves without publishing.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "ptx.cuh"

namespace rmm {
namespace {

constexpr int kGvWarps = 8;                              // consumer warps
constexpr int kGvThreads = (kGvWarps + 1) * 32;          // + one producer warp
constexpr int kGvStages = 5;
static_assert(kGvStageK == kGvWarps * kGvBK, "one MMA step per consumer warp per stage");
constexpr uint32_t kGvWBytes = kGvStageK * kGvBN * 2;    // 16 KB
constexpr uint32_t kGvXBytes = kGvMaxM * kGvStageK * 2;  // 4 KB
constexpr uint32_t kGvGBytes = kGvStageK * 2;            // 256 B
constexpr uint32_t kGvOffW = 0;
constexpr uint32_t kGvOffX = kGvOffW + kGvStages * kGvWBytes;
constexpr uint32_t kGvOffG = kGvOffX + kGvStages * kGvXBytes;
constexpr uint32_t kGvOffBar = kGvOffG + kGvStages * kGvGBytes;
constexpr uint32_t kGvOffSs = kGvOffBar + 2 * kGvStages * 8;
constexpr uint32_t kGvOffMisc = kGvOffSs + kGvWarps * kGvMaxM * 4;
constexpr uint32_t kGvSmem = kGvOffMisc + 16 + 1024;     // + alignment slack
// the warps' accumulators while they are combined, over the W ring:
// [warp][16 rows][64 + 8 columns] fp32 (8 columns of padding against bank conflicts)
constexpr int kGvRedLd = kGvBN + 8;
static_assert(kGvWarps * kGvMaxM * kGvRedLd * 4 <= kGvStages * kGvWBytes, "reduction area");
constexpr int kGvPiece = kGvPieceFloats;

// Position in a ring of n stages: the slot and the parity of the current pass.
struct Ring {
    uint32_t idx = 0, phase = 0, n;
    __device__ explicit Ring(uint32_t n_) : n(n_) {}
    __device__ __forceinline__ void advance() {
        if (++idx == n) {
            idx = 0;
            phase ^= 1;
        }
    }
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
// D (16 x 8 fp32) += A (16 x 16 bf16, row-major) * B (16 x 8 bf16, column-major).
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Byte address of 16-byte chunk `chunk` of row `row` in a tile of 128-byte
// rows written by TMA with the 128-byte swizzle (chunk index XOR row % 8).
__device__ __forceinline__ uint32_t swz128(uint32_t tile, int row, int chunk) {
    return tile + row * 128 + ((chunk ^ (row & 7)) << 4);
}

template <bool kFused>
__global__ void __launch_bounds__(kGvThreads, 2)
    gemv_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                const __grid_constant__ CUtensorMap tmG, __nv_bfloat16* __restrict__ Y, GemvLaunch a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const uint32_t sw = sb + kGvOffW, sx = sb + kGvOffX, sg = sb + kGvOffG, bar0 = sb + kGvOffBar;
    auto full = [&](uint32_t s) { return bar0 + 8 * s; };
    auto empty = [&](uint32_t s) { return bar0 + 8 * (kGvStages + s); };
    float* red_ss = reinterpret_cast<float*>(smem + kGvOffSs);   // [warp][row]
    volatile int* abort = reinterpret_cast<volatile int*>(smem + kGvOffMisc);
    int* is_last = reinterpret_cast<int*>(smem + kGvOffMisc + 8);

    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int unit = blockIdx.x / a.splits, piece = blockIdx.x - unit * a.splits;
    const int n0 = unit * kGvBN;
    const int st0 = piece * a.stages_per_piece;                              // first stage of the piece
    const int nst = max(0, min(a.kstages, st0 + a.stages_per_piece) - st0);  // its stages

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGvStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), kGvWarps);   // one elected lane per consumer warp
        }
        abort[0] = 0;
        abort[1] = a.wait_limit_us;
        fence_mbar_init();
    }
    __syncthreads();
    // X, g and W may be the previous kernel's output: wait for it; the next
    // kernel on the stream may be scheduled at once (it waits for this one).
    grid_dep_wait();

    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    float ss0 = 0.f, ss1 = 0.f;   // rows lane/4 and lane/4 + 8 (consumers)

    if (w == kGvWarps) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            grid_dep_launch();
            prefetch_tmap(&tmW);
            prefetch_tmap(&tmX);
            if (kFused) prefetch_tmap(&tmG);
            Ring ring(kGvStages);
            int issued = 0;
            for (int i = 0; i < nst; ++i) {
                if (!mbar_wait(empty(ring.idx), ring.phase ^ 1, abort)) break;
                const uint32_t f = full(ring.idx);
                const int k0 = (st0 + i) * kGvStageK;
                mbar_arrive_expect_tx(f, kGvWBytes + kGvXBytes + (kFused ? kGvGBytes : 0));
                const uint32_t dw = sw + ring.idx * kGvWBytes, dx = sx + ring.idx * kGvXBytes;
                tma_load_2d_nohint(dw, &tmW, f, n0, k0);
                tma_load_2d_nohint(dw + kGvWBytes / 2, &tmW, f, n0, k0 + 64);
                tma_load_2d_nohint(dx, &tmX, f, k0, 0);
                tma_load_2d_nohint(dx + kGvXBytes / 2, &tmX, f, k0 + 64, 0);
                if (kFused) {
                    tma_load_1d(sg + ring.idx * kGvGBytes, &tmG, f, k0);
                    tma_load_1d(sg + ring.idx * kGvGBytes + kGvGBytes / 2, &tmG, f, k0 + 64);
                }
                ring.advance();
                ++issued;
            }
            // never leave with copies still landing in shared memory
            for (int i = issued > kGvStages ? issued - kGvStages : 0; i < issued; ++i)
                mbar_wait_teardown(full(i % kGvStages), (i / kGvStages) & 1);
        }
    } else {
        // ------------------------------------------------ consumers: k-step w of every stage
        const int q = lane & 3;
        // ldmatrix row addresses: lane l gives row l % 8 of matrix l / 8
        const int mj = lane >> 3, mr = lane & 7;
        // A (X [16 rows][64 k] box w / 4, k-step (w % 4) * 16): matrices (rows 0-7 | 8-15) x (k 0-7 | 8-15)
        const int xrow = mr + 8 * (mj & 1);
        const int xchunk = 2 * (w & 3) + (mj >> 1);
        const uint32_t xoff = (w >> 2) * (kGvXBytes / 2);
        // B (W [64 k][64 n] box w / 4): matrices (k 0-7 | 8-15) x (n 16x + 0-7 | 16x + 8-15)
        const int wrow = 16 * (w & 3) + mr + 8 * (mj & 1);
        const uint32_t woff = (w >> 2) * (kGvWBytes / 2);
        Ring ring(kGvStages);
        for (int i = 0; i < nst; ++i) {
            if (!warp_wait(full(ring.idx), ring.phase, abort)) break;
            const uint32_t xt = sx + ring.idx * kGvXBytes + xoff;
            const uint32_t wt = sw + ring.idx * kGvWBytes + woff;
            uint32_t af[4];
            ldsm_x4(swz128(xt, xrow, xchunk), af);
            if (kFused) {
                // rows lane/4 (af[0], af[2]) and lane/4 + 8 (af[1], af[3]); k pairs 2q and 2q + 8
                ss0 = fmaf(bf16lo(af[0]), bf16lo(af[0]), ss0);
                ss0 = fmaf(bf16hi(af[0]), bf16hi(af[0]), ss0);
                ss0 = fmaf(bf16lo(af[2]), bf16lo(af[2]), ss0);
                ss0 = fmaf(bf16hi(af[2]), bf16hi(af[2]), ss0);
                ss1 = fmaf(bf16lo(af[1]), bf16lo(af[1]), ss1);
                ss1 = fmaf(bf16hi(af[1]), bf16hi(af[1]), ss1);
                ss1 = fmaf(bf16lo(af[3]), bf16lo(af[3]), ss1);
                ss1 = fmaf(bf16hi(af[3]), bf16hi(af[3]), ss1);
                const uint32_t gt = sg + ring.idx * kGvGBytes + (16 * w + 2 * q) * 2;
                const uint32_t g01 = lds32(gt), g89 = lds32(gt + 16);
                af[0] = mul_bf16x2(af[0], g01);
                af[1] = mul_bf16x2(af[1], g01);
                af[2] = mul_bf16x2(af[2], g89);
                af[3] = mul_bf16x2(af[3], g89);
            }
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                uint32_t b[4];
                ldsm_x4_trans(swz128(wt, wrow, 2 * x + (mj >> 1)), b);
                mma_16816(acc[2 * x], af, b[0], b[1]);
                mma_16816(acc[2 * x + 1], af, b[2], b[3]);
            }
            // every lane's ldmatrix has returned: the stage may be refilled
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(ring.idx));
            ring.advance();
        }
    }

    // ---- combine the warps in warp order (over the idle W ring)
    __syncthreads();   // every stage consumed, every copy landed
    const bool ok = !*abort;
    float* red = reinterpret_cast<float*>(smem + kGvOffW);
    if (w < kGvWarps) {
        const int gi = lane >> 2, q = lane & 3;
        float* mine = red + w * kGvMaxM * kGvRedLd;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            *reinterpret_cast<float2*>(mine + gi * kGvRedLd + 8 * i + 2 * q) = make_float2(acc[i][0], acc[i][1]);
            *reinterpret_cast<float2*>(mine + (gi + 8) * kGvRedLd + 8 * i + 2 * q) =
                make_float2(acc[i][2], acc[i][3]);
        }
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
    }
    __syncthreads();
    if (!ok) return;   // a wait ran out: the status word says so; publish nothing
    // thread t < 128: row m = t / 8, columns n0 + nl .. + 7
    const int m = threadIdx.x >> 3, nl = 8 * (threadIdx.x & 7);
    const bool worker = threadIdx.x < kGvMaxM * 8;
    float v[8];
    float ssm = 0.f;
    if (worker) {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kGvWarps; ++w2) {
            const float* src = red + (w2 * kGvMaxM + m) * kGvRedLd + nl;
            const float4 lo = *reinterpret_cast<const float4*>(src);
            const float4 hi = *reinterpret_cast<const float4*>(src + 4);
            v[0] += lo.x; v[1] += lo.y; v[2] += lo.z; v[3] += lo.w;
            v[4] += hi.x; v[5] += hi.y; v[6] += hi.z; v[7] += hi.w;
            if (kFused) ssm += red_ss[w2 * kGvMaxM + m];
        }
    }
    const float inv_k = 1.f / static_cast<float>(a.K);
    auto store8 = [&](const float (&t)[8], float r) {
        uint4 o;
        o.x = pack_bf16x2(t[0] * r, t[1] * r);
        o.y = pack_bf16x2(t[2] * r, t[3] * r);
        o.z = pack_bf16x2(t[4] * r, t[5] * r);
        o.w = pack_bf16x2(t[6] * r, t[7] * r);
        *reinterpret_cast<uint4*>(Y + static_cast<size_t>(m) * a.N + n0 + nl) = o;
    };
    if (a.splits == 1) {
        if (worker && m < a.M && n0 + nl < a.N) store8(v, kFused ? rsqrtf(ssm * inv_k + a.eps) : 1.f);
        return;
    }

    // ---- K pieces: publish, and the last CTA of the unit adds them in order
    float* mine = a.ws + static_cast<size_t>(blockIdx.x) * kGvPiece;
    if (worker) {
        __stcg(reinterpret_cast<float4*>(mine + m * kGvBN + nl), make_float4(v[0], v[1], v[2], v[3]));
        __stcg(reinterpret_cast<float4*>(mine + m * kGvBN + nl + 4), make_float4(v[4], v[5], v[6], v[7]));
        if (nl == 0) __stcg(mine + kGvMaxM * kGvBN + m, ssm);
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        *is_last = atomicAdd(a.counters + unit, 1) == a.splits - 1;
        __threadfence();
    }
    __syncthreads();
    if (!*is_last) return;
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
        if (m < a.M && n0 + nl < a.N) store8(t, kFused ? rsqrtf(tss * inv_k + a.eps) : 1.f);
    }
    // every piece of this unit has arrived: reset its counter for the next launch
    if (threadIdx.x == 0) a.counters[unit] = 0;
}

// Raises the kernel's dynamic shared-memory limit, once per (variant, device).
cudaError_t gemv_smem_attr(bool fused) {
    static int done[2][64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && done[fused][dev]) return cudaSuccess;
    e = fused ? cudaFuncSetAttribute(gemv_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGvSmem)
              : cudaFuncSetAttribute(gemv_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGvSmem);
    if (e == cudaSuccess && dev < 64) done[fused][dev] = 1;
    return e;
}

}  // namespace

cudaError_t launch_gemv(bool fused, const CUtensorMap& tmX, const CUtensorMap& tmW, const CUtensorMap& tmG,
                        void* Y, const GemvLaunch& a, cudaStream_t s) {
    cudaError_t e = gemv_smem_attr(fused);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.units * a.splits);
    cfg.blockDim = dim3(kGvThreads);
    cfg.dynamicSmemBytes = kGvSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    auto* y = static_cast<__nv_bfloat16*>(Y);
    e = fused ? cudaLaunchKernelEx(&cfg, gemv_kernel<true>, tmX, tmW, tmG, y, a)
              : cudaLaunchKernelEx(&cfg, gemv_kernel<false>, tmX, tmW, tmG, y, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

int gemv_ctas_per_sm(bool fused) {
    if (gemv_smem_attr(fused) != cudaSuccess) return 0;
    int n = 0;
    const cudaError_t e =
        fused ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gemv_kernel<true>, kGvThreads, kGvSmem)
              : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gemv_kernel<false>, kGvThreads, kGvSmem);
    return e == cudaSuccess ? n : 0;
}

cudaError_t gemv_read_and_clear_status(int* out) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_status, sizeof(int));
    if (e != cudaSuccess) return e;
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
    *out = v;
    return e;
}

}  // namespace rmm
