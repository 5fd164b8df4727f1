// attention.cu -- QK-normalised attention on sm_103a.
//
// The operation is the "QKNorm + Attention" workload of the Mirage review
// page's benchmark table (section 5): per-head RMSNorm with a gain on every
// query and key head, then softmax attention (causal or full) with grouped
// key/value heads.  Two kernels:
//
//   rmsnorm_heads_kernel    normalises every key head once (memory-bound; one
//                           warp per head row), into a bf16 workspace;
//   qknorm_attention_kernel one CTA per 128-row query tile of one head:
//                           normalises the query tile in shared memory (with
//                           scale * log2(e) folded in), then for each 128-key
//                           tile S = Qn Kn^T and O += P V on the tensor cores
//                           (tcgen05, accumulators in tensor memory), with the
//                           online softmax between them.
//
// Normalising each key once, not once per query tile that reads it, is the
// choice for GB300: a key tile is read by S/128 query tiles of every head in
// its group, and the workspace round trip costs two reads of K.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "launch.h"
#include "ptx.cuh"

namespace rmm {
namespace {

struct Ring {   // index and phase of a circular buffer of mbarrier-guarded slots
    uint32_t idx = 0, phase = 0, n;
    __device__ explicit Ring(uint32_t n_) : n(n_) {}
    __device__ __forceinline__ void advance() {
        if (++idx == n) {
            idx = 0;
            phase ^= 1;
        }
    }
};

// ------------------------------------------------------------ key rmsnorm
constexpr int kHeadsWarps = 8;

// Y[t,h,:] = bf16(X[t,h,:] * g * rsqrt(mean(X[t,h,:]^2) + eps)), one warp per
// (t, h).  D is a multiple of 8 and at most 256: lane l holds elements
// [8l, 8l + 8) when 8l < D.
__global__ void __launch_bounds__(kHeadsWarps * 32)
    rmsnorm_heads_kernel(const __nv_bfloat16* __restrict__ X, int64_t ldx,
                         const __nv_bfloat16* __restrict__ g, __nv_bfloat16* __restrict__ Y,
                         int64_t ldy, int64_t T, int H, int D, float eps) {
    // X may be the output of the previous kernel on the stream
    grid_dep_wait();
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t item = static_cast<int64_t>(blockIdx.x) * kHeadsWarps + warp;
    if (item >= T * H) return;
    const int64_t t = item / H;
    const int h = static_cast<int>(item - t * H);
    const bool active = lane * 8 < D;
    float v[8];
    float ss = 0.f;
    if (active) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(X + t * ldx + h * D + lane * 8));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = bf16lo(w[i]);
            v[2 * i + 1] = bf16hi(w[i]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(v[i], v[i], ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = rsqrtf(ss / static_cast<float>(D) + eps);
    if (active) {
        const uint4 gu = __ldg(reinterpret_cast<const uint4*>(g + lane * 8));
        const uint32_t gw[4] = {gu.x, gu.y, gu.z, gu.w};
        uint32_t out[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            out[i] = pack_bf16x2(v[2 * i] * bf16lo(gw[i]) * r, v[2 * i + 1] * bf16hi(gw[i]) * r);
        *reinterpret_cast<uint4*>(Y + t * ldy + h * D + lane * 8) =
            make_uint4(out[0], out[1], out[2], out[3]);
    }
}

// ------------------------------------------------------- attention kernel
constexpr int kAttThreads = 256;     // warp 0 TMA, 1 MMA, 2 TMEM, 3 idle, 4-7 rows
constexpr int kAttKStages = 3;
constexpr int kAttVStages = 2;
constexpr uint32_t kAttTile = kAttBM * kAttD * 2;   // 32 KB: a Q, K or V tile
constexpr uint32_t kAttHalf = kAttTile / 2;         // 64 columns of a tile (SW128 box)
constexpr uint32_t kAttOffQ = 0;                    // Q tile, later the O staging
constexpr uint32_t kAttOffK = kAttOffQ + kAttTile;
constexpr uint32_t kAttOffV = kAttOffK + kAttKStages * kAttTile;
constexpr uint32_t kAttOffG = kAttOffV + kAttVStages * kAttTile;   // gq as fp32 [128]
constexpr uint32_t kAttOffBar = kAttOffG + kAttD * 4;
constexpr uint32_t kAttNumBars = 18;
constexpr uint32_t kAttOffMisc = kAttOffBar + 256;
constexpr uint32_t kAttSmem = kAttOffMisc + 16 + 1024;   // + alignment slack
static_assert(kAttNumBars * 8 <= 256, "barrier area");
// Tensor memory: two S buffers (P overwrites the first 64 columns of its S
// buffer, two bf16 per column) and the O accumulator.
constexpr uint32_t kAttColS = 0, kAttColO = 256, kAttTmemCols = 512;
constexpr float kAttRescale = 8.f;   // rescale O only when the row max grows by > 2^8

__global__ void __launch_bounds__(kAttThreads, 1)
    qknorm_attention_kernel(const __grid_constant__ CUtensorMap tmQ,
                            const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV,
                            const __grid_constant__ CUtensorMap tmO,
                            const __nv_bfloat16* __restrict__ gq, AttnLaunch a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sq = sbase + kAttOffQ, sk = sbase + kAttOffK, sv = sbase + kAttOffV;
    float* sg = reinterpret_cast<float*>(smem + kAttOffG);
    const uint32_t bar0 = sbase + kAttOffBar;
    const uint32_t q_full = bar0, q_ready = bar0 + 8;
    auto k_full = [&](uint32_t i) { return bar0 + 16 + 8 * i; };
    auto k_empty = [&](uint32_t i) { return bar0 + 40 + 8 * i; };
    auto v_full = [&](uint32_t i) { return bar0 + 64 + 8 * i; };
    auto v_empty = [&](uint32_t i) { return bar0 + 80 + 8 * i; };
    auto s_full = [&](uint32_t i) { return bar0 + 96 + 8 * i; };
    auto p_full = [&](uint32_t i) { return bar0 + 112 + 8 * i; };
    const uint32_t o_done = bar0 + 128, mmadone = bar0 + 136;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kAttOffMisc);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + kAttOffMisc + 4);

    // the tile: query rows [q0, q0 + 128) of head h in sequence b; causal
    // launches take the longest rows (the last query tiles) first
    const int bid = blockIdx.x;
    const int qt = a.causal ? a.n_qt - 1 - bid / a.n_hb : bid / a.n_hb;
    const int hb = bid % a.n_hb;
    const int h = hb % a.Hq, b = hb / a.Hq;
    const int c = h / a.group;
    const int q0 = qt * kAttBM;
    const int n_kv_all = (a.S + kAttBN - 1) / kAttBN;
    const int n_kv = a.causal ? min(qt + 1, n_kv_all) : n_kv_all;

    if (threadIdx.x == 0) {
        if (blockDim.x != kAttThreads) atomicCAS(&g_status, 0, kStatusInternal);
        mbar_init(q_full, 1);
        mbar_init(q_ready, 4);   // one elected lane per row warp
        for (int i = 0; i < kAttKStages; ++i) {
            mbar_init(k_full(i), 1);
            mbar_init(k_empty(i), 1);
        }
        for (int i = 0; i < kAttVStages; ++i) {
            mbar_init(v_full(i), 1);
            mbar_init(v_empty(i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(s_full(i), 1);
            mbar_init(p_full(i), 4);
        }
        mbar_init(o_done, 1);
        mbar_init(mmadone, 1);
        abort[0] = blockDim.x != kAttThreads;
        abort[1] = a.wait_limit_us;
        fence_mbar_init();
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmO);
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_holder), kAttTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    // Inputs (the key workspace above all) are written by the previous
    // kernel on the stream: wait for it before the first read.
    grid_dep_wait();
    grid_dep_launch();

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0 && !*abort) {
            const uint64_t keep = policy_evict_last();   // K and V tiles are re-read
            const uint64_t once = policy_evict_first();  // the query tile is read once
            mbar_arrive_expect_tx(q_full, kAttTile);
            tma_load_3d(sq, &tmQ, q_full, h * kAttD, q0, b, once);
            tma_load_3d(sq + kAttHalf, &tmQ, q_full, h * kAttD + 64, q0, b, once);
            Ring kr(kAttKStages), vr(kAttVStages);
            int k_issued = 0, v_issued = 0;
            for (int j = 0; j < n_kv; ++j) {
                if (!mbar_wait(k_empty(kr.idx), kr.phase ^ 1, abort)) break;
                mbar_arrive_expect_tx(k_full(kr.idx), kAttTile);
                const uint32_t kd = sk + kr.idx * kAttTile;
                tma_load_3d(kd, &tmK, k_full(kr.idx), c * kAttD, j * kAttBN, b, keep);
                tma_load_3d(kd + kAttHalf, &tmK, k_full(kr.idx), c * kAttD + 64, j * kAttBN, b, keep);
                kr.advance();
                ++k_issued;
                if (!mbar_wait(v_empty(vr.idx), vr.phase ^ 1, abort)) break;
                mbar_arrive_expect_tx(v_full(vr.idx), kAttTile);
                const uint32_t vd = sv + vr.idx * kAttTile;
                // four boxes of [64 keys][64 dims]: box (kk, n) at (2 kk + n) * 8 KB
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                    for (int n = 0; n < 2; ++n)
                        tma_load_3d(vd + (2 * kk + n) * (kAttTile / 4), &tmV, v_full(vr.idx),
                                    c * kAttD + n * 64, j * kAttBN + kk * 64, b, keep);
                vr.advance();
                ++v_issued;
            }
            // never leave with copies still landing in shared memory
            mbar_wait_teardown(q_full, 0);
            for (int i = k_issued > kAttKStages ? k_issued - kAttKStages : 0; i < k_issued; ++i)
                mbar_wait_teardown(k_full(i % kAttKStages), (i / kAttKStages) & 1);
            for (int i = v_issued > kAttVStages ? v_issued - kAttVStages : 0; i < v_issued; ++i)
                mbar_wait_teardown(v_full(i % kAttVStages), (i / kAttVStages) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(kAttBM, kAttBN, false, false);
            constexpr uint32_t idesc_o = idesc_bf16_f32(kAttBM, kAttD, false, true);
            Ring kr(kAttKStages), vr(kAttVStages);
            // S_j = Qn K_j^T into S buffer j & 1: A and B K-major, 8 steps of 16 dims
            auto issue_s = [&](int j) -> bool {
                if (!mbar_wait(k_full(kr.idx), kr.phase, abort)) return false;
                tc_fence_after();
                const uint32_t d = tmem + kAttColS + (j & 1) * kAttBN;
                const uint32_t kb = sk + kr.idx * kAttTile;
#pragma unroll
                for (int kk = 0; kk < kAttD / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kAttHalf + (kk & 3) * 32;
                    mma_bf16_ss(d, sdesc_sw128(sq + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024),
                                idesc_s, kk > 0);
                }
                mma_commit(k_empty(kr.idx));
                mma_commit(s_full(j & 1));
                kr.advance();
                return true;
            };
            bool ok = mbar_wait(q_ready, 0, abort);
            if (ok) {
                tc_fence_after();
                ok = issue_s(0);
            }
            for (int j = 0; ok && j < n_kv; ++j) {
                // the next scores first, so the softmax of tile j + 1 overlaps P_j V_j
                if (j + 1 < n_kv && !issue_s(j + 1)) break;
                if (!mbar_wait(p_full(j & 1), (j >> 1) & 1, abort)) break;
                if (!mbar_wait(v_full(vr.idx), vr.phase, abort)) break;
                tc_fence_after();
                // O += P_j V_j: A = P from tensor memory (keys 16kk.. in columns
                // 8kk..), B = V MN-major (dims contiguous), 8 steps of 16 keys
                const uint32_t pa = tmem + kAttColS + (j & 1) * kAttBN;
                const uint32_t vb = sv + vr.idx * kAttTile;
#pragma unroll
                for (int kk = 0; kk < kAttBN / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * (kAttTile / 2) + (kk & 3) * 2048;
                    mma_bf16_ts(tmem + kAttColO, pa + kk * 8, sdesc_sw128(vb + off, kAttTile / 4, 1024),
                                idesc_o, j > 0 || kk > 0);
                }
                mma_commit(v_empty(vr.idx));
                mma_commit(o_done);
                vr.advance();
            }
            mma_commit(mmadone);
            mbar_wait_teardown(mmadone, 0);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------ rows: norm, softmax, epilogue
        const int q = warp - 4;                  // lane quarter of tensor memory
        const int row = q * 32 + lane;           // query row of the tile
        const int qpos = q0 + row;
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t swz = static_cast<uint32_t>(row & 7);
        const uint32_t srow = sq + static_cast<uint32_t>(row) * 128;
        sg[row] = __bfloat162float(gq[row]);
        named_bar_sync(1, 128);
        bool ok = warp_wait(q_full, 0, abort);
        if (ok) {
            // Qn * scale * log2(e) in place, bf16 (the swizzled K-major tile layout)
            float ss = 0.f;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const uint4 u = lds128(srow + hf * kAttHalf + ((cc ^ swz) << 4));
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        ss = fmaf(bf16lo(w[i]), bf16lo(w[i]), ss);
                        ss = fmaf(bf16hi(w[i]), bf16hi(w[i]), ss);
                    }
                }
            const float f = rsqrtf(ss * (1.f / kAttD) + a.eps) * a.qscale;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const uint32_t addr = srow + hf * kAttHalf + ((cc ^ swz) << 4);
                    const uint4 u = lds128(addr);
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
                    const float* gg = sg + hf * 64 + cc * 8;
                    uint32_t o4[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        o4[i] = pack_bf16x2(bf16lo(w[i]) * gg[2 * i] * f,
                                            bf16hi(w[i]) * gg[2 * i + 1] * f);
                    sts128(addr, make_uint4(o4[0], o4[1], o4[2], o4[3]));
                }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(q_ready);
        }
        const uint32_t obuf = tmem + kAttColO + lane_base;
        float m_ref = 0.f, l = 0.f;
        for (int j = 0; ok && j < n_kv; ++j) {
            if (!warp_wait(s_full(j & 1), (j >> 1) & 1, abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t sbuf = tmem + kAttColS + (j & 1) * kAttBN + lane_base;
            float s[kAttBN];
#pragma unroll
            for (int cc = 0; cc < kAttBN / 32; ++cc) {
                uint32_t v[32];
                tmem_ld_32x32(sbuf + cc * 32, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) s[cc * 32 + i] = __uint_as_float(v[i]);
            }
            // keys past the sequence end, and after the query when causal
            const int kbase = j * kAttBN;
            int lim = min(kAttBN, a.S - kbase);
            if (a.causal && j == qt) lim = min(lim, qpos - kbase + 1);
            if (lim < kAttBN) {
#pragma unroll
                for (int i = 0; i < kAttBN; ++i)
                    if (i >= lim) s[i] = -INFINITY;
            }
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int i = 0; i < kAttBN; i += 4) {
                mx[0] = fmaxf(mx[0], s[i]);
                mx[1] = fmaxf(mx[1], s[i + 1]);
                mx[2] = fmaxf(mx[2], s[i + 2]);
                mx[3] = fmaxf(mx[3], s[i + 3]);
            }
            const float m_tile = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
            float alpha = 1.f;
            bool rescale = false;
            if (j == 0) {
                m_ref = m_tile == -INFINITY ? 0.f : m_tile;
            } else if (m_tile > m_ref + kAttRescale) {
                // weights stay below 2^8 relative to m_ref; beyond that the
                // reference moves and O and l are scaled down to it
                alpha = ex2_approx(m_ref - m_tile);
                m_ref = m_tile;
                l *= alpha;
                rescale = true;
            }
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float p0 = ex2_approx(s[half * 64 + 2 * i] - m_ref);
                    const float p1 = ex2_approx(s[half * 64 + 2 * i + 1] - m_ref);
                    ls[i & 3] += p0 + p1;
                    pk[i] = pack_bf16x2(p0, p1);
                }
                tmem_st_32x32(sbuf + half * 32, pk);
            }
            l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            if (__any_sync(0xffffffffu, rescale)) {
                // O holds P_0..P_{j-1} V: wait for the last product, then scale.
                // S_j completed, and it was issued after P_{j-2} V, so o_done is
                // at most one phase behind: the parity wait is exact.
                if (!warp_wait(o_done, (j - 1) & 1, abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int cc = 0; cc < kAttD / 32; ++cc) {
                    uint32_t v[32];
                    tmem_ld_32x32(obuf + cc * 32, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
                    tmem_st_32x32(obuf + cc * 32, v);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full(j & 1));
        }
        // ------------------------------------------------ epilogue: O / l -> bf16 -> TMA store
        // The last product's completion, from the single-use barrier the MMA
        // issuer commits after its last instruction: a parity wait on o_done
        // could be two phases behind here (S_{n-1} is issued before P_{n-2} V).
        if (ok) ok = warp_wait(mmadone, 0, abort);
        if (ok) {
            tc_fence_after();
            const float inv_l = 1.f / l;
            // staging in the Q area (every MMA that read it has completed):
            // 128-byte swizzle, two 64-column halves
#pragma unroll
            for (int cc = 0; cc < kAttD / 32; ++cc) {
                uint32_t v[32];
                tmem_ld_32x32(obuf + cc * 32, v);
                const uint32_t dst = srow + (cc >> 1) * kAttHalf;
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    uint32_t o4[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        o4[i] = pack_bf16x2(__uint_as_float(v[8 * t + 2 * i]) * inv_l,
                                            __uint_as_float(v[8 * t + 2 * i + 1]) * inv_l);
                    const uint32_t chunk = static_cast<uint32_t>((cc & 1) * 4 + t);
                    sts128(dst + ((chunk ^ swz) << 4), make_uint4(o4[0], o4[1], o4[2], o4[3]));
                }
            }
            fence_proxy_async_smem();
        }
        named_bar_sync(1, 128);
        if (row == 0 && !*abort) {
            tma_store_3d(&tmO, sq, h * kAttD, q0, b);
            tma_store_3d(&tmO, sq + kAttHalf, h * kAttD + 64, q0, b);
            bulk_commit_group();
            bulk_wait_group_all();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, kAttTmemCols);
    }
}

template <typename... Args>
cudaError_t launch_pdl(void (*kern)(Args...), int grid, int block, size_t smem, cudaStream_t s,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace

size_t attn_smem_bytes() { return kAttSmem; }

cudaError_t launch_rmsnorm_heads(const void* X, int64_t ldx, const void* g, void* Y, int64_t ldy,
                                 int64_t T, int H, int D, float eps, cudaStream_t s) {
    const int64_t items = T * H;
    if (items <= 0) return cudaSuccess;
    const int64_t grid = (items + kHeadsWarps - 1) / kHeadsWarps;
    if (grid > INT32_MAX) return cudaErrorInvalidValue;
    return launch_pdl(rmsnorm_heads_kernel, static_cast<int>(grid), kHeadsWarps * 32, 0, s,
                      static_cast<const __nv_bfloat16*>(X), ldx,
                      static_cast<const __nv_bfloat16*>(g), static_cast<__nv_bfloat16*>(Y), ldy, T,
                      H, D, eps);
}

cudaError_t launch_qknorm_attention(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                    const CUtensorMap& tmV, const CUtensorMap& tmO,
                                    const void* gq, const AttnLaunch& a, cudaStream_t s) {
    // the shared-memory limit is a per-device attribute of the function
    static std::atomic<bool> attr_set[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load()) {
        e = cudaFuncSetAttribute(qknorm_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kAttSmem);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true);
    }
    return launch_pdl(qknorm_attention_kernel, a.grid, kAttThreads, kAttSmem, s, tmQ, tmK, tmV, tmO,
                      static_cast<const __nv_bfloat16*>(gq), a);
}

cudaError_t attn_read_and_clear_status(int* out) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_status, sizeof(int));
    if (e != cudaSuccess) return e;
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
    *out = v;
    return e;
}

}  // namespace rmm
