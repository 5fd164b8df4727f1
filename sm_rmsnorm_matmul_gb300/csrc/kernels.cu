// kernels.cu -- sm_103a kernels for RMSNorm followed by MatMul.
//
// The fusion follows the Mirage review page ("Mirage: A Multi-Level
// Superoptimizer for Tensor Programs" review, section 3, "muGraph example"
// and "core formula" E(O) = sum(k, div(mul(E(I1), E(I2)), E(I3)))): the
// per-row divisor I3 = sqrt(mean_k X^2 + eps) does not depend on k, so it is
// applied after the k-sum, in the epilogue, and the normalised X is never
// written to memory.  I1 = X*g is formed while each X tile sits in shared
// memory, in the same pass that accumulates the row sum of squares.
//
// Two tensor-core kernels (tcgen05, accumulators in tensor memory, operands
// staged by TMA through an mbarrier ring), one warp-specialised CTA per SM:
//   rows_kernel: CTA tile = 128 rows of X x 256 columns of W.  A = X*g
//     (K-major), B = W (N-major).  For large M (prefill-like shapes).
//   cols_kernel: CTA tile = 128 columns of W x MP rows of X (MP <= 128).
//     A = W^T (N-major, the same shared-memory tile layout), B = X*g
//     (K-major).  W is streamed once; when N alone gives too few tiles the
//     K range is split and fp32 partials are combined in a fixed order by
//     the last CTA to finish a column tile.  For small M (decode-like shapes).
// Warp roles (384 threads): warp 0 TMA producer, warp 1 MMA issuer, warp 2
// tensor-memory allocator, warps 4-7 transform (X*g, sum of squares),
// warps 8-11 epilogue (tensor memory -> registers -> scale by r -> bf16).
// A third kernel, rmsnorm_kernel, is the unfused RMSNorm kept for comparison.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "ptx.cuh"

namespace rmm {
namespace {

constexpr int kThreads = 384;
constexpr uint32_t kGBytes = kBK * 2;            // one g slice per stage: 128 B
constexpr uint32_t kWBoxBytes = 64 * kBK * 2;    // one [64 k][64 n] W box: 8 KB

// ------------------------------------------------------------ row-tile path
constexpr int kRowsStages = 4;
constexpr uint32_t kRowsXBytes = kRowsBM * kBK * 2;   // 16 KB
constexpr uint32_t kRowsWBytes = kRowsBN * kBK * 2;   // 32 KB
constexpr uint32_t kRowsOffX = 0;
constexpr uint32_t kRowsOffW = kRowsOffX + kRowsStages * kRowsXBytes;
constexpr uint32_t kRowsOffG = kRowsOffW + kRowsStages * kRowsWBytes;
constexpr uint32_t kRowsOffBar = kRowsOffG + kRowsStages * kGBytes;
// barriers: full[S], xform[S], empty[S], accfull[2], accempty[2], srfull[2], mmadone
constexpr uint32_t kRowsNumBars = 3 * kRowsStages + 7;
constexpr uint32_t kRowsOffSr = kRowsOffBar + ((kRowsNumBars * 8 + 15) / 16) * 16;
constexpr uint32_t kRowsOffMisc = kRowsOffSr + 2 * kRowsBM * 4;
constexpr uint32_t kRowsSmem = kRowsOffMisc + 16 + 1024;   // + alignment slack
constexpr uint32_t kRowsTmemCols = 2 * kRowsBN;            // double-buffered accumulator

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Tile order: groups of 8 row-blocks; inside a group the row-block index
// varies fastest, so the CTAs resident at one time share W column panels
// and X row panels in L2.
__device__ __forceinline__ void rows_tile_coords(int t, int m_tiles, int n_tiles, int& mb,
                                                 int& nb) {
    constexpr int G = 8;
    const int per_group = G * n_tiles;
    const int group = t / per_group;
    const int first = group * G;
    const int gsz = min(m_tiles - first, G);
    const int local = t - group * per_group;
    mb = first + local % gsz;
    nb = local / gsz;
}

// x*g for 8 bf16 values (one 16-byte chunk), rounded to bf16; accumulates the
// sum of squares of the unscaled x.
__device__ __forceinline__ uint4 gain8(uint4 xv, uint4 gv, float& ss) {
    uint4 o;
    const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w};
    const uint32_t gs[4] = {gv.x, gv.y, gv.z, gv.w};
    uint32_t os[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float x0 = bf16lo(xs[i]), x1 = bf16hi(xs[i]);
        ss = fmaf(x0, x0, ss);
        ss = fmaf(x1, x1, ss);
        os[i] = pack_bf16x2(x0 * bf16lo(gs[i]), x1 * bf16hi(gs[i]));
    }
    o.x = os[0]; o.y = os[1]; o.z = os[2]; o.w = os[3];
    return o;
}

template <bool kFused>
__global__ void __launch_bounds__(kThreads, 1)
    rows_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                const __grid_constant__ CUtensorMap tmG, __nv_bfloat16* __restrict__ Y, int M,
                int N, int K, float eps, int m_tiles, int n_tiles, int k_blocks) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    const uint32_t sb = smem_u32(smem);
    const uint32_t sx = sb + kRowsOffX, sw = sb + kRowsOffW, sg = sb + kRowsOffG;
    const uint32_t bar0 = sb + kRowsOffBar;
    auto full = [&](uint32_t s) { return bar0 + 8 * s; };
    auto xform = [&](uint32_t s) { return bar0 + 8 * (kRowsStages + s); };
    auto empty = [&](uint32_t s) { return bar0 + 8 * (2 * kRowsStages + s); };
    auto accfull = [&](uint32_t b) { return bar0 + 8 * (3 * kRowsStages + b); };
    auto accempty = [&](uint32_t b) { return bar0 + 8 * (3 * kRowsStages + 2 + b); };
    auto srfull = [&](uint32_t b) { return bar0 + 8 * (3 * kRowsStages + 4 + b); };
    const uint32_t mmadone = bar0 + 8 * (3 * kRowsStages + 6);
    float* sr = reinterpret_cast<float*>(smem + kRowsOffSr);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kRowsOffMisc);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + kRowsOffMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRowsStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(xform(s), 128);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accfull(b), 1);
            mbar_init(accempty(b), 128);
            mbar_init(srfull(b), 128);
        }
        mbar_init(mmadone, 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
        if (kFused) prefetch_tmap(&tmG);
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_holder), kRowsTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const int num_tiles = m_tiles * n_tiles;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
                int mb, nb;
                rows_tile_coords(t, m_tiles, n_tiles, mb, nb);
                const int n0 = nb * kRowsBN;
                const int nbox = min(4, (N - n0 + 63) / 64);
                const uint32_t bytes = kRowsXBytes + nbox * kWBoxBytes + (kFused ? kGBytes : 0);
                for (int kb = 0; kb < k_blocks; ++kb) {
                    const uint32_t s = it % kRowsStages, ph = (it / kRowsStages) & 1;
                    if (!mbar_wait(empty(s), ph ^ 1, abort)) { ok = false; break; }
                    mbar_arrive_expect_tx(full(s), bytes);
                    tma_load_2d_nohint(sx + s * kRowsXBytes, &tmX, full(s), kb * kBK, mb * kRowsBM);
                    for (int j = 0; j < nbox; ++j)
                        tma_load_2d_nohint(sw + s * kRowsWBytes + j * kWBoxBytes, &tmW, full(s),
                                           n0 + 64 * j, kb * kBK);
                    if (kFused) tma_load_1d(sg + s * kGBytes, &tmG, full(s), kb * kBK);
                    ++it;
                }
            }
            // never leave with copies still landing in shared memory
            const uint32_t pending = it < kRowsStages ? it : kRowsStages;
            for (uint32_t i = it - pending; i < it; ++i)
                mbar_wait_teardown(full(i % kRowsStages), (i / kRowsStages) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kRowsBM, kRowsBN, false, true);
            uint32_t it = 0, tl = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x, ++tl) {
                const uint32_t buf = tl & 1, use = tl >> 1;
                if (!mbar_wait(accempty(buf), (use & 1) ^ 1, abort)) break;
                tc_fence_after();
                const uint32_t d = tmem + buf * kRowsBN;
                for (int kb = 0; kb < k_blocks; ++kb) {
                    const uint32_t s = it % kRowsStages, ph = (it / kRowsStages) & 1;
                    if (!mbar_wait(kFused ? xform(s) : full(s), ph, abort)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a0 = sx + s * kRowsXBytes, b0 = sw + s * kRowsWBytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        mma_bf16_ss(d, sdesc_sw128(a0 + kk * 32, 16, 1024),
                                    sdesc_sw128(b0 + kk * 2048, kWBoxBytes, 1024), idesc,
                                    (kb | kk) != 0);
                    mma_commit(empty(s));
                    ++it;
                }
                if (!ok) break;
                mma_commit(accfull(buf));
            }
            mma_commit(mmadone);
            mbar_wait_teardown(mmadone, 0);
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------ transform: X*g, sum of squares
        if (kFused) {
            // 8 consecutive threads cover the 8 16-byte chunks of one 128-byte
            // row, so each warp access touches 4 whole rows (no bank conflicts).
            const int t = threadIdx.x - 128;
            const int kc = t & 7;           // chunk of the row
            const int rb = t >> 3;          // rows rb + 16 i, i = 0..7
            const uint32_t swz_off = static_cast<uint32_t>((kc ^ (rb & 7)) << 4);
            uint32_t it = 0, tl = 0;
            bool ok = true;
            for (int t_ = blockIdx.x; ok && t_ < num_tiles; t_ += gridDim.x, ++tl) {
                const uint32_t buf = tl & 1, use = tl >> 1;
                // sr[buf] is free once the epilogue released this accumulator
                if (!warp_wait(accempty(buf), (use & 1) ^ 1, abort)) break;
                float ss[kRowsBM / 16];
#pragma unroll
                for (int i = 0; i < kRowsBM / 16; ++i) ss[i] = 0.f;
                for (int kb = 0; kb < k_blocks; ++kb) {
                    const uint32_t s = it % kRowsStages, ph = (it / kRowsStages) & 1;
                    if (!warp_wait(full(s), ph, abort)) { ok = false; break; }
                    const uint4 gv = lds128(sg + s * kGBytes + kc * 16);
                    const uint32_t xt = sx + s * kRowsXBytes + swz_off;
#pragma unroll
                    for (int i = 0; i < kRowsBM / 16; ++i) {
                        // row rb + 16 i has the same (row & 7) as rb
                        const uint32_t a = xt + (rb + 16 * i) * 128;
                        sts128(a, gain8(lds128(a), gv, ss[i]));
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(xform(s));
                    ++it;
                }
                if (!ok) break;
#pragma unroll
                for (int i = 0; i < kRowsBM / 16; ++i) {
                    float v = ss[i];
                    v += __shfl_xor_sync(0xffffffffu, v, 1);
                    v += __shfl_xor_sync(0xffffffffu, v, 2);
                    v += __shfl_xor_sync(0xffffffffu, v, 4);
                    if (kc == 0) sr[buf * kRowsBM + rb + 16 * i] = rsqrtf(v / static_cast<float>(K) + eps);
                }
                mbar_arrive(srfull(buf));
            }
        }
    } else if (warp >= 8) {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;             // tensor-memory lane quarter of this warp
        const int row = q * 32 + lane;
        uint32_t tl = 0;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++tl) {
            const uint32_t buf = tl & 1, use = tl >> 1;
            if (!warp_wait(accfull(buf), use & 1, abort)) break;
            float r = 1.f;
            if (kFused) {
                if (!warp_wait(srfull(buf), use & 1, abort)) break;
                r = sr[buf * kRowsBM + row];
            }
            tc_fence_after();
            int mb, nb;
            rows_tile_coords(t, m_tiles, n_tiles, mb, nb);
            const int m = mb * kRowsBM + row;
            const int n0 = nb * kRowsBN;
            const int ncols = min(kRowsBN, N - n0);
            __nv_bfloat16* yrow = Y + static_cast<size_t>(m) * N + n0;
            const uint32_t taddr = tmem + buf * kRowsBN + (static_cast<uint32_t>(q * 32) << 16);
            for (int c = 0; c < kRowsBN / 32; ++c) {
                if (c * 32 >= ncols) break;   // warp-uniform
                uint32_t v[32];
                tmem_ld_32x32(taddr + c * 32, v);
                if (m < M) {
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const int col = c * 32 + g * 8;
                        if (col < ncols) {
                            uint4 o;
                            o.x = pack_bf16x2(__uint_as_float(v[g * 8 + 0]) * r,
                                              __uint_as_float(v[g * 8 + 1]) * r);
                            o.y = pack_bf16x2(__uint_as_float(v[g * 8 + 2]) * r,
                                              __uint_as_float(v[g * 8 + 3]) * r);
                            o.z = pack_bf16x2(__uint_as_float(v[g * 8 + 4]) * r,
                                              __uint_as_float(v[g * 8 + 5]) * r);
                            o.w = pack_bf16x2(__uint_as_float(v[g * 8 + 6]) * r,
                                              __uint_as_float(v[g * 8 + 7]) * r);
                            *reinterpret_cast<uint4*>(yrow + col) = o;
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(accempty(buf));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, kRowsTmemCols);
    }
}

// ------------------------------------------------------------ small-M path
struct ColsLayout {
    uint32_t off_w, off_x, off_g, off_bar, off_ss, off_r, off_misc, total;
};

__host__ __device__ inline ColsLayout cols_layout(int MP, int stages) {
    ColsLayout L;
    L.off_w = 0;
    L.off_x = L.off_w + stages * (kColsBN * kBK * 2);
    L.off_g = L.off_x + stages * (MP * kBK * 2);
    L.off_bar = L.off_g + stages * kGBytes;
    const uint32_t nbars = 3 * kColsMaxStages + 8;
    L.off_ss = L.off_bar + ((nbars * 8 + 15) / 16) * 16;
    L.off_r = L.off_ss + 2 * kColsMaxMP * 4;
    L.off_misc = L.off_r + kColsMaxMP * 4;
    L.total = L.off_misc + 16 + 1024;
    return L;
}

template <bool kFused>
__global__ void __launch_bounds__(kThreads, 1)
    cols_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                const __grid_constant__ CUtensorMap tmG, __nv_bfloat16* __restrict__ Y,
                ColsLaunch a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    const int MP = a.MP, S = a.stages;
    const ColsLayout L = cols_layout(MP, S);
    const uint32_t sb = smem_u32(smem);
    const uint32_t sw = sb + L.off_w, sx = sb + L.off_x, sg = sb + L.off_g;
    const uint32_t xbytes = MP * kBK * 2;
    constexpr uint32_t wbytes = kColsBN * kBK * 2;
    const uint32_t bar0 = sb + L.off_bar;
    auto full = [&](uint32_t s) { return bar0 + 8 * s; };
    auto xform = [&](uint32_t s) { return bar0 + 8 * (kColsMaxStages + s); };
    auto empty = [&](uint32_t s) { return bar0 + 8 * (2 * kColsMaxStages + s); };
    auto accfull = [&](uint32_t b) { return bar0 + 8 * (3 * kColsMaxStages + b); };
    auto accempty = [&](uint32_t b) { return bar0 + 8 * (3 * kColsMaxStages + 2 + b); };
    auto srfull = [&](uint32_t b) { return bar0 + 8 * (3 * kColsMaxStages + 4 + b); };
    const uint32_t mmadone = bar0 + 8 * (3 * kColsMaxStages + 6);
    const uint32_t episync = bar0 + 8 * (3 * kColsMaxStages + 7);
    float* ss_s = reinterpret_cast<float*>(smem + L.off_ss);    // [2][128]
    float* r_red = reinterpret_cast<float*>(smem + L.off_r);    // [128]
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L.off_misc);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + L.off_misc + 4);
    volatile int* last_flag = reinterpret_cast<volatile int*>(smem + L.off_misc + 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(xform(s), 128);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accfull(b), 1);
            mbar_init(accempty(b), 128);
            mbar_init(srfull(b), 128);
        }
        mbar_init(mmadone, 1);
        mbar_init(episync, 128);
        *abort = 0;
        *last_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
        if (kFused) prefetch_tmap(&tmG);
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_holder), a.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const int units = a.n_tiles * a.splits;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();   // W is read exactly once
            const uint64_t pol_x = policy_evict_last();    // X is re-read by every column tile
            uint32_t it = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
                const int nt = u / a.splits, sp = u - nt * a.splits;
                const int kb0 = sp * a.kb_per_split, kb1 = min(a.k_blocks, kb0 + a.kb_per_split);
                const int n0 = nt * kColsBN;
                const int nbox = min(2, (a.N - n0 + 63) / 64);
                const uint32_t bytes = nbox * kWBoxBytes + xbytes + (kFused ? kGBytes : 0);
                for (int kb = kb0; kb < kb1; ++kb) {
                    const uint32_t s = it % S, ph = (it / S) & 1;
                    if (!mbar_wait(empty(s), ph ^ 1, abort)) { ok = false; break; }
                    mbar_arrive_expect_tx(full(s), bytes);
                    for (int j = 0; j < nbox; ++j)
                        tma_load_2d(sw + s * wbytes + j * kWBoxBytes, &tmW, full(s), n0 + 64 * j,
                                    kb * kBK, pol_w);
                    tma_load_2d(sx + s * xbytes, &tmX, full(s), kb * kBK, 0, pol_x);
                    if (kFused) tma_load_1d(sg + s * kGBytes, &tmG, full(s), kb * kBK);
                    ++it;
                }
            }
            const uint32_t pending = it < static_cast<uint32_t>(S) ? it : S;
            for (uint32_t i = it - pending; i < it; ++i) mbar_wait_teardown(full(i % S), (i / S) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kColsBN, MP, true, false);
            uint32_t it = 0, tl = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < units; u += gridDim.x, ++tl) {
                const int nt = u / a.splits, sp = u - nt * a.splits;
                const int kb0 = sp * a.kb_per_split, kb1 = min(a.k_blocks, kb0 + a.kb_per_split);
                const uint32_t buf = tl & 1, use = tl >> 1;
                if (!mbar_wait(accempty(buf), (use & 1) ^ 1, abort)) break;
                tc_fence_after();
                const uint32_t d = tmem + buf * MP;
                for (int kb = kb0; kb < kb1; ++kb) {
                    const uint32_t s = it % S, ph = (it / S) & 1;
                    if (!mbar_wait(kFused ? xform(s) : full(s), ph, abort)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a0 = sw + s * wbytes, b0 = sx + s * xbytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        mma_bf16_ss(d, sdesc_sw128(a0 + kk * 2048, kWBoxBytes, 1024),
                                    sdesc_sw128(b0 + kk * 32, 16, 1024), idesc,
                                    (kb != kb0 || kk != 0));
                    mma_commit(empty(s));
                    ++it;
                }
                if (!ok) break;
                mma_commit(accfull(buf));
            }
            mma_commit(mmadone);
            mbar_wait_teardown(mmadone, 0);
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------ transform: X*g, sum of squares
        if (kFused) {
            const int t = threadIdx.x - 128;
            const int kc = t & 7;         // 16-byte chunk of the 128-byte row
            const int rb = t >> 3;        // rows rb, rb + 16, rb + 32, ...
            const int groups = MP / 16;
            const uint32_t swz_off = static_cast<uint32_t>((kc ^ (rb & 7)) << 4);
            uint32_t it = 0, tl = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < units; u += gridDim.x, ++tl) {
                const int nt = u / a.splits, sp = u - nt * a.splits;
                const int kb0 = sp * a.kb_per_split, kb1 = min(a.k_blocks, kb0 + a.kb_per_split);
                const uint32_t buf = tl & 1, use = tl >> 1;
                if (!warp_wait(accempty(buf), (use & 1) ^ 1, abort)) break;
                float ss[kColsMaxMP / 16];
#pragma unroll
                for (int i = 0; i < kColsMaxMP / 16; ++i) ss[i] = 0.f;
                for (int kb = kb0; kb < kb1; ++kb) {
                    const uint32_t s = it % S, ph = (it / S) & 1;
                    if (!warp_wait(full(s), ph, abort)) { ok = false; break; }
                    const uint4 gv = lds128(sg + s * kGBytes + kc * 16);
                    const uint32_t xt = sx + s * xbytes;
#pragma unroll
                    for (int i = 0; i < kColsMaxMP / 16; ++i) {
                        if (i < groups) {
                            // row = rb + 16 i has the same (row & 7) as rb
                            const uint32_t addr = xt + (rb + 16 * i) * 128 + swz_off;
                            sts128(addr, gain8(lds128(addr), gv, ss[i]));
                        }
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(xform(s));
                    ++it;
                }
                if (!ok) break;
#pragma unroll
                for (int i = 0; i < kColsMaxMP / 16; ++i) {
                    float v = ss[i];
                    v += __shfl_xor_sync(0xffffffffu, v, 1);
                    v += __shfl_xor_sync(0xffffffffu, v, 2);
                    v += __shfl_xor_sync(0xffffffffu, v, 4);
                    if (i < groups && kc == 0) ss_s[buf * kColsMaxMP + rb + 16 * i] = v;
                }
                mbar_arrive(srfull(buf));
            }
        }
    } else if (warp >= 8) {
        // ------------------------------------------------ epilogue
        const int e = threadIdx.x - 256;     // == tensor-memory lane == column within the tile
        const int q = warp & 3;
        // bounded barrier over the 4 epilogue warps (an mbarrier, so that a
        // timeout elsewhere cannot leave a warp waiting forever)
        uint32_t ep = 0;
        auto epi_sync = [&]() {
            mbar_arrive(episync);
            return warp_wait(episync, (ep++) & 1, abort);
        };
        uint32_t tl = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x, ++tl) {
            const int nt = u / a.splits, sp = u - nt * a.splits;
            const uint32_t buf = tl & 1, use = tl >> 1;
            if (!warp_wait(accfull(buf), use & 1, abort)) break;
            if (kFused && !warp_wait(srfull(buf), use & 1, abort)) break;
            tc_fence_after();
            const int n = nt * kColsBN + e;
            const bool n_ok = n < a.N;
            const uint32_t taddr = tmem + buf * MP + (static_cast<uint32_t>(q * 32) << 16);
            const int jmax = (a.M + 15) / 16;   // column groups that hold real rows
            if (a.splits == 1) {
                for (int j = 0; j < jmax; ++j) {
                    uint32_t v[16];
                    tmem_ld_32x16(taddr + j * 16, v);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int m = j * 16 + i;
                        if (m < a.M && n_ok) {
                            float r = 1.f;
                            if (kFused)
                                r = rsqrtf(ss_s[buf * kColsMaxMP + m] / static_cast<float>(a.K) +
                                           a.eps);
                            Y[static_cast<size_t>(m) * a.N + n] =
                                __float2bfloat16_rn(__uint_as_float(v[i]) * r);
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(accempty(buf));
            } else {
                // publish this split's partial sums, then the last CTA to finish
                // the column tile adds all splits in split order (its own from
                // tensor memory, which it still holds) and writes Y.
                float* part = a.ws_acc + static_cast<size_t>(sp) * a.M * a.N;
                for (int j = 0; j < jmax; ++j) {
                    uint32_t v[16];
                    tmem_ld_32x16(taddr + j * 16, v);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int m = j * 16 + i;
                        if (m < a.M && n_ok)
                            part[static_cast<size_t>(m) * a.N + n] = __uint_as_float(v[i]);
                    }
                }
                if (kFused && e < a.M)
                    a.ws_ss[(static_cast<size_t>(nt) * a.splits + sp) * kColsMaxMP + e] =
                        ss_s[buf * kColsMaxMP + e];
                __threadfence();
                bool go = epi_sync();
                if (go && e == 0) *last_flag = (atomicAdd(&a.counters[nt], 1) == a.splits - 1);
                go = go && epi_sync();
                if (go && *last_flag) {
                    __threadfence();
                    if (kFused && e < a.M) {
                        float tot = 0.f;
#pragma unroll 4
                        for (int s2 = 0; s2 < a.splits; ++s2)
                            tot += __ldcg(&a.ws_ss[(static_cast<size_t>(nt) * a.splits + s2) *
                                                       kColsMaxMP + e]);
                        r_red[e] = rsqrtf(tot / static_cast<float>(a.K) + a.eps);
                    }
                    go = epi_sync();
                    for (int j = 0; go && j < jmax; ++j) {
                        uint32_t v[16];
                        tmem_ld_32x16(taddr + j * 16, v);
                        float acc[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) acc[i] = 0.f;
                        if (n_ok) {
#pragma unroll 2
                            for (int s2 = 0; s2 < a.splits; ++s2) {
                                const float* p2 = a.ws_acc + static_cast<size_t>(s2) * a.M * a.N + n;
                                float pv[16];
#pragma unroll
                                for (int i = 0; i < 16; ++i) {
                                    const int m = j * 16 + i;
                                    pv[i] = (s2 == sp) ? __uint_as_float(v[i])
                                            : (m < a.M ? __ldcg(p2 + static_cast<size_t>(m) * a.N) : 0.f);
                                }
#pragma unroll
                                for (int i = 0; i < 16; ++i) acc[i] += pv[i];
                            }
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const int m = j * 16 + i;
                                if (m < a.M) {
                                    const float r = kFused ? r_red[m] : 1.f;
                                    Y[static_cast<size_t>(m) * a.N + n] = __float2bfloat16_rn(acc[i] * r);
                                }
                            }
                        }
                    }
                    if (e == 0) a.counters[nt] = 0;
                }
                tc_fence_before();
                mbar_arrive(accempty(buf));
                if (!go || !epi_sync()) break;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, a.tmem_cols);
    }
}

// ------------------------------------------------------------ unfused RMSNorm
constexpr int kNormThreads = 256;

__global__ void __launch_bounds__(kNormThreads)
    rmsnorm_kernel(const __nv_bfloat16* __restrict__ X, const __nv_bfloat16* __restrict__ g,
                   __nv_bfloat16* __restrict__ Xn, int K, float eps) {
    const size_t m = blockIdx.x;
    const uint4* xr = reinterpret_cast<const uint4*>(X + m * K);
    const uint4* gr = reinterpret_cast<const uint4*>(g);
    uint4* yr = reinterpret_cast<uint4*>(Xn + m * K);
    const int chunks = K / 8;
    float ss = 0.f;
    for (int c = threadIdx.x; c < chunks; c += kNormThreads) {
        const uint4 v = __ldg(xr + c);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float x0 = bf16lo(w[i]), x1 = bf16hi(w[i]);
            ss = fmaf(x0, x0, ss);
            ss = fmaf(x1, x1, ss);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    __shared__ float part[kNormThreads / 32];
    __shared__ float r_sh;
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float tot = 0.f;
        for (int i = 0; i < kNormThreads / 32; ++i) tot += part[i];
        r_sh = rsqrtf(tot / static_cast<float>(K) + eps);
    }
    __syncthreads();
    const float r = r_sh;
    for (int c = threadIdx.x; c < chunks; c += kNormThreads) {
        const uint4 v = __ldg(xr + c);
        const uint4 gv = __ldg(gr + c);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            o[i] = pack_bf16x2(bf16lo(w[i]) * bf16lo(gw[i]) * r, bf16hi(w[i]) * bf16hi(gw[i]) * r);
        yr[c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// Raises a kernel's dynamic shared-memory limit to the device's opt-in
// maximum, once per (kernel slot, device).
cudaError_t ensure_smem_attr(const void* func, int slot) {
    static int done[4][64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && done[slot][dev]) return cudaSuccess;
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
    if (e == cudaSuccess && dev < 64) done[slot][dev] = 1;
    return e;
}

}  // namespace

size_t rows_smem_bytes() { return kRowsSmem; }
size_t cols_smem_bytes(int MP, int stages) { return cols_layout(MP, stages).total; }
size_t cols_fixed_smem_bytes() { return cols_layout(16, 0).total; }
size_t cols_stage_bytes(int MP) { return kColsBN * kBK * 2 + MP * kBK * 2 + kGBytes; }

cudaError_t launch_rows(bool fused, const CUtensorMap& tmX, const CUtensorMap& tmW,
                        const CUtensorMap& tmG, void* Y, const RowsLaunch& a, cudaStream_t s) {
    auto* y = static_cast<__nv_bfloat16*>(Y);
    cudaError_t e;
    if (fused) {
        e = ensure_smem_attr(reinterpret_cast<const void*>(rows_kernel<true>), 0);
        if (e != cudaSuccess) return e;
        rows_kernel<true><<<a.grid, kThreads, kRowsSmem, s>>>(tmX, tmW, tmG, y, a.M, a.N, a.K,
                                                              a.eps, a.m_tiles, a.n_tiles,
                                                              a.k_blocks);
    } else {
        e = ensure_smem_attr(reinterpret_cast<const void*>(rows_kernel<false>), 1);
        if (e != cudaSuccess) return e;
        rows_kernel<false><<<a.grid, kThreads, kRowsSmem, s>>>(tmX, tmW, tmG, y, a.M, a.N, a.K,
                                                               a.eps, a.m_tiles, a.n_tiles,
                                                               a.k_blocks);
    }
    return cudaGetLastError();
}

cudaError_t launch_cols(bool fused, const CUtensorMap& tmX, const CUtensorMap& tmW,
                        const CUtensorMap& tmG, void* Y, const ColsLaunch& a, cudaStream_t s) {
    auto* y = static_cast<__nv_bfloat16*>(Y);
    const size_t smem = cols_smem_bytes(a.MP, a.stages);
    cudaError_t e;
    if (fused) {
        e = ensure_smem_attr(reinterpret_cast<const void*>(cols_kernel<true>), 2);
        if (e != cudaSuccess) return e;
        cols_kernel<true><<<a.grid, kThreads, smem, s>>>(tmX, tmW, tmG, y, a);
    } else {
        e = ensure_smem_attr(reinterpret_cast<const void*>(cols_kernel<false>), 3);
        if (e != cudaSuccess) return e;
        cols_kernel<false><<<a.grid, kThreads, smem, s>>>(tmX, tmW, tmG, y, a);
    }
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const void* X, const void* g, void* Xn, int M, int K, float eps,
                           cudaStream_t s) {
    rmsnorm_kernel<<<M, kNormThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(X),
                                             static_cast<const __nv_bfloat16*>(g),
                                             static_cast<__nv_bfloat16*>(Xn), K, eps);
    return cudaGetLastError();
}

cudaError_t read_and_clear_status(int* out) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_status, sizeof(int));
    if (e != cudaSuccess) return e;
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
    *out = v;
    return e;
}

}  // namespace rmm
