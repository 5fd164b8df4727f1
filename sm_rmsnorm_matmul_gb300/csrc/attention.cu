// attention.cu -- QK-normalised attention on sm_103a.
//
// The operation is the "QKNorm + Attention" workload of the Mirage review
// page's benchmark table (section 5): per-head RMSNorm with a gain on every
// query and key head, then softmax attention (causal or full) with grouped
// key/value heads.  Two kernels:
//
//   rmsnorm_heads_kernel    normalises every key head once (memory-bound; one
//                           warp per head row), into a bf16 workspace, with
//                           the query gain gq folded in: Kg = bf16(Kn * gq);
//   qknorm_attention_kernel one CTA per 256 query rows of one head (two
//                           128-row tiles): for each 128-key tile S' = Q Kg^T
//                           (the raw bf16 queries) and O += P V on the tensor
//                           cores (tcgen05, accumulators in tensor memory),
//                           with the online softmax between them.
//
// The query normalisation is a row scale: <Qn_i, Kn_j> = r_i <Q_i * gq, Kn_j>
// = r_i <Q_i, Kg_j> with r_i = 1 / sqrt(mean(Q_i^2) + eps), so the kernel
// multiplies row i of S' by r_i * scale * log2(e) inside the softmax (one
// fused multiply-add that also subtracts the running maximum), and the MMA
// reads the query tile as it was loaded.  Normalising each key once, not
// once per query tile that reads it, is the choice for GB300: a key tile is
// read by S/128 query tiles of every head in its group, and the workspace
// round trip costs two reads of K.
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

// Y[t,h,:] = bf16(X[t,h,:] * g * g2 * rsqrt(mean(X[t,h,:]^2) + eps)), one
// warp per (t, h); g2 is an optional second gain (nullptr: none), the
// products in fp32 and one rounding.  D is a multiple of 8 and at most 256:
// lane l holds elements [8l, 8l + 8) when 8l < D.
__global__ void __launch_bounds__(kHeadsWarps * 32)
    rmsnorm_heads_kernel(const __nv_bfloat16* __restrict__ X, int64_t ldx,
                         const __nv_bfloat16* __restrict__ g, const __nv_bfloat16* __restrict__ g2,
                         __nv_bfloat16* __restrict__ Y, int64_t ldy, int64_t T, int H, int D,
                         float eps) {
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
        float gf[8] = {bf16lo(gu.x), bf16hi(gu.x), bf16lo(gu.y), bf16hi(gu.y),
                       bf16lo(gu.z), bf16hi(gu.z), bf16lo(gu.w), bf16hi(gu.w)};
        if (g2 != nullptr) {
            const uint4 hu = __ldg(reinterpret_cast<const uint4*>(g2 + lane * 8));
            const float hf[8] = {bf16lo(hu.x), bf16hi(hu.x), bf16lo(hu.y), bf16hi(hu.y),
                                 bf16lo(hu.z), bf16hi(hu.z), bf16lo(hu.w), bf16hi(hu.w)};
#pragma unroll
            for (int i = 0; i < 8; ++i) gf[i] *= hf[i];
        }
        uint32_t out[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            out[i] = pack_bf16x2(v[2 * i] * gf[2 * i] * r, v[2 * i + 1] * gf[2 * i + 1] * r);
        *reinterpret_cast<uint4*>(Y + t * ldy + h * D + lane * 8) =
            make_uint4(out[0], out[1], out[2], out[3]);
    }
}

// ------------------------------------------------------- attention kernel
// One CTA per block of 256 query rows of one head: two 128-row query tiles,
// A (rows q0 .. q0 + 127) and B (q0 + 128 .. q0 + 255), each with its own
// score buffer, output accumulator, group of four softmax warps and MMA
// issuing thread.  The issuers take turns, A then B for every key tile
// (a pair of turn barriers): that keeps the two tiles half a period apart, so
// the tensor cores work on one tile's products while the other tile's
// softmax runs, and each issuer does its waits and releases while the other
// one issues (an issuing thread stalls whenever the tensor pipe's queue is
// full, so a single issuer's own waits leave the pipe idle).  Without the
// turns the two issuers drift into step and both softmaxes run while the
// pipe idles.  Both tiles read the same K and V tiles, loaded once: stage j
// of the ring holds V_j and K_{j+1} (K_0 has a barrier of its own).
constexpr int kAttThreads = 352;    // warp 0 TMA, 1 MMA A + TMEM, 2-5 softmax A, 6-9 softmax B, 10 MMA B
constexpr int kAttStages = 2;       // K and V slots
constexpr uint32_t kAttTile = kAttBM * kAttD * 2;   // 32 KB: a Q, K or V tile
constexpr uint32_t kAttHalf = kAttTile / 2;         // 64 columns of a tile (SW128 box)
constexpr uint32_t kAttOffQ = 0;                    // Q tiles A and B, later the O staging
constexpr uint32_t kAttOffK = kAttOffQ + 2 * kAttTile;
constexpr uint32_t kAttOffV = kAttOffK + kAttStages * kAttTile;
constexpr uint32_t kAttOffBar = kAttOffV + kAttStages * kAttTile;
constexpr uint32_t kAttNumBars = 15;
constexpr uint32_t kAttOffMisc = kAttOffBar + 256;
constexpr uint32_t kAttSmem = kAttOffMisc + 16 + 1024;   // + alignment slack
static_assert(kAttNumBars * 8 <= 256, "barrier area");
// Tensor memory, per query tile X (columns X * 256 ..): the score buffer S
// (P overwrites its first 64 columns, two bf16 per column), then O.
constexpr uint32_t kAttColO = 128, kAttTmemCols = 512;
constexpr float kAttRescale = 8.f;   // rescale O only when the row max grows by > 2^8

__global__ void __launch_bounds__(kAttThreads, 1)
    qknorm_attention_kernel(const __grid_constant__ CUtensorMap tmQ,
                            const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV,
                            const __grid_constant__ CUtensorMap tmO, AttnLaunch a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sq = sbase + kAttOffQ, sk = sbase + kAttOffK, sv = sbase + kAttOffV;
    const uint32_t bar0 = sbase + kAttOffBar;
    const uint32_t q_full = bar0, k0_full = bar0 + 8;
    auto turn = [&](int x) { return bar0 + 16 + 8 * x; };   // issuer x may issue
    auto kv_full = [&](uint32_t i) { return bar0 + 32 + 8 * i; };
    auto kv_empty = [&](uint32_t i) { return bar0 + 48 + 8 * i; };
    auto s_full = [&](int x) { return bar0 + 64 + 8 * x; };
    auto p_full = [&](int x) { return bar0 + 80 + 8 * x; };
    auto o_final = [&](int x) { return bar0 + 96 + 8 * x; };
    const uint32_t mmadone = bar0 + 112;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kAttOffMisc);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + kAttOffMisc + 4);

    // the block: query rows [q0, q0 + 256) of head h in sequence b; causal
    // launches take the longest rows (the last blocks) first
    const int bid = blockIdx.x;
    const int qb = a.causal ? a.n_qb - 1 - bid / a.n_hb : bid / a.n_hb;
    const int hb = bid % a.n_hb;
    const int h = hb % a.Hq, b = hb / a.Hq;
    const int c = h / a.group;
    const int q0 = qb * 2 * kAttBM;
    const int n_kv_all = (a.S + kAttBN - 1) / kAttBN;
    // key tiles each query tile visits (tile B may lie past the sequence end)
    auto tiles_of = [&](int x) {
        const int qt = 2 * qb + x;
        return q0 + x * kAttBM >= a.S ? 0 : a.causal ? min(qt + 1, n_kv_all) : n_kv_all;
    };
    const int n_a = tiles_of(0), n_b = tiles_of(1);
    auto n_x = [&](int x) { return x ? n_b : n_a; };
    const int n_kv = max(n_a, n_b);

    if (threadIdx.x == 0) {
        if (blockDim.x != kAttThreads) atomicCAS(&g_status, 0, kStatusInternal);
        mbar_init(q_full, 1);
        mbar_init(k0_full, 1);
        for (int x = 0; x < 2; ++x) {
            mbar_init(s_full(x), 1);
            mbar_init(p_full(x), 4);
            mbar_init(o_final(x), 1);
        }
        for (int i = 0; i < kAttStages; ++i) {
            mbar_init(kv_full(i), 1);
            mbar_init(kv_empty(i), 2);   // one commit per issuer
        }
        mbar_init(turn(0), 1);
        mbar_init(turn(1), 1);
        mbar_init(mmadone, 2);
        abort[0] = blockDim.x != kAttThreads;
        abort[1] = a.wait_limit_us;
        fence_mbar_init();
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmO);
    }
    if (warp == 1) {
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
            const uint64_t once = policy_evict_first();  // the query tiles are read once
            mbar_arrive_expect_tx(q_full, 2 * kAttTile);
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                tma_load_3d(sq + x * kAttTile, &tmQ, q_full, h * kAttD, q0 + x * kAttBM, b, once);
                tma_load_3d(sq + x * kAttTile + kAttHalf, &tmQ, q_full, h * kAttD + 64,
                            q0 + x * kAttBM, b, once);
            }
            mbar_arrive_expect_tx(k0_full, kAttTile);
            tma_load_3d(sk, &tmK, k0_full, c * kAttD, 0, b, keep);
            tma_load_3d(sk + kAttHalf, &tmK, k0_full, c * kAttD + 64, 0, b, keep);
            int issued = 0;
            for (int j = 0; j < n_kv; ++j) {
                const uint32_t st = j & 1;
                // V slot j & 1 held V_{j-2} and K slot (j+1) & 1 held K_{j-1};
                // both are released by the issuers' commits after key tile
                // j - 2 (for j = 1: after S(0), which read K_0)
                if (j >= 1) {
                    const uint32_t par = (j & 1) ? ((j - 1) >> 1) & 1 : ((j >> 1) - 1) & 1;
                    if (!mbar_wait(kv_empty(st), par, abort)) break;
                }
                const bool kn = j + 1 < n_kv;
                mbar_arrive_expect_tx(kv_full(st), kn ? 2 * kAttTile : kAttTile);
                const uint32_t vd = sv + st * kAttTile;
                // four boxes of [64 keys][64 dims]: box (kk, n) at (2 kk + n) * 8 KB
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                    for (int n = 0; n < 2; ++n)
                        tma_load_3d(vd + (2 * kk + n) * (kAttTile / 4), &tmV, kv_full(st),
                                    c * kAttD + n * 64, j * kAttBN + kk * 64, b, keep);
                if (kn) {
                    const uint32_t kd = sk + ((j + 1) & 1) * kAttTile;
                    tma_load_3d(kd, &tmK, kv_full(st), c * kAttD, (j + 1) * kAttBN, b, keep);
                    tma_load_3d(kd + kAttHalf, &tmK, kv_full(st), c * kAttD + 64, (j + 1) * kAttBN, b,
                                keep);
                }
                ++issued;
            }
            // never leave with copies still landing in shared memory
            mbar_wait_teardown(q_full, 0);
            mbar_wait_teardown(k0_full, 0);
            for (int i = issued > kAttStages ? issued - kAttStages : 0; i < issued; ++i)
                mbar_wait_teardown(kv_full(i & 1), (i >> 1) & 1);
        }
    } else if (warp == 1 || warp == 10) {
        // ------------------------------------------------ MMA issuer of tile x
        if (lane == 0) {
            const int x = warp == 1 ? 0 : 1;
            const int n = n_x(x);
            constexpr uint32_t idesc_s = idesc_bf16_f32(kAttBM, kAttBN, false, false);
            constexpr uint32_t idesc_o = idesc_bf16_f32(kAttBM, kAttD, false, true);
            // Descriptors are built once; a step adds its byte offset >> 4 to
            // the start-address field (every tile lies below 256 KB, so the
            // 14-bit field never carries).
            const uint64_t dq = sdesc_sw128(sq + x * kAttTile, 16, 1024);
            const uint64_t dk0 = sdesc_sw128(sk, 16, 1024), dk1 = sdesc_sw128(sk + kAttTile, 16, 1024);
            const uint64_t dv0 = sdesc_sw128(sv, kAttTile / 4, 1024);
            const uint64_t dv1 = sdesc_sw128(sv + kAttTile, kAttTile / 4, 1024);
            const uint32_t dS = tmem + x * 256;
            // S = Q_x Kg^T into the tile's score buffer: A and B K-major, 8 steps of 16 dims
            auto issue_s = [&](uint32_t kslot) {
                const uint64_t b0 = kslot ? dk1 : dk0;
#pragma unroll
                for (int kk = 0; kk < kAttD / 16; ++kk) {
                    const uint64_t off = ((kk >> 2) * kAttHalf + (kk & 3) * 32) >> 4;
                    mma_bf16_ss(dS, dq + off, b0 + off, idesc_s, kk > 0);
                }
                mma_commit(s_full(x));
            };
            // O_x += P V: A = P from tensor memory (keys 16kk.. in columns
            // 8kk..), B = V MN-major (dims contiguous), 8 steps of 16 keys
            auto issue_pv = [&](uint32_t vslot, bool acc) {
                const uint64_t b0 = vslot ? dv1 : dv0;
#pragma unroll
                for (int kk = 0; kk < kAttBN / 16; ++kk) {
                    const uint64_t off = ((kk >> 2) * (kAttTile / 2) + (kk & 3) * 2048) >> 4;
                    mma_bf16_ts(dS + kAttColO, dS + kk * 8, b0 + off, idesc_o, acc || kk > 0);
                }
            };
            bool ok = mbar_wait(k0_full, 0, abort) && mbar_wait(q_full, 0, abort);
            if (ok) {
                tc_fence_after();
                if (n > 0) issue_s(0);
                mma_commit(kv_empty(1));   // K_0 read: "key tile -1" of stage 1
            }
            // Each issuer waits for stage j before releasing it, so neither
            // releases a stage twice before the other released it once.  The
            // turn passes A -> B -> A every key tile, also through an issuer
            // that has nothing left to issue.
            for (int j = 0; ok && j < n_kv; ++j) {
                const uint32_t st = j & 1;
                if (!mbar_wait(kv_full(st), (j >> 1) & 1, abort)) break;
                if (j < n && !mbar_wait(p_full(x), j & 1, abort)) break;
                // A's turn for tile j is B's hand-back from tile j - 1 (none for j = 0)
                if ((x == 1 || j > 0) && !mbar_wait(turn(x), (x == 0 ? j - 1 : j) & 1, abort)) break;
                if (j < n) {
                    tc_fence_after();
                    issue_pv(st, j > 0);
                    if (j + 1 < n) issue_s((j + 1) & 1);
                    else mma_commit(o_final(x));
                }
                mbar_arrive(turn(x ^ 1));
                mma_commit(kv_empty(st));
            }
            mma_commit(mmadone);
            mbar_wait_teardown(mmadone, 0);
        }
    } else {
        // ------------------------------------------------ softmax warps of tile x
        const int x = (warp - 2) >> 2;          // 0: tile A (warps 2-5), 1: tile B (6-9)
        const int q = warp & 3;                  // lane quarter of tensor memory
        const int row = q * 32 + lane;           // query row of the tile
        const int qt = 2 * qb + x;
        const int qpos = qt * kAttBM + row;
        const int n = n_x(x);
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t swz = static_cast<uint32_t>(row & 7);
        const uint32_t srow = sq + x * kAttTile + static_cast<uint32_t>(row) * 128;
        bool ok = warp_wait(q_full, 0, abort);
        // the row's scale r * scale * log2(e) (the query tile is only read:
        // the first products run on it meanwhile)
        float ss[4] = {0.f, 0.f, 0.f, 0.f};
        if (ok) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const uint4 u = lds128(srow + hf * kAttHalf + ((cc ^ swz) << 4));
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        ss[i] = fmaf(bf16lo(w[i]), bf16lo(w[i]), ss[i]);
                        ss[i] = fmaf(bf16hi(w[i]), bf16hi(w[i]), ss[i]);
                    }
                }
        }
        const float rc = rsqrtf(((ss[0] + ss[1]) + (ss[2] + ss[3])) * (1.f / kAttD) + a.eps) * a.qscale;
        const uint64_t rc2 = pack_f32x2(rc, rc);
        const uint32_t sbuf = tmem + x * 256 + lane_base;
        const uint32_t obuf = sbuf + kAttColO;
        float m_ref = 0.f, l = 0.f;
        for (int j = 0; ok && j < n; ++j) {
            if (!warp_wait(s_full(x), j & 1, abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t v[kAttBN];
            tmem_ld_32x32_x128(sbuf, v);
            // keys past the sequence end, and after the query when causal
            const int kbase = j * kAttBN;
            int lim = min(kAttBN, a.S - kbase);
            if (a.causal && j == qt) lim = min(lim, qpos - kbase + 1);
            if (lim < kAttBN) {
#pragma unroll
                for (int i = 0; i < kAttBN; ++i)
                    if (i >= lim) v[i] = 0xff800000u;   // -inf
            }
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int i = 0; i < kAttBN; i += 8) {
                mx[0] = max3f(mx[0], __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
                mx[1] = max3f(mx[1], __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
                mx[2] = max3f(mx[2], __uint_as_float(v[i + 4]), __uint_as_float(v[i + 5]));
                mx[3] = max3f(mx[3], __uint_as_float(v[i + 6]), __uint_as_float(v[i + 7]));
            }
            // rc > 0: the maximum of the scaled scores is rc times the maximum
            const float m_tile = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * rc;
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
            const uint64_t negm = pack_f32x2(-m_ref, -m_ref);
            uint64_t acc[4] = {0, 0, 0, 0};   // packed partial row sums (0.0f pairs)
            uint32_t pk[kAttBN / 2];
#pragma unroll
            for (int i = 0; i < kAttBN / 2; ++i) {
                const uint64_t d = fma_f32x2(pack_f32x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])),
                                             rc2, negm);
                const float p0 = ex2_approx(lo_f32(d)), p1 = ex2_approx(hi_f32(d));
                acc[i & 3] = add_f32x2(acc[i & 3], pack_f32x2(p0, p1));
                pk[i] = pack_bf16x2(p0, p1);
            }
            tmem_st_32x32_x64(sbuf, pk);
            const uint64_t t = add_f32x2(add_f32x2(acc[0], acc[1]), add_f32x2(acc[2], acc[3]));
            l += lo_f32(t) + hi_f32(t);
            if (__any_sync(0xffffffffu, rescale)) {
                // O holds P_0..P_{j-1} V, complete: S_j was issued after the
                // last of those products and has completed
#pragma unroll 1
                for (int cc = 0; cc < kAttD / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld_32x32(obuf + cc * 32, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st_32x32(obuf + cc * 32, o);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full(x));
        }
        // ------------------------------------------------ epilogue: O / l -> bf16 -> TMA store
        if (ok && n > 0) ok = warp_wait(o_final(x), 0, abort);
        if (ok && n > 0) {
            tc_fence_after();
            const float inv_l = 1.f / l;
            // staging in this tile's Q area (every MMA that read it has
            // completed): 128-byte swizzle, two 64-column halves
#pragma unroll
            for (int cc = 0; cc < kAttD / 32; ++cc) {
                uint32_t o[32];
                tmem_ld_32x32(obuf + cc * 32, o);
                const uint32_t dst = srow + (cc >> 1) * kAttHalf;
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    uint32_t o4[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        o4[i] = pack_bf16x2(__uint_as_float(o[8 * t + 2 * i]) * inv_l,
                                            __uint_as_float(o[8 * t + 2 * i + 1]) * inv_l);
                    const uint32_t chunk = static_cast<uint32_t>((cc & 1) * 4 + t);
                    sts128(dst + ((chunk ^ swz) << 4), make_uint4(o4[0], o4[1], o4[2], o4[3]));
                }
            }
            fence_proxy_async_smem();
        }
        named_bar_sync(2 + x, 128);
        if (row == 0 && n > 0 && !*abort) {
            const uint32_t src = sq + x * kAttTile;
            tma_store_3d(&tmO, src, h * kAttD, qt * kAttBM, b);
            tma_store_3d(&tmO, src + kAttHalf, h * kAttD + 64, qt * kAttBM, b);
            bulk_commit_group();
            bulk_wait_group_read<0>();   // the staging area is read; the writes complete on their own
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
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

cudaError_t launch_rmsnorm_heads(const void* X, int64_t ldx, const void* g, const void* g2, void* Y,
                                 int64_t ldy, int64_t T, int H, int D, float eps, cudaStream_t s) {
    const int64_t items = T * H;
    if (items <= 0) return cudaSuccess;
    const int64_t grid = (items + kHeadsWarps - 1) / kHeadsWarps;
    if (grid > INT32_MAX) return cudaErrorInvalidValue;
    return launch_pdl(rmsnorm_heads_kernel, static_cast<int>(grid), kHeadsWarps * 32, 0, s,
                      static_cast<const __nv_bfloat16*>(X), ldx,
                      static_cast<const __nv_bfloat16*>(g), static_cast<const __nv_bfloat16*>(g2),
                      static_cast<__nv_bfloat16*>(Y), ldy, T, H, D, eps);
}

cudaError_t launch_qknorm_attention(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                    const CUtensorMap& tmV, const CUtensorMap& tmO,
                                    const AttnLaunch& a, cudaStream_t s) {
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
    return launch_pdl(qknorm_attention_kernel, a.grid, kAttThreads, kAttSmem, s, tmQ, tmK, tmV, tmO, a);
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
