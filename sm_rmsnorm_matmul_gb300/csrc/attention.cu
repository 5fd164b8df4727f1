// attention.cu -- QK-normalised attention on sm_103a.
//
// The operation is the "QKNorm + Attention" workload of the Mirage review
// page's benchmark table (section 5): per-head RMSNorm with a gain on every
// query and key head, then softmax attention (causal or full) with grouped
// key/value heads.  Two launches:
//
//   rmsnorm_rows_kernel     normalises every key head once (memory-bound; one
//   (rmsnorm_heads_kernel   warp per token and all its heads, or one warp per
//    for other D)           head when D is not a power of two), into a bf16
//                           workspace, with the query gain gq folded in:
//                           Kg = bf16(Kn * gq);
//   qknorm_attention_kernel persistent, one CTA per SM walking blocks of 256
//                           query rows of one head (two 128-row tiles): for
//                           each 128-key tile S' = Q Kg^T (the raw bf16
//                           queries) and O += P V on the tensor cores
//                           (tcgen05, accumulators in tensor memory), with
//                           the online softmax between them.
//
// The query normalisation is a row scale: <Qn_i, Kn_j> = r_i <Q_i * gq, Kn_j>
// = r_i <Q_i, Kg_j> with r_i = 1 / sqrt(mean(Q_i^2) + eps), so the kernel
// multiplies row i of S' by r_i * scale * log2(e) inside the softmax (one
// fused multiply-add that also subtracts the running maximum), and the MMA
// reads the query tile as it was loaded.  Normalising each key once, not
// once per query tile that reads it, is the choice for GB300: a key tile is
// read by S/128 query tiles of every head in its group, and the workspace
// round trip costs one write and one read of the normalised keys.
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

// The same for head dimensions D = 8 << s (D / 8 chunks of 16 bytes divide
// a warp's 32 lanes): one warp per row t, all H heads at once.  The row's
// H * D elements are contiguous; lane l takes chunks l, l + 32, ... (so
// every 512 bytes of the row are one coalesced warp access, and all of a
// lane's loads are issued before any arithmetic), and a head's D / 8 chunks
// sit in D / 8 consecutive lanes, summed with xor shuffles inside that group.
template <int kChunksMax>
__global__ void __launch_bounds__(kHeadsWarps * 32)
    rmsnorm_rows_kernel(const __nv_bfloat16* __restrict__ X, int64_t ldx,
                        const __nv_bfloat16* __restrict__ g, const __nv_bfloat16* __restrict__ g2,
                        __nv_bfloat16* __restrict__ Y, int64_t ldy, int64_t T, int H, int D,
                        float eps) {
    grid_dep_wait();
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kHeadsWarps + warp;
    if (t >= T) return;
    const int gsz = D >> 3;                    // lanes (chunks) per head: 1 .. 32
    const int n_chunks = H * gsz;
    const int n_iter = (n_chunks + 31) >> 5;   // <= kChunksMax
    const __nv_bfloat16* x = X + t * ldx;
    __nv_bfloat16* y = Y + t * ldy;
    uint4 u[kChunksMax];
#pragma unroll
    for (int i = 0; i < kChunksMax; ++i) {
        const int ch = lane + 32 * i;
        u[i] = (i < n_iter && ch < n_chunks) ? __ldg(reinterpret_cast<const uint4*>(x) + ch)
                                             : make_uint4(0, 0, 0, 0);
    }
    const float inv_d = 1.f / static_cast<float>(D);
#pragma unroll
    for (int i = 0; i < kChunksMax; ++i) {
        if (i >= n_iter) break;
        const int ch = lane + 32 * i;
        const uint32_t w[4] = {u[i].x, u[i].y, u[i].z, u[i].w};
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            ss = fmaf(bf16lo(w[k]), bf16lo(w[k]), ss);
            ss = fmaf(bf16hi(w[k]), bf16hi(w[k]), ss);
        }
        for (int o = 1; o < gsz; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (ch >= n_chunks) continue;
        const float r = rsqrtf(ss * inv_d + eps);
        const int d0 = (ch % gsz) * 8;        // position of the chunk within its head
        const uint4 gu = __ldg(reinterpret_cast<const uint4*>(g + d0));
        float gf[8] = {bf16lo(gu.x), bf16hi(gu.x), bf16lo(gu.y), bf16hi(gu.y),
                       bf16lo(gu.z), bf16hi(gu.z), bf16lo(gu.w), bf16hi(gu.w)};
        if (g2 != nullptr) {
            const uint4 hu = __ldg(reinterpret_cast<const uint4*>(g2 + d0));
            const float hf[8] = {bf16lo(hu.x), bf16hi(hu.x), bf16lo(hu.y), bf16hi(hu.y),
                                 bf16lo(hu.z), bf16hi(hu.z), bf16lo(hu.w), bf16hi(hu.w)};
#pragma unroll
            for (int k = 0; k < 8; ++k) gf[k] *= hf[k];
        }
        uint32_t out[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            out[k] = pack_bf16x2(bf16lo(w[k]) * gf[2 * k] * r, bf16hi(w[k]) * gf[2 * k + 1] * r);
        reinterpret_cast<uint4*>(y)[ch] = make_uint4(out[0], out[1], out[2], out[3]);
    }
}

// ------------------------------------------------------- attention kernel
// A persistent CTA per SM walks its blocks of 256 query rows.  Blocks are
// numbered longest first when causal; CTA c of G takes block r G + c from
// each even band r of G blocks and (r + 1) G - 1 - c from each odd band (a
// zig-zag, so that every CTA gets a similar total of key tiles: a plain
// stride left the heaviest CTA 30% above the mean).  A block holds
// two 128-row query tiles, A (rows q0 .. q0 + 127) and B (q0 + 128 ..), each
// with its own score buffer, output accumulator, group of four softmax warps
// and MMA issuing thread.  The softmax hands P over in two halves of 64
// keys, so the P V of the first half runs during the second half's
// exponentials.  For D = 128, where P overwrites half of the score buffer,
// the issuers take turns, A then B for every key tile (a pair of turn
// barriers): that keeps the two tiles half a period apart, so the tensor
// cores work on one tile's products while the other tile's softmax runs, and
// each issuer does its waits and releases while the other one issues (an
// issuing thread stalls whenever the tensor pipe's queue is full).  Without
// the turns the two issuers drift into step and both softmaxes run while the
// pipe idles.  For D = 64, P has tensor-memory columns of its own: the next
// score product runs as soon as the softmax has read the scores, the softmax
// never waits for a P V of its own tile, and the issuers take no turns.
//
// Both tiles read the same K and V tiles, loaded once, as one stream across
// the CTA's blocks: stage g of a two-deep ring holds V_j of the current
// block and the next K tile of the stream, K_{j+1}, or for the block's last
// stage the next block's K_0 (the very first K_0 has a barrier of its own).
// The next block's query tiles load as soon as the current block's last
// score products have completed and its row norms have been read, during the
// block's last key tile; an issuer starts the next block's first products
// right after its last ones of the current block, and O leaves through plain
// stores from the softmax threads, so blocks follow each other without a
// gap.  Every barrier's parity is a count kept by the roles that use it.
constexpr int kAttThreads = 352;    // warp 0 TMA, 1 MMA A + TMEM, 2-5 softmax A, 6-9 softmax B, 10 MMA B
constexpr int kAttStages = 2;       // K and V slots
constexpr uint32_t kAttBox = kAttBM * 64 * 2;      // 16 KB: [128 rows][64 columns], one SW128 box
constexpr uint32_t kAttNumBars = 26;
static_assert(kAttNumBars * 8 <= 256, "barrier area");
// Shared memory for head dimension D: query tiles A and B, two K and two V
// tiles (each [128][D]), barriers, the TMEM address and abort words.
constexpr uint32_t att_tile_bytes(int D) { return kAttBM * D * 2; }
constexpr uint32_t att_off_bar(int D) { return (2 + 2 * kAttStages) * att_tile_bytes(D); }
constexpr uint32_t att_smem_bytes(int D) { return att_off_bar(D) + 256 + 16 + 1024; }   // + alignment slack
// Tensor memory, per query tile x (columns x * 256 ..): the score buffer S
// (128 columns), then O (D columns).  P (two bf16 per column, 64 columns)
// overwrites the first half of S for D = 128; for D = 64 it has the last 64
// columns to itself, so the next S can be computed while P is.
constexpr uint32_t kAttColO = 128, kAttTmemCols = 512;
constexpr uint32_t att_col_p(int D) { return D == 64 ? kAttColO + 64 : 0; }
constexpr float kAttRescale = 8.f;   // rescale O only when the row max grows by > 2^8
// Scores of normalised queries and keys are bounded (Cauchy-Schwarz): with
// G = max_i |gq_i gk_i|, |rc S| <= qscale * D * G.  Up to a bound of 50 (in
// log2 units) every softmax weight 2^(s - bound) stays above 2^-100, a normal
// float, and the bound serves as the reference instead of a running maximum.
constexpr float kAttBoundMax = 50.f;

// One block of 256 query rows of one head of one sequence.
struct AttnBlock {
    int qb, h, b, c, q0;
    int n0, n1;  // key tiles query tiles A and B visit (0: tile past the sequence end)
    int nkv;     // max(n0, n1)
    __device__ __forceinline__ int n(int x) const { return x ? n1 : n0; }
};

__device__ __forceinline__ AttnBlock attn_block(const AttnLaunch& a, int k) {
    AttnBlock B;
    B.qb = a.causal ? a.n_qb - 1 - k / a.n_hb : k / a.n_hb;
    const int hb = k % a.n_hb;
    B.h = hb % a.Hq;
    B.b = hb / a.Hq;
    B.c = B.h / a.group;
    B.q0 = B.qb * 2 * kAttBM;
    const int n_all = (a.S + kAttBN - 1) / kAttBN;
    auto tiles = [&](int x) {
        const int qt = 2 * B.qb + x;
        return B.q0 + x * kAttBM >= a.S ? 0 : a.causal ? min(qt + 1, n_all) : n_all;
    };
    B.n0 = tiles(0);
    B.n1 = tiles(1);
    B.nkv = max(B.n0, B.n1);
    return B;
}

template <int kD>   // head dimension: 64 or 128
__global__ void __launch_bounds__(kAttThreads, 1)
    qknorm_attention_kernel(const __grid_constant__ CUtensorMap tmQ,
                            const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, AttnLaunch a) {
    static_assert(kD == 64 || kD == 128, "head dimension");
    // P apart from S: the next score product does not wait for this P V
    constexpr bool kPSep = att_col_p(kD) != 0;
    constexpr uint32_t kTile = att_tile_bytes(kD);   // a Q, K or V tile
    constexpr int kBoxes = kD / 64;                  // SW128 boxes of 64 columns per tile
    constexpr uint32_t kOffK = 2 * kTile, kOffV = kOffK + kAttStages * kTile;
    constexpr uint32_t kOffBar = att_off_bar(kD), kOffMisc = kOffBar + 256;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sq = sbase, sk = sbase + kOffK, sv = sbase + kOffV;
    const uint32_t bar0 = sbase + kOffBar;
    const uint32_t q_full = bar0, q_empty = bar0 + 8, k0_full = bar0 + 16;
    auto kv_full = [&](uint32_t i) { return bar0 + 24 + 8 * i; };
    auto kv_empty = [&](uint32_t i) { return bar0 + 40 + 8 * i; };
    auto turn = [&](int x) { return bar0 + 56 + 8 * x; };      // issuer x may issue
    auto s_full = [&](int x) { return bar0 + 72 + 8 * x; };
    // P of keys 64h .. 64h + 63 of tile x is in tensor memory
    auto p_full = [&](int x, int h) { return h ? bar0 + 144 + 8 * x : bar0 + 88 + 8 * x; };
    // (P apart from S) the softmax has read S / the P V of key half h has completed
    auto s_empty = [&](int x) { return bar0 + 160 + 8 * x; };
    auto pv_done = [&](int x, int h) { return bar0 + 176 + 8 * (2 * x + h); };
    auto o_final = [&](int x) { return bar0 + 104 + 8 * x; };
    auto o_empty = [&](int x) { return bar0 + 120 + 8 * x; };
    const uint32_t mmadone = bar0 + 136;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
    // the CTA's r-th block, or -1 (once a band has none, no later band has)
    auto block_id = [&](int r) {
        const int G = gridDim.x, c = blockIdx.x;
        const int k = (r & 1) ? (r + 1) * G - 1 - c : r * G + c;
        return k < a.n_blocks ? k : -1;
    };

    if (threadIdx.x == 0) {
        if (blockDim.x != kAttThreads) atomicCAS(&g_status, 0, kStatusInternal);
        mbar_init(q_full, 1);
        mbar_init(q_empty, 2 + 8);   // a commit per issuer + one lane per softmax warp
        mbar_init(k0_full, 1);
        for (int x = 0; x < 2; ++x) {
            mbar_init(kv_full(x), 1);
            mbar_init(kv_empty(x), 2);   // one commit per issuer
            mbar_init(turn(x), 1);
            mbar_init(s_full(x), 1);
            mbar_init(p_full(x, 0), 4);  // one lane per softmax warp
            mbar_init(p_full(x, 1), 4);
            mbar_init(s_empty(x), 4);
            mbar_init(pv_done(x, 0), 1);
            mbar_init(pv_done(x, 1), 1);
            mbar_init(o_final(x), 1);
            mbar_init(o_empty(x), 4);
        }
        mbar_init(mmadone, 2);
        abort[0] = blockDim.x != kAttThreads;
        abort[1] = a.wait_limit_us;
        fence_mbar_init();
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
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
        if (lane == 0 && !*abort && block_id(0) >= 0) {
            const uint64_t keep = policy_evict_last();   // K and V tiles are re-read
            const uint64_t once = policy_evict_first();  // the query tiles are read once
            auto load_q = [&](const AttnBlock& B) {
                mbar_arrive_expect_tx(q_full, 2 * kTile);
#pragma unroll
                for (int x = 0; x < 2; ++x)
#pragma unroll
                    for (int bx = 0; bx < kBoxes; ++bx)
                        tma_load_3d(sq + x * kTile + bx * kAttBox, &tmQ, q_full, B.h * kD + bx * 64,
                                    B.q0 + x * kAttBM, B.b, once);
            };
            AttnBlock cur = attn_block(a, block_id(0));
            load_q(cur);
            mbar_arrive_expect_tx(k0_full, kTile);
#pragma unroll
            for (int bx = 0; bx < kBoxes; ++bx)
                tma_load_3d(sk + bx * kAttBox, &tmK, k0_full, cur.c * kD + bx * 64, 0, cur.b, keep);
            uint32_t g = 0;   // stages issued
            uint32_t t = 0;   // blocks begun
            bool ok = true;
            for (int r = 0; ok && block_id(r) >= 0; ++r, ++t) {
                const bool has_next = block_id(r + 1) >= 0;
                const AttnBlock nxt = has_next ? attn_block(a, block_id(r + 1)) : cur;
                for (int j = 0; j < cur.nkv; ++j, ++g) {
                    const uint32_t st = g & 1;
                    // V slot g & 1 held the V of stage g - 2 and K slot (g+1) & 1
                    // the K of stage g - 2 (the first K_0 for g = 1): both are
                    // released by the issuers' commits after stage g - 2
                    if (g >= 1) {
                        const uint32_t par = (g & 1) ? ((g - 1) >> 1) & 1 : ((g >> 1) - 1) & 1;
                        if (!mbar_wait(kv_empty(st), par, abort)) { ok = false; break; }
                    }
                    // test hook: leave out the first stage, so that the issuers'
                    // waits for it run out (the timeout path, without a fault)
                    if (a.test_skip_loads && g == 0) continue;
                    const bool last = j + 1 == cur.nkv;
                    const bool kn = !last || has_next;
                    mbar_arrive_expect_tx(kv_full(st), kn ? 2 * kTile : kTile);
                    const uint32_t vd = sv + st * kTile;
                    // boxes of [64 keys][64 dims]: box (kk, n) at (kBoxes kk + n) * 8 KB
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                        for (int n = 0; n < kBoxes; ++n)
                            tma_load_3d(vd + (kBoxes * kk + n) * (kAttBox / 2), &tmV, kv_full(st),
                                        cur.c * kD + n * 64, j * kAttBN + kk * 64, cur.b, keep);
                    if (kn) {
                        const uint32_t kd = sk + ((g + 1) & 1) * kTile;
                        const int kc = last ? nxt.c : cur.c, kj = last ? 0 : j + 1, kb = last ? nxt.b : cur.b;
#pragma unroll
                        for (int bx = 0; bx < kBoxes; ++bx)
                            tma_load_3d(kd + bx * kAttBox, &tmK, kv_full(st), kc * kD + bx * 64, kj * kAttBN,
                                        kb, keep);
                    }
                }
                if (!ok || !has_next) break;
                // the next block's query tiles, once this block's score
                // products have completed and its row norms have been read
                if (!mbar_wait(q_empty, t & 1, abort)) break;
                load_q(nxt);
                cur = nxt;
            }
            // never leave with copies still landing in shared memory
            mbar_wait_teardown(q_full, t & 1);
            mbar_wait_teardown(k0_full, 0);
            for (uint32_t i = g > kAttStages ? g - kAttStages : 0; i < g; ++i)
                mbar_wait_teardown(kv_full(i & 1), (i >> 1) & 1);
        }
    } else if (warp == 1 || warp == 10) {
        // ------------------------------------------------ MMA issuer of tile x
        if (lane == 0) {
            const int x = warp == 1 ? 0 : 1;
            constexpr uint32_t idesc_s = idesc_bf16_f32(kAttBM, kAttBN, false, false);
            constexpr uint32_t idesc_o = idesc_bf16_f32(kAttBM, kD, false, true);
            // Descriptors are built once; a step adds its byte offset >> 4 to
            // the start-address field (every tile lies below 256 KB, so the
            // 14-bit field never carries).
            const uint64_t dq = sdesc_sw128(sq + x * kTile, 16, 1024);
            const uint64_t dk0 = sdesc_sw128(sk, 16, 1024), dk1 = sdesc_sw128(sk + kTile, 16, 1024);
            const uint64_t dv0 = sdesc_sw128(sv, kAttBox / 2, 1024);
            const uint64_t dv1 = sdesc_sw128(sv + kTile, kAttBox / 2, 1024);
            const uint32_t dS = tmem + x * 256;
            // S = Q_x Kg^T into the tile's score buffer: A and B K-major, steps
            // k0 .. k1 - 1 of 8 (16 dims each)
            auto s_steps = [&](uint32_t kslot, int k0, int k1) {
                const uint64_t b0 = kslot ? dk1 : dk0;
#pragma unroll
                for (int kk = k0; kk < k1; ++kk) {
                    const uint64_t off = ((kk >> 2) * kAttBox + (kk & 3) * 32) >> 4;
                    mma_bf16_ss(dS, dq + off, b0 + off, idesc_s, kk > 0);
                }
            };
            uint32_t ns = 0;   // score tiles issued (P apart from S)
            auto issue_s = [&](uint32_t kslot) -> bool {
                if constexpr (kPSep) {
                    // the score buffer is free once the softmax has read the last S
                    if (ns > 0) {
                        if (!mbar_wait(s_empty(x), (ns - 1) & 1, abort)) return false;
                        tc_fence_after();
                    }
                    ++ns;
                }
                s_steps(kslot, 0, kD / 16);
                mma_commit(s_full(x));
                return true;
            };
            // O_x += P V: A = P from tensor memory (keys 16kk.. in columns
            // 8kk..), B = V MN-major (dims contiguous), steps k0 .. k1 - 1 of 8
            auto pv_steps = [&](uint32_t vslot, bool acc, int k0, int k1) {
                const uint64_t b0 = vslot ? dv1 : dv0;
#pragma unroll
                for (int kk = k0; kk < k1; ++kk) {
                    const uint64_t off = ((kk >> 2) * (kTile / 2) + (kk & 3) * 2048) >> 4;
                    mma_bf16_ts(dS + kAttColO, dS + att_col_p(kD) + kk * 8, b0 + off, idesc_o, acc || kk > 0);
                }
            };
            // the first score product of a block; a query tile with at most
            // one key tile has then read its query tile for the last time
            auto begin_block = [&](const AttnBlock& B, uint32_t kslot) -> bool {
                if (B.n(x) > 0 && !issue_s(kslot)) return false;
                if (B.n(x) <= 1) mma_commit(q_empty);
                return true;
            };
            uint32_t g = 0, t = 0, pi = 0;   // stages, blocks, P tiles consumed
            const bool any = block_id(0) >= 0;
            AttnBlock cur = attn_block(a, any ? block_id(0) : 0);
            bool ok = any && mbar_wait(k0_full, 0, abort) && mbar_wait(q_full, 0, abort);
            if (ok) {
                tc_fence_after();
                ok = begin_block(cur, 0);
                mma_commit(kv_empty(1));   // the first K_0 read: "stage -1" of slot 1
            }
            // Each issuer waits for stage g before releasing it, so neither
            // releases a stage twice before the other released it once.  The
            // turn passes A -> B -> A every stage, also through an issuer that
            // has nothing to issue in it.
            for (int r = 0; ok && block_id(r) >= 0; ++r, ++t) {
                const bool has_next = block_id(r + 1) >= 0;
                const AttnBlock nxt = has_next ? attn_block(a, block_id(r + 1)) : cur;
                const int n = cur.n(x);
                for (int j = 0; j < cur.nkv; ++j, ++g) {
                    const uint32_t st = g & 1;
                    if (!mbar_wait(kv_full(st), (g >> 1) & 1, abort)) { ok = false; break; }
                    if constexpr (kPSep) {
                        // S_{j+1} as soon as the softmax has read S_j, then
                        // P_j V in two halves as P_j's halves arrive (no turns:
                        // the softmax does not wait for P V)
                        if (j < n) {
                            if (j + 1 < n) {
                                if (!issue_s((g + 1) & 1)) { ok = false; break; }
                                if (j + 2 == n) mma_commit(q_empty);   // the last score product
                            }
                            if (j == 0 && t > 0 && !mbar_wait(o_empty(x), (t - 1) & 1, abort)) {
                                ok = false;
                                break;
                            }
                            if (!mbar_wait(p_full(x, 0), pi & 1, abort)) { ok = false; break; }
                            tc_fence_after();
                            pv_steps(st, j > 0, 0, 4);
                            mma_commit(pv_done(x, 0));
                            if (!mbar_wait(p_full(x, 1), pi & 1, abort)) { ok = false; break; }
                            tc_fence_after();
                            ++pi;
                            pv_steps(st, true, 4, kAttBN / 16);
                            mma_commit(pv_done(x, 1));
                            if (j + 1 == n) mma_commit(o_final(x));
                        }
                        if (j + 1 == cur.nkv && has_next) {
                            if (!mbar_wait(q_full, (t + 1) & 1, abort)) { ok = false; break; }
                            tc_fence_after();
                            if (!begin_block(nxt, (g + 1) & 1)) { ok = false; break; }
                        }
                        mma_commit(kv_empty(st));
                        continue;
                    }
                    if (j < n && !mbar_wait(p_full(x, 0), pi & 1, abort)) { ok = false; break; }
                    // the first P V of a block overwrites O: the previous
                    // block's epilogue has read it (one arrival per block)
                    if (j == 0 && n > 0 && t > 0 && !mbar_wait(o_empty(x), (t - 1) & 1, abort)) {
                        ok = false;
                        break;
                    }
                    // A's turn at stage g is B's hand-back from stage g - 1 (none at g = 0)
                    if ((x == 1 || g > 0) && !mbar_wait(turn(x), (x == 0 ? g - 1 : g) & 1, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // The turn passes four MMAs before the end of this issuer's
                    // work for the stage: the other issuer wakes while they
                    // are issued (its own MMAs do not depend on these).
                    // The P V of the first 64 keys runs while the softmax
                    // computes the second half of P.
                    if (j < n) {
                        pv_steps(st, j > 0, 0, 4);
                        if (!mbar_wait(p_full(x, 1), pi & 1, abort)) { ok = false; break; }
                        tc_fence_after();
                        ++pi;
                        if (j + 1 < n) {
                            pv_steps(st, true, 4, kAttBN / 16);
                            s_steps((g + 1) & 1, 0, 4);
                            mbar_arrive(turn(x ^ 1));
                            s_steps((g + 1) & 1, 4, kD / 16);
                            mma_commit(s_full(x));
                            if (j + 2 == n) mma_commit(q_empty);   // that was the last score product
                        } else {
                            mbar_arrive(turn(x ^ 1));
                            pv_steps(st, true, 4, kAttBN / 16);
                            mma_commit(o_final(x));
                        }
                    } else {
                        mbar_arrive(turn(x ^ 1));
                    }
                    if (j + 1 == cur.nkv && has_next) {
                        // the next block's first product (after the turn is
                        // handed over, so the other tile's last products do
                        // not wait for the load): its query tiles, loaded
                        // during this stage, and its K_0, in this stage
                        if (!mbar_wait(q_full, (t + 1) & 1, abort)) { ok = false; break; }
                        tc_fence_after();
                        if (!begin_block(nxt, (g + 1) & 1)) { ok = false; break; }
                    }
                    mma_commit(kv_empty(st));
                }
                cur = nxt;
            }
            mma_commit(mmadone);
            mbar_wait_teardown(mmadone, 0);
        }
    } else if (warp >= 2 && warp < 10) {
        // ------------------------------------------------ softmax warps of tile x
        const int x = (warp - 2) >> 2;          // 0: tile A (warps 2-5), 1: tile B (6-9)
        const int q = warp & 3;                  // lane quarter of tensor memory
        const int row = q * 32 + lane;           // query row of the tile
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t swz = static_cast<uint32_t>(row & 7);
        const uint32_t srow = sq + x * kTile + static_cast<uint32_t>(row) * 128;
        const uint32_t sbuf = tmem + x * 256 + lane_base;
        const uint32_t obuf = sbuf + kAttColO;
        uint32_t t = 0, si = 0, ob = 0;   // blocks, S tiles consumed, blocks with output
        // G = max |gq_i gk_i| (the same in every CTA, so is the choice below)
        float gm = 0.f;
        for (int i = lane; i < kD; i += 32)
            gm = fmaxf(gm, fabsf(__bfloat162float(static_cast<const __nv_bfloat16*>(a.gq)[i]) *
                                 __bfloat162float(static_cast<const __nv_bfloat16*>(a.gk)[i])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, o));
        // the bound, with a margin for the bf16 rounding of the keys and the
        // accumulation order
        gm *= 1.f + 1.f / 64;
        const bool bounded = a.qscale * kD * gm <= kAttBoundMax;
        bool ok = true;
        for (int r = 0; ok && block_id(r) >= 0; ++r, ++t) {
            const AttnBlock B = attn_block(a, block_id(r));
            const int n = B.n(x);
            const int qt = 2 * B.qb + x;
            const int qpos = qt * kAttBM + row;
            if (!warp_wait(q_full, t & 1, abort)) break;
            // the row's scale r * scale * log2(e); the query tile is only read
            float ss[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int hf = 0; hf < kBoxes; ++hf)
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const uint4 u = lds128(srow + hf * kAttBox + ((cc ^ swz) << 4));
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        ss[i] = fmaf(bf16lo(w[i]), bf16lo(w[i]), ss[i]);
                        ss[i] = fmaf(bf16hi(w[i]), bf16hi(w[i]), ss[i]);
                    }
                }
            __syncwarp();
            if (lane == 0) mbar_arrive(q_empty);
            const float rc = rsqrtf(((ss[0] + ss[1]) + (ss[2] + ss[3])) * (1.f / kD) + a.eps) * a.qscale;
            const uint64_t rc2 = pack_f32x2(rc, rc);
            // bounded: this row's own bound, rc |Q_row| sqrt(D) G (at most qscale D G)
            float m_ref = bounded ? rc * sqrtf(((ss[0] + ss[1]) + (ss[2] + ss[3])) * kD) * gm : 0.f;
            float l = 0.f;
            for (int j = 0; j < n; ++j, ++si) {
                if (!warp_wait(s_full(x), si & 1, abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t v[kAttBN];
                tmem_ld_32x32_x128(sbuf, v);
                if constexpr (kPSep) {   // S is in registers: the buffer may take the next S
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(s_empty(x));
                }
                // keys past the sequence end, and after the query when causal
                const int kbase = j * kAttBN;
                int lim = min(kAttBN, a.S - kbase);
                if (a.causal && j == qt) lim = min(lim, qpos - kbase + 1);
                if (lim < kAttBN) {
#pragma unroll
                    for (int i = 0; i < kAttBN; ++i)
                        if (i >= lim) v[i] = 0xff800000u;   // -inf
                }
                float alpha = 1.f;
                bool rescale = false;
                if (!bounded) {
                    // a running maximum: eight independent chains of three-input maxima
                    float mx[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        mx[c] = max3f(__uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1]),
                                      __uint_as_float(v[16 + 2 * c]));
#pragma unroll
                    for (int i = 32; i < kAttBN; i += 16)
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            mx[c] = max3f(mx[c], __uint_as_float(v[i + 2 * c]), __uint_as_float(v[i + 2 * c + 1]));
#pragma unroll
                    for (int c = 0; c < 8; ++c) mx[c] = fmaxf(mx[c], __uint_as_float(v[17 + 2 * c]));
                    // rc > 0: the maximum of the scaled scores is rc times the maximum
                    const float m_tile = fmaxf(fmaxf(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], mx[5])),
                                               fmaxf(mx[6], mx[7])) * rc;
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
                }
                // P in two halves of 64 keys (32 columns each), each handed
                // over as soon as it is stored: the P V of the first half
                // runs during the second half's exponentials
                const uint64_t negm = pack_f32x2(-m_ref, -m_ref);
                uint64_t acc[4] = {0, 0, 0, 0};   // packed partial row sums (0.0f pairs)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t pk[kAttBN / 4];
#pragma unroll
                    for (int i = 0; i < kAttBN / 4; ++i) {
                        const int e = hf * (kAttBN / 2) + 2 * i;
                        const uint64_t d = fma_f32x2(pack_f32x2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])),
                                                     rc2, negm);
                        const float p0 = ex2_approx(lo_f32(d)), p1 = ex2_approx(hi_f32(d));
                        acc[i & 3] = add_f32x2(acc[i & 3], pack_f32x2(p0, p1));
                        pk[i] = pack_bf16x2(p0, p1);
                    }
                    // (P apart from S) the last tile's P V has read this half
                    if (kPSep && si > 0 && !warp_wait(pv_done(x, hf), (si - 1) & 1, abort)) {
                        ok = false;
                        break;
                    }
                    tmem_st_32x32(sbuf + att_col_p(kD) + hf * (kAttBN / 4), pk);
                    if (hf == 0 && __any_sync(0xffffffffu, rescale)) {
                        // (P apart from S) O must hold all of the last tile's P V
                        if (kPSep && !warp_wait(pv_done(x, 1), (si - 1) & 1, abort)) {
                            ok = false;
                            break;
                        }
                        // O holds this block's P_0..P_{j-1} V, complete (with P
                        // in S: S_j was issued after the last of those products
                        // and has completed); P_j V starts once the first half
                        // is handed over
#pragma unroll 1
                        for (int cc = 0; cc < kD / 32; ++cc) {
                            uint32_t o[32];
                            tmem_ld_32x32(obuf + cc * 32, o);
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                            tmem_st_32x32(obuf + cc * 32, o);
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(p_full(x, hf));
                }
                if (!ok) break;
                const uint64_t tsum = add_f32x2(add_f32x2(acc[0], acc[1]), add_f32x2(acc[2], acc[3]));
                l += lo_f32(tsum) + hi_f32(tsum);
            }
            if (!ok) break;
            // ------------------------------------------------ epilogue: O / l -> bf16 -> global
            if (n > 0) {
                if (!warp_wait(o_final(x), ob & 1, abort)) break;
                ++ob;
                tc_fence_after();
                const float inv_l = 1.f / l;
                __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.O) +
                                      (static_cast<int64_t>(B.b) * a.S + qpos) * a.ldo + B.h * kD;
                const bool valid = qpos < a.S;
#pragma unroll
                for (int cc = 0; cc < kD / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld_32x32(obuf + cc * 32, o);
#pragma unroll
                    for (int t4 = 0; t4 < 4; ++t4) {
                        uint32_t o4[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            o4[i] = pack_bf16x2(__uint_as_float(o[8 * t4 + 2 * i]) * inv_l,
                                                __uint_as_float(o[8 * t4 + 2 * i + 1]) * inv_l);
                        if (valid)
                            *reinterpret_cast<uint4*>(orow + cc * 32 + t4 * 8) =
                                make_uint4(o4[0], o4[1], o4[2], o4[3]);
                    }
                }
                tc_fence_before();
            }
            // O of this tile is free for the next block's first product
            __syncwarp();
            if (lane == 0) mbar_arrive(o_empty(x));
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

size_t attn_smem_bytes(int D) { return att_smem_bytes(D); }

cudaError_t launch_rmsnorm_heads(const void* X, int64_t ldx, const void* g, const void* g2, void* Y,
                                 int64_t ldy, int64_t T, int H, int D, float eps, cudaStream_t s) {
    const int64_t items = T * H;
    if (items <= 0) return cudaSuccess;
    // D a power of two from 8 to 256 and a row of at most 8 warp-wide chunks:
    // one warp per row (the common case, e.g. 8 key heads of 128)
    const bool pow2 = D >= 8 && D <= 256 && (D & (D - 1)) == 0;
    if (pow2 && (static_cast<int64_t>(H) * (D / 8) + 31) / 32 <= 8) {
        const int64_t grid_r = (T + kHeadsWarps - 1) / kHeadsWarps;
        if (grid_r > INT32_MAX) return cudaErrorInvalidValue;
        return launch_pdl(rmsnorm_rows_kernel<8>, static_cast<int>(grid_r), kHeadsWarps * 32, 0, s,
                          static_cast<const __nv_bfloat16*>(X), ldx,
                          static_cast<const __nv_bfloat16*>(g), static_cast<const __nv_bfloat16*>(g2),
                          static_cast<__nv_bfloat16*>(Y), ldy, T, H, D, eps);
    }
    const int64_t grid = (items + kHeadsWarps - 1) / kHeadsWarps;
    if (grid > INT32_MAX) return cudaErrorInvalidValue;
    return launch_pdl(rmsnorm_heads_kernel, static_cast<int>(grid), kHeadsWarps * 32, 0, s,
                      static_cast<const __nv_bfloat16*>(X), ldx,
                      static_cast<const __nv_bfloat16*>(g), static_cast<const __nv_bfloat16*>(g2),
                      static_cast<__nv_bfloat16*>(Y), ldy, T, H, D, eps);
}

cudaError_t launch_qknorm_attention(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                    const CUtensorMap& tmV, const AttnLaunch& a, cudaStream_t s) {
    // the shared-memory limit is a per-device attribute of each function
    static std::atomic<bool> attr_set[2][64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (a.D != 64 && a.D != 128) return cudaErrorInvalidValue;
    const int v = a.D == 128;
    auto kern = v ? qknorm_attention_kernel<128> : qknorm_attention_kernel<64>;
    const uint32_t smem = att_smem_bytes(a.D);
    if (!attr_set[v][dev].load()) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_set[v][dev].store(true);
    }
    return launch_pdl(kern, a.grid, kAttThreads, smem, s, tmQ, tmK, tmV, a);
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
