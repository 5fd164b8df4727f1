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
// staged by TMA through an mbarrier ring), one warp-specialised CTA per SM,
// CTA tile = 128 rows of X x 256 columns of W, A = X*g (K-major), B = W:
//   rows_kernel: one row tile (M <= 128); when the column tiles alone give
//     too few CTAs the K range is split over the CTAs of a cluster, whose
//     partial sums meet in shared memory in a fixed order.
//   rows_ta_kernel: several row tiles (prefill-like shapes), persistent, the
//     A operand written into tensor memory as X*g is formed.
// Warp roles (384 threads): TMA producers, one MMA issuer, a tensor-memory
// allocator, four transform warps (X*g, sum of squares) and four epilogue
// warps (tensor memory -> registers -> scale by r -> bf16).
// A third kernel, rmsnorm_kernel, is the unfused RMSNorm kept for comparison.
// The small-M path (at most 16 rows of X) is in gemv.cu.
#include <algorithm>

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
constexpr uint32_t kRowsWBytes = kRowsBN * kBK * 2;   // 32 KB: four [64 k][64 n] W boxes
constexpr uint32_t kRowsTmemCols = 2 * kRowsBN;       // double-buffered accumulator

// Position in a ring of n pipeline stages: the slot and the parity of the
// current pass over the ring (flips each time the slot wraps to 0).
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

// The low-rank adapter's T enters the contraction as two bf16 stages, its hi
// and lo halves.
constexpr int kLoraStages = 2;

// Two outputs a, b as bf16 pairs: hi = bf16(v) and lo = bf16(v - hi) (v - hi
// is exact in fp32), so that hi + lo carries v to about 2^-16 relative.
__device__ __forceinline__ void hilo_pack(float a, float b, uint32_t& hi, uint32_t& lo) {
    hi = pack_bf16x2(a, b);
    lo = pack_bf16x2(a - bf16lo(hi), b - bf16hi(hi));
}
// Four consecutive outputs of a row at column col (< 64) of a hilo output
// [rows][128]: hi at col, lo at 64 + col.
__device__ __forceinline__ void store_hilo4(__nv_bfloat16* yrow, int col, float v0, float v1, float v2,
                                            float v3) {
    uint2 h, l;
    hilo_pack(v0, v1, h.x, l.x);
    hilo_pack(v2, v3, h.y, l.y);
    *reinterpret_cast<uint2*>(yrow + col) = h;
    *reinterpret_cast<uint2*>(yrow + kBK + col) = l;
}

struct RowsLayout {
    uint32_t xbytes, off_x, off_w, off_g, off_red, red_block, off_bar, off_sr, off_misc, total;
};

// Column chunks of 32 in a row tile.  With a cluster K split of S, the
// chunks are reduced in units: one chunk each, or, for the gated form, a
// gate chunk and the up chunk 128 columns further (the tile's 256 columns are
// 128 gate columns then the 128 matching up columns).  Unit u is reduced by
// CTA u % S, which therefore owns at most ceil(units / S) units.
constexpr int kRowsChunks = kRowsBN / 32;
// (chunks: of the tile, 8 for 256 columns, 4 for the 128-column tile)
__host__ __device__ inline int rows_red_units(bool glu, int chunks = kRowsChunks) {
    return glu ? chunks / 2 : chunks;
}
__host__ __device__ inline int rows_owned_max(int splits, bool glu, int chunks = kRowsChunks) {
    return (rows_red_units(glu, chunks) + splits - 1) / splits;
}

// Swish gate, single precision: silu(z) = z * sigmoid(z) = h (1 + tanh h)
// with h = z / 2 (sigmoid(z) = (1 + tanh(z/2)) / 2), on the hardware tanh
// approximation (relative error about 2^-11, below the bf16 rounding of Y).
__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float silu_f(float z) {
    const float h = 0.5f * z;
    return fmaf(h, tanh_approx(h), h);
}
// Output of the gated form from the gate and up accumulators of a row whose
// reciprocal RMS is r.
__device__ __forceinline__ float glu_out(float gate, float up, float r) {
    return silu_f(gate * r) * (up * r);
}

// One W stage: k-block kb by the tile's kBN (256, or 128 for the plain
// [K, N] form) accumulator columns, into the slot at dst (kBN * 128 bytes).  Weights stored [K, N] (N contiguous): [64 k][64 n] boxes,
// N-major for the MMA, as many as fall inside N.  Weights stored [N, K] (K
// contiguous, the layout of a linear layer's weight): one [256 n][64 k] box,
// K-major, rows past N read as zeros.  Gated: accumulator columns 0..127 come
// from the gate columns n0.. and 128..255 from the up columns Nout + n0.. (a
// box past the gate half reads up columns, one past N zeros; neither reaches
// an output).  w_stage_bytes() gives the bytes the copies deliver.
template <bool kGlu, bool kWnk, int kBN = kRowsBN>
__device__ __forceinline__ uint32_t w_stage_bytes(int n0, int N) {
    static_assert(kBN == kRowsBN || (!kGlu && !kWnk), "128-column W stages: plain [K, N] form only");
    if constexpr (kWnk || kGlu) return kRowsWBytes;
    else return static_cast<uint32_t>(min(kBN / 64, (N - n0 + 63) / 64)) * kWBoxBytes;
}
template <bool kGlu, bool kWnk, int kBN = kRowsBN>
__device__ __forceinline__ void load_w_stage(uint32_t dst, const CUtensorMap* tm, uint32_t bar, int n0,
                                             int kb, int N, int Nout) {
    if constexpr (kWnk) {
        if constexpr (kGlu) {
            tma_load_2d_nohint(dst, tm, bar, kb * kBK, n0);
            tma_load_2d_nohint(dst + kRowsWBytes / 2, tm, bar, kb * kBK, Nout + n0);
        } else {
            tma_load_2d_nohint(dst, tm, bar, kb * kBK, n0);
        }
    } else {
        const int nbox = static_cast<int>(w_stage_bytes<kGlu, kWnk, kBN>(n0, N) / kWBoxBytes);
        for (int j = 0; j < nbox; ++j)
            tma_load_2d_nohint(dst + j * kWBoxBytes, tm, bar, kGlu && j >= 2 ? Nout + n0 + 64 * (j - 2) : n0 + 64 * j,
                               kb * kBK);
    }
}
// Shared-memory descriptor of the W stage at b0 for the MMA's k-step kk.
template <bool kWnk>
__device__ __forceinline__ uint64_t w_desc(uint32_t b0, int kk) {
    return kWnk ? sdesc_sw128(b0 + kk * 32, 16, 1024) : sdesc_sw128(b0 + kk * 2048, kWBoxBytes, 1024);
}

// Shared-memory layout of rows_kernel.  xrows: rows of X each stage loads
// (128, or M rounded up to 16 when one row tile covers M).  X tiles come
// first: the MMA always reads a 128-row window from an X tile, whose rows
// past xrows (discarded results) fall on the following tiles.  red_slots:
// with a cluster K split of S = red_slots, each CTA receives one block per
// split, [MP] fp32 row sums of squares followed by [ceil(units/S)][1 or 2
// chunks][MP][32] fp32 partial rows of the units it owns (the 16-byte pieces
// of a row rotated by row & 7 against bank conflicts).  With overlay, the
// receive blocks occupy the start of the pipeline buffers, which are idle by
// the time they fill.
__host__ __device__ inline RowsLayout rows_layout(int xrows, int stages, int red_slots, int MP,
                                                  bool overlay = false, bool glu = false, int bn = kRowsBN) {
    RowsLayout L;
    L.xbytes = xrows * kBK * 2;
    L.off_x = 0;
    L.off_w = ((stages * L.xbytes + 1023) / 1024) * 1024;
    L.off_g = L.off_w + stages * static_cast<uint32_t>(bn) * kBK * 2;
    L.red_block = red_slots > 0 ? MP * (4 + rows_owned_max(red_slots, glu, bn / 32) * (glu ? 2 : 1) * 128) : 0;
    L.off_red = overlay ? 0 : ((L.off_g + stages * kGBytes + 15) / 16) * 16;
    L.off_bar = overlay ? ((L.off_g + stages * kGBytes + 15) / 16) * 16 : L.off_red + red_slots * L.red_block;
    const uint32_t nbars = 4 * kRowsMaxStages + 10;
    L.off_sr = L.off_bar + ((nbars * 8 + 15) / 16) * 16;
    L.off_misc = L.off_sr + 2 * kRowsBM * 4;
    L.total = L.off_misc + 16 + 1024;
    return L;
}


// kBN: accumulator columns of a tile, 256, or 128 (plain [K, N] form with a
// K split: twice the CTAs for the same K split, half the partial sums each
// CTA exchanges).
template <bool kFused, bool kSplit, bool kGlu, bool kWnk, bool kLora, int kBN = kRowsBN>
__global__ void __launch_bounds__(kThreads, 1)
    rows_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmT,
                const __grid_constant__ CUtensorMap tmB, __nv_bfloat16* __restrict__ Y, RowsLaunch a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    const int S = a.stages;
    const int split = kSplit ? a.splits : 1;
    static_assert(kBN == kRowsBN || (kSplit && !kGlu && !kWnk && !kLora), "128-column tiles: plain K split only");
    constexpr uint32_t kWBytes = kBN * kBK * 2;    // one W stage
    constexpr int kChunks = kBN / 32;              // 32-column chunks of a tile
    const RowsLayout L = rows_layout(a.xrows, S, kSplit ? split : 0, a.MP, kSplit && a.red_overlay, kGlu, kBN);
    // Output columns: N, or F = N / 2 for the gated form, whose tile covers
    // 128 output columns from two W column ranges (gate, then up).
    const int Nout = kGlu ? a.N / 2 : a.N;
    constexpr int kOutBN = kGlu ? kBN / 2 : kBN;
    const uint32_t xbytes = L.xbytes;
    const uint32_t sb = smem_u32(smem);
    const uint32_t sx = sb + L.off_x, sw = sb + L.off_w, sg = sb + L.off_g;
    const uint32_t bar0 = sb + L.off_bar;
    auto full = [&](uint32_t s) { return bar0 + 8 * s; };
    auto xform = [&](uint32_t s) { return bar0 + 8 * (kRowsMaxStages + s); };
    auto empty = [&](uint32_t s) { return bar0 + 8 * (2 * kRowsMaxStages + s); };
    auto accfull = [&](uint32_t b) { return bar0 + 8 * (3 * kRowsMaxStages + b); };
    auto accempty = [&](uint32_t b) { return bar0 + 8 * (3 * kRowsMaxStages + 2 + b); };
    auto srfull = [&](uint32_t b) { return bar0 + 8 * (3 * kRowsMaxStages + 4 + b); };
    const uint32_t mmadone = bar0 + 8 * (3 * kRowsMaxStages + 6);
    // the other splits' blocks (partials of the chunks this CTA owns, row
    // sums of squares) have arrived
    const uint32_t redfull = bar0 + 8 * (3 * kRowsMaxStages + 8);
    // with the receive blocks over the pipeline buffers: every other split's
    // buffers are idle, so its blocks may be stored
    const uint32_t redgo = bar0 + 8 * (3 * kRowsMaxStages + 9);
    // fused: stage s's X tile and g slice have landed (its W lands on
    // full(s)), so the transform of a stage runs while its W is still on
    // the way, and the MMA waits for both
    auto xland = [&](uint32_t s) { return bar0 + 8 * (3 * kRowsMaxStages + 10 + s); };
    float* sr = reinterpret_cast<float*>(smem + L.off_sr);         // [2][128] row sums of squares
    const uint32_t red_addr = sb + L.off_red;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L.off_misc);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + L.off_misc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // units = (tile, K split); with a cluster, blockIdx.x = cluster * splits +
    // rank and the splits of one tile are the CTAs of one cluster, one unit
    // per CTA (a launch that breaks this does no work and reports an
    // internal error)
    int units = a.m_tiles * a.n_tiles * split;
    const bool bad_launch = kSplit && (units > static_cast<int>(gridDim.x) ||
                                       (a.red_overlay && split * L.red_block > L.off_g));
    if (bad_launch) units = 0;
    // W boxes of 64 columns for the tile whose output columns start at n0:
    // plain, the columns themselves (as many as fall inside N); gated, two
    // boxes of gate columns n0.. and two of up columns Nout + n0.. (always
    // four: a box past the gate half reads up columns, one past N reads
    // zeros, and neither reaches an output column).
    // Low-rank adapter: the unit holding split 0 of a tile runs two more
    // stages after its k-blocks, at k-block indices k_blocks + e, e = 0, 1,
    // whose A tiles are the hi (e = 0) and lo (e = 1) halves of T = (X*g) @ A
    // (columns [64e, 64e + 64) of tmT, zeros past R in each half) and whose B
    // tile is the adapter's B both times (rows of tmB, zeros past R); they get
    // no gain and add nothing to the row statistic.  T_hi @ B + T_lo @ B
    // carries T to about 2^-16 relative, far below the output's rounding.
    // (its own instantiations: kLora, fused [K, N] form only; the others
    // carry none of it)
    static_assert(!kLora || (kFused && !kGlu && !kWnk), "the adapter stage is for the plain fused form");
    auto lora_extra = [&](int sp) { return kLora && sp == 0 ? kLoraStages : 0; };
    // Loads of stage s = k-block kb of the unit whose tile starts at row block
    // mb and output column n0 (kb >= k_blocks: adapter stage kb - k_blocks).
    // (Fused: X and g complete on xland(s), W on full(s).)
    auto issue = [&](uint32_t s, int kb, int mb, int n0) {
        const bool ext = kLora && kb >= a.k_blocks;
        const uint32_t xbar = kFused ? xland(s) : full(s);
        if (kFused) {
            mbar_arrive_expect_tx(xbar, xbytes + (!ext ? kGBytes : 0));
            mbar_arrive_expect_tx(full(s), w_stage_bytes<kGlu, kWnk, kBN>(n0, a.N));
        } else {
            mbar_arrive_expect_tx(full(s), xbytes + w_stage_bytes<kGlu, kWnk, kBN>(n0, a.N));
        }
        tma_load_2d_nohint(sx + s * xbytes, ext ? &tmT : &tmX, xbar, (ext ? kb - a.k_blocks : kb) * kBK,
                           mb * kRowsBM);
        if (kFused && !ext) tma_load_1d(sg + s * kGBytes, &tmG, xbar, kb * kBK);
        load_w_stage<kGlu, kWnk, kBN>(sw + s * kWBytes, ext ? &tmB : &tmW, full(s), n0, ext ? 0 : kb, a.N, Nout);
    };
    // k-blocks of the first unit that thread 0 (the producer) issues before
    // the CTA-wide set-up barrier, as soon as its barriers exist and the
    // previous kernel on the stream has completed
    uint32_t pro = 0;
    if (threadIdx.x == 0) {
        if (bad_launch) atomicCAS(&g_status, 0, kStatusInternal);
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(xform(s), 4);   // one elected lane per transform warp
            mbar_init(empty(s), 1);
            mbar_init(xland(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accfull(b), 1);
            mbar_init(accempty(b), 4);  // one elected lane per epilogue warp
            mbar_init(srfull(b), 4);    // one elected lane per transform warp
        }
        mbar_init(mmadone, 1);
        mbar_init(redfull, 1);   // own expect_tx (+ the peers' bytes)
        mbar_init(redgo, split > 1 ? split - 1 : 1);   // one remote arrive per other split
        abort[0] = 0;
        abort[1] = a.wait_limit_us;
        fence_mbar_init();
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
        if (kFused) prefetch_tmap(&tmG);
        // The previous kernel's writes are visible after grid_dep_wait(); the
        // next kernel may then be scheduled (its set-up overlaps this one).
        // With the adapter the previous kernel is the launch that computes T,
        // which itself waited for its own predecessor before letting this one
        // start: X, g, W and B are then visible already, and only the adapter
        // stage (which reads T) waits for it.
        if (!kLora) grid_dep_wait();
        grid_dep_launch();
        if (static_cast<int>(blockIdx.x) < units) {
            const int u = blockIdx.x, t = u / split, sp = u - t * split;
            const int kb0 = sp * a.kb_per_split, kb1 = min(a.k_blocks, kb0 + a.kb_per_split);
            int mb, nb;
            rows_tile_coords(t, a.m_tiles, a.n_tiles, mb, nb);
            const int n0 = nb * kOutBN;
            const int kend = kb1 + lora_extra(sp);
            pro = static_cast<uint32_t>(min(S, kend - kb0));
            for (uint32_t i = 0; i < pro; ++i) {
                const int kb = kb0 + static_cast<int>(i);
                if (kLora && kb >= kb1) grid_dep_wait();
                issue(i, kb < kb1 ? kb : a.k_blocks + (kb - kb1), mb, n0);
            }
        }
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_holder), kRowsTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // peers' barriers must be initialised before the first remote access:
    // announce it here, wait for the peers just before that access
    if (kSplit) cluster_arrive();
    if (!kLora) grid_dep_wait();   // with the adapter only the producer reads T (see above)
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t it = pro;
            Ring ring(S);
            for (uint32_t i = 0; i < pro; ++i) ring.advance();
            bool ok = true;
            for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
                const int t = u / split, sp = u - t * split;
                const int kb0 = sp * a.kb_per_split, kb1 = min(a.k_blocks, kb0 + a.kb_per_split);
                int mb, nb;
                rows_tile_coords(t, a.m_tiles, a.n_tiles, mb, nb);
                const int n0 = nb * kOutBN;
                const int first = kb0 + (u == static_cast<int>(blockIdx.x) ? static_cast<int>(pro) : 0);
                const int kend = kb1 + lora_extra(sp);
                for (int kb = first; kb < kend; ++kb) {
                    const uint32_t s = ring.idx, ph = ring.phase;
                    if (!mbar_wait(empty(s), ph ^ 1, abort)) { ok = false; break; }
                    if (kLora && kb >= kb1) grid_dep_wait();   // the adapter stage reads T
                    issue(s, kb < kb1 ? kb : a.k_blocks + (kb - kb1), mb, n0);
                    ++it;
                    ring.advance();
                }
            }
            // never leave with copies still landing in shared memory
            const uint32_t pending = it < static_cast<uint32_t>(S) ? it : S;
            for (uint32_t i = it - pending; i < it; ++i) {
                if (!mbar_wait_teardown(full(i % S), (i / S) & 1)) break;
                if (kFused && !mbar_wait_teardown(xland(i % S), (i / S) & 1)) break;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kRowsBM, kBN, false, !kWnk);
            uint32_t it = 0, tl = 0;
            Ring ring(S);
            bool ok = true;
            for (int u = blockIdx.x; ok && u < units; u += gridDim.x, ++tl) {
                const int t = u / split, sp = u - t * split;
                const int kb0 = sp * a.kb_per_split, kb1 = min(a.k_blocks, kb0 + a.kb_per_split);
                const uint32_t buf = tl & 1, use = tl >> 1;
                if (!mbar_wait(accempty(buf), (use & 1) ^ 1, abort)) break;
                tc_fence_after();
                const uint32_t d = tmem + buf * kBN;
                const int kend = kb1 + lora_extra(sp);
                for (int kb = kb0; kb < kend; ++kb) {
                    const uint32_t s = ring.idx, ph = ring.phase;
                    if (!mbar_wait(full(s), ph, abort) || (kFused && !mbar_wait(xform(s), ph, abort))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = sx + s * xbytes, b0 = sw + s * kWBytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        mma_bf16_ss(d, sdesc_sw128(a0 + kk * 32, 16, 1024), w_desc<kWnk>(b0, kk), idesc,
                                    (kb != kb0 || kk != 0));
                    mma_commit(empty(s));
                    ++it;
                    ring.advance();
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
            const int rb = t >> 3;          // rows rb + 16 i
            const int groups = a.xrows / 16;
            const uint32_t swz_off = static_cast<uint32_t>((kc ^ (rb & 7)) << 4);
            uint32_t it = 0, tl = 0;
            Ring ring(S);
            bool ok = true;
            for (int u = blockIdx.x; ok && u < units; u += gridDim.x, ++tl) {
                const int tt = u / split, sp = u - tt * split;
                const int kb0 = sp * a.kb_per_split, kb1 = min(a.k_blocks, kb0 + a.kb_per_split);
                const uint32_t buf = tl & 1, use = tl >> 1;
                // sr[buf] is free once the epilogue released this accumulator
                if (!warp_wait(accempty(buf), (use & 1) ^ 1, abort)) break;
                float ss[kRowsBM / 16];
#pragma unroll
                for (int i = 0; i < kRowsBM / 16; ++i) ss[i] = 0.f;
                const int kend = kb1 + lora_extra(sp);
                for (int kb = kb0; kb < kend; ++kb) {
                    const uint32_t s = ring.idx, ph = ring.phase;
                    if (!warp_wait(xland(s), ph, abort)) { ok = false; break; }
                    if (!kLora || kb < kb1) {   // (the adapter stage needs no transform)
                        const uint4 gv = lds128(sg + s * kGBytes + kc * 16);
                        const uint32_t xt = sx + s * xbytes + swz_off;
                        // rows rb + 16 i all have (row & 7) == (rb & 7)
                        // all loads first, then the stores (the shared-memory
                        // accesses keep program order), so the loads overlap
                        uint4 xv[kRowsBM / 16];
#pragma unroll
                        for (int i = 0; i < kRowsBM / 16; ++i)
                            if (i < groups) xv[i] = lds128(xt + (rb + 16 * i) * 128);
#pragma unroll
                        for (int i = 0; i < kRowsBM / 16; ++i)
                            if (i < groups) sts128(xt + (rb + 16 * i) * 128, gain8(xv[i], gv, ss[i]));
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(xform(s));
                    ++it;
                    ring.advance();
                }
                if (!ok) break;
#pragma unroll
                for (int i = 0; i < kRowsBM / 16; ++i) {
                    float v = ss[i];
                    v += __shfl_xor_sync(0xffffffffu, v, 1);
                    v += __shfl_xor_sync(0xffffffffu, v, 2);
                    v += __shfl_xor_sync(0xffffffffu, v, 4);
                    if (kc == 0) sr[buf * kRowsBM + rb + 16 * i] = v;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(srfull(buf));
            }
        }
    } else if (warp >= 8 && !kSplit) {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;             // tensor-memory lane quarter of this warp
        const int row = q * 32 + lane;
        const float inv_k = 1.f / static_cast<float>(a.K);
        uint32_t tl = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x, ++tl) {
            const uint32_t buf = tl & 1, use = tl >> 1;
            if (!warp_wait(accfull(buf), use & 1, abort)) break;
            if (kFused && !warp_wait(srfull(buf), use & 1, abort)) break;
            tc_fence_after();
            int mb, nb;
            rows_tile_coords(u, a.m_tiles, a.n_tiles, mb, nb);
            const int n0 = nb * kOutBN;
            // a hilo output writes all 64 columns of each half (zeros past N)
            const int ncols = !kGlu && a.hilo ? kBK : min(kOutBN, Nout - n0);
            const int rows_here = min(kRowsBM, a.M - mb * kRowsBM);   // valid rows of this tile
            const uint32_t taddr = tmem + buf * kBN + (static_cast<uint32_t>(q * 32) << 16);
            const bool warp_has_rows = q * 32 < rows_here;              // warp-uniform
            const int m = mb * kRowsBM + row;
            const float r = kFused && !a.unscaled ? rsqrtf(sr[buf * kRowsBM + row] * inv_k + a.eps) : 1.f;
            const int ldy = !kGlu && a.hilo ? 2 * kBK : Nout;   // row stride of Y
            __nv_bfloat16* yrow = Y + static_cast<size_t>(m) * ldy + n0;
            for (int c = 0; warp_has_rows && c < kOutBN / 32; ++c) {
                if (c * 32 >= ncols) break;   // warp-uniform
                uint32_t v[32], w2[kGlu ? 32 : 1];
                tmem_ld_32x32(taddr + c * 32, v);
                if constexpr (kGlu) tmem_ld_32x32(taddr + kOutBN + c * 32, w2);
                auto out = [&](int i) {
                    if constexpr (kGlu) return glu_out(__uint_as_float(v[i]), __uint_as_float(w2[i]), r);
                    else return __uint_as_float(v[i]) * r;
                };
                if (row < rows_here) {
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const int col = c * 32 + g * 8;
                        if (col < ncols) {
                            if (!kGlu && a.hilo) {
                                store_hilo4(yrow, col, out(g * 8 + 0), out(g * 8 + 1), out(g * 8 + 2),
                                            out(g * 8 + 3));
                                store_hilo4(yrow, col + 4, out(g * 8 + 4), out(g * 8 + 5), out(g * 8 + 6),
                                            out(g * 8 + 7));
                                continue;
                            }
                            uint4 o;
                            o.x = pack_bf16x2(out(g * 8 + 0), out(g * 8 + 1));
                            o.y = pack_bf16x2(out(g * 8 + 2), out(g * 8 + 3));
                            o.z = pack_bf16x2(out(g * 8 + 4), out(g * 8 + 5));
                            o.w = pack_bf16x2(out(g * 8 + 6), out(g * 8 + 7));
                            *reinterpret_cast<uint4*>(yrow + col) = o;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(accempty(buf));
        }
    }

    if (kSplit) {
        // ---------------------------------------- K split: reduce by scatter
        // One (tile, split) unit per CTA, one row tile (M <= 128); the K
        // splits of the tile are the CTAs of this cluster.  Chunk c of 32
        // columns belongs to CTA c % splits.  Every warp takes part:
        //  1. warps 4..11 of each tensor-memory lane quarter that holds rows
        //     (two per quarter, taking every other chunk) read the
        //     accumulator and store each chunk straight from registers into
        //     its owner's receive block for this split (st.async; the bytes
        //     complete on the owner's redfull) or, for their own chunks, into
        //     their own block; with it go the row sums of squares.  Warps 0
        //     and 1 (producer, MMA) are left out: they reach this point last,
        //     and their first cluster-barrier wait (~0.6 us even when every
        //     peer has long arrived) would hold up the sends;
        //  2. once every split's block has arrived, all threads add the
        //     blocks in split order (fixed, whatever the arrival order),
        //     scale by 1/rms and write this CTA's chunks of Y.
        // The 16-byte pieces of a row are rotated by row & 7 in the blocks,
        // against bank conflicts.  The cluster barrier's second phase is
        // entered once this CTA's blocks have all arrived (nothing is stored
        // into it after that) and left before exit, so that no CTA leaves
        // while its stores to a peer are in flight.
        __syncwarp();
        const int u = blockIdx.x;
        const bool have = u < units;
        const uint32_t rank = cluster_ctarank();
        const int me = static_cast<int>(rank);
        int mb = 0, nb = 0;
        if (have) rows_tile_coords(u / split, a.m_tiles, a.n_tiles, mb, nb);
        const int n0 = nb * kOutBN;
        // output columns of this tile (a hilo output: all 64 of each half, zeros past N)
        const int ncols = !kGlu && a.hilo ? kBK : min(kOutBN, Nout - n0);
        const int rows_here = min(kRowsBM, a.M - mb * kRowsBM);
        // reduction units of 32 output columns: accumulator chunk u, or (gated)
        // gate chunk u with up chunk u + 4
        constexpr int kUnitChunks = kGlu ? 2 : 1;
        const int nunits = (ncols + 31) / 32;
        const int owned = nunits > me ? (nunits - 1 - me) / split + 1 : 0;
        const uint32_t blk = L.red_block;
        const uint32_t my_block = red_addr + rank * blk;   // this split's block in every CTA
        const int q = warp & 3, team = warp >> 2;
        const int row = q * 32 + lane;
        const bool send = a.test_skip_sends == 0;
        if (have && threadIdx.x == 0)
            mbar_arrive_expect_tx(redfull,
                                  static_cast<uint32_t>((split - 1) * rows_here * (4 + owned * kUnitChunks * 128)));
        cluster_wait();    // the peers' barriers are initialised
        // 1. tensor memory -> owners
        const int wteam = team - 1;   // chunk team of warps 4..11
        if (have && team >= 1 && q * 32 < rows_here &&
            warp_wait(accfull(0), 0, abort) && (!kFused || warp_wait(srfull(0), 0, abort)) &&
            (!a.red_overlay || [&] {
                // The last MMA is done, so this CTA's pipeline buffers, which
                // hold its receive blocks, are idle: tell the other splits,
                // then wait until theirs are idle too.
                if (threadIdx.x == 128)
                    for (int p = 0; p < split; ++p)
                        if (p != me) mbar_arrive_remote(mapa_shared(redgo, p));
                return warp_wait_cluster(redgo, 0, abort);
            }())) {
            tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16);
            const uint32_t swz = static_cast<uint32_t>(row & 7);
            for (int c = wteam; c < kChunks; c += 2) {
                const int unit = kGlu ? (c & (kChunks / 2 - 1)) : c, half = kGlu ? c / (kChunks / 2) : 0;
                if (unit >= nunits) continue;   // warp-uniform
                uint32_t v[32];
                tmem_ld_32x32(taddr + c * 32, v);
                if (row < rows_here) {
                    const int owner = unit % split;
                    const uint32_t dst =
                        my_block + a.MP * 4 + (((unit / split) * kUnitChunks + half) * a.MP + row) * 128;
                    if (owner == me) {
#pragma unroll
                        for (int g = 0; g < 8; ++g)
                            sts128(dst + ((g ^ swz) << 4),
                                   make_uint4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]));
                    } else if (send) {
                        const uint32_t rdst = mapa_shared(dst, owner);
                        const uint32_t rbar = mapa_shared(redfull, owner);
#pragma unroll
                        for (int g = 0; g < 8; ++g)
                            st_async_v4(rdst + ((g ^ swz) << 4),
                                        make_uint4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]), rbar);
                    }
                }
            }
            if (team == 1 && row < rows_here) {
                const float ssv = kFused ? sr[row] : 0.f;
                const uint32_t dst = my_block + row * 4;
                *reinterpret_cast<float*>(smem + (dst - sb)) = ssv;
                for (int p = 0; p < split && send; ++p)
                    if (p != me) st_async_b32(mapa_shared(dst, p), __float_as_uint(ssv), mapa_shared(redfull, p));
            }
        }
        // 2. sum once every block has arrived (this CTA's own block: after
        // the barrier below)
        const bool ok = have && warp_wait_cluster(redfull, 0, abort);
        cluster_arrive();
        __syncthreads();
        if (ok && !*abort) {
            const float inv_k = 1.f / static_cast<float>(a.K);
            const int n3 = rows_here * owned * 8;
            for (int i = threadIdx.x; i < n3; i += kThreads) {
                const int g = i & 7, j = (i >> 3) % owned, rr = (i >> 3) / owned;
                const uint32_t piece = static_cast<uint32_t>((g ^ (rr & 7)) << 4);
                // every split's pieces and row sum in flight before the first add
                float ssv[kClusterMaxSplits];
                uint4 t4[kClusterMaxSplits][kUnitChunks];
#pragma unroll
                for (int s2 = 0; s2 < kClusterMaxSplits; ++s2)
                    if (s2 < split) {
                        ssv[s2] = *reinterpret_cast<const float*>(smem + L.off_red + s2 * blk + rr * 4);
#pragma unroll
                        for (int h = 0; h < kUnitChunks; ++h)
                            t4[s2][h] = lds128(red_addr + s2 * blk + a.MP * 4 +
                                               ((j * kUnitChunks + h) * a.MP + rr) * 128 + piece);
                    }
                float tot = 0.f;
                float4 acc[kUnitChunks];
#pragma unroll
                for (int h = 0; h < kUnitChunks; ++h) acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int s2 = 0; s2 < kClusterMaxSplits; ++s2)
                    if (s2 < split) {
                        tot += ssv[s2];
#pragma unroll
                        for (int h = 0; h < kUnitChunks; ++h) {
                            acc[h].x += __uint_as_float(t4[s2][h].x);
                            acc[h].y += __uint_as_float(t4[s2][h].y);
                            acc[h].z += __uint_as_float(t4[s2][h].z);
                            acc[h].w += __uint_as_float(t4[s2][h].w);
                        }
                    }
                const float r = kFused && !a.unscaled ? rsqrtf(tot * inv_k + a.eps) : 1.f;
                const int col = (me + j * split) * 32 + g * 4;
                if (col < ncols) {
                    float o4[4];
                    if constexpr (kGlu) {
                        o4[0] = glu_out(acc[0].x, acc[kUnitChunks - 1].x, r);
                        o4[1] = glu_out(acc[0].y, acc[kUnitChunks - 1].y, r);
                        o4[2] = glu_out(acc[0].z, acc[kUnitChunks - 1].z, r);
                        o4[3] = glu_out(acc[0].w, acc[kUnitChunks - 1].w, r);
                    } else {
                        o4[0] = acc[0].x * r;
                        o4[1] = acc[0].y * r;
                        o4[2] = acc[0].z * r;
                        o4[3] = acc[0].w * r;
                        if (a.hilo) {
                            store_hilo4(Y + static_cast<size_t>(mb * kRowsBM + rr) * (2 * kBK), col, o4[0], o4[1],
                                        o4[2], o4[3]);
                            continue;
                        }
                    }
                    uint2 o;
                    o.x = pack_bf16x2(o4[0], o4[1]);
                    o.y = pack_bf16x2(o4[2], o4[3]);
                    *reinterpret_cast<uint2*>(Y + static_cast<size_t>(mb * kRowsBM + rr) * Nout + n0 + col) = o;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    // every CTA of the cluster has received all its blocks (the arrive above)
    if (kSplit) cluster_wait();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, kRowsTmemCols);
    }
}

// ------------------------------------------- row-tile path, A in tensor memory
// The fused kernel for several row tiles (prefill-like shapes).  The gain is
// applied on the way from shared to tensor memory: each transform thread
// reads its row of the X tile once, multiplies by g in bf16x2 and stores the
// row straight into a tensor-memory A slot with tcgen05.st, and the MMA reads
// A from there.  Compared with writing X*g back into shared memory for the
// MMA to read, this removes two of the three passes over each X tile in
// shared memory, whose bandwidth bounds this kernel.  X and W have separate
// rings: an X slot is released as soon as its rows are in tensor memory.
// Tensor memory: columns [0, 256) hold the accumulator (single buffer; the
// epilogue holds it only while it reads it out), [256, 512) eight A slots of
// 32 columns (128 rows x 64 bf16 each).
constexpr int kTaXStages = 4;
constexpr int kTaWStages = 4;
// Paired: a CTA's W slot holds half a stage (16 KB); the same 192 KB then
// hold six X slots and six W half-slots.
constexpr int kTaXStagesPair = 6;
constexpr int kTaWStagesPair = 6;
constexpr int kTaAStages = 8;
constexpr uint32_t kTaXBytes = kRowsBM * kBK * 2;    // 16 KB
constexpr uint32_t kTaStageOut = kRowsBM * 32 * 2;   // 8 KB: 128 rows x 32 bf16 of Y
constexpr uint32_t kTaOffX = 0;
constexpr uint32_t kTaOffW = kTaOffX + kTaXStages * kTaXBytes;
constexpr uint32_t kTaOffWPair = kTaOffX + kTaXStagesPair * kTaXBytes;
constexpr uint32_t kTaOffOut = kTaOffW + kTaWStages * kRowsWBytes;   // 2 staging buffers
static_assert(kTaOffWPair + kTaWStagesPair * (kRowsWBytes / 2) == kTaOffOut, "paired rings fill the same memory");
constexpr uint32_t kTaOffG = kTaOffOut + 2 * kTaStageOut;
constexpr uint32_t kTaOffBar = kTaOffG + kTaXStagesPair * kGBytes;
// xfull, xempty, wfull, wempty, afull, aempty, accfull, accempty, srfull[2], srempty[2],
// mmadone, episync
constexpr uint32_t kTaNumBars = 2 * kTaXStagesPair + 2 * kTaWStagesPair + 2 * kTaAStages + 8;
constexpr uint32_t kTaOffSr = kTaOffBar + ((kTaNumBars * 8 + 15) / 16) * 16;
constexpr uint32_t kTaOffRr = kTaOffSr + 2 * kRowsBM * 4;    // 1/rms of a piece's rows
constexpr uint32_t kTaOffMisc = kTaOffRr + kRowsBM * 4;
constexpr uint32_t kTaSmem = kTaOffMisc + 16 + 1024;
constexpr uint32_t kTaAccCol = 0, kTaACol = 256;

// Work of CTA slot b of G in rows_ta_kernel (a slot is one CTA, or a pair of
// CTAs that share W: their tiles are the two row blocks of a "unit" of
// kC = 2 row blocks x one column tile), in order: whole units b, b + G, ...
// below full = units - tail_tiles; then, if b < tail_tiles * tail_pieces, K
// piece b % tail_pieces of tail unit b / tail_pieces (unit full + that).
struct TaUnit {
    int t, kb0, kb1, piece;   // piece < 0: the whole K range
    int extra;                // adapter stages that follow (whole tile, or piece 0 of a tail tile)
};
template <int kC>
__device__ __forceinline__ bool ta_unit(const RowsLaunch& a, int i, TaUnit& u) {
    const int G = static_cast<int>(gridDim.x) / kC, b = static_cast<int>(blockIdx.x) / kC;
    const int full = ((a.m_tiles + kC - 1) / kC) * a.n_tiles - a.tail_tiles;
    const int t = b + i * G;
    if (t < full) {
        u.t = t;
        u.kb0 = 0;
        u.kb1 = a.k_blocks;
        u.piece = -1;
        u.extra = a.lora ? kLoraStages : 0;
        return true;
    }
    const int whole = b < full ? (full - b + G - 1) / G : 0;
    if (i != whole || b >= a.tail_tiles * a.tail_pieces) return false;
    u.piece = b % a.tail_pieces;
    u.t = full + b / a.tail_pieces;
    u.kb0 = u.piece * a.tail_kbp;
    u.kb1 = min(a.k_blocks, u.kb0 + a.tail_kbp);
    u.extra = a.lora && u.piece == 0 ? kLoraStages : 0;
    return true;
}

template <bool kGlu, bool kWnk, bool kLora, bool kHilo, bool kPair>
__global__ void __launch_bounds__(kThreads, 1)
    rows_ta_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                   const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmT,
                   const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmY,
                   __nv_bfloat16* __restrict__ Y, RowsLaunch a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    const uint32_t sb = smem_u32(smem);
    // rings: X, W (paired: half stages), A (tensor memory)
    constexpr int kXSt = kPair ? kTaXStagesPair : kTaXStages;
    constexpr int kWSt = kPair ? kTaWStagesPair : kTaWStages;
    constexpr uint32_t kWSlot = kPair ? kRowsWBytes / 2 : kRowsWBytes;
    const uint32_t sx = sb + kTaOffX, sw = sb + (kPair ? kTaOffWPair : kTaOffW), sg = sb + kTaOffG;
    const uint32_t bar0 = sb + kTaOffBar;
    uint32_t nb_ = 0;
    const uint32_t xfull0 = bar0 + 8 * nb_; nb_ += kTaXStagesPair;
    const uint32_t xempty0 = bar0 + 8 * nb_; nb_ += kTaXStagesPair;
    const uint32_t wfull0 = bar0 + 8 * nb_; nb_ += kTaWStagesPair;
    const uint32_t wempty0 = bar0 + 8 * nb_; nb_ += kTaWStagesPair;
    const uint32_t afull0 = bar0 + 8 * nb_; nb_ += kTaAStages;
    const uint32_t aempty0 = bar0 + 8 * nb_; nb_ += kTaAStages;
    const uint32_t accfull = bar0 + 8 * nb_++;
    const uint32_t accempty = bar0 + 8 * nb_++;
    const uint32_t srfull0 = bar0 + 8 * nb_; nb_ += 2;
    const uint32_t srempty0 = bar0 + 8 * nb_; nb_ += 2;
    const uint32_t mmadone = bar0 + 8 * nb_++;
    const uint32_t episync = bar0 + 8 * nb_++;
    const uint32_t sout = sb + kTaOffOut;
    float* sr = reinterpret_cast<float*>(smem + kTaOffSr);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kTaOffMisc);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + kTaOffMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Paired: launched as clusters of two, or not at all (a launch without
    // them reports an internal error and does no work: no cluster or
    // tensor-memory operation may run, the pair allocation least of all).
    if (kPair) {
        uint32_t nct;
        asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(nct));
        if (nct != 2 || a.tail_tiles != 0) {
            if (threadIdx.x == 0) atomicCAS(&g_status, 0, kStatusInternal);
            return;
        }
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kXSt; ++s) {
            mbar_init(xfull0 + 8 * s, 1);
            mbar_init(xempty0 + 8 * s, 4);
        }
        for (int s = 0; s < kWSt; ++s) {
            mbar_init(wfull0 + 8 * s, 1);
            mbar_init(wempty0 + 8 * s, 1);
        }
        for (int s = 0; s < kTaAStages; ++s) {
            // paired, rank 0: the k-block's one "ready" barrier for the MMA: this CTA's W
            // copies (one arrival and their bytes), its four transform warps and rank 1's signal
            mbar_init(afull0 + 8 * s, kPair && cluster_ctarank() == 0 ? 6 : 4);
            mbar_init(aempty0 + 8 * s, 1);
        }
        mbar_init(accfull, 1);
        mbar_init(accempty, kPair ? 8 : 4);   // paired: both CTAs' epilogue warps release it
        for (int b = 0; b < 2; ++b) {
            mbar_init(srfull0 + 8 * b, 4);
            mbar_init(srempty0 + 8 * b, 4);
        }
        mbar_init(mmadone, 1);
        mbar_init(episync, 4);
        abort[0] = 0;
        abort[1] = a.wait_limit_us;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
        prefetch_tmap(&tmG);
        prefetch_tmap(&tmY);
    }
    if (warp == 2) {
        if constexpr (kPair) {
            tmem_alloc_pair(smem_u32(tmem_holder), 512);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_holder), 512);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // paired: the peer's barriers exist before any signal or commit targets them
    if (kPair) cluster_sync_all();
    // Set-up above overlaps the previous kernel on the stream; its writes are
    // visible after grid_dep_wait().  The next kernel may then be scheduled.
    // With the adapter the previous kernel is the launch that computes T,
    // which itself waited for its own predecessor before letting this one
    // start: X, g, W and B are visible already, and only the loads of T (the
    // adapter stages) and the K pieces' workspace (which that launch may use
    // too) wait for it.
    if (!kLora) grid_dep_wait();
    if (threadIdx.x == 0) grid_dep_launch();
    const uint32_t tmem = *tmem_holder;
    // Paired (kPair): the two CTAs of a cluster take the two row blocks of each
    // unit (256 x 256) as one pair MMA of M = 256: each loads its own X rows
    // and half of every W stage (columns [128 rank, 128 rank + 128) of the
    // tile) and keeps its rows' A slots and accumulator in its own tensor
    // memory; rank 0 issues the MMAs once its own stage and rank 1's (which
    // rank 1's MMA warp signals) are ready.  Per 128 x 256 x 64 of work a CTA
    // takes in 32 KB (its X rows and half a W stage) instead of 48 KB.  Units
    // are counted in pairs of row blocks.
    constexpr int kC = kPair ? 2 : 1;
    const int rank = kPair ? static_cast<int>(cluster_ctarank()) : 0;
    const int m_units = (a.m_tiles + kC - 1) / kC;
    const int num_tiles = m_units * a.n_tiles;
    static_assert(!kPair || !kHilo, "the hi/lo output runs unpaired");
    // Output columns: N, or F = N / 2 for the gated form, whose tile covers
    // 128 output columns read from gate columns n0.. and up columns F + n0..
    const int Nout = kGlu ? a.N / 2 : a.N;
    constexpr int kOutBN = kGlu ? kRowsBN / 2 : kRowsBN;
    // the low-rank adapter stage: its own instantiations (kLora), plain [K, N] form only
    static_assert(!kLora || (!kGlu && !kWnk), "the adapter stage is for the plain form");
    // the hi/lo output of the adapter's T: its own instantiation (kHilo), unscaled plain form
    static_assert(!kHilo || (!kGlu && !kWnk && !kLora), "the hi/lo output is for the plain form");

    if (warp == 0 || warp == 3) {
        // ------------------------------------------------ TMA producers
        // Two threads, so that X (released as soon as it is in tensor memory)
        // runs ahead on its own ring instead of behind the W ring: warp 0
        // loads W, warp 3 loads X and g.
        if (lane == 0) {
            const bool load_x = warp == 3;
            Ring ring(load_x ? kXSt : kWSt);
            Ring rr(kTaAStages);   // paired, rank 0, W: the k-block's ready barrier (its A slot's)
            uint32_t issued = 0;
            const uint32_t full0 = load_x ? xfull0 : wfull0, empty0 = load_x ? xempty0 : wempty0;
            bool ok = true;
            TaUnit un;
            for (int i = 0; ok && ta_unit<kC>(a, i, un); ++i) {
                int mb, nb;
                rows_tile_coords(un.t, m_units, a.n_tiles, mb, nb);
                mb = mb * kC + rank;
                const int n0 = nb * kOutBN;
                for (int kb = un.kb0; kb < un.kb1 + (kLora ? un.extra : 0); ++kb) {
                    const bool ext = kLora && kb >= un.kb1;   // the adapter stages: T (hi, lo) and B
                    // (paired: rank 0's commit releases W slots in both CTAs)
                    if (!(kPair && !load_x ? mbar_wait_cluster(empty0 + 8 * ring.idx, ring.phase ^ 1, abort)
                                           : mbar_wait(empty0 + 8 * ring.idx, ring.phase ^ 1, abort))) {
                        ok = false;
                        break;
                    }
                    const uint32_t f = full0 + 8 * ring.idx;
                    if (kLora && ext && load_x) grid_dep_wait();   // T is the previous launch's output
                    if (load_x) {
                        mbar_arrive_expect_tx(f, kTaXBytes + (ext ? 0 : kGBytes));
                        tma_load_2d_nohint(sx + ring.idx * kTaXBytes, ext ? &tmT : &tmX, f,
                                           (ext ? kb - un.kb1 : kb) * kBK, mb * kRowsBM);
                        if (!ext) tma_load_1d(sg + ring.idx * kGBytes, &tmG, f, kb * kBK);
                    } else if constexpr (kPair) {
                        // this CTA's half of the stage: columns n0 + 128 rank + [0, 128), the boxes inside N;
                        // rank 0's copies complete on the k-block's ready barrier (its A slot's)
                        // (adapter stages: the same columns of B's rows; gated: rank 0 the
                        // tile's gate columns, rank 1 its up columns, so that each CTA's
                        // accumulator row holds both, as unpaired)
                        // Weights stored [N, K]: one [128 n][64 k] box of those columns' rows,
                        // K-major (the tensor map's box is 128 rows for paired launches).
                        const int c0 = kGlu ? (rank == 0 ? n0 : Nout + n0) : n0 + 128 * rank;
                        const uint32_t fw = rank == 0 ? afull0 + 8 * rr.idx : f;
                        if constexpr (kWnk) {
                            mbar_arrive_expect_tx(fw, kWSlot);
                            tma_load_2d_nohint(sw + ring.idx * kWSlot, &tmW, fw, kb * kBK, c0);
                        } else {
                            const int nbox = kGlu ? 2 : c0 >= a.N ? 0 : min(2, (a.N - c0 + 63) / 64);
                            mbar_arrive_expect_tx(fw, static_cast<uint32_t>(nbox) * kWBoxBytes);
                            for (int j = 0; j < nbox; ++j)
                                tma_load_2d_nohint(sw + ring.idx * kWSlot + j * kWBoxBytes, ext ? &tmB : &tmW, fw,
                                                   c0 + 64 * j, ext ? 0 : kb * kBK);
                        }
                    } else {
                        mbar_arrive_expect_tx(f, w_stage_bytes<kGlu, kWnk>(n0, a.N));
                        load_w_stage<kGlu, kWnk>(sw + ring.idx * kRowsWBytes, ext ? &tmB : &tmW, f, n0,
                                                 ext ? 0 : kb, a.N, Nout);
                    }
                    ring.advance();
                    rr.advance();
                    ++issued;
                }
            }
            // never leave with copies still landing in shared memory (paired,
            // rank 0's W: they complete on the ready barriers)
            const bool on_ready = kPair && !load_x && rank == 0;
            const uint32_t tn = on_ready ? rr.n : ring.n, tfull0 = on_ready ? afull0 : full0;
            // (after a timed-out wait the rest are not waited for: an aborted launch stays short)
            for (uint32_t i = issued > tn ? issued - tn : 0; i < issued; ++i)
                if (!mbar_wait_teardown(tfull0 + 8 * (i % tn), (i / tn) & 1)) break;
            const uint32_t n = ring.n;
            // Paired: rank 0's MMAs release every W slot of both CTAs (commit
            // multicast), and those arrivals land asynchronously.  Wait until
            // the last use of each slot has been released, so that after the
            // exit barrier no arrival is still in flight towards this CTA.
            if (kPair && !load_x)
                for (uint32_t i = issued > n ? issued - n : 0; i < issued; ++i)
                    if (!mbar_wait_teardown(empty0 + 8 * (i % n), (i / n) & 1)) break;
        }
    } else if (warp == 1) {
        if constexpr (kPair) {
            if (rank == 1) {
                // ------------------------------------------------ paired, rank 1: stage-ready signals
                // Each k-block's W half and A slot of this CTA, once in place, are
                // announced on rank 0's ready barrier of the k-block (its A slot's).
                if (lane == 0) {
                    Ring wr(kWSt), ar(kTaAStages);
                    const uint32_t ready_r0 = mapa_shared(afull0, 0);
                    bool ok = true;
                    TaUnit un;
                    for (int i = 0; ok && ta_unit<kC>(a, i, un); ++i) {
                        for (int kb = un.kb0; kb < un.kb1 + (kLora ? un.extra : 0); ++kb) {
                            if (!mbar_wait(wfull0 + 8 * wr.idx, wr.phase, abort)) { ok = false; break; }
                            if (!mbar_wait(afull0 + 8 * ar.idx, ar.phase, abort)) { ok = false; break; }
                            // (test hook: leave out the first signal, so that rank 0's wait runs out)
                            if (!(a.test_skip_sends && i == 0 && kb == un.kb0))
                                mbar_arrive_remote_relaxed(ready_r0 + 8 * ar.idx);
                            wr.advance();
                            ar.advance();
                        }
                    }
                }
            } else {
                // ------------------------------------------------ paired, rank 0: pair MMA issuer
                if (lane == 0) {
                    constexpr uint32_t idesc = idesc_bf16_f32(2 * kRowsBM, kRowsBN, false, !kWnk);
                    Ring wr(kWSt), ar(kTaAStages);
                    uint32_t tl = 0;
                    bool ok = true;
                    TaUnit un;
                    for (int i = 0; ok && ta_unit<kC>(a, i, un); ++i, ++tl) {
                        // both CTAs' epilogues have read the accumulator
                        if (!mbar_wait_cluster(accempty, (tl & 1) ^ 1, abort)) break;
                        tc_fence_after();
                        const uint32_t d = tmem + kTaAccCol;
                        for (int kb = un.kb0; kb < un.kb1 + (kLora ? un.extra : 0); ++kb) {
                            // both CTAs' W halves and A slots of this k-block
                            if (!mbar_wait_cluster(afull0 + 8 * ar.idx, ar.phase, abort)) { ok = false; break; }
                            tc_fence_after();
                            const uint32_t a0 = tmem + kTaACol + ar.idx * 32;
                            const uint32_t b0 = sw + wr.idx * kWSlot;
#pragma unroll
                            for (int kk = 0; kk < kBK / 16; ++kk)
                                mma_bf16_ts_pair(d, a0 + kk * 8, w_desc<kWnk>(b0, kk), idesc, kb != un.kb0 || kk != 0);
                            mma_commit_pair_mc(wempty0 + 8 * wr.idx, 0x3);   // both CTAs' W halves
                            mma_commit_pair_mc(aempty0 + 8 * ar.idx, 0x3);   // both CTAs' A slots
                            wr.advance();
                            ar.advance();
                        }
                        if (!ok) break;
                        mma_commit_pair_mc(accfull, 0x3);
                    }
                    mma_commit_pair_mc(mmadone, 0x1);
                    mbar_wait_teardown(mmadone, 0);
                }
            }
        } else {
            // ------------------------------------------------ MMA issuer
            if (lane == 0) {
                // the hi/lo output (N <= 64) multiplies one 64-column box of W, not a 256-wide padded tile
                constexpr uint32_t idesc = idesc_bf16_f32(kRowsBM, kHilo ? kBK : kRowsBN, false, !kWnk);
                Ring wr(kTaWStages), ar(kTaAStages);
                uint32_t tl = 0;
                bool ok = true;
                TaUnit un;
                for (int i = 0; ok && ta_unit<kC>(a, i, un); ++i, ++tl) {
                    if (!mbar_wait(accempty, (tl & 1) ^ 1, abort)) break;
                    tc_fence_after();
                    const uint32_t d = tmem + kTaAccCol;
                    for (int kb = un.kb0; kb < un.kb1 + (kLora ? un.extra : 0); ++kb) {
                        if (!mbar_wait(wfull0 + 8 * wr.idx, wr.phase, abort)) { ok = false; break; }
                        if (!mbar_wait(afull0 + 8 * ar.idx, ar.phase, abort)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t a0 = tmem + kTaACol + ar.idx * 32;
                        const uint32_t b0 = sw + wr.idx * kRowsWBytes;
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)
                            mma_bf16_ts(d, a0 + kk * 8, w_desc<kWnk>(b0, kk), idesc, kb != un.kb0 || kk != 0);
                        mma_commit(wempty0 + 8 * wr.idx);
                        mma_commit(aempty0 + 8 * ar.idx);
                        wr.advance();
                        ar.advance();
                    }
                    if (!ok) break;
                    mma_commit(accfull);
                }
                mma_commit(mmadone);
                mbar_wait_teardown(mmadone, 0);
            }
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------ transform: X*g -> tensor memory
        const int q = warp - 4;               // lane quarter this warp may access
        const int row = q * 32 + lane;        // row of the X tile
        const uint32_t xrow = static_cast<uint32_t>(row) * 128;
        const uint32_t swz = static_cast<uint32_t>(row & 7);
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        Ring xr(kXSt), ar(kTaAStages);
        uint32_t tl = 0, a_used = 0;
        bool ok = true;
        TaUnit un;
        for (int i = 0; ok && ta_unit<kC>(a, i, un); ++i, ++tl) {
            const uint32_t buf = tl & 1, use = tl >> 1;
            // sr[buf] is free once the epilogue read it for the tile two back
            if (!warp_wait(srempty0 + 8 * buf, (use & 1) ^ 1, abort)) break;
            float ssp[8];   // independent partial sums: no long dependency chain
#pragma unroll
            for (int c = 0; c < 8; ++c) ssp[c] = 0.f;
            // The X rows of block kb + 1 are loaded from shared memory before
            // block kb's store into tensor memory, so that the two overlap.
            const int kend = un.kb1 + (kLora ? un.extra : 0);
            uint4 xv[8];
            if (!warp_wait(xfull0 + 8 * xr.idx, xr.phase, abort)) { ok = false; break; }
#pragma unroll
            for (int c = 0; c < 8; ++c) xv[c] = lds128(sx + xr.idx * kTaXBytes + xrow + ((c ^ swz) << 4));
            for (int kb = un.kb0; kb < kend; ++kb) {
                const bool ext = kLora && kb >= un.kb1;   // the adapter stages: T rows, no gain, no statistic
                const uint32_t gt = sg + xr.idx * kGBytes;   // g of this block (the slot of its X)
                uint32_t out[32];
                if (!ext) {
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint4 gv = lds128(gt + c * 16);
                        const uint32_t xs[4] = {xv[c].x, xv[c].y, xv[c].z, xv[c].w};
                        const uint32_t gs[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            ssp[c] = fma_sq_bf16x2(xs[i], ssp[c]);
                            out[c * 4 + i] = mul_bf16x2(xs[i], gs[i]);
                        }
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        out[c * 4 + 0] = xv[c].x;
                        out[c * 4 + 1] = xv[c].y;
                        out[c * 4 + 2] = xv[c].z;
                        out[c * 4 + 3] = xv[c].w;
                    }
                }
                // the X slot has been read (values are in registers)
                __syncwarp();
                if (lane == 0) mbar_arrive(xempty0 + 8 * xr.idx);
                xr.advance();
                if (kb + 1 < kend) {
                    if (!warp_wait(xfull0 + 8 * xr.idx, xr.phase, abort)) { ok = false; break; }
#pragma unroll
                    for (int c = 0; c < 8; ++c) xv[c] = lds128(sx + xr.idx * kTaXBytes + xrow + ((c ^ swz) << 4));
                }
                // (paired: rank 0's commit releases A slots in both CTAs)
                if (!(kPair ? warp_wait_cluster(aempty0 + 8 * ar.idx, ar.phase ^ 1, abort)
                            : warp_wait(aempty0 + 8 * ar.idx, ar.phase ^ 1, abort))) {
                    ok = false;
                    break;
                }
                tmem_st_32x32(tmem + kTaACol + ar.idx * 32 + lane_base, out);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(afull0 + 8 * ar.idx);
                ar.advance();
                ++a_used;
            }
            if (!ok) break;
            sr[buf * kRowsBM + row] = ((ssp[0] + ssp[1]) + (ssp[2] + ssp[3])) +
                                      ((ssp[4] + ssp[5]) + (ssp[6] + ssp[7]));
            __syncwarp();
            if (lane == 0) mbar_arrive(srfull0 + 8 * buf);
        }
        // Paired: the commits that release the last use of each A slot land
        // asynchronously; wait for them, so that after the exit barrier no
        // arrival is still in flight towards this CTA.
        if (kPair && warp == 4 && lane == 0) {
            const uint32_t n = ar.n;
            for (uint32_t i = a_used > n ? a_used - n : 0; i < a_used; ++i)
                if (!mbar_wait_teardown(aempty0 + 8 * (i % n), (i / n) & 1)) break;
        }
    } else if (warp >= 8) {
        // ------------------------------------------------ epilogue
        // Read the whole accumulator row (scaled, bf16) into registers and
        // release tensor memory at once; then store Y through two 8 KB
        // staging buffers with TMA stores (64-byte swizzle: the 16-byte chunk
        // j of row r sits at chunk j ^ ((r >> 1) & 3)), overlapped with the
        // next tile's main loop.
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const int e = threadIdx.x - 256;
        const float inv_k = 1.f / static_cast<float>(a.K);
        uint32_t ep = 0;
        auto epi_sync = [&]() {
            __syncwarp();
            if (lane == 0) mbar_arrive(episync);
            return warp_wait(episync, (ep++) & 1, abort);
        };
        const uint32_t rswz = static_cast<uint32_t>((row >> 1) & 3);
        uint32_t chunks = 0;   // staging buffer uses so far
        uint32_t tl = 0;
        TaUnit un;
        for (int i = 0; ta_unit<kC>(a, i, un); ++i, ++tl) {
            const uint32_t buf = tl & 1, use = tl >> 1;
            // (paired: rank 0's commit signals both CTAs)
            if (!(kPair ? warp_wait_cluster(accfull, tl & 1, abort) : warp_wait(accfull, tl & 1, abort))) break;
            if (!warp_wait(srfull0 + 8 * buf, use & 1, abort)) break;
            tc_fence_after();
            const float ss_row = sr[buf * kRowsBM + row];
            __syncwarp();
            if (lane == 0) mbar_arrive(srempty0 + 8 * buf);
            int mb, nb;
            rows_tile_coords(un.t, m_units, a.n_tiles, mb, nb);
            mb = mb * kC + rank;
            const int n0 = nb * kOutBN;
            const uint32_t taddr = tmem + kTaAccCol + (static_cast<uint32_t>(q * 32) << 16);
            if (un.piece >= 0) {
                // A K piece of a tail tile: publish the fp32 partial and the
                // partial row sums of squares, wait for the tile's other
                // pieces, then reduce rows [r0, r1) of the tile over all
                // pieces in piece order and write them to Y.
                const int P = a.tail_pieces;
                const int tail = (un.t - (num_tiles - a.tail_tiles)) * kC + rank;   // tail tile
                const size_t slot = static_cast<size_t>(tail) * P;
                if (kLora) grid_dep_wait();   // the launch that computes T may use the workspace
                float* wrow = a.ws_acc + ((slot + un.piece) * kRowsBM + row) * kRowsBN;
                // accumulator columns the reduction reads (a hi/lo output has 64)
                constexpr int kPartCols = kHilo ? kBK : kRowsBN;
#pragma unroll 4
                for (int c = 0; c < kPartCols / 16; ++c) {
                    uint32_t v[16];
                    tmem_ld_32x16(taddr + c * 16, v);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        __stcg(reinterpret_cast<float4*>(wrow + c * 16 + 4 * j),
                               make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                           __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3])));
                }
                __stcg(a.ws_ss + (slot + un.piece) * kRowsBM + row, ss_row);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(accempty);
                __threadfence();
                int* cnt = a.ws_count + 2 * tail;
                bool ok = epi_sync();
                if (e == 0) {
                    atomicAdd(cnt, 1);
                    ok = spin_until_ge(cnt, P, abort) && ok;
                }
                ok = epi_sync() && ok && !*abort;
                const int r0 = (un.piece * kRowsBM) / P, r1 = ((un.piece + 1) * kRowsBM) / P;
                float* rr = reinterpret_cast<float*>(smem + kTaOffRr);
                if (ok && e < r1 - r0) {
                    float tot = 0.f;
                    for (int p2 = 0; p2 < P; ++p2) tot += __ldcg(a.ws_ss + (slot + p2) * kRowsBM + r0 + e);
                    rr[e] = a.unscaled ? 1.f : rsqrtf(tot * inv_k + a.eps);
                }
                ok = epi_sync() && ok;
                // items: 4 output columns of one row; gated, from the gate
                // partial at accumulator column col and the up partial 128
                // columns further
                constexpr int kHalves = kGlu ? 2 : 1;
                constexpr int kRedBN = kHilo ? kBK : kOutBN;   // output columns of the tile
                const int items = (r1 - r0) * (kRedBN / 4);
                for (int it = e; ok && it < items; it += 128) {
                    const int rl = it / (kRedBN / 4), col = (it % (kRedBN / 4)) * 4;
                    const int m = mb * kRowsBM + r0 + rl;
                    const float* src = a.ws_acc + (slot * kRowsBM + r0 + rl) * kRowsBN + col;
                    float4 acc[kHalves];
#pragma unroll
                    for (int h = 0; h < kHalves; ++h) acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
                    int p2 = 0;
                    for (; p2 + 4 <= P; p2 += 4) {
                        float4 t4[4][kHalves];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
#pragma unroll
                            for (int h = 0; h < kHalves; ++h)
                                t4[j][h] = __ldcg(reinterpret_cast<const float4*>(
                                    src + static_cast<size_t>(p2 + j) * kRowsBM * kRowsBN + h * kOutBN));
#pragma unroll
                        for (int j = 0; j < 4; ++j)
#pragma unroll
                            for (int h = 0; h < kHalves; ++h) {
                                acc[h].x += t4[j][h].x;
                                acc[h].y += t4[j][h].y;
                                acc[h].z += t4[j][h].z;
                                acc[h].w += t4[j][h].w;
                            }
                    }
                    for (; p2 < P; ++p2)
#pragma unroll
                        for (int h = 0; h < kHalves; ++h) {
                            const float4 t4 = __ldcg(reinterpret_cast<const float4*>(
                                src + static_cast<size_t>(p2) * kRowsBM * kRowsBN + h * kOutBN));
                            acc[h].x += t4.x;
                            acc[h].y += t4.y;
                            acc[h].z += t4.z;
                            acc[h].w += t4.w;
                        }
                    if (m < a.M && n0 + col < (kHilo ? kBK : Nout)) {
                        const float r = rr[rl];
                        float o4[4];
                        if constexpr (kGlu) {
                            o4[0] = glu_out(acc[0].x, acc[kHalves - 1].x, r);
                            o4[1] = glu_out(acc[0].y, acc[kHalves - 1].y, r);
                            o4[2] = glu_out(acc[0].z, acc[kHalves - 1].z, r);
                            o4[3] = glu_out(acc[0].w, acc[kHalves - 1].w, r);
                        } else {
                            o4[0] = acc[0].x * r;
                            o4[1] = acc[0].y * r;
                            o4[2] = acc[0].z * r;
                            o4[3] = acc[0].w * r;
                            if constexpr (kHilo) {
                                store_hilo4(Y + static_cast<size_t>(m) * (2 * kBK), col, o4[0], o4[1], o4[2], o4[3]);
                                continue;
                            }
                        }
                        uint2 o;
                        o.x = pack_bf16x2(o4[0], o4[1]);
                        o.y = pack_bf16x2(o4[2], o4[3]);
                        *reinterpret_cast<uint2*>(Y + static_cast<size_t>(m) * Nout + n0 + col) = o;
                    }
                }
                // the last piece through resets the tile's counters for the next launch
                epi_sync();
                if (e == 0 && atomicAdd(cnt + 1, 1) == P - 1) {
                    atomicExch(cnt, 0);
                    atomicExch(cnt + 1, 0);
                }
                continue;
            }
            const float r = a.unscaled ? 1.f : rsqrtf(ss_row * inv_k + a.eps);
            uint32_t pk[kOutBN / 2];   // the row's outputs, packed as bf16x2
            // a hilo output: the first 64 accumulator columns as hi (words
            // 0..31, columns 0..63 of Y) and lo (words 32..63, columns 64..127)
            constexpr bool hilo = kHilo;
            if constexpr (hilo) {
#pragma unroll
                for (int c = 0; c < kBK / 16; ++c) {
                    uint32_t v[16];
                    tmem_ld_32x16(taddr + c * 16, v);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        hilo_pack(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]), pk[c * 8 + i],
                                  pk[kBK / 2 + c * 8 + i]);
                }
            }
#pragma unroll
            for (int c = 0; c < (hilo ? 0 : kOutBN / 16); ++c) {
                uint32_t v[16];
                tmem_ld_32x16(taddr + c * 16, v);
                if constexpr (kGlu) {
                    uint32_t w2[16];
                    tmem_ld_32x16(taddr + kOutBN + c * 16, w2);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        pk[c * 8 + i] = pack_bf16x2(
                            glu_out(__uint_as_float(v[2 * i]), __uint_as_float(w2[2 * i]), r),
                            glu_out(__uint_as_float(v[2 * i + 1]), __uint_as_float(w2[2 * i + 1]), r));
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        pk[c * 8 + i] = pack_bf16x2(__uint_as_float(v[2 * i]) * r,
                                                    __uint_as_float(v[2 * i + 1]) * r);
                }
            }
            tc_fence_before();
            __syncwarp();
            // the MMA may start the next tile (paired: rank 0's, once both CTAs' epilogues are here)
            if (lane == 0) {
                if constexpr (kPair) mbar_arrive_remote(mapa_shared(accempty, 0));
                else mbar_arrive(accempty);
            }
            bool ok = true;
            const int nstore = hilo ? 2 * kBK : Nout;   // columns of Y
#pragma unroll
            for (int c = 0; c < kOutBN / 32; ++c) {
                if (n0 + c * 32 < nstore) {             // block-uniform
                    const uint32_t sbuf = sout + (chunks & 1) * kTaStageOut;
                    // the store issued two chunks ago must have read this buffer
                    if (e == 0) bulk_wait_group_read<1>();
                    if (!(ok = epi_sync())) break;
                    const uint32_t rbase = sbuf + row * 64;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        sts128(rbase + ((j ^ rswz) << 4),
                               make_uint4(pk[c * 16 + 4 * j], pk[c * 16 + 4 * j + 1],
                                          pk[c * 16 + 4 * j + 2], pk[c * 16 + 4 * j + 3]));
                    fence_proxy_async_smem();
                    if (!(ok = epi_sync())) break;
                    if (e == 0 && mb < a.m_tiles) {   // (a paired unit's second row block may lie past M)
                        tma_store_2d(&tmY, sbuf, n0 + c * 32, mb * kRowsBM);
                        bulk_commit_group();
                    }
                    ++chunks;
                }
            }
            if (!ok) break;
        }
        if (e == 0) bulk_wait_group_all();   // Y is written before the CTA exits
    }

    tc_fence_before();
    __syncthreads();
    // paired: the peer may still signal this CTA, or rank 0's MMAs read this
    // CTA's memory, until it is done
    if (kPair) cluster_sync_all();
    if (warp == 2) {
        tc_fence_after();
        if constexpr (kPair) tmem_dealloc_pair(tmem, 512);
        else tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------- tall tiles: 256 rows per CTA
// The unfused contraction for many row tiles (prefill-like shapes): each CTA
// computes a tile of 256 rows (two halves of 128, one M = 128 MMA each) by
// 256 columns, so that every W stage it loads feeds both halves.  Per
// 128 x 256 x 64 of work a CTA then takes in 32 KB (16 KB of A, half of a
// 32 KB W stage) instead of the 48 KB of a 128-row tile; on GB300 the operand
// delivery into each SM, not the tensor pipe, bounds the 128-row kernels.
// The two accumulators fill tensor memory (2 x 256 columns) and the MMAs read
// A from shared memory as the copy wrote it; A and W of a k-block share one
// stage, which the MMAs' commit releases.  (The fused form would have to
// multiply each A stage by g in place first, which holds the stage through
// that transform: measured slower than the 128-row fused kernel.)  Warps:
// 0 TMA producer, 1 MMA issuer, 2 tensor-memory allocation, 4-11 epilogue
// (warps 4-7 the first half's rows, 8-11 the second's).  Tiles and tail
// pieces are those of the 128-row kernel with 256-row tiles.
//
// kStat: RMSNorm with the gain already folded into the weights (W' = diag(g)
// W, prepared once; (X diag(g)) W = X W'): A is raw X as the copy wrote it,
// and warps 2-3 read every A stage once more for the row sums of squares
// (each of their 64 threads four rows of the tile; the stage is released
// when both the MMAs and they are done).  The epilogue scales row m by
// 1/rms_m; tail pieces publish their partial row sums with their partial
// products and the reducing piece adds both in piece order.
constexpr uint32_t kTtXBytes = kTtBM * kBK * 2;               // 32 KB
constexpr uint32_t kTtStageBytes = kTtXBytes + kRowsWBytes;   // 64 KB: A, then W
constexpr uint32_t kTtOutBytes = kRowsBM * 32 * 2;            // 8 KB: 128 rows x 32 bf16 of C
constexpr uint32_t kTtOffOut = kTtStages * kTtStageBytes;     // two staging buffers per half
constexpr uint32_t kTtOffBar = kTtOffOut + 4 * kTtOutBytes;
// full, empty per stage; accfull, accempty, mmadone, episync[2], tailsync,
// srfull, srempty
constexpr uint32_t kTtNumBars = 2 * kTtStages + 8;
constexpr uint32_t kTtOffSr = kTtOffBar + ((kTtNumBars * 8 + 15) / 16) * 16;   // [256] row sums (kStat)
constexpr uint32_t kTtOffMisc = kTtOffSr + kTtBM * 4;
constexpr uint32_t kTtSmem = kTtOffMisc + 16 + 1024;
static_assert(kTtSmem <= 232448, "the tall-tile kernel's shared memory exceeds the opt-in limit");

// kStat: how a tile gets its rows' statistic.  A row block's first column
// tile (nb = 0), when whole, forms it and publishes r to the workspace
// (kTtPublish); the row block's other whole tiles read it there (kTtRead) and
// skip the extra pass over X; tail pieces form their partial sums
// (kTtPiece).  A whole tile whose row block's first tile were a tail tile
// would form its own (kTtSelf); with tail tiles the last indices and a row
// block's first tile its smallest, that does not arise, but the check costs
// nothing.  A reader waits for the flag of a tile with a smaller index, which
// every CTA reaches before any larger one of its own, so the launch (all CTAs
// resident: cooperative) cannot deadlock.
enum { kTtSelf = 0, kTtPublish = 1, kTtRead = 2, kTtPiece = 3 };
__device__ __forceinline__ int tt_tile_index(int mb, int nb, int m_tiles, int n_tiles) {
    constexpr int G = 8;   // as rows_tile_coords
    const int group = mb / G, first = group * G, gsz = min(m_tiles - first, G);
    return group * G * n_tiles + nb * gsz + (mb - first);
}
__device__ __forceinline__ int tt_stat_mode(const RowsLaunch& a, const TaUnit& un, int mb, int nb) {
    if (un.piece >= 0) return kTtPiece;
    const int limit = a.m_tiles * a.n_tiles - a.tail_tiles;   // whole tiles: index < limit
    if (tt_tile_index(mb, 0, a.m_tiles, a.n_tiles) >= limit) return kTtSelf;
    return nb == 0 ? kTtPublish : kTtRead;
}
// whole tiles of row block mb that read its published r
__device__ __forceinline__ int tt_readers(const RowsLaunch& a, int mb) {
    const int limit = a.m_tiles * a.n_tiles - a.tail_tiles;
    int n = 0;
    for (int nb = 1; nb < a.n_tiles; ++nb) n += tt_tile_index(mb, nb, a.m_tiles, a.n_tiles) < limit;
    return n;
}
// [m_tiles][256] published r, after the tail pieces' row sums
__device__ __forceinline__ float* tt_r_base(const RowsLaunch& a) {
    return a.ws_ss + static_cast<size_t>(a.tail_tiles) * a.tail_pieces * kTtBM;
}
// [m_tiles] flags, then [m_tiles] reader counts, after the tail counters
__device__ __forceinline__ int* tt_flags(const RowsLaunch& a) { return a.ws_count + 2 * a.tail_tiles; }

template <bool kStat>
__global__ void __launch_bounds__(kThreads, 1)
    tall_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                const __grid_constant__ CUtensorMap tmY, __nv_bfloat16* __restrict__ Y, RowsLaunch a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    const uint32_t sb = smem_u32(smem);
    const uint32_t sout = sb + kTtOffOut;
    const uint32_t bar0 = sb + kTtOffBar;
    const uint32_t full0 = bar0, empty0 = bar0 + 8 * kTtStages;
    const uint32_t accfull = bar0 + 16 * kTtStages, accempty = accfull + 8, mmadone = accfull + 16;
    const uint32_t episync0 = accfull + 24, tailsync = accfull + 40;
    // kStat: the tile's row sums of squares are in sr / have been read
    const uint32_t srfull = accfull + 48, srempty = accfull + 56;
    float* sr = reinterpret_cast<float*>(smem + kTtOffSr);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kTtOffMisc);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + kTtOffMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kTtStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kStat ? 3 : 1);   // the MMAs' commit (+ warps 2-3)
        }
        mbar_init(accfull, 1);
        mbar_init(accempty, 8);
        mbar_init(mmadone, 1);
        mbar_init(episync0, 4);
        mbar_init(episync0 + 8, 4);
        mbar_init(tailsync, 8);
        mbar_init(srfull, 2);    // one lane of each of warps 2-3
        mbar_init(srempty, 8);   // one lane of each epilogue warp
        abort[0] = 0;
        abort[1] = a.wait_limit_us;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
        prefetch_tmap(&tmY);
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_holder), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Set-up above overlaps the previous kernel on the stream; its writes are
    // visible after grid_dep_wait().  The next kernel may then be scheduled.
    grid_dep_wait();
    if (threadIdx.x == 0) grid_dep_launch();
    const uint32_t tmem = *tmem_holder;
    const int num_tiles = a.m_tiles * a.n_tiles;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            Ring ring(kTtStages);
            uint32_t issued = 0;
            bool ok = true;
            TaUnit un;
            for (int i = 0; ok && ta_unit<1>(a, i, un); ++i) {
                int mb, nb;
                rows_tile_coords(un.t, a.m_tiles, a.n_tiles, mb, nb);
                const int n0 = nb * kRowsBN;
                const uint32_t wbytes = w_stage_bytes<false, false>(n0, a.N);
                for (int kb = un.kb0; kb < un.kb1; ++kb) {
                    if (!mbar_wait(empty0 + 8 * ring.idx, ring.phase ^ 1, abort)) { ok = false; break; }
                    const uint32_t f = full0 + 8 * ring.idx;
                    const uint32_t st = sb + ring.idx * kTtStageBytes;
                    mbar_arrive_expect_tx(f, kTtXBytes + wbytes);
                    // two boxes of 128 rows (a box past M reads zeros)
                    tma_load_2d_nohint(st, &tmX, f, kb * kBK, mb * kTtBM);
                    tma_load_2d_nohint(st + kTtXBytes / 2, &tmX, f, kb * kBK, mb * kTtBM + kRowsBM);
                    load_w_stage<false, false>(st + kTtXBytes, &tmW, f, n0, kb, a.N, a.N);
                    ring.advance();
                    ++issued;
                }
            }
            // never leave with copies still landing in shared memory
            const uint32_t n = ring.n;
            for (uint32_t i = issued > n ? issued - n : 0; i < issued; ++i)
                mbar_wait_teardown(full0 + 8 * (i % n), (i / n) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kRowsBM, kRowsBN, false, true);
            Ring ring(kTtStages);
            uint32_t tl = 0;
            bool ok = true;
            TaUnit un;
            for (int i = 0; ok && ta_unit<1>(a, i, un); ++i, ++tl) {
                if (!mbar_wait(accempty, (tl & 1) ^ 1, abort)) break;
                tc_fence_after();
                for (int kb = un.kb0; kb < un.kb1; ++kb) {
                    if (!mbar_wait(full0 + 8 * ring.idx, ring.phase, abort)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t st = sb + ring.idx * kTtStageBytes;
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)
                            mma_bf16_ss(tmem + h * kRowsBN, sdesc_sw128(st + h * (kTtXBytes / 2) + kk * 32, 16, 1024),
                                        w_desc<false>(st + kTtXBytes, kk), idesc, kb != un.kb0 || kk != 0);
                    mma_commit(empty0 + 8 * ring.idx);
                    ring.advance();
                }
                if (!ok) break;
                mma_commit(accfull);
            }
            mma_commit(mmadone);
            mbar_wait_teardown(mmadone, 0);
        }
    } else if (kStat && (warp == 2 || warp == 3)) {
        // ------------------------------------------------ row sums of squares
        // Thread st of 64 takes rows st + 64 j of every A stage: the whole
        // row, its eight 16-byte pieces read from lane-rotated positions so
        // that the eight lanes of an access phase hit distinct banks.  Tiles
        // that read their row block's published r skip the reads (but keep
        // step with the stages).
        const int st = threadIdx.x - 64;
        Ring ring(kTtStages);
        uint32_t ts = 0;   // tiles whose sums went through sr
        bool ok = true;
        TaUnit un;
        for (int i = 0; ok && ta_unit<1>(a, i, un); ++i) {
            int mb, nb;
            rows_tile_coords(un.t, a.m_tiles, a.n_tiles, mb, nb);
            const int mode = tt_stat_mode(a, un, mb, nb);
            float ss[4] = {0.f, 0.f, 0.f, 0.f};
            for (int kb = un.kb0; kb < un.kb1; ++kb) {
                if (!warp_wait(full0 + 8 * ring.idx, ring.phase, abort)) { ok = false; break; }
                const uint32_t stg = sb + ring.idx * kTtStageBytes;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (mode == kTtRead) break;
                    const int r = st + 64 * j;
                    const uint32_t rowp = stg + (r >> 7) * (kTtXBytes / 2) + (r & 127) * 128;
#pragma unroll
                    for (int c0 = 0; c0 < 8; c0 += 4) {
                        uint4 v[4];
#pragma unroll
                        for (int c = 0; c < 4; ++c) v[c] = lds128(rowp + (((c0 + c + lane) & 7) << 4));
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            ss[j] = fma_sq_bf16x2(v[c].x, ss[j]);
                            ss[j] = fma_sq_bf16x2(v[c].y, ss[j]);
                            ss[j] = fma_sq_bf16x2(v[c].z, ss[j]);
                            ss[j] = fma_sq_bf16x2(v[c].w, ss[j]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty0 + 8 * ring.idx);
                ring.advance();
            }
            if (!ok) break;
            if (mode == kTtRead) continue;
            // the epilogue has read the previous tile's sums
            if (ts > 0 && !warp_wait(srempty, (ts - 1) & 1, abort)) break;
#pragma unroll
            for (int j = 0; j < 4; ++j) sr[st + 64 * j] = ss[j];
            __syncwarp();
            if (lane == 0) mbar_arrive(srfull);
            ++ts;
            if (mode == kTtPublish && tt_readers(a, mb) > 0) {
                // the row block's r for its other tiles: values, then the flag
                // (which the last of them resets)
                float* rb = tt_r_base(a) + static_cast<size_t>(mb) * kTtBM;
#pragma unroll
                for (int j = 0; j < 4; ++j) __stcg(rb + st + 64 * j, rsqrtf(ss[j] * (1.f / a.K) + a.eps));
                named_bar_sync(1, 64);
                if (st == 0) {
                    __threadfence();
                    atomicExch(tt_flags(a) + mb, 1);
                }
            }
        }
    } else if (warp >= 4) {
        // ------------------------------------------------ epilogue
        // Read this thread's accumulator row (bf16) into registers and
        // release tensor memory at once; then store C through the half's two
        // 8 KB staging buffers with TMA stores (64-byte swizzle: the 16-byte
        // chunk j of row r sits at chunk j ^ ((r >> 1) & 3)), overlapped with
        // the next tile's main loop.
        const int hh = (warp - 4) >> 2;                // half of the tile
        const int q = warp & 3;                        // lane quarter this warp may access
        const int rh = q * 32 + lane;                  // row within the half (tensor-memory lane)
        const int row = hh * kRowsBM + rh;             // row of the tile
        const int et = threadIdx.x - 128;              // 0..255
        const uint32_t taddr = tmem + hh * kRowsBN + (static_cast<uint32_t>(q * 32) << 16);
        const uint32_t episync = episync0 + 8 * hh;
        uint32_t ep = 0, tp = 0;
        // the four warps of this half; all eight warps
        auto half_sync = [&]() {
            __syncwarp();
            if (lane == 0) mbar_arrive(episync);
            return warp_wait(episync, (ep++) & 1, abort);
        };
        auto all_sync = [&]() {
            __syncwarp();
            if (lane == 0) mbar_arrive(tailsync);
            return warp_wait(tailsync, (tp++) & 1, abort);
        };
        const uint32_t rswz = static_cast<uint32_t>((rh >> 1) & 3);
        uint32_t chunks = 0;   // staging buffer uses so far (per half)
        uint32_t tl = 0;
        TaUnit un;
        const float inv_k = 1.f / static_cast<float>(a.K);
        uint32_t ts = 0;   // (kStat) tiles whose sums came through sr
        for (int i = 0; ta_unit<1>(a, i, un); ++i, ++tl) {
            if (!warp_wait(accfull, tl & 1, abort)) break;
            int mb, nb;
            rows_tile_coords(un.t, a.m_tiles, a.n_tiles, mb, nb);
            const int n0 = nb * kRowsBN, m0 = mb * kTtBM;
            // kStat: this tile's (or piece's) row sum of squares, or the
            // row block's r as its first tile published it
            float ssr = 0.f, rr = 1.f;
            if (kStat) {
                if (tt_stat_mode(a, un, mb, nb) == kTtRead) {
                    int* flag = tt_flags(a) + mb;
                    if (!spin_until_ge(flag, 1, abort)) break;
                    rr = __ldcg(tt_r_base(a) + static_cast<size_t>(mb) * kTtBM + row);
                    // the last of the row block's readers resets its flag for the next call
                    __syncwarp();
                    if (lane == 0 && atomicAdd(flag + a.m_tiles, 1) == 8 * tt_readers(a, mb) - 1) {
                        atomicExch(flag + a.m_tiles, 0);
                        atomicExch(flag, 0);
                    }
                } else {
                    if (!warp_wait(srfull, ts & 1, abort)) break;
                    ssr = sr[row];
                    __syncwarp();
                    if (lane == 0) mbar_arrive(srempty);
                    ++ts;
                    rr = rsqrtf(ssr * inv_k + a.eps);
                }
            }
            tc_fence_after();
            if (un.piece >= 0) {
                // A K piece of a tail tile: publish the fp32 partial, wait for
                // the tile's other pieces, then reduce rows [r0, r1) of the
                // tile over all pieces in piece order and write them to C.
                const int P = a.tail_pieces;
                const int tail = un.t - (num_tiles - a.tail_tiles);
                const size_t slot = static_cast<size_t>(tail) * P;
                float* wrow = a.ws_acc + ((slot + un.piece) * kTtBM + row) * kRowsBN;
#pragma unroll 4
                for (int c = 0; c < kRowsBN / 16; ++c) {
                    uint32_t v[16];
                    tmem_ld_32x16(taddr + c * 16, v);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        __stcg(reinterpret_cast<float4*>(wrow + c * 16 + 4 * j),
                               make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                           __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3])));
                }
                if (kStat) __stcg(a.ws_ss + (slot + un.piece) * kTtBM + row, ssr);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(accempty);
                __threadfence();
                int* cnt = a.ws_count + 2 * tail;
                bool ok = all_sync();
                if (et == 0) {
                    atomicAdd(cnt, 1);
                    ok = spin_until_ge(cnt, P, abort) && ok;
                }
                ok = all_sync() && ok && !*abort;
                const int r0 = (un.piece * kTtBM) / P, r1 = ((un.piece + 1) * kTtBM) / P;
                // items: 4 output columns of one row
                const int items = (r1 - r0) * (kRowsBN / 4);
                for (int it = et; ok && it < items; it += 256) {
                    const int rl = it / (kRowsBN / 4), col = (it % (kRowsBN / 4)) * 4;
                    const int m = m0 + r0 + rl;
                    const float* src = a.ws_acc + (slot * kTtBM + r0 + rl) * kRowsBN + col;
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    int p2 = 0;
                    for (; p2 + 4 <= P; p2 += 4) {
                        float4 t4[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            t4[j] = __ldcg(reinterpret_cast<const float4*>(
                                src + static_cast<size_t>(p2 + j) * kTtBM * kRowsBN));
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            acc.x += t4[j].x;
                            acc.y += t4[j].y;
                            acc.z += t4[j].z;
                            acc.w += t4[j].w;
                        }
                    }
                    for (; p2 < P; ++p2) {
                        const float4 t4 =
                            __ldcg(reinterpret_cast<const float4*>(src + static_cast<size_t>(p2) * kTtBM * kRowsBN));
                        acc.x += t4.x;
                        acc.y += t4.y;
                        acc.z += t4.z;
                        acc.w += t4.w;
                    }
                    if (kStat) {
                        // the row's sum of squares over the pieces, in piece order
                        const float* ssrc = a.ws_ss + slot * kTtBM + r0 + rl;
                        float tot = 0.f;
                        for (int p3 = 0; p3 < P; ++p3) tot += __ldcg(ssrc + static_cast<size_t>(p3) * kTtBM);
                        const float rr = rsqrtf(tot * inv_k + a.eps);
                        acc.x *= rr;
                        acc.y *= rr;
                        acc.z *= rr;
                        acc.w *= rr;
                    }
                    if (m < a.M && n0 + col < a.N) {
                        uint2 o;
                        o.x = pack_bf16x2(acc.x, acc.y);
                        o.y = pack_bf16x2(acc.z, acc.w);
                        *reinterpret_cast<uint2*>(Y + static_cast<size_t>(m) * a.N + n0 + col) = o;
                    }
                }
                // the last piece through resets the tile's counters for the next launch
                all_sync();
                if (et == 0 && atomicAdd(cnt + 1, 1) == P - 1) {
                    atomicExch(cnt, 0);
                    atomicExch(cnt + 1, 0);
                }
                if (!ok) break;
                continue;
            }
            uint32_t pk[kRowsBN / 2];   // the row's outputs, packed as bf16x2
#pragma unroll
            for (int c = 0; c < kRowsBN / 16; ++c) {
                uint32_t v[16];
                tmem_ld_32x16(taddr + c * 16, v);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    pk[c * 8 + j] = pack_bf16x2(__uint_as_float(v[2 * j]) * rr, __uint_as_float(v[2 * j + 1]) * rr);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(accempty);   // the MMA may start the next tile
            bool ok = true;
            const bool rows_in = m0 + hh * kRowsBM < a.M;   // (a half past M is not stored)
#pragma unroll
            for (int c = 0; c < kRowsBN / 32; ++c) {
                if (n0 + c * 32 < a.N) {             // block-uniform
                    const uint32_t sbuf = sout + (2 * hh + (chunks & 1)) * kTtOutBytes;
                    // the store issued two chunks ago must have read this buffer
                    if (rh == 0) bulk_wait_group_read<1>();
                    if (!(ok = half_sync())) break;
                    const uint32_t rbase = sbuf + rh * 64;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        sts128(rbase + ((j ^ rswz) << 4),
                               make_uint4(pk[c * 16 + 4 * j], pk[c * 16 + 4 * j + 1], pk[c * 16 + 4 * j + 2],
                                          pk[c * 16 + 4 * j + 3]));
                    fence_proxy_async_smem();
                    if (!(ok = half_sync())) break;
                    if (rh == 0 && rows_in) {
                        tma_store_2d(&tmY, sbuf, n0 + c * 32, m0 + hh * kRowsBM);
                        bulk_commit_group();
                    }
                    ++chunks;
                }
            }
            if (!ok) break;
        }
        if (rh == 0) bulk_wait_group_all();   // C is written before the CTA exits
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
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

// ------------------------------------------------------------ gain folding
// W'[k, n] = bf16(g[k] W[k, n]): the product of two bf16 values is exact in
// fp32, so W' holds one rounding of it.  One thread per 8 columns of a row
// (N a multiple of 8).
__global__ void __launch_bounds__(kNormThreads)
    fold_gain_kernel(const __nv_bfloat16* __restrict__ g, const __nv_bfloat16* W, __nv_bfloat16* Wg,
                     int64_t K, int64_t N) {
    const int64_t per_row = N / 8, total = K * per_row;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kNormThreads + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * kNormThreads) {
        const int64_t k = i / per_row;
        const float gk = __bfloat162float(g[k]);
        const uint4 v = reinterpret_cast<const uint4*>(W)[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = pack_bf16x2(bf16lo(w[j]) * gk, bf16hi(w[j]) * gk);
        reinterpret_cast<uint4*>(Wg)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// Raises a kernel's dynamic shared-memory limit to the device's opt-in
// maximum, once per (kernel slot, device).
cudaError_t ensure_smem_attr(const void* func, int slot) {
    static int done[32][64] = {};
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

size_t rows_smem_bytes(int xrows, int stages, int red_slots, int MP, bool overlay, bool glu, int bn) {
    return rows_layout(xrows, stages, red_slots, MP, overlay, glu, bn).total;
}
bool rows_overlay_fits(int xrows, int stages, int splits, int MP, bool glu, int bn) {
    const RowsLayout L = rows_layout(xrows, stages, splits, MP, true, glu, bn);
    return static_cast<uint32_t>(splits) * L.red_block <= L.off_g;
}
size_t rows_stage_bytes(int xrows, int bn) { return xrows * kBK * 2 + static_cast<size_t>(bn) * kBK * 2 + kGBytes; }
// Launch with programmatic dependent launch (the kernel's set-up may overlap
// the previous kernel on the stream) and, optionally, a 1-D cluster, or as a
// cooperative grid (all CTAs resident at once, or the launch fails).
template <typename... Args>
cudaError_t launch_ex(void (*kern)(Args...), int grid, size_t smem, int cluster, cudaStream_t s,
                      bool cooperative, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[3];
    int n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cooperative) {
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n].val.cooperative = 1;
        ++n;
    }
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

cudaError_t launch_rows(bool fused, const CUtensorMap& tmX, const CUtensorMap& tmW,
                        const CUtensorMap& tmG, const CUtensorMap& tmT, const CUtensorMap& tmB, void* Y,
                        const RowsLaunch& a, cudaStream_t s) {
    auto* y = static_cast<__nv_bfloat16*>(Y);
    const bool split = a.cluster != 0;
    const bool glu = a.glu != 0, wnk = a.w_nk != 0, lora = a.lora != 0;
    if ((glu || wnk || lora) && !fused) return cudaErrorInvalidValue;
    if (lora && (glu || wnk)) return cudaErrorInvalidValue;
    if (a.tall) {
        if (fused || glu || wnk || lora || a.hilo || a.unscaled || split) return cudaErrorInvalidValue;
        auto tk = a.fold ? tall_kernel<true> : tall_kernel<false>;
        cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(tk), a.fold ? 28 : 22);
        if (e != cudaSuccess) return e;
        // cooperative with tail pieces, as the 128-row kernel
        // (folded: tiles wait for their row block's first tile, in another CTA)
        e = launch_ex(tk, a.grid, kTtSmem, 1, s, a.tail_tiles > 0 || a.fold != 0, tmX, tmW, *a.tmY, y, a);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    if (fused && !split && a.xrows == kRowsBM) {
        const bool hilo = a.hilo != 0;
        if (hilo && (glu || wnk || lora)) return cudaErrorInvalidValue;
        const bool pair = a.pair != 0;
        if (pair && hilo) return cudaErrorInvalidValue;
        auto ta = pair ? (lora  ? rows_ta_kernel<false, false, true, false, true>
                          : wnk ? (glu ? rows_ta_kernel<true, true, false, false, true>
                                       : rows_ta_kernel<false, true, false, false, true>)
                          : glu ? rows_ta_kernel<true, false, false, false, true>
                                : rows_ta_kernel<false, false, false, false, true>)
                : hilo ? rows_ta_kernel<false, false, false, true, false>
                : lora ? rows_ta_kernel<false, false, true, false, false>
                : wnk  ? (glu ? rows_ta_kernel<true, true, false, false, false>
                              : rows_ta_kernel<false, true, false, false, false>)
                       : (glu ? rows_ta_kernel<true, false, false, false, false>
                              : rows_ta_kernel<false, false, false, false, false>);
        cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(ta),
                                         pair ? (lora ? 23 : wnk ? (glu ? 25 : 24) : glu ? 21 : 20) : hilo ? 19 : lora ? 18 : wnk ? (glu ? 15 : 14) : (glu ? 9 : 6));
        if (e != cudaSuccess) return e;
        // The pieces of a tail tile wait for one another: launched as a
        // cooperative grid, every CTA is resident at once (or the launch
        // fails), whatever else shares the device.
        e = launch_ex(ta, a.grid, kTaSmem, pair ? 2 : 1, s, a.tail_tiles > 0, tmX, tmW, tmG, tmT, tmB, *a.tmY, y, a);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    const int bn = a.bn ? a.bn : kRowsBN;   // (0: the default width)
    decltype(&rows_kernel<true, true, true, true, false>) kern;
    int slot;
    if (lora) {
        kern = split ? rows_kernel<true, true, false, false, true> : rows_kernel<true, false, false, false, true>;
        slot = split ? 17 : 16;
    } else if (wnk) {
        kern = glu ? (split ? rows_kernel<true, true, true, true, false> : rows_kernel<true, false, true, true, false>)
                   : (split ? rows_kernel<true, true, false, true, false> : rows_kernel<true, false, false, true, false>);
        slot = 10 + (glu ? 2 : 0) + (split ? 1 : 0);
    } else if (glu) {
        kern = split ? rows_kernel<true, true, true, false, false> : rows_kernel<true, false, true, false, false>;
        slot = split ? 8 : 7;
    } else if (bn == kRowsBN / 2) {
        if (!split) return cudaErrorInvalidValue;   // 128-column tiles: K split only
        kern = fused ? rows_kernel<true, true, false, false, false, kRowsBN / 2>
                     : rows_kernel<false, true, false, false, false, kRowsBN / 2>;
        slot = fused ? 26 : 27;
    } else {
        kern = fused ? (split ? rows_kernel<true, true, false, false, false> : rows_kernel<true, false, false, false, false>)
                     : (split ? rows_kernel<false, true, false, false, false> : rows_kernel<false, false, false, false, false>);
        slot = (fused ? 0 : 1) + (split ? 4 : 0);
    }
    if (bn != kRowsBN && bn != kRowsBN / 2) return cudaErrorInvalidValue;
    if (bn != kRowsBN && (glu || wnk || lora)) return cudaErrorInvalidValue;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), slot);
    if (e != cudaSuccess) return e;
    const size_t smem =
        rows_smem_bytes(a.xrows, a.stages, split ? a.splits : 0, a.MP, split && a.red_overlay, glu, bn);
    e = launch_ex(kern, a.grid, smem, split ? a.splits : 1, s, false, tmX, tmW, tmG, tmT, tmB, y, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <typename Kern>
int max_active_clusters(Kern kern, int slot, int splits, size_t smem) {
    if (ensure_smem_attr(reinterpret_cast<const void*>(kern), slot) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(splits);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = splits;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return 0;
    return n;
}

int rows_pair_max_active_clusters() {
    return max_active_clusters(rows_ta_kernel<false, false, false, false, true>, 20, 2, kTaSmem);
}

int rows_max_active_clusters(bool fused, int splits, size_t smem, bool glu, bool wnk, bool lora, int bn) {
    if (bn == kRowsBN / 2)
        return fused ? max_active_clusters(rows_kernel<true, true, false, false, false, kRowsBN / 2>, 26, splits, smem)
                     : max_active_clusters(rows_kernel<false, true, false, false, false, kRowsBN / 2>, 27, splits, smem);
    if (lora) return max_active_clusters(rows_kernel<true, true, false, false, true>, 17, splits, smem);
    if (wnk)
        return glu ? max_active_clusters(rows_kernel<true, true, true, true, false>, 13, splits, smem)
                   : max_active_clusters(rows_kernel<true, true, false, true, false>, 11, splits, smem);
    if (glu) return max_active_clusters(rows_kernel<true, true, true, false, false>, 8, splits, smem);
    return fused ? max_active_clusters(rows_kernel<true, true, false, false, false>, 4, splits, smem)
                 : max_active_clusters(rows_kernel<false, true, false, false, false>, 5, splits, smem);
}

cudaError_t launch_rmsnorm(const void* X, const void* g, void* Xn, int M, int K, float eps,
                           cudaStream_t s) {
    rmsnorm_kernel<<<M, kNormThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(X),
                                             static_cast<const __nv_bfloat16*>(g),
                                             static_cast<__nv_bfloat16*>(Xn), K, eps);
    return cudaGetLastError();
}

cudaError_t launch_fold_gain(const void* g, const void* W, void* Wg, int64_t K, int64_t N, cudaStream_t s) {
    const int64_t total = K * (N / 8);
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorInvalidDevice;
    const int64_t want = (total + kNormThreads - 1) / kNormThreads;
    const int grid = static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(sms) * 8));
    fold_gain_kernel<<<grid > 0 ? grid : 1, kNormThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(g),
                                                                static_cast<const __nv_bfloat16*>(W),
                                                                static_cast<__nv_bfloat16*>(Wg), K, N);
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
