// launch.h -- internal interface between the host API (api.cu) and the
// kernels (kernels.cu).  Not part of the public C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime_api.h>
#include <stddef.h>
#include <stdint.h>

namespace rmm {

constexpr int kBK = 64;          // K extent of one pipeline stage (128 B of bf16)

// Row-tile path: CTA tile 128 (rows of X) x 256 (columns of W).
constexpr int kRowsBM = 128;
constexpr int kRowsBN = 256;
constexpr int kRowsMaxStages = 12;

constexpr int kClusterMaxSplits = 8;   // portable cluster size

// 256-row path (the plain form over many row tiles): CTA tile 256 x 256, two
// M = 128 halves sharing each W stage, in three pipeline stages.
constexpr int kTtBM = 2 * kRowsBM;
constexpr int kTtStages = 3;

// Row-tile path shared memory: xrows = rows of X loaded per stage (128, or
// M rounded up to 16 for a single row tile); red_slots = K splits reduced
// through a cluster (0 without); MP = M rounded up to 16; overlay: the
// splits' receive blocks reuse the pipeline buffers instead of an area of
// their own.
// glu: the gated form (reduction units of two chunks).  bn: columns of a
// tile, kRowsBN or kRowsBN / 2 (the plain [K, N] form with a K split).
size_t rows_smem_bytes(int xrows, int stages, int red_slots, int MP, bool overlay = false,
                       bool glu = false, int bn = kRowsBN);
// The receive blocks of a K split over `splits` CTAs fit the pipeline buffers.
bool rows_overlay_fits(int xrows, int stages, int splits, int MP, bool glu = false, int bn = kRowsBN);
size_t rows_stage_bytes(int xrows, int bn = kRowsBN);
int rows_max_active_clusters(bool fused, int splits, size_t smem, bool glu = false, bool wnk = false,
                             bool lora = false, int bn = kRowsBN);
// Clusters of two CTAs of the paired fused kernel that fit on the device at once.
int rows_pair_max_active_clusters();
struct RowsLaunch {
    int M, N, K;
    float eps;
    int m_tiles, n_tiles, k_blocks;
    int splits, kb_per_split;  // K split of each tile (splits > 1 needs m_tiles == 1
                               // and one (tile, split) unit per CTA)
    int red_overlay;           // 1: the splits' receive blocks reuse the pipeline buffers
    int glu;                   // 1: gated form: W [K, N = 2F] holds gate then up columns,
                               // Y [M, F] = silu(gate) * up; output tiles of 128 columns
    int w_nk;                  // 1: W stored [N, K] (K contiguous), read K-major
    int unscaled;              // 1: no division by the row RMS (Y = (X*g) @ W)
    int hilo;                  // 1 (with unscaled, N <= 64): each output v is written as the
                               // bf16 pair hi = bf16(v), lo = bf16(v - hi), Y [M, 128] with
                               // hi in columns [0, 64) and lo in [64, 128) (zeros past N)
    int lora;                  // 1: two more stages per tile, the adapter's T (hi, then lo
                               // columns of a hilo output) times B
    int wait_limit_us;         // limit of one bounded in-kernel wait
    int test_skip_sends;       // test hook: the K-split reduction skips its stores
    int cluster;               // 1: the splits of a tile form a cluster
    int bn;                    // columns of a tile of the row-tile kernel: kRowsBN (or 0), or
                               // kRowsBN / 2 (plain [K, N] form with a K split)
    int xrows, MP, stages;
    int grid;
    int tall;                  // 1: the 256-row kernel (plain form; m_tiles then counts 256-row tiles)
    int fold;                  // 1 (with tall): W holds the gain folded in (W' = diag(g) W); the kernel
                               // forms the row sums of squares and scales Y by 1/rms
    int pair;                  // 1: fused kernel for several row tiles, CTAs in clusters of two that
                               // take the two row blocks of each unit and share its W stages
                               // (tiles and tail tiles then count units of two row blocks)
    const CUtensorMap* tmY;    // Y in boxes of [128 rows][32 columns], 64-byte swizzle
                               // (used by the fused kernel for several row tiles)
    // Fused kernel for several row tiles, and the 256-row kernel: the last tail_tiles tiles (those a
    // whole wave of CTAs would leave mostly idle) are cut along K into
    // tail_pieces pieces of tail_kbp k-blocks, one per CTA, and reduced
    // through global memory.  0 tail tiles: every tile is whole.
    int tail_tiles, tail_pieces, tail_kbp;
    float* ws_acc;             // [tail_tiles][tail_pieces][128][256] fp32 partials
    float* ws_ss;              // [tail_tiles][tail_pieces][128] partial row sums of squares
    int* ws_count;             // [tail_tiles][2] arrival counters, zero between launches
};

// tmT, tmB: the low-rank adapter's T [M, R] and B [R, N] (used with a.lora).
cudaError_t launch_rows(bool fused, const CUtensorMap& tmX, const CUtensorMap& tmW,
                        const CUtensorMap& tmG, const CUtensorMap& tmT, const CUtensorMap& tmB, void* Y,
                        const RowsLaunch& a, cudaStream_t s);
cudaError_t launch_rmsnorm(const void* X, const void* g, void* Xn, int M, int K, float eps,
                           cudaStream_t s);
// W'[k, n] = bf16(g[k] * W[k, n]) for W, W' [K, N] (N a multiple of 8).
cudaError_t launch_fold_gain(const void* g, const void* W, void* Wg, int64_t K, int64_t N, cudaStream_t s);

// Copies the in-kernel status word to *out and clears it (synchronous).
cudaError_t read_and_clear_status(int* out);

// ------------------------------------------------ small-M path (gemv.cu)
constexpr int kGvMaxM = 16;      // rows of X: one m16 tile of mma.sync.m16n8k16
constexpr int kGvBN = 64;        // columns of W per unit
constexpr int kGvBK = 16;        // k per MMA step
constexpr int kGvStageK = 128;   // k per pipeline stage (one MMA step per consumer warp)
constexpr int kGvPieceFloats = kGvMaxM * kGvBN + kGvMaxM;   // one published piece: tile, then row sums

struct GemvLaunch {
    int M, N, K;
    float eps;
    int units;              // ceil(N / 64)
    int kstages;            // ceil(K / 128)
    int splits;             // K pieces per unit, one CTA each (grid = units * splits)
    int stages_per_piece;   // stages of a piece (the last may have fewer)
    float* ws;              // [units][splits][16 * 64 + 16] fp32 partials (splits > 1)
    int* counters;          // [units] arrival counters, zero between launches (splits > 1)
    int wait_limit_us;      // limit of one bounded in-kernel wait
};
// tmX: X [M, K] in boxes of [16 rows][64 k]; tmW: W [K, N] in boxes of
// [64 k][64 n]; tmG: g [K] in boxes of 64 (fused only); 128-byte swizzle.
cudaError_t launch_gemv(bool fused, const CUtensorMap& tmX, const CUtensorMap& tmW, const CUtensorMap& tmG,
                        void* Y, const GemvLaunch& a, cudaStream_t s);
// CTAs of the small-M kernel that fit on one SM.
int gemv_ctas_per_sm(bool fused);
// The small-M kernel's own status word (as read_and_clear_status).
cudaError_t gemv_read_and_clear_status(int* out);

// ------------------------------------------------ QK-normalised attention (attention.cu)
constexpr int kAttBM = 128;   // query rows per tile
constexpr int kAttBN = 128;   // keys per tile

struct AttnLaunch {
    int S;            // sequence length (queries and keys)
    int D;            // head dimension, 64 or 128
    int Hq, group;    // query heads; query heads per key/value head
    int n_qb;         // blocks of 256 query rows per sequence, ceil(S / 256)
    int n_hb;         // Hq * B
    int causal;
    int n_blocks;     // n_qb * n_hb
    int grid;         // persistent CTAs, min(n_blocks, SMs)
    float eps;
    float qscale;     // scale * log2(e), applied with each query row's 1/RMS to its scores
    int wait_limit_us;
    void* O;          // output [B, S, Hq, D], row stride ldo elements
    long long ldo;
    int test_skip_loads;   // test hook: the producer leaves out its first K/V stage
    const void* gq;   // the query and key gains [D] (bf16): they bound the scores
    const void* gk;
};

// Y[t,h,:] = RMSNorm(X[t,h,:]; g, eps) * g2 for T rows of H heads of D
// (8..256); g2 may be nullptr (no second gain).
cudaError_t launch_rmsnorm_heads(const void* X, int64_t ldx, const void* g, const void* g2, void* Y,
                                 int64_t ldy, int64_t T, int H, int D, float eps, cudaStream_t s);
// tmQ, tmK (normalised keys times gq), tmV: 3-D maps [B][S][heads*128] read
// in boxes of [128 rows][64] (V: [64][64]).
cudaError_t launch_qknorm_attention(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                    const CUtensorMap& tmV, const AttnLaunch& a, cudaStream_t s);
size_t attn_smem_bytes(int D);
// The attention translation unit's own status word (as read_and_clear_status).
cudaError_t attn_read_and_clear_status(int* out);


}  // namespace rmm
