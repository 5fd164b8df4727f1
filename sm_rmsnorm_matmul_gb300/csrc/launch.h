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

// Small-M path: CTA tile 128 (columns of W) x MP (rows of X, padded to 16).
constexpr int kColsBN = 128;
constexpr int kColsMaxMP = 128;
constexpr int kColsMaxStages = 8;
constexpr int kColsMaxSplits = 16;

size_t rows_smem_bytes();
size_t cols_smem_bytes(int MP, int stages);
size_t cols_fixed_smem_bytes();
size_t cols_stage_bytes(int MP);

struct RowsLaunch {
    int M, N, K;
    float eps;
    int m_tiles, n_tiles, k_blocks;
    int grid;
};

struct ColsLaunch {
    int M, N, K;
    float eps;
    int MP, n_tiles, k_blocks, splits, kb_per_split, stages, grid;
    uint32_t tmem_cols;
    float* ws_acc;    // [splits][M][N] fp32 partials (splits > 1 only)
    float* ws_ss;     // [n_tiles][splits][128] fp32 partial sums of squares
    int* counters;    // [n_tiles] arrival counters, zero between launches
};

cudaError_t launch_rows(bool fused, const CUtensorMap& tmX, const CUtensorMap& tmW,
                        const CUtensorMap& tmG, void* Y, const RowsLaunch& a, cudaStream_t s);
cudaError_t launch_cols(bool fused, const CUtensorMap& tmX, const CUtensorMap& tmW,
                        const CUtensorMap& tmG, void* Y, const ColsLaunch& a, cudaStream_t s);
cudaError_t launch_rmsnorm(const void* X, const void* g, void* Xn, int M, int K, float eps,
                           cudaStream_t s);

// Copies the in-kernel status word to *out and clears it (synchronous).
cudaError_t read_and_clear_status(int* out);

}  // namespace rmm
