// api.cu -- the C ABI declared in include/rmsnorm_matmul.h: argument
// validation, the shape dispatcher, TMA tensor-map encoding, the per-(device,
// stream) split-K workspace, and launches.  Every step of the computation
// runs in the kernels of kernels.cu; nothing here touches tensor data.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <vector>
#include <tuple>
#include <mutex>
#include <utility>

#include "launch.h"
#include "qknorm_attention.h"
#include "rmsnorm_matmul.h"

namespace {

using rmm::kBK;

std::atomic<int> g_force_path{0};
// Test hooks (rmm_test_hooks): the limit of one bounded in-kernel wait and
// whether the K-split reduction skips its stores; passed in every launch.
constexpr int64_t kDefaultWaitUs = 2000000;
std::atomic<int> g_wait_limit_us{static_cast<int>(kDefaultWaitUs)};
std::atomic<int> g_skip_sends{0};

constexpr int kPathRows = 1;
constexpr int kPathSmallM = 2;

// ------------------------------------------------------------------ device
struct DeviceInfo {
    bool known = false;
    bool supported = false;
    int sm_count = 0;
    int smem_optin = 0;
};

std::mutex g_dev_mu;
std::map<int, DeviceInfo> g_dev;

int current_device(int* dev, DeviceInfo* info) {
    if (cudaGetDevice(dev) != cudaSuccess) return RMM_ERR_LAUNCH;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[*dev];
    if (!d.known) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, *dev) !=
                cudaSuccess)
            return RMM_ERR_LAUNCH;
        d.supported = (major == 10 && minor == 3);
        d.known = true;
    }
    *info = d;
    return d.supported ? RMM_OK : RMM_ERR_UNSUPPORTED_DEVICE;
}

// ------------------------------------------------------------- tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Row-major bf16 matrix [rows, cols] read in boxes of [box_rows, 64 columns]
// with the 128-byte swizzle; out-of-range elements read as zero.
bool map_2d(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major bf16 matrix [rows, cols] written in boxes of [128 rows, 32
// columns] from shared memory with the 64-byte swizzle; writes outside the
// matrix are dropped.
bool map_2d_store(CUtensorMap* m, void* ptr, uint64_t rows, uint64_t cols) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {32, static_cast<cuuint32_t>(rmm::kRowsBM)};
    const cuuint32_t estr[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 vector [n] read in boxes of 64 elements.
bool map_1d(CUtensorMap* m, const void* ptr, uint64_t n) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    const cuuint64_t dims[1] = {n};
    const cuuint64_t strides[1] = {n * 2};  // not read for rank 1
    const cuuint32_t box[1] = {64};
    const cuuint32_t estr[1] = {1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 1, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 tensor [B][S][width] with row stride ld (elements) and sequence
// stride S * ld, read or written in boxes of [box_rows][64] with the
// 128-byte swizzle; outside the tensor loads read zero and stores are dropped.
bool map_3d(CUtensorMap* m, const void* ptr, uint64_t B, uint64_t S, uint64_t width, uint64_t ld,
            uint32_t box_rows) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    const cuuint64_t dims[3] = {width, S, B};
    const cuuint64_t strides[2] = {ld * 2, S * ld * 2};
    const cuuint32_t box[3] = {64, box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// -------------------------------------------------------------- validation
bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const auto pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + nb && pb < pa + na;
}
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kNoop = -1;

// Shared checks for (M, K, N) and eps.  Returns kNoop for an empty output.
int check_sizes(int64_t M, int64_t K, int64_t N, float eps, bool has_eps) {
    if (M < 0 || N < 0 || K < 1) return RMM_ERR_INVALID_ARG;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return RMM_ERR_INVALID_ARG;
    if (has_eps && (!std::isfinite(eps) || eps < 0.f)) return RMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return kNoop;
    if (K % 8 != 0 || N % 8 != 0) return RMM_ERR_ALIGNMENT;
    return RMM_OK;
}

int check_ptrs(const void* out, size_t out_bytes, std::initializer_list<std::pair<const void*, size_t>> ins) {
    if (!out) return RMM_ERR_INVALID_ARG;
    for (auto& in : ins)
        if (!in.first) return RMM_ERR_INVALID_ARG;
    if (!aligned16(out)) return RMM_ERR_ALIGNMENT;
    for (auto& in : ins)
        if (!aligned16(in.first)) return RMM_ERR_ALIGNMENT;
    for (auto& in : ins)
        if (overlaps(out, out_bytes, in.first, in.second)) return RMM_ERR_INVALID_ARG;
    return RMM_OK;
}

// --------------------------------------------------------------- workspace
struct Workspace {
    float* acc = nullptr;
    size_t acc_bytes = 0;
    float* ss = nullptr;
    size_t ss_bytes = 0;
    int* counters = nullptr;
    size_t n_counters = 0;
    void* lora_t = nullptr;   // the low-rank adapter's T = (X*g) @ A as bf16 hi | lo, [M, 128]
    size_t lora_t_bytes = 0;
    void* khat = nullptr;     // normalised keys of qknorm_attention, [B, S, Hkv, D]
    size_t khat_bytes = 0;
};

std::mutex g_ws_mu;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;

size_t round_up_pow2(size_t v) {
    size_t p = 1 << 20;
    while (p < v) p <<= 1;
    return p;
}

// Returns the split-K workspace of (dev, stream), grown to at least the given
// sizes.  Growing synchronises the stream and is refused during capture.
int get_workspace(int dev, cudaStream_t s, size_t acc_bytes, size_t ss_bytes, size_t ncount,
                  Workspace* out) {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    Workspace& w = g_ws[{dev, s}];
    if (w.acc_bytes >= acc_bytes && w.ss_bytes >= ss_bytes && w.n_counters >= ncount) {
        *out = w;
        return RMM_OK;
    }
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
        return RMM_ERR_INTERNAL;  // first use of a shape must happen outside capture
    if (cudaStreamSynchronize(s) != cudaSuccess) return RMM_ERR_LAUNCH;
    Workspace n;
    n.acc_bytes = round_up_pow2(std::max(acc_bytes, w.acc_bytes));
    n.ss_bytes = round_up_pow2(std::max(ss_bytes, w.ss_bytes));
    n.n_counters = std::max<size_t>(std::max(ncount, w.n_counters), 4096);
    if (cudaMalloc(&n.acc, n.acc_bytes) != cudaSuccess) return RMM_ERR_INTERNAL;
    if (cudaMalloc(&n.ss, n.ss_bytes) != cudaSuccess) {
        cudaFree(n.acc);
        return RMM_ERR_INTERNAL;
    }
    if (cudaMalloc(&n.counters, n.n_counters * sizeof(int)) != cudaSuccess) {
        cudaFree(n.acc);
        cudaFree(n.ss);
        return RMM_ERR_INTERNAL;
    }
    if (cudaMemsetAsync(n.counters, 0, n.n_counters * sizeof(int), s) != cudaSuccess)
        return RMM_ERR_LAUNCH;
    if (w.acc) cudaFree(w.acc);
    if (w.ss) cudaFree(w.ss);
    if (w.counters) cudaFree(w.counters);
    // the adapter's T and the normalised keys keep their own buffers
    w.acc = n.acc;
    w.acc_bytes = n.acc_bytes;
    w.ss = n.ss;
    w.ss_bytes = n.ss_bytes;
    w.counters = n.counters;
    w.n_counters = n.n_counters;
    *out = w;
    return RMM_OK;
}

// Zeroes the arrival counters of every workspace of the current device, after
// a kernel that gave up may have left some of them set.  Synchronous.
cudaError_t clear_workspace_counters() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_ws_mu);
    for (auto& kv : g_ws) {
        if (kv.first.first != dev || !kv.second.counters) continue;
        e = cudaMemset(kv.second.counters, 0, kv.second.n_counters * sizeof(int));
        if (e != cudaSuccess) return e;
    }
    return cudaDeviceSynchronize();
}

// The T buffer of (dev, stream) for the low-rank adapter, grown to `bytes`.
// Growing synchronises the stream and is refused during capture.
int get_lora_buffer(int dev, cudaStream_t s, size_t bytes, void** out) {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    Workspace& w = g_ws[{dev, s}];
    if (w.lora_t_bytes < bytes) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
            return RMM_ERR_INTERNAL;
        if (cudaStreamSynchronize(s) != cudaSuccess) return RMM_ERR_LAUNCH;
        void* p = nullptr;
        const size_t n = round_up_pow2(bytes);
        if (cudaMalloc(&p, n) != cudaSuccess) return RMM_ERR_INTERNAL;
        if (w.lora_t) cudaFree(w.lora_t);
        w.lora_t = p;
        w.lora_t_bytes = n;
    }
    *out = w.lora_t;
    return RMM_OK;
}

int get_khat_buffer(int dev, cudaStream_t s, size_t bytes, void** out) {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    Workspace& w = g_ws[{dev, s}];
    if (w.khat_bytes < bytes) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
            return RMM_ERR_INTERNAL;
        if (cudaStreamSynchronize(s) != cudaSuccess) return RMM_ERR_LAUNCH;
        void* p = nullptr;
        const size_t n = round_up_pow2(bytes);
        if (cudaMalloc(&p, n) != cudaSuccess) return RMM_ERR_INTERNAL;
        if (w.khat) cudaFree(w.khat);
        w.khat = p;
        w.khat_bytes = n;
    }
    *out = w.khat;
    return RMM_OK;
}

// ---------------------------------------------------------------- planning
// Small-M path (gemv.cu): units of 64 columns, K cut into `splits` pieces of
// stages_per_piece 128-deep stages, one CTA per piece.
struct GemvPlan {
    int units, kstages, splits, stages_per_piece;
};

std::mutex g_gv_mu;
std::map<std::pair<int, bool>, int> g_gv_occ;

int gemv_slots_per_sm(int dev, bool fused) {
    std::lock_guard<std::mutex> lk(g_gv_mu);
    auto key = std::make_pair(dev, fused);
    auto it = g_gv_occ.find(key);
    if (it != g_gv_occ.end()) return it->second;
    const int n = std::max(1, rmm::gemv_ctas_per_sm(fused));
    g_gv_occ[key] = n;
    return n;
}

// K split of the small-M path: the pieces of one launch run as waves of
// (SMs x CTAs per SM); a piece of P stages costs its CTA time in proportion
// to P, and a split adds the publication of the pieces and the last CTA's sum
// over them, about two stages' time plus one per batch of 8 pieces.
GemvPlan plan_gemv(int dev, bool fused, int64_t K, int64_t N, const DeviceInfo& d) {
    GemvPlan p{};
    p.units = static_cast<int>((N + rmm::kGvBN - 1) / rmm::kGvBN);
    p.kstages = static_cast<int>((K + rmm::kGvStageK - 1) / rmm::kGvStageK);
    const long slots = static_cast<long>(d.sm_count > 0 ? d.sm_count : 1) * gemv_slots_per_sm(dev, fused);
    p.splits = 1;
    p.stages_per_piece = p.kstages;
    long best = -1;
    for (int s = 1; s <= 32 && s <= p.kstages; ++s) {
        const int spp = (p.kstages + s - 1) / s;
        if ((p.kstages + spp - 1) / spp != s) continue;
        const long waves = (static_cast<long>(p.units) * s + slots - 1) / slots;
        const long cost = 4 * waves * spp + (s > 1 ? 8 + 4 * ((s + 7) / 8) : 0);   // quarter stages
        if (best < 0 || cost < best) {
            best = cost;
            p.splits = s;
            p.stages_per_piece = spp;
        }
    }
    return p;
}

struct RowsPlan {
    int m_tiles, n_tiles, k_blocks, splits, kb_per_split, cluster, xrows, MP, stages, grid;
    int overlay;
    int bn = rmm::kRowsBN;   // columns of a tile
};

int rows_stages(int xrows, int red_slots, int MP, const DeviceInfo& d, bool overlay = false,
                bool glu = false, int bn = rmm::kRowsBN) {
    const size_t fixed = rmm::rows_smem_bytes(xrows, 0, red_slots, MP, overlay, glu, bn);
    const size_t per = rmm::rows_stage_bytes(xrows, bn);
    const size_t avail = d.smem_optin > 0 ? static_cast<size_t>(d.smem_optin) : 227 * 1024;
    int st = avail > fixed ? static_cast<int>((avail - fixed) / per) : 0;
    st = std::min(rmm::kRowsMaxStages, st);
    // the X tiles are padded to 1 KB as a whole
    while (st > 0 && rmm::rows_smem_bytes(xrows, st, red_slots, MP, overlay, glu, bn) > avail) --st;
    return st;
}

std::mutex g_rows_occ_mu;
std::map<std::tuple<int, bool, int, size_t, bool, bool, bool, int>, int> g_rows_occ;

int rows_max_clusters(int dev, bool fused, int splits, size_t smem, bool glu, bool wnk, bool lora,
                      int bn = rmm::kRowsBN) {
    std::lock_guard<std::mutex> lk(g_rows_occ_mu);
    auto key = std::make_tuple(dev, fused, splits, smem, glu, wnk, lora, bn);
    auto it = g_rows_occ.find(key);
    if (it != g_rows_occ.end()) return it->second;
    const int n = rmm::rows_max_active_clusters(fused, splits, smem, glu, wnk, lora, bn);
    g_rows_occ[key] = n;
    return n;
}

// Row-tile path plan.  More than one row tile: no K split, 128-row X boxes.
// One row tile (M <= 128, the W-streaming regime): X boxes of M rounded up to
// 16 rows, and K split over 1..8 CTAs of a cluster chosen with a model of one
// launch in microseconds (fitted to GB300 measurements): each CTA streams W at
// about 55 GB/s, the GPU at about 6 TB/s, a unit costs about 1 us of fill and
// drain, and the cluster reduction about 1.5 us.  glu: the gated form, whose
// tiles cover 128 output columns (256 columns of W, N = 2F).
RowsPlan plan_rows(int dev, bool fused, int64_t M, int64_t K, int64_t N, const DeviceInfo& d,
                   bool glu = false, bool wnk = false, bool lora = false) {
    RowsPlan p{};
    p.m_tiles = static_cast<int>((M + rmm::kRowsBM - 1) / rmm::kRowsBM);
    p.n_tiles = glu ? static_cast<int>((N / 2 + rmm::kRowsBN / 2 - 1) / (rmm::kRowsBN / 2))
                    : static_cast<int>((N + rmm::kRowsBN - 1) / rmm::kRowsBN);
    p.k_blocks = static_cast<int>((K + kBK - 1) / kBK);
    p.MP = static_cast<int>(std::min<int64_t>(rmm::kRowsBM, ((M + 15) / 16) * 16));
    const int sms = d.sm_count > 0 ? d.sm_count : 1;
    p.splits = 1;
    p.kb_per_split = p.k_blocks;
    p.cluster = 0;
    if (p.m_tiles > 1) {
        p.xrows = rmm::kRowsBM;
        p.stages = rows_stages(p.xrows, 0, p.MP, d);
        p.grid = static_cast<int>(std::min<long>(static_cast<long>(p.m_tiles) * p.n_tiles, sms));
        return p;
    }
    p.xrows = p.MP;
    double best = 1e300;
    const double w_total = static_cast<double>(K) * N * 2;
    // Tiles of 256 columns, or (plain [K, N] form, K split, at most 32 rows)
    // of 128: twice the CTAs for a K split, and half the partial sums each
    // CTA exchanges; with more rows the X tile, loaded again for every W
    // stage, would grow to the size of the stage's W.  (Measured: 8 x 1024 x
    // 1024 5.30 -> 4.72 us; 16 x 4096 x 6144 keeps 256 columns, as three
    // splits of 48 tiles do not fit as clusters, and two splits took 17.3 us
    // against 11.7: a CTA streams W at ~55-60 GB/s whatever its stage count.)
    for (int bn : {rmm::kRowsBN, rmm::kRowsBN / 2}) {
    const bool narrow = bn != rmm::kRowsBN;
    if (narrow && (glu || wnk || lora || p.MP > 32)) continue;
    const int n_tiles = glu ? static_cast<int>((N / 2 + bn / 2 - 1) / (bn / 2)) : static_cast<int>((N + bn - 1) / bn);
    for (int s = narrow ? 2 : 1; s <= rmm::kClusterMaxSplits && s <= p.k_blocks; ++s) {
        const int kbps = (p.k_blocks + s - 1) / s;
        if ((p.k_blocks + kbps - 1) / kbps != s) continue;
        const int red_slots = s > 1 ? s : 0;
        int st = rows_stages(p.xrows, red_slots, p.MP, d, false, glu, bn);
        // A receive area of its own that leaves fewer than 3 stages: put the
        // receive blocks over the pipeline buffers instead.  The extra
        // handshake measured ~0.5 us, more than going from 3 to 5 stages
        // bought (M = 64), less than going from 2 stages or none (M > 64).
        bool overlay = false;
        if (s > 1 && st < 3) {
            const int so = rows_stages(p.xrows, red_slots, p.MP, d, true, glu, bn);
            if (so > st && so >= 2 && rmm::rows_overlay_fits(p.xrows, so, s, p.MP, glu, bn)) {
                st = so;
                overlay = true;
            }
        }
        if (st < 2) continue;
        int resident = sms;
        if (s > 1) {
            resident = rows_max_clusters(dev, fused, s,
                                         rmm::rows_smem_bytes(p.xrows, st, red_slots, p.MP, overlay, glu, bn),
                                         glu, wnk, lora, bn) * s;
            if (resident <= 0) continue;
        }
        const long units = static_cast<long>(n_tiles) * s;
        // a K split runs one (tile, split) unit per CTA, all resident at once
        if (s > 1 && units > resident) continue;
        const long waves = (units + resident - 1) / resident;
        const double per_cta = static_cast<double>(waves) * kbps * bn * kBK * 2 / 55e9;
        // the reduction: ~0.5 us, plus ~1 us for the exchange of a 256-column
        // tile's partial sums (proportional to the tile's columns)
        const double red = s > 1 ? 0.5 + 1.0 * bn / rmm::kRowsBN : 0.5;
        const double cost = std::max(per_cta, w_total / 6.0e12) * 1e6 + waves * 1.0 + red + (overlay ? 0.7 : 0.0);
        if (cost < best - 1e-9) {
            best = cost;
            p.splits = s;
            p.kb_per_split = kbps;
            p.cluster = s > 1 ? 1 : 0;
            p.stages = st;
            p.overlay = overlay ? 1 : 0;
            p.bn = bn;
            p.n_tiles = n_tiles;
            p.grid = static_cast<int>(std::min<long>(units, resident));
        }
    }
    }
    if (p.cluster) p.grid = (p.grid / p.splits) * p.splits;
    return p;
}

// K split of the last units of the fused kernel for several row tiles.  A
// unit is one tile, or (paired) the two row blocks of one column tile, taken
// by one CTA slot (a CTA or a cluster of two).  When the units leave a last
// wave at most half full, those units are cut along K so that every slot has
// a share of them.  When all the units fill at most half the slots (one
// partial wave, e.g. a contraction with a narrow N such as the adapter's T),
// every unit is cut, one piece per slot, up to one slot per SM or pair of SMs.
// The pieces of a tile wait for one another, so the launch is cooperative.
struct TailPlan {
    int tiles = 0;    // tail units (0: every unit whole)
    int pieces = 1;   // K pieces per tail unit
    int kbp = 0;      // k-blocks per piece
    int grid = 0;     // slots of the launch
};
TailPlan plan_tail(int units, int grid, int k_blocks, int slots) {
    TailPlan t;
    t.grid = grid;
    const bool few = units <= grid && 2 * units <= slots;
    const int g = few ? slots : grid;
    const int rem = units % g;
    if (!((units > g || few) && rem > 0 && 2 * rem <= g && k_blocks >= 2)) return t;
    const int pmax = g / rem;
    const int kbp = (k_blocks + pmax - 1) / pmax;
    const int pieces = (k_blocks + kbp - 1) / kbp;
    if (pieces < 2) return t;
    t.tiles = rem;
    t.pieces = pieces;
    t.kbp = kbp;
    if (few) t.grid = units * pieces;   // every unit cut: one slot per piece
    return t;
}

std::mutex g_pair_mu;
std::map<int, int> g_pair_occ;

// Clusters of two of the paired fused kernel resident at once on `dev`.
int pair_clusters(int dev) {
    std::lock_guard<std::mutex> lk(g_pair_mu);
    auto it = g_pair_occ.find(dev);
    if (it != g_pair_occ.end()) return it->second;
    const int n = rmm::rows_pair_max_active_clusters();
    g_pair_occ[dev] = n;
    return n;
}

// Launch shape of the fused kernel for several row tiles: its units, the K
// split of its last units, and whether it runs paired (clusters of two CTAs,
// one pair MMA per 256-row unit, for the plain form).  The paired kernel
// never cuts units along K: a launch that is both a cluster launch and
// cooperative is not used (two such launches faulted the GPU when replayed
// under the profiler, though none did otherwise).  It is chosen where clusters
// of two can be resident and either its units need no K-split tail or at
// most a fifth of its cluster-rounds would sit idle in the last round (on
// GB300 a paired round is ~7% shorter than the 128-row kernel's wave, and the
// K-split tail costs more than that: 4096 x 4096 x 6144, six paired rounds
// of which the last is 5% busy, 158 us against 163 us with the tail cut).
struct TaPlan {
    bool pair;
    int kc;        // CTAs per slot
    int units;     // units of kc row blocks x one column tile
    TailPlan tail;
    int ctas;      // grid size
};
TaPlan plan_ta(int dev, const RowsPlan& p, const DeviceInfo& d, bool plain) {
    const int sms = d.sm_count > 0 ? d.sm_count : 1;
    const int clusters = plain ? pair_clusters(dev) : 0;
    TaPlan t{};
    if (clusters > 0) {
        t.pair = true;
        t.kc = 2;
        t.units = ((p.m_tiles + 1) / 2) * p.n_tiles;
        t.tail = plan_tail(t.units, std::min(t.units, clusters), p.k_blocks, clusters);
        const int rounds = (t.units + clusters - 1) / clusters;
        if (t.tail.tiles == 0 || 5 * t.units >= 4 * rounds * clusters) {
            t.tail = TailPlan{};
            t.tail.grid = std::min(t.units, clusters);
            t.ctas = t.tail.grid * 2;
            return t;
        }
    }
    t.pair = false;
    t.kc = 1;
    t.units = p.m_tiles * p.n_tiles;
    t.tail = plan_tail(t.units, std::min(t.units, sms), p.k_blocks, sms);
    t.ctas = t.tail.grid;
    return t;
}

// The 256-row kernel (two M = 128 halves per CTA sharing each W stage) for
// the unfused contraction from two of its tiles (512 rows of X) up; shorter
// shapes keep the 128-row kernel.  (Fused, its in-place X*g holds each 64 KB
// stage through the transform, and the 128-row kernel with A in tensor
// memory measured faster: 166 against 201 us on 4096 x 4096 x 6144.)
bool use_tall(bool fused, int64_t M) { return !fused && M >= 2 * rmm::kTtBM; }

// Shape-based dispatch.  Up to 16 rows of X both kernels stream W; the
// row-tile kernel runs one CTA per (256-column tile, K split) with at most 8
// splits (a portable cluster), each CTA streaming about 55 GB/s, while the
// small-M kernel's 64-column units and unbounded K pieces reach the HBM rate
// (~6 TB/s) at a fixed cost about 1.5 us higher.  The model that picks the
// faster, fitted to eleven shapes timed on GB300 (cold L2, back-to-back calls;
// every one on the side it predicts): small-M for 16 x 8192 x 1024 (9.7 vs
// 12.4 us), 16 x 14336 x 2048 (14.4 vs 17.8), 4 x 2048 x 512 (5.5 vs 6.4);
// row-tile for 16 x 2048 x 2048 (6.7 vs 7.4), decode QKV 16 x 4096 x 6144
// (11.9 vs 12.5), 16 x 4096 x 28672 (37 vs 49).
int choose_path(int64_t M, int64_t K, int64_t N, int sms) {
    const int f = g_force_path.load();
    if (f == kPathRows || f == kPathSmallM) return f;
    if (M > rmm::kGvMaxM) return kPathRows;
    const double wbytes = 2.0 * static_cast<double>(K) * static_cast<double>(N);
    const int64_t tiles = (N + rmm::kRowsBN - 1) / rmm::kRowsBN;
    const int64_t ctas = std::min<int64_t>(std::max(1, sms),
                                           tiles * std::min<int64_t>(rmm::kClusterMaxSplits, (K + kBK - 1) / kBK));
    const double rows_us = wbytes / (static_cast<double>(ctas) * 55e9) * 1e6;
    const double small_us = wbytes / 6e12 * 1e6 + 1.5;
    return small_us < rows_us ? kPathSmallM : kPathRows;
}

// Device memory for K-split partials that the caller provides instead of the
// per-(device, stream) workspace: a fixed area with its capacities.  The plan
// is the one the workspace would get; a plan whose partials do not fit is
// refused with RMM_ERR_SCRATCH_LIMIT.  The arrival counters are cleared on the
// stream before each launch that uses them (the area keeps the previous
// call's contents).
struct FixedScratch {
    unsigned char* area;   // fp32 partial sums, then the partial row sums of squares
    size_t area_bytes;
    int* counters;
    size_t counter_bytes;
    // The partials of a plan (acc_bytes of sums, then ss_bytes) placed in
    // `area`; false if they do not fit.
    bool place(size_t acc_bytes, size_t ss_bytes, float** acc, float** ss) const {
        const size_t ss_off = (acc_bytes + 255) / 256 * 256;
        if (ss_off + ss_bytes > area_bytes) return false;
        *acc = reinterpret_cast<float*>(area);
        *ss = reinterpret_cast<float*>(area + ss_off);
        return true;
    }
};

// One launch of the tensor-core contraction, fused (RMSNorm folded in) or not.
// fixed: never allocate; K-split partials go to that area (RMM_ERR_SCRATCH_LIMIT
// if the plan's partials do not fit).
// glu: the gated form (fused only; always the row-tile path), Y [M, N / 2].
// wnk: W stored [N, K] (fused only; always the row-tile path).
// unscaled: no division by the row RMS; hilo (with unscaled, N <= 64): Y is
// [M, 128], each output written as the bf16 pair hi (columns [0, 64)) and lo
// (columns [64, 128)).  lora_t, lora_b: the low-rank adapter's T [M, 128] (a
// hilo output) and B [R, N], added as two more stages per tile (row-tile
// path).
int run_contraction(bool fused, const void* X, const void* g, const void* W, void* Y, int64_t M,
                    int64_t K, int64_t N, float eps, cudaStream_t stream, const FixedScratch* fixed = nullptr,
                    bool glu = false, bool wnk = false, bool unscaled = false,
                    const void* lora_t = nullptr, const void* lora_b = nullptr, int64_t R = 0,
                    bool hilo = false, bool fold = false) {
    // fold: W holds the gain folded in (fused must be false): the 256-row
    // kernel with the row statistic, for every shape
    const bool lora = lora_t != nullptr;
    int dev = 0;
    DeviceInfo d;
    int rc = current_device(&dev, &d);
    if (rc != RMM_OK) return rc;
    const int path =
        glu || wnk || lora || unscaled || fold ? static_cast<int>(kPathRows) : choose_path(M, K, N, d.sm_count);
    if (path == kPathSmallM) {
        if (M > rmm::kGvMaxM) return RMM_ERR_INVALID_ARG;
        const GemvPlan p = plan_gemv(dev, fused, K, N, d);
        CUtensorMap tmX, tmW, tmG;
        if (!map_2d(&tmX, X, M, K, rmm::kGvMaxM) || !map_2d(&tmW, W, K, N, kBK)) return RMM_ERR_INTERNAL;
        if (fused ? !map_1d(&tmG, g, K) : false) return RMM_ERR_INTERNAL;
        if (!fused) tmG = tmX;   // unused by the kernel
        rmm::GemvLaunch a{};
        a.M = static_cast<int>(M);
        a.N = static_cast<int>(N);
        a.K = static_cast<int>(K);
        a.eps = eps;
        a.units = p.units;
        a.kstages = p.kstages;
        a.splits = p.splits;
        a.stages_per_piece = p.stages_per_piece;
        a.wait_limit_us = g_wait_limit_us.load();
        if (p.splits > 1) {
            const size_t ws_bytes = static_cast<size_t>(p.units) * p.splits * rmm::kGvPieceFloats * sizeof(float);
            const size_t ncount = static_cast<size_t>(p.units);
            if (fixed) {
                float* unused = nullptr;
                if (!fixed->place(ws_bytes, 0, &a.ws, &unused) || ncount * sizeof(int) > fixed->counter_bytes)
                    return RMM_ERR_SCRATCH_LIMIT;
                if (cudaMemsetAsync(fixed->counters, 0, ncount * sizeof(int), stream) != cudaSuccess)
                    return RMM_ERR_LAUNCH;
                a.counters = fixed->counters;
            } else {
                Workspace w;
                rc = get_workspace(dev, stream, ws_bytes, 0, ncount, &w);
                if (rc != RMM_OK) return rc;
                a.ws = w.acc;
                a.counters = w.counters;
            }
        }
        return rmm::launch_gemv(fused, tmX, tmW, tmG, Y, a, stream) == cudaSuccess ? RMM_OK : RMM_ERR_LAUNCH;
    }
    CUtensorMap tmX, tmW, tmG;
    // [K, N]: boxes of [64 k][64 n]; [N, K]: boxes of [256 n][64 k], or 128 rows
    // each for the gate and up halves of the gated form
    if (!(wnk ? map_2d(&tmW, W, N, K, glu ? rmm::kRowsBN / 2 : rmm::kRowsBN) : map_2d(&tmW, W, K, N, kBK)))
        return RMM_ERR_INTERNAL;
    if (fused) {
        if (!map_1d(&tmG, g, K)) return RMM_ERR_INTERNAL;
    }
    const RowsPlan p = plan_rows(dev, fused, M, K, N, d, glu, wnk, lora);
    if (!map_2d(&tmX, X, M, K, fold ? rmm::kRowsBM : p.xrows)) return RMM_ERR_INTERNAL;
    if (!fused) tmG = tmX;
    rmm::RowsLaunch a{};
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.eps = eps;
    a.m_tiles = p.m_tiles;
    a.n_tiles = p.n_tiles;
    a.k_blocks = p.k_blocks;
    a.splits = p.splits;
    a.kb_per_split = p.kb_per_split;
    a.cluster = p.cluster;
    a.xrows = p.xrows;
    a.MP = p.MP;
    a.stages = p.stages;
    a.grid = p.grid;
    a.red_overlay = p.overlay;
    a.bn = p.bn;
    a.glu = glu ? 1 : 0;
    a.w_nk = wnk ? 1 : 0;
    a.unscaled = unscaled ? 1 : 0;
    a.hilo = hilo ? 1 : 0;
    a.lora = lora ? 1 : 0;
    a.wait_limit_us = g_wait_limit_us.load();
    a.test_skip_sends = g_skip_sends.load();
    CUtensorMap tmT = tmX, tmB = tmW;   // unused without the adapter
    if (lora) {
        if (!map_2d(&tmT, lora_t, M, 2 * kBK, p.xrows) || !map_2d(&tmB, lora_b, R, N, kBK))
            return RMM_ERR_INTERNAL;
    }
    CUtensorMap tmY;
    a.tail_tiles = 0;
    a.tail_pieces = 1;
    a.tail_kbp = p.k_blocks;
    const bool tall =
        fold || (!glu && !wnk && !lora && !unscaled && !p.cluster && p.xrows == rmm::kRowsBM && use_tall(fused, M));
    if (tall) {
        // tiles of 256 rows, the last ones cut along K as for the 128-row kernel
        if (!map_2d_store(&tmY, Y, M, N)) return RMM_ERR_INTERNAL;
        a.tmY = &tmY;
        a.tall = 1;
        a.fold = fold ? 1 : 0;
        a.m_tiles = static_cast<int>((M + rmm::kTtBM - 1) / rmm::kTtBM);
        a.n_tiles = static_cast<int>((N + rmm::kRowsBN - 1) / rmm::kRowsBN);
        a.bn = rmm::kRowsBN;
        a.splits = 1;
        a.cluster = 0;
        const int sms = d.sm_count > 0 ? d.sm_count : 1;
        const int units = a.m_tiles * a.n_tiles;
        const TailPlan t = plan_tail(units, std::min(units, sms), p.k_blocks, sms);
        a.grid = t.grid;
        if (t.tiles > 0 || fold) {
            constexpr size_t kPieceBytes = static_cast<size_t>(rmm::kTtBM) * rmm::kRowsBN * sizeof(float);
            const size_t pieces = static_cast<size_t>(t.tiles) * t.pieces;
            // the folded form: the pieces' partial row sums of squares, then each
            // row block's published r; counters: two per tail tile, then a flag
            // and a reader count per row block (unfused: pieces' counters only)
            const size_t rblocks = fold ? static_cast<size_t>(a.m_tiles) : 0;
            const size_t ss_bytes = fold ? (pieces + rblocks) * rmm::kTtBM * sizeof(float) : 0;
            const size_t ncount = static_cast<size_t>(t.tiles) * 2 + 2 * rblocks;
            if (fixed) {
                if (!fixed->place(pieces * kPieceBytes, ss_bytes, &a.ws_acc, &a.ws_ss) ||
                    ncount * sizeof(int) > fixed->counter_bytes)
                    return RMM_ERR_SCRATCH_LIMIT;
                if (cudaMemsetAsync(fixed->counters, 0, ncount * sizeof(int), stream) != cudaSuccess)
                    return RMM_ERR_LAUNCH;
                a.ws_count = fixed->counters;
            } else {
                Workspace w;
                rc = get_workspace(dev, stream, pieces * kPieceBytes, ss_bytes, ncount, &w);
                if (rc != RMM_OK) return rc;
                a.ws_acc = w.acc;
                a.ws_ss = w.ss;
                a.ws_count = w.counters;
            }
            if (t.tiles > 0) {
                a.tail_tiles = t.tiles;
                a.tail_pieces = t.pieces;
                a.tail_kbp = t.kbp;
            }
        }
    } else if (fused && !p.cluster && p.xrows == rmm::kRowsBM) {
        if (!map_2d_store(&tmY, Y, M, hilo ? 2 * kBK : glu ? N / 2 : N)) return RMM_ERR_INTERNAL;
        a.tmY = &tmY;
        const TaPlan tp = plan_ta(dev, p, d, !hilo);   // (paired: every form but T's hi/lo output)
        const TailPlan& t = tp.tail;
        a.pair = tp.pair ? 1 : 0;
        // paired, weights stored [N, K]: each CTA loads boxes of 128 weight rows
        if (tp.pair && wnk && !map_2d(&tmW, W, N, K, rmm::kRowsBN / 2)) return RMM_ERR_INTERNAL;
        a.grid = tp.ctas;
        if (t.tiles > 0) {
            const int rem = t.tiles * tp.kc, pieces = t.pieces;   // tail tiles
            {
                constexpr size_t kPieceBytes = static_cast<size_t>(rmm::kRowsBM) * rmm::kRowsBN * sizeof(float);
                const size_t units = static_cast<size_t>(rem) * pieces;
                if (fixed) {
                    if (!fixed->place(units * kPieceBytes, units * rmm::kRowsBM * sizeof(float), &a.ws_acc,
                                      &a.ws_ss) ||
                        static_cast<size_t>(rem) * 2 * sizeof(int) > fixed->counter_bytes)
                        return RMM_ERR_SCRATCH_LIMIT;
                    if (cudaMemsetAsync(fixed->counters, 0, static_cast<size_t>(rem) * 2 * sizeof(int), stream) !=
                        cudaSuccess)
                        return RMM_ERR_LAUNCH;
                    a.ws_count = fixed->counters;
                } else {
                    Workspace w;
                    rc = get_workspace(dev, stream, units * kPieceBytes, units * rmm::kRowsBM * sizeof(float),
                                       static_cast<size_t>(rem) * 2, &w);
                    if (rc != RMM_OK) return rc;
                    a.ws_acc = w.acc;
                    a.ws_ss = w.ss;
                    a.ws_count = w.counters;
                }
                a.tail_tiles = t.tiles;   // in units
                a.tail_pieces = pieces;
                a.tail_kbp = t.kbp;
            }
        }
    }
    return rmm::launch_rows(fused, tmX, tmW, tmG, tmT, tmB, Y, a, stream) == cudaSuccess ? RMM_OK
                                                                              : RMM_ERR_LAUNCH;
}

}  // namespace

extern "C" {

int rmsnorm_matmul(const void* X, const void* g, const void* W, void* Y, int64_t M, int64_t K,
                   int64_t N, float eps, cudaStream_t stream) {
    int rc = check_sizes(M, K, N, eps, true);
    if (rc == kNoop) return RMM_OK;
    if (rc != RMM_OK) return rc;
    rc = check_ptrs(Y, static_cast<size_t>(M) * N * 2,
                    {{X, static_cast<size_t>(M) * K * 2}, {g, static_cast<size_t>(K) * 2},
                     {W, static_cast<size_t>(K) * N * 2}});
    if (rc != RMM_OK) return rc;
    return run_contraction(true, X, g, W, Y, M, K, N, eps, stream);
}

int rmsnorm_matmul_ex(const void* X, const void* g, const void* W, void* Y, int64_t M, int64_t K,
                      int64_t N, float eps, unsigned flags, cudaStream_t stream) {
    if (flags & ~static_cast<unsigned>(RMM_WEIGHT_NK | RMM_GATED_SILU)) return RMM_ERR_INVALID_ARG;
    const bool glu = (flags & RMM_GATED_SILU) != 0, wnk = (flags & RMM_WEIGHT_NK) != 0;
    int rc = check_sizes(M, K, N, eps, true);
    if (rc == kNoop) return RMM_OK;
    if (rc != RMM_OK) return rc;
    if (glu && N % 16 != 0) return RMM_ERR_ALIGNMENT;   // F = N / 2 must be a multiple of 8
    const int64_t out_cols = glu ? N / 2 : N;
    rc = check_ptrs(Y, static_cast<size_t>(M) * out_cols * 2,
                    {{X, static_cast<size_t>(M) * K * 2}, {g, static_cast<size_t>(K) * 2},
                     {W, static_cast<size_t>(K) * N * 2}});
    if (rc != RMM_OK) return rc;
    return run_contraction(true, X, g, W, Y, M, K, N, eps, stream, nullptr, glu, wnk);
}

int rmsnorm_matmul_lora(const void* X, const void* g, const void* W, const void* A, const void* B,
                        void* Y, int64_t M, int64_t K, int64_t N, int64_t R, float eps,
                        cudaStream_t stream) {
    int rc = check_sizes(M, K, N, eps, true);
    if (rc == kNoop) return RMM_OK;
    if (rc != RMM_OK) return rc;
    if (R < 1 || R > kBK) return RMM_ERR_INVALID_ARG;
    if (R % 8 != 0) return RMM_ERR_ALIGNMENT;
    rc = check_ptrs(Y, static_cast<size_t>(M) * N * 2,
                    {{X, static_cast<size_t>(M) * K * 2}, {g, static_cast<size_t>(K) * 2},
                     {W, static_cast<size_t>(K) * N * 2}, {A, static_cast<size_t>(K) * R * 2},
                     {B, static_cast<size_t>(R) * N * 2}});
    if (rc != RMM_OK) return rc;
    int dev = 0;
    DeviceInfo d;
    rc = current_device(&dev, &d);
    if (rc != RMM_OK) return rc;
    void* T = nullptr;
    rc = get_lora_buffer(dev, stream, static_cast<size_t>(M) * 2 * kBK * 2, &T);
    if (rc != RMM_OK) return rc;
    // T = (X*g) @ A over the same gained, bf16-rounded rows the MMA sees,
    // without the division by the RMS (applied once, to the sum, below),
    // kept as the bf16 pair hi = bf16(T), lo = bf16(T - hi): [M, 128]
    rc = run_contraction(true, X, g, A, T, M, K, R, eps, stream, nullptr, false, false, true, nullptr, nullptr, 0,
                         true);
    if (rc != RMM_OK) return rc;
    return run_contraction(true, X, g, W, Y, M, K, N, eps, stream, nullptr, false, false, false, T, B, R);
}

int rmsnorm_matmul_swiglu(const void* X, const void* g, const void* W, void* Y, int64_t M,
                          int64_t K, int64_t N, float eps, cudaStream_t stream) {
    return rmsnorm_matmul_ex(X, g, W, Y, M, K, N, eps, RMM_GATED_SILU, stream);
}

int matmul(const void* A, const void* B, void* C, int64_t M, int64_t K, int64_t N,
           cudaStream_t stream) {
    int rc = check_sizes(M, K, N, 0.f, false);
    if (rc == kNoop) return RMM_OK;
    if (rc != RMM_OK) return rc;
    rc = check_ptrs(C, static_cast<size_t>(M) * N * 2,
                    {{A, static_cast<size_t>(M) * K * 2}, {B, static_cast<size_t>(K) * N * 2}});
    if (rc != RMM_OK) return rc;
    return run_contraction(false, A, nullptr, B, C, M, K, N, 0.f, stream);
}

}  // extern "C"

// A gain of ones, [K] bf16, per device: the folded form of a single row tile
// runs the fused row-tile kernels with it (X * 1 = X exactly).  Grown when a
// longer K arrives; an outgrown buffer is kept, since calls on other streams
// may still read it.  Returns nullptr if it has to grow during stream capture.
std::mutex g_ones_mu;
std::map<int, std::pair<void*, int64_t>> g_ones;

const void* ones_gain(int dev, int64_t K, cudaStream_t s) {
    std::lock_guard<std::mutex> lk(g_ones_mu);
    auto& e = g_ones[dev];
    if (e.first && e.second >= K) return e.first;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return nullptr;
    const int64_t n = std::max<int64_t>(round_up_pow2(static_cast<size_t>(K)), 4096);
    void* p = nullptr;
    if (cudaMalloc(&p, static_cast<size_t>(n) * 2) != cudaSuccess) return nullptr;
    std::vector<uint16_t> one(static_cast<size_t>(n), 0x3F80);   // bf16 1.0
    if (cudaMemcpy(p, one.data(), static_cast<size_t>(n) * 2, cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaFree(p);
        return nullptr;
    }
    e = {p, n};
    return p;
}

extern "C" {

int fold_gain(const void* g, const void* W, void* Wg, int64_t K, int64_t N, cudaStream_t stream) {
    if (K < 1 || N < 1 || K > (int64_t(1) << 31) || N > (int64_t(1) << 31) || N % 8 != 0)
        return RMM_ERR_INVALID_ARG;
    int rc = check_ptrs(Wg, static_cast<size_t>(K) * N * 2,
                        {{g, static_cast<size_t>(K) * 2}, {W, static_cast<size_t>(K) * N * 2}});
    if (rc != RMM_OK) return rc;
    return rmm::launch_fold_gain(g, W, Wg, K, N, stream) == cudaSuccess ? RMM_OK : RMM_ERR_LAUNCH;
}

int rmsnorm_matmul_folded(const void* X, const void* Wg, void* Y, int64_t M, int64_t K, int64_t N, float eps,
                          cudaStream_t stream) {
    int rc = check_sizes(M, K, N, eps, true);
    if (rc == kNoop) return RMM_OK;
    if (rc != RMM_OK) return rc;
    rc = check_ptrs(Y, static_cast<size_t>(M) * N * 2,
                    {{X, static_cast<size_t>(M) * K * 2}, {Wg, static_cast<size_t>(K) * N * 2}});
    if (rc != RMM_OK) return rc;
    if (M <= rmm::kRowsBM) {
        // one row tile: the fused row-tile (or small-M) kernel with a gain of ones
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return RMM_ERR_UNSUPPORTED_DEVICE;
        const void* ones = ones_gain(dev, K, stream);
        if (!ones) return RMM_ERR_INTERNAL;
        return run_contraction(true, X, ones, Wg, Y, M, K, N, eps, stream);
    }
    return run_contraction(false, X, nullptr, Wg, Y, M, K, N, eps, stream, nullptr, false, false, false, nullptr,
                           nullptr, 0, false, true);
}

int rmsnorm(const void* X, const void* g, void* Xn, int64_t M, int64_t K, float eps,
            cudaStream_t stream) {
    // N plays no part; pass K so that the N checks pass trivially.
    int rc = check_sizes(M, K, K, eps, true);
    if (rc == kNoop) return RMM_OK;
    if (rc != RMM_OK) return rc;
    rc = check_ptrs(Xn, static_cast<size_t>(M) * K * 2,
                    {{X, static_cast<size_t>(M) * K * 2}, {g, static_cast<size_t>(K) * 2}});
    if (rc != RMM_OK) return rc;
    int dev = 0;
    DeviceInfo d;
    rc = current_device(&dev, &d);
    if (rc != RMM_OK) return rc;
    return rmm::launch_rmsnorm(X, g, Xn, static_cast<int>(M), static_cast<int>(K), eps, stream) ==
                   cudaSuccess
               ? RMM_OK
               : RMM_ERR_LAUNCH;
}

int rmm_force_path(int path) {
    if (path < 0 || path > 2) return -1;
    return g_force_path.exchange(path);
}

int rmm_describe_plan(int64_t M, int64_t K, int64_t N, int fused, int* info) {
    if (!info || M < 1 || K < 1 || N < 1 || fused < 0 || fused > 2) return RMM_ERR_INVALID_ARG;
    const bool glu = fused == 2;
    int dev = 0;
    DeviceInfo d;
    int rc = current_device(&dev, &d);
    if (rc != RMM_OK) return rc;
    for (int i = 0; i < 8; ++i) info[i] = 0;
    info[0] = glu ? static_cast<int>(kPathRows) : choose_path(M, K, N, d.sm_count);
    if (info[0] == kPathSmallM) {
        if (M > rmm::kGvMaxM) return RMM_ERR_INVALID_ARG;
        const GemvPlan p = plan_gemv(dev, fused != 0, K, N, d);
        info[1] = p.splits;
        info[2] = 0;
        info[3] = p.units * p.splits;
        info[4] = 5;   // pipeline stages of 128 k
        info[5] = rmm::kGvMaxM;
        info[6] = p.units;
        info[7] = p.stages_per_piece * (rmm::kGvStageK / kBK);   // k-blocks of 64 per piece
    } else {
        const RowsPlan p = plan_rows(dev, fused != 0, M, K, N, d, glu);
        info[1] = p.splits;
        info[2] = p.cluster;
        info[3] = p.grid;
        info[4] = p.stages;
        info[5] = p.xrows;
        info[6] = p.m_tiles * p.n_tiles;
        info[7] = p.kb_per_split;
        if (fused != 2 && !p.cluster && p.xrows == rmm::kRowsBM && use_tall(fused != 0, M)) {
            // the 256-row kernel: its grid, stages, rows per tile, tiles and tail pieces
            const int sms = d.sm_count > 0 ? d.sm_count : 1;
            const int mt = static_cast<int>((M + rmm::kTtBM - 1) / rmm::kTtBM);
            const int units = mt * p.n_tiles;
            const TailPlan t = plan_tail(units, std::min(units, sms), p.k_blocks, sms);
            info[1] = t.tiles > 0 ? t.pieces : 1;
            info[3] = t.grid;
            info[4] = rmm::kTtStages;
            info[5] = rmm::kTtBM;
            info[6] = units;
            info[7] = t.tiles > 0 ? t.kbp : p.k_blocks;
        } else if (fused != 0 && !p.cluster && p.xrows == rmm::kRowsBM) {
            // the fused kernel for several row tiles: its grid and its tail tiles' K pieces
            const TaPlan tp = plan_ta(dev, p, d, true);
            info[3] = tp.ctas;
            if (tp.tail.tiles > 0) {
                info[1] = tp.tail.pieces;
                info[7] = tp.tail.kbp;
            }
        }
    }
    return RMM_OK;
}

int rmm_dispatch_path(int64_t M, int64_t K, int64_t N) {
    if (M < 1 || K < 1 || N < 1) return RMM_ERR_INVALID_ARG;
    int dev = 0;
    DeviceInfo d;
    // without a usable device, the dispatch of a 152-SM GB300
    const int sms = current_device(&dev, &d) == RMM_OK ? d.sm_count : 152;
    return choose_path(M, K, N, sms);
}

int rmm_device_status(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return RMM_ERR_LAUNCH;
    int v = 0, va = 0, vg = 0;
    if (rmm::read_and_clear_status(&v) != cudaSuccess) return RMM_ERR_LAUNCH;
    if (rmm::attn_read_and_clear_status(&va) != cudaSuccess) return RMM_ERR_LAUNCH;
    if (rmm::gemv_read_and_clear_status(&vg) != cudaSuccess) return RMM_ERR_LAUNCH;
    if (v == RMM_OK) v = va;
    if (v == RMM_OK) v = vg;
    if (v != RMM_OK && clear_workspace_counters() != cudaSuccess) return RMM_ERR_LAUNCH;
    return v;
}

int rmsnorm_heads(const void* X, int64_t ldx, const void* g, void* Y, int64_t ldy, int64_t T,
                  int64_t H, int64_t D, float eps, cudaStream_t stream) {
    if (T < 0 || H < 1 || D < 8 || D > 256 || D % 8 != 0) return RMM_ERR_INVALID_ARG;
    if (!std::isfinite(eps) || eps < 0.f) return RMM_ERR_INVALID_ARG;
    if (H > INT32_MAX / D || ldx < H * D || ldy < H * D) return RMM_ERR_INVALID_ARG;
    if (T == 0) return RMM_OK;
    if (ldx % 8 != 0 || ldy % 8 != 0) return RMM_ERR_ALIGNMENT;
    const size_t xb = static_cast<size_t>((T - 1) * ldx + H * D) * 2;
    const size_t yb = static_cast<size_t>((T - 1) * ldy + H * D) * 2;
    int rc = check_ptrs(Y, yb, {{X, xb}, {g, static_cast<size_t>(D) * 2}});
    if (rc != RMM_OK) return rc;
    int dev = 0;
    DeviceInfo d;
    rc = current_device(&dev, &d);
    if (rc != RMM_OK) return rc;
    return rmm::launch_rmsnorm_heads(X, ldx, g, nullptr, Y, ldy, T, static_cast<int>(H),
                                     static_cast<int>(D), eps, stream) == cudaSuccess
               ? RMM_OK
               : RMM_ERR_LAUNCH;
}

int qknorm_attention(const void* Q, int64_t ldq, const void* K, int64_t ldk, const void* V,
                     int64_t ldv, const void* gq, const void* gk, void* O, int64_t ldo, int64_t B,
                     int64_t S, int64_t Hq, int64_t Hkv, int64_t D, float eps, float scale,
                     int causal, cudaStream_t stream) {
    if (B < 0 || S < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return RMM_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return RMM_ERR_INVALID_ARG;
    if (!std::isfinite(eps) || eps < 0.f || !std::isfinite(scale)) return RMM_ERR_INVALID_ARG;
    if (Hq > 4096 || ldq < Hq * D || ldo < Hq * D || ldk < Hkv * D || ldv < Hkv * D)
        return RMM_ERR_INVALID_ARG;
    if (B == 0 || S == 0) return RMM_OK;
    if (S > INT32_MAX / 2 || B * Hq > INT32_MAX) return RMM_ERR_INVALID_ARG;
    const int64_t n_qb = (S + 2 * rmm::kAttBM - 1) / (2 * rmm::kAttBM);
    if (n_qb * B * Hq > INT32_MAX) return RMM_ERR_INVALID_ARG;
    if (ldq % 8 != 0 || ldk % 8 != 0 || ldv % 8 != 0 || ldo % 8 != 0) return RMM_ERR_ALIGNMENT;
    auto span = [&](int64_t ld, int64_t heads) {
        return static_cast<size_t>((B * S - 1) * ld + heads * D) * 2;
    };
    int rc = check_ptrs(O, span(ldo, Hq),
                        {{Q, span(ldq, Hq)}, {K, span(ldk, Hkv)}, {V, span(ldv, Hkv)},
                         {gq, static_cast<size_t>(D) * 2}, {gk, static_cast<size_t>(D) * 2}});
    if (rc != RMM_OK) return rc;
    int dev = 0;
    DeviceInfo d;
    rc = current_device(&dev, &d);
    if (rc != RMM_OK) return rc;
    if (static_cast<size_t>(d.smem_optin) < rmm::attn_smem_bytes(static_cast<int>(D)))
        return RMM_ERR_UNSUPPORTED_DEVICE;
    void* khat = nullptr;
    rc = get_khat_buffer(dev, stream, static_cast<size_t>(B * S * Hkv * D) * 2, &khat);
    if (rc != RMM_OK) return rc;
    CUtensorMap tmQ, tmK, tmV;
    if (!map_3d(&tmQ, Q, B, S, Hq * D, ldq, rmm::kAttBM) ||
        !map_3d(&tmK, khat, B, S, Hkv * D, Hkv * D, rmm::kAttBN) ||
        !map_3d(&tmV, V, B, S, Hkv * D, ldv, 64))
        return RMM_ERR_INTERNAL;
    // the keys once: RMSNorm(K; gk) * gq per head, into the workspace (the
    // query gain moves onto the keys; the query rows keep only their 1/RMS)
    if (rmm::launch_rmsnorm_heads(K, ldk, gk, gq, khat, Hkv * D, B * S, static_cast<int>(Hkv),
                                  static_cast<int>(D), eps, stream) != cudaSuccess)
        return RMM_ERR_LAUNCH;
    rmm::AttnLaunch a{};
    a.S = static_cast<int>(S);
    a.D = static_cast<int>(D);
    a.Hq = static_cast<int>(Hq);
    a.group = static_cast<int>(Hq / Hkv);
    a.n_qb = static_cast<int>(n_qb);
    a.n_hb = static_cast<int>(B * Hq);
    a.causal = causal != 0;
    a.n_blocks = static_cast<int>(n_qb * B * Hq);
    a.grid = std::min(a.n_blocks, d.sm_count);
    a.eps = eps;
    const double sc = scale > 0.f ? static_cast<double>(scale) : 1.0 / std::sqrt(static_cast<double>(D));
    a.qscale = static_cast<float>(sc * 1.4426950408889634);   // log2(e)
    a.wait_limit_us = g_wait_limit_us.load();
    a.O = O;
    a.ldo = ldo;
    a.test_skip_loads = g_skip_sends.load();
    a.gq = gq;
    a.gk = gk;
    return rmm::launch_qknorm_attention(tmQ, tmK, tmV, a, stream) == cudaSuccess
               ? RMM_OK
               : RMM_ERR_LAUNCH;
}

int rmm_test_hooks(int skip_sends, int64_t wait_limit_ns) {
    if (wait_limit_ns < 0) return RMM_ERR_INVALID_ARG;
    const int64_t us = wait_limit_ns > 0 ? std::max<int64_t>(1, wait_limit_ns / 1000) : kDefaultWaitUs;
    g_wait_limit_us.store(static_cast<int>(std::min<int64_t>(us, kDefaultWaitUs)));
    g_skip_sends.store(skip_sends != 0 ? 1 : 0);
    return RMM_OK;
}

const char* rmm_status_string(int code) {
    switch (code) {
        case RMM_OK: return "RMM_OK";
        case RMM_ERR_INVALID_ARG: return "RMM_ERR_INVALID_ARG";
        case RMM_ERR_ALIGNMENT: return "RMM_ERR_ALIGNMENT";
        case RMM_ERR_UNSUPPORTED_DEVICE: return "RMM_ERR_UNSUPPORTED_DEVICE";
        case RMM_ERR_LAUNCH: return "RMM_ERR_LAUNCH";
        case RMM_ERR_DEVICE_TIMEOUT: return "RMM_ERR_DEVICE_TIMEOUT";
        case RMM_ERR_INTERNAL: return "RMM_ERR_INTERNAL";
        case RMM_ERR_SCRATCH_LIMIT: return "RMM_ERR_SCRATCH_LIMIT";
        default: return "RMM_UNKNOWN_STATUS";
    }
}

}  // extern "C"

// ============================================================================
// Allocation-free variant of rmsnorm_matmul().
//
// Some callers cannot let a library allocate device memory during a call:
// inference runtimes and plugin hosts that own every byte of device memory
// through their own pool and forbid allocation inside their enqueue step;
// processes that fix their device-memory budget at start-up; and
// latency-critical paths where cudaMalloc, which may synchronise the device,
// is not acceptable.  rmsnorm_matmul_noalloc() runs the same kernels with the
// same plans, but the K-split partial sums that rmsnorm_matmul() keeps in a
// workspace allocated on first use (the prefill kernel's tail pieces, the
// small-M path's global split) live in the fixed array below.  20 MiB holds
// the tail pieces of any shape on a 152-SM device (at most one 128 x 256
// fp32 piece per SM: 19.1 MiB); a plan that needs more is refused.
// ============================================================================
namespace {

constexpr size_t kScratchBytes = size_t(20) << 20;          // 20 MiB in total
constexpr size_t kScratchCounterBytes = size_t(64) << 10;   // arrival counters first
constexpr size_t kScratchAreaBytes = kScratchBytes - kScratchCounterBytes;

// Held on every device where this module is loaded, until the process exits.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_scratch_mu;
std::map<int, unsigned char*> g_scratch_addr;

// Device address of g_scratch on `dev`, which must be the current device.
// Looked up once per device (the first call may load this library's device
// code on that device) and kept for the life of the process: a device reset
// while the library is in use leaves it (like the workspaces) dangling.
int scratch_address(int dev, unsigned char** out) {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    auto it = g_scratch_addr.find(dev);
    if (it != g_scratch_addr.end()) {
        *out = it->second;
        return RMM_OK;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return RMM_ERR_LAUNCH;
    g_scratch_addr[dev] = static_cast<unsigned char*>(p);
    *out = static_cast<unsigned char*>(p);
    return RMM_OK;
}

}  // namespace

extern "C" int rmsnorm_matmul_noalloc(const void* X, const void* g, const void* W, void* Y,
                                      int64_t M, int64_t K, int64_t N, float eps,
                                      cudaStream_t stream) {
    int rc = check_sizes(M, K, N, eps, true);
    if (rc == kNoop) return RMM_OK;
    if (rc != RMM_OK) return rc;
    rc = check_ptrs(Y, static_cast<size_t>(M) * N * 2,
                    {{X, static_cast<size_t>(M) * K * 2}, {g, static_cast<size_t>(K) * 2},
                     {W, static_cast<size_t>(K) * N * 2}});
    if (rc != RMM_OK) return rc;
    int dev = 0;
    DeviceInfo d;
    rc = current_device(&dev, &d);
    if (rc != RMM_OK) return rc;
    unsigned char* base = nullptr;
    rc = scratch_address(dev, &base);
    if (rc != RMM_OK) return rc;
    const FixedScratch f{base + kScratchCounterBytes, kScratchAreaBytes, reinterpret_cast<int*>(base),
                         kScratchCounterBytes};
    return run_contraction(true, X, g, W, Y, M, K, N, eps, stream, &f);
}
