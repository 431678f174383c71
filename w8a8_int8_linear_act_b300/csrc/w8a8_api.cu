// C ABI of the guarded W8A8 linear layer (declared in include/w8a8.h).
// Host-side argument checks, the shape guard, tensor-map encoding and kernel
// launches.  No allocation, no synchronisation (except w8a8_read_status).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/w8a8.h"
#include "gemm_tcgen05.cuh"
#include "gemm_kcluster.cuh"
#include "quant_rows.cuh"
#include "quant_blocks.cuh"
#include "norm_quant.cuh"

namespace {

constexpr int kVersion = 1;
constexpr size_t kAlign = 1024;
constexpr int kMaxDevices = 64;

std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
std::atomic<int> g_skip_loads{0};
std::atomic<int> g_force_single{0};
std::atomic<int> g_force_form{-1};   // -1: the planner decides; 0: persistent form; 1: cluster-K form
std::atomic<int> g_force_bn{0};      // cluster-K form under the switch: tile width (0: planner's)
std::atomic<int> g_force_ks{0};      // cluster-K form under the switch: cluster size (0: planner's)

// Tile widths and cluster sizes of the cluster-K form (gemm_kcluster.cuh).
constexpr int kKcWidths[3] = {64, 128, 256};
constexpr int kKcSizes[4] = {1, 2, 4, 8};

struct DeviceInfo {
    bool ready = false;
    bool supported = false;
    int num_sms = 0;
    bool gemm_attr_set = false;
    int pair_workers = 0;   // co-resident CTA pairs of the 2-CTA GEMM (0: form unavailable)
    bool kc_ready = false;
    int kc_clusters[3][4] = {};   // co-resident clusters of the cluster-K form per (width, cluster size)
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Raises a kernel's dynamic shared-memory limit on the current device, once
// per device (the attribute belongs to each device's context).  `done` is
// the kernel's own per-device flag array.  A failure leaves the flag clear
// (the launch then fails and reports W8A8_ERR_CUDA).
void set_dynamic_smem_once(const void* func, int bytes, std::atomic<bool>* done)
{
    int dev = -1;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices && !done[dev].load()) {
        if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess)
            done[dev].store(true);
    }
    cudaGetLastError();
}

// Per-device facts, queried once.  Returns nullptr when the current device
// cannot run sm_103a code.
const DeviceInfo* device_info(int* dev_out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaGetLastError();
        d.supported = (major == 10 && minor == 3);
        d.num_sms = sms;
        d.ready = true;
    }
    if (dev_out) *dev_out = dev;
    return d.supported ? &d : nullptr;
}

bool load_encode_fn()
{
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        cudaGetLastError();
    });
    return g_encode != nullptr;
}

// 2-D bf16 tensor [rows][inner] (inner contiguous), boxes of box_rows x 64
// elements (128 bytes) with 128-byte swizzling; loads zero-fill outside the
// tensor, stores skip it.
bool encode_bf16_2d(CUtensorMap* map, const void* base, int64_t rows, int64_t inner, uint32_t box_rows)
{
    if (!load_encode_fn()) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * 2u};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(w8a8::kBK), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Workspace layout, relative to the first 1024-byte boundary at or after the
// caller's pointer (the caller only guarantees 16 bytes; kAlign bytes of
// slack are part of the size):
//   header  1 KB: status word (word 0), split-tile arrival counters (words
//           16 ..), cleared by the first kernel of every call
//   sx      M fp32 row scales
//   codes   M x K activation codes as bf16
//   slots   INT32 partial tiles of the GEMM's K-split last wave, as many as
//           fit in what the caller gave (none is fine: no split then)
constexpr size_t kCounterOffWords = 16;
constexpr int kMaxSplitTiles = 256 - static_cast<int>(kCounterOffWords);   // counters: split tiles x CTAs per tile
constexpr size_t kSlotBytes = static_cast<size_t>(w8a8::kPartialInt4) * 16u;

struct WsLayout {
    size_t status_off, sx_off, codes_off, slots_off, min_total;
};

bool ws_layout(int64_t M, int64_t K, WsLayout* L)
{
    if (M < 1 || K < 1 || M > INT32_MAX || K > INT32_MAX) return false;
    L->status_off = 0;
    L->sx_off = kAlign;
    L->codes_off = L->sx_off + align_up(static_cast<size_t>(M) * 4u, kAlign);
    L->slots_off = L->codes_off + align_up(static_cast<size_t>(M) * static_cast<size_t>(K) * 2u, kAlign);
    L->min_total = kAlign + L->slots_off;
    return true;
}

// Workspace of the BF16 linear: the 1 KB header (status word and split-tile
// counters) and the partial-tile slots; no codes, no scales.
void bf16_ws_layout(WsLayout* L)
{
    L->status_off = 0;
    L->sx_off = L->codes_off = 0;   // unused
    L->slots_off = kAlign;
    L->min_total = kAlign + L->slots_off;
}

// Largest M, N (and the BF16 path's K) the GEMM takes: its tile and k-block
// counts are formed as (dim + tile - 1) / tile in 32-bit arithmetic.
constexpr int64_t kMaxDim = int64_t(1) << 30;

int bf16_guard_reasons(int64_t M, int64_t N, int64_t K, int bias_dtype)
{
    int r = 0;
    if (M < 1 || M > kMaxDim) r |= W8A8_REASON_M;
    if (N < 8 || N % 8 != 0 || N > kMaxDim) r |= W8A8_REASON_N;
    if (K < 8 || K % 8 != 0 || K > kMaxDim) r |= W8A8_REASON_K;
    if (bias_dtype != W8A8_F32 && bias_dtype != W8A8_BF16) r |= W8A8_REASON_BIAS_DTYPE;
    return r;
}

// Partial-tile slots that fit in a workspace of ws_bytes.
int64_t ws_slots(const WsLayout& L, size_t ws_bytes)
{
    return ws_bytes > L.min_total ? static_cast<int64_t>((ws_bytes - L.min_total) / kSlotBytes) : 0;
}

uint8_t* ws_base(const void* ws)
{
    return reinterpret_cast<uint8_t*>(align_up(reinterpret_cast<uintptr_t>(ws), kAlign));
}

// How the GEMM deals its output tiles to its workers (see gemm_tcgen05.cuh).
// A worker is a CTA pair on two SMs (256-row tiles) or, where pairs cannot
// be resident or the single-CTA test switch is on, one CTA (128-row tiles).
// Full waves run whole tiles.  When the last wave would be at most half
// full, its `rem` tiles are cut along K into `splits` segments so that all
// workers share that wave.  The last segment of a tile
// to finish adds the other partials (each one 128 x 256 INT32 block read
// from L2), so more segments cost more fix-up: splits stays near
// sqrt(k-blocks), which balances the segment's MMA time (k-blocks / splits)
// against that fix-up ((splits - 1) reads).
struct GemmPlan {
    int pair;          // CTAs per tile: 1 or 2
    int64_t dp_tiles;
    int splits;
    int64_t tail_units;
    int grid;          // CTAs launched
};

constexpr int kMinKbPerSplit = 2;
// Tiles shorter than this many k-blocks are never split: measured on the
// B300, the fix-up (partials written, fenced, copied back) then costs more
// than the shorter segments save (K = 2048 shapes ran 1-2 us slower split,
// a 256-deep tile 5 us slower; K = 4096 and 16384 ran 3 and 47 us faster).
constexpr int64_t kMinKbToSplit = 48;

// `workers`: CTAs (pair 1) or co-resident CTA pairs (pair 2).
// `max_slots`: partial-tile slots (128 x 256 INT32 each) in the workspace.
GemmPlan plan_gemm(int64_t M, int64_t N, int64_t K, int pair, int workers, int64_t max_slots)
{
    const int64_t tile_rows = static_cast<int64_t>(w8a8::kBM) * pair;
    const int64_t tiles = ((M + tile_rows - 1) / tile_rows) * ((N + w8a8::kBN - 1) / w8a8::kBN);
    const int64_t num_kb = (K + w8a8::kBK - 1) / w8a8::kBK;
    GemmPlan g;
    g.pair = pair;
    g.dp_tiles = tiles;
    g.splits = 1;
    g.tail_units = 0;
    g.grid = static_cast<int>(tiles < workers ? tiles : workers) * pair;
    const int64_t rem = tiles % workers;
    if (rem == 0 || 2 * rem > workers || rem * pair > kMaxSplitTiles || num_kb < kMinKbToSplit) return g;
    int64_t s = workers / rem;
    int64_t root = 1;
    while ((root + 1) * (root + 1) <= num_kb) ++root;
    if (s > root) s = root;
    if (s > num_kb / kMinKbPerSplit) s = num_kb / kMinKbPerSplit;
    if (s > max_slots / pair / rem) s = max_slots / pair / rem;
    if (s < 2) return g;
    g.dp_tiles = tiles - rem;
    g.splits = static_cast<int>(s);
    g.tail_units = rem * s;
    g.grid = static_cast<int>(tiles >= workers ? workers : g.tail_units) * pair;
    return g;
}

// The 2-CTA form whenever clusters of two can be resident and the single-CTA
// test switch is off, also for M <= 128 (the
// odd CTA's rows are then all outside X and Y: its copies fill zeros and it
// stores nothing), because per SM they move a third fewer operand bytes:
// 126-row GEMMs ran 8 % faster that way than on single CTAs.
GemmPlan choose_plan(int64_t M, int64_t N, int64_t K, int num_sms, int pair_workers, int64_t max_slots)
{
    if (pair_workers >= 1 && !g_force_single.load())
        return plan_gemm(M, N, K, 2, pair_workers, max_slots);
    return plan_gemm(M, N, K, 1, num_sms, max_slots);
}

// ---------------------------------------------------------------- cluster-K form
//
// For problems whose output has few tiles (a partial first wave of the
// persistent form), gemm_kcluster.cuh computes each 128 x bn tile with a
// cluster of ks CTAs that split K and add their INT32 partials through
// distributed shared memory.  The choice compares estimated kernel times,
// fitted to a sweep of every (bn, ks) on B300 at the audio and tiny shapes
// (hot L2, CUDA-graph replays):
//   cluster-K:  a fixed cost per launch (set-up, first copies, exchange and
//               store latency), plus per CTA its operand stream (A rows
//               that exist + bn rows of B, 128 B per row and k-block) at the
//               rate one SM sustains, or its MMA time if longer, plus its
//               share of the epilogue, plus the cluster exchange (two
//               cluster barriers) when ks > 1, times the waves of clusters;
//   persistent: the same fixed cost plus waves of 256 x 256 pair tiles,
//               each the MMA time of a tile.
// Widths of 256 and clusters of 8 measured slower than the estimate in
// every case (the 256-wide epilogue spills, clusters of 8 wait longer at
// their barriers), so the planner uses them only under the test switch.
struct KcPlan {
    int bn = 0, ks = 0;
    int64_t tiles_m = 0, tiles = 0, ctas = 0;
    double cost_us = 0.0;
};

constexpr double kSmMmaFlopsPerUs = 1.75e9 / 148.0;    // bf16 tcgen05 operations per microsecond per SM
constexpr double kSmStreamBytesPerUs = 110e3;          // operand bytes per microsecond one SM streams
constexpr double kLaunchFixedUs = 4.0;                 // per launch: set-up, first copies, last stores
constexpr double kItemUs = 0.1;                        // per 8-column epilogue item of one thread
constexpr double kExchangeUs = 1.5;                    // the cluster exchange (ks > 1)
constexpr double kExchange4Us = 0.5;                   // ... and more for clusters of 4
constexpr int kMinKbPerCta = 4;                        // at least 256 of K per CTA of a cluster

int kc_width_index(int bn) { return bn == 64 ? 0 : bn == 128 ? 1 : bn == 256 ? 2 : -1; }
int kc_size_index(int ks) { return ks == 1 ? 0 : ks == 2 ? 1 : ks == 4 ? 2 : ks == 8 ? 3 : -1; }

// Estimated time (microseconds) of the cluster-K form with (bn, ks);
// `clusters`: how many such clusters are co-resident.
double kc_cost(int64_t M, int64_t N, int64_t K, int bn, int ks, int clusters, KcPlan* out)
{
    const int64_t tiles_m = (M + w8a8::kBM - 1) / w8a8::kBM;
    const int64_t tiles = tiles_m * ((N + bn - 1) / bn);
    const int64_t num_kb = (K + w8a8::kBK - 1) / w8a8::kBK;
    const double kb = static_cast<double>((num_kb + ks - 1) / ks);   // k-blocks per CTA
    const double a_rows = static_cast<double>(M < w8a8::kBM ? M : w8a8::kBM);
    const double t_load = kb * (a_rows + bn) * 128.0 / kSmStreamBytesPerUs;
    const double t_mma = kb * 2.0 * w8a8::kBM * bn * w8a8::kBK / kSmMmaFlopsPerUs;
    const double items = static_cast<double>(w8a8::kBM / ks) * (bn / 8) / (32.0 * w8a8::kEpiWarps);
    const double t_x = ks > 1 ? kExchangeUs + (ks >= 4 ? kExchange4Us : 0.0) : 0.0;
    const int64_t waves = (tiles + clusters - 1) / (clusters > 0 ? clusters : 1);
    const double cost =
        kLaunchFixedUs + static_cast<double>(waves) * ((t_mma > t_load ? t_mma : t_load) + items * kItemUs + t_x);
    if (out) {
        out->bn = bn;
        out->ks = ks;
        out->tiles_m = tiles_m;
        out->tiles = tiles;
        out->ctas = tiles * ks;
        out->cost_us = cost;
    }
    return cost;
}

// The cluster-K plan for (M, N, K), or bn == 0 when the persistent form is
// expected to be faster.  clusters[w][s]: co-resident clusters per (width,
// size) index.  force_bn / force_ks (nonzero) pin the width / size; `force`
// takes the cluster-K form whatever the estimate.
KcPlan plan_kcluster(int64_t M, int64_t N, int64_t K, int num_sms, int pair_workers, const int (*clusters)[4],
                     bool force, int force_bn, int force_ks)
{
    KcPlan best;
    const int64_t num_kb = (K + w8a8::kBK - 1) / w8a8::kBK;
    const int64_t ptiles = ((M + 255) / 256) * ((N + w8a8::kBN - 1) / w8a8::kBN);
    // Only problems that leave the persistent form's only wave mostly idle.
    if (!force && (pair_workers < 1 || ptiles * 10 > static_cast<int64_t>(pair_workers) * 6)) return best;
    double best_cost = 1e30;
    for (int wi = 0; wi < 3; ++wi) {
        const int bn = kKcWidths[wi];
        if (force_bn ? bn != force_bn : (!force && bn == 256)) continue;
        for (int si = 0; si < 4; ++si) {
            const int ks = kKcSizes[si];
            if (force_ks ? ks != force_ks : (!force && ks == 8)) continue;
            if (!force_ks && ks > 1 && num_kb < static_cast<int64_t>(ks) * kMinKbPerCta) continue;
            const int cl = clusters[wi][si];
            if (cl < 1) continue;
            KcPlan cand;
            const double c = kc_cost(M, N, K, bn, ks, cl, &cand);
            if (!force && cand.ctas > num_sms) continue;   // one wave of CTAs at most, unless forced
            if (c < best_cost) {
                best_cost = c;
                best = cand;
            }
        }
    }
    if (best.bn == 0 || force) return best;
    // Keep the persistent form where it is estimated faster: waves of pair
    // tiles, each 256 x 256 x K of MMA work on two SMs.
    const int64_t pwaves = (ptiles + pair_workers - 1) / pair_workers;
    const double t_pair = kLaunchFixedUs + static_cast<double>(pwaves) * 2.0 * 256.0 * w8a8::kBN *
                                               static_cast<double>(num_kb * w8a8::kBK) / (2.0 * kSmMmaFlopsPerUs);
    if (best.cost_us >= t_pair) best = KcPlan();
    return best;
}

// Co-resident clusters when no device is current: every SM takes one CTA.
void default_kc_clusters(int num_sms, int (*clusters)[4])
{
    for (int wi = 0; wi < 3; ++wi)
        for (int si = 0; si < 4; ++si) clusters[wi][si] = num_sms / kKcSizes[si];
}

template <int kMode, int BN>
cudaError_t set_kc_smem()
{
    return cudaFuncSetAttribute(w8a8::gemm_kcluster_kernel<kMode, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(w8a8::KClusterCfg<BN>::kSmemBytes));
}

template <int BN>
int kc_max_clusters(int ks, int num_sms)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(ks);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms / ks * ks));
    cfg.blockDim = dim3(w8a8::kGemmThreads);
    cfg.dynamicSmemBytes = w8a8::KClusterCfg<BN>::kSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, w8a8::gemm_kcluster_kernel<w8a8::kModeW8A8, BN>, &cfg) != cudaSuccess)
        n = 0;
    cudaGetLastError();
    return n;
}

// Shared-memory attributes of the cluster-K instantiations and their
// cluster occupancy, once per device.
bool ensure_kcluster_ready(DeviceInfo* dev)
{
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (dev->kc_ready) return true;
    using namespace w8a8;
    if (set_kc_smem<kModeW8A8, 64>() != cudaSuccess || set_kc_smem<kModeW8A8, 128>() != cudaSuccess ||
        set_kc_smem<kModeW8A8, 256>() != cudaSuccess || set_kc_smem<kModeS32, 64>() != cudaSuccess ||
        set_kc_smem<kModeS32, 128>() != cudaSuccess || set_kc_smem<kModeS32, 256>() != cudaSuccess ||
        set_kc_smem<kModeBf16, 64>() != cudaSuccess || set_kc_smem<kModeBf16, 128>() != cudaSuccess ||
        set_kc_smem<kModeBf16, 256>() != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    for (int si = 0; si < 4; ++si) {
        dev->kc_clusters[0][si] = kc_max_clusters<64>(kKcSizes[si], dev->num_sms);
        dev->kc_clusters[1][si] = kc_max_clusters<128>(kKcSizes[si], dev->num_sms);
        dev->kc_clusters[2][si] = kc_max_clusters<256>(kKcSizes[si], dev->num_sms);
    }
    dev->kc_ready = true;
    return true;
}

template <int kMode, int kPair>
cudaError_t set_gemm_smem()
{
    return cudaFuncSetAttribute(w8a8::gemm_w8a8_tcgen05_kernel<kMode, kPair>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(w8a8::GemmCfg<kPair>::kSmemBytes));
}

// Shared-memory attributes of the four GEMM instantiations, and how many CTA
// pairs the 2-CTA form can hold at once on this device; once per device.
bool ensure_gemm_ready(DeviceInfo* dev)
{
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (dev->gemm_attr_set) return true;
    using namespace w8a8;
    if (set_gemm_smem<kModeW8A8, 1>() != cudaSuccess || set_gemm_smem<kModeS32, 1>() != cudaSuccess ||
        set_gemm_smem<kModeBf16, 1>() != cudaSuccess || set_gemm_smem<kModeW8A8, 2>() != cudaSuccess ||
        set_gemm_smem<kModeS32, 2>() != cudaSuccess || set_gemm_smem<kModeBf16, 2>() != cudaSuccess ||
        set_gemm_smem<kModeW8A8RowMax, 1>() != cudaSuccess || set_gemm_smem<kModeW8A8RowMax, 2>() != cudaSuccess ||
        set_gemm_smem<kModeW8A8Fused, 1>() != cudaSuccess || set_gemm_smem<kModeW8A8Fused, 2>() != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * static_cast<unsigned>(dev->num_sms / 2 > 0 ? dev->num_sms / 2 : 1));
    cfg.blockDim = dim3(w8a8::kGemmThreads);
    cfg.dynamicSmemBytes = w8a8::GemmCfg<2>::kSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, w8a8::gemm_w8a8_tcgen05_kernel<w8a8::kModeW8A8, 2>, &cfg) !=
        cudaSuccess)
        clusters = 0;
    cudaGetLastError();
    dev->pair_workers = clusters > dev->num_sms / 2 ? dev->num_sms / 2 : clusters;
    dev->gemm_attr_set = true;
    return true;
}

// Plan for the current device (a 148-SM device with 74 pairs when none is
// current), as the launch will make it.
GemmPlan current_plan(int64_t M, int64_t N, int64_t K, int64_t max_slots)
{
    int dno = 0;
    DeviceInfo* d = const_cast<DeviceInfo*>(device_info(&dno));
    if (d && ensure_gemm_ready(d)) return choose_plan(M, N, K, d->num_sms, d->pair_workers, max_slots);
    return choose_plan(M, N, K, 148, 74, max_slots);
}

int guard_reasons(int64_t M, int64_t N, int64_t K, int x_dtype, int bias_dtype)
{
    int r = 0;
    if (M < 1 || M > kMaxDim) r |= W8A8_REASON_M;
    if (N < 8 || N % 8 != 0 || N > kMaxDim) r |= W8A8_REASON_N;
    if (K < 16 || K % 16 != 0) r |= W8A8_REASON_K;
    if (K > W8A8_MAX_K) r |= W8A8_REASON_K_RANGE;
    if (x_dtype != W8A8_F32 && x_dtype != W8A8_BF16) r |= W8A8_REASON_X_DTYPE;
    if (bias_dtype != W8A8_F32 && bias_dtype != W8A8_BF16) r |= W8A8_REASON_BIAS_DTYPE;
    return r;
}

w8a8_status last_launch_status()
{
    return cudaGetLastError() == cudaSuccess ? W8A8_OK : W8A8_ERR_CUDA;
}

// ---------------------------------------------------------------- row quant

template <typename TIn, bool kBf16Codes, int NV, int kRows>
void launch_quant_cfg(const TIn* A, int64_t R, int64_t K, void* Q, float* S, uint32_t* header, unsigned threads,
                      cudaStream_t stream, uint32_t* zero_rows)
{
    constexpr int64_t kPer = kRows > 0 ? kRows : 1;   // rows per CTA (0: the CTA-per-row form)
    const int64_t blocks = (R + kPer - 1) / kPer;
    w8a8::quant_rows_kernel<TIn, kBf16Codes, NV, kRows>
        <<<static_cast<unsigned>(blocks), threads, 0, stream>>>(A, R, K, Q, S, header, zero_rows);
}

// Rows of up to 512 16-byte vectors: a warp per row, kQuantRows rows per
// CTA, each lane holding up to 16 vectors.  Up to 4096 vectors: a CTA per
// row of ceil(V / 16) threads rounded to warps.  Longer: a CTA of 1024
// threads per row reading it twice.
constexpr int kQuantRows = 4;

// Up to this many rows per SM: a CTA per row of at most 256 threads with 2,
// 4 or 8 vectors a thread (rows of 64 to 2048 vectors).  A warp per row
// walks its row's vectors one after another, and with few warps per SM that
// serial chain, not HBM, sets the time (297 rows of 4096: 15.1 µs against
// 4.5 µs with a CTA per row).  Measured on B300 with L2 flushed, the CTA per
// row is as fast or faster up to 6144 rows for rows of 128 to 512 vectors
// (6144 x 4096 with outlier columns: 21.3 against 22.5 µs; 1001 x 2048:
// 4.6 against 8.9 µs), the warp per row from about 9500 rows on (28672 x
// 4096: 75.0 against 85.3 µs).
constexpr int64_t kFewRowsPerSm = 48;

template <typename TIn, bool kBf16Codes>
w8a8_status launch_quant_typed(const TIn* A, int64_t R, int64_t K, void* Q, float* S, uint32_t* header,
                               cudaStream_t stream, uint32_t* zero_rows, int num_sms)
{
    constexpr int E = w8a8::InVec<TIn>::kElems;
    const int64_t V = K / E;  // vectors per row
    if (R <= kFewRowsPerSm * num_sms && V >= 64 && V <= 2048) {
        // Rows of up to 256 vectors: 2 a thread; up to 1024: 4 a thread (at
        // 512 vectors, 128 threads of 4 measured 3-8 % faster than 256 of 2
        // from 1536 to 6144 rows); longer: 8.
        if (V <= 256)
            launch_quant_cfg<TIn, kBf16Codes, 2, 0>(A, R, K, Q, S, header,
                                                    static_cast<unsigned>(((V + 1) / 2 + 31) / 32 * 32), stream,
                                                    zero_rows);
        else if (V <= 1024)
            launch_quant_cfg<TIn, kBf16Codes, 4, 0>(A, R, K, Q, S, header,
                                                    static_cast<unsigned>(((V + 3) / 4 + 31) / 32 * 32), stream,
                                                    zero_rows);
        else
            launch_quant_cfg<TIn, kBf16Codes, 8, 0>(A, R, K, Q, S, header,
                                                    static_cast<unsigned>(((V + 7) / 8 + 31) / 32 * 32), stream,
                                                    zero_rows);
        return last_launch_status();
    }
    if (V <= 32)
        launch_quant_cfg<TIn, kBf16Codes, 1, kQuantRows>(A, R, K, Q, S, header, 32 * kQuantRows, stream, zero_rows);
    else if (V <= 64)
        launch_quant_cfg<TIn, kBf16Codes, 2, kQuantRows>(A, R, K, Q, S, header, 32 * kQuantRows, stream, zero_rows);
    else if (V <= 128)
        launch_quant_cfg<TIn, kBf16Codes, 4, kQuantRows>(A, R, K, Q, S, header, 32 * kQuantRows, stream, zero_rows);
    else if (V <= 256)
        launch_quant_cfg<TIn, kBf16Codes, 8, kQuantRows>(A, R, K, Q, S, header, 32 * kQuantRows, stream, zero_rows);
    else if (V <= 512)
        launch_quant_cfg<TIn, kBf16Codes, 16, kQuantRows>(A, R, K, Q, S, header, 32 * kQuantRows, stream, zero_rows);
    else if (V <= 4096) {
        const unsigned T = static_cast<unsigned>(((V + 15) / 16 + 31) / 32 * 32);
        launch_quant_cfg<TIn, kBf16Codes, 16, 0>(A, R, K, Q, S, header, T, stream, zero_rows);
    } else
        launch_quant_cfg<TIn, kBf16Codes, 0, 0>(A, R, K, Q, S, header, 1024, stream, zero_rows);
    return last_launch_status();
}

template <bool kBf16Codes>
w8a8_status launch_quant(const void* A, int dtype, int64_t R, int64_t K, void* Q, float* S, uint32_t* status,
                         cudaStream_t stream, uint32_t* zero_rows = nullptr)
{
    const DeviceInfo* dev = device_info(nullptr);
    const int num_sms = dev ? dev->num_sms : 148;
    if (dtype == W8A8_BF16)
        return launch_quant_typed<__nv_bfloat16, kBf16Codes>(static_cast<const __nv_bfloat16*>(A), R, K, Q, S,
                                                             status, stream, zero_rows, num_sms);
    return launch_quant_typed<float, kBf16Codes>(static_cast<const float*>(A), R, K, Q, S, status, stream,
                                                 zero_rows, num_sms);
}

w8a8_status check_quant_args(const void* A, int dtype, int64_t R, int64_t K, const void* Q, const float* S)
{
    if (R < 0 || K < 0) return W8A8_ERR_INVALID_ARG;
    if (R == 0 && dtype == W8A8_F32) return W8A8_OK;   // empty input: nothing to do, pointers may be NULL
    if (R == 0 && dtype == W8A8_BF16) return W8A8_OK;
    if (!A || !Q || !S) return W8A8_ERR_INVALID_ARG;
    if (dtype != W8A8_F32 && dtype != W8A8_BF16) return W8A8_ERR_DTYPE;
    if (R > INT32_MAX || K < 16 || K % 16 != 0 || K > W8A8_MAX_K) return W8A8_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(A, 16) || !aligned(Q, 16) || !aligned(S, 4)) return W8A8_ERR_ALIGNMENT;
    return W8A8_OK;
}

w8a8_status quantize_rows_entry(const void* A, int dtype, int64_t R, int64_t K, int8_t* Q, float* S, void* stream)
{
    w8a8_status st = check_quant_args(A, dtype, R, K, Q, S);
    if (st != W8A8_OK) return st;
    if (!device_info(nullptr)) return W8A8_ERR_NO_DEVICE;
    if (R == 0) return W8A8_OK;
    return launch_quant<false>(A, dtype, R, K, Q, S, nullptr, static_cast<cudaStream_t>(stream));
}

w8a8_status launch_codes_to_bf16(const int8_t* Qi, uint16_t* Qb, int64_t n, uint32_t* status, int num_sms,
                                 cudaStream_t stream)
{
    const int64_t n16 = n / 16;
    int64_t blocks = (n16 + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    w8a8::codes_to_bf16_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(Qi, Qb, n16, status);
    return last_launch_status();
}

// ---------------------------------------------------------------- GEMM

// The cluster-K plan the GEMM launch takes for (M, N, K) on this device
// (bn == 0: the persistent form), honouring the test switch.
KcPlan current_kc_plan(DeviceInfo* dev, int64_t M, int64_t N, int64_t K)
{
    const int ff = g_force_form.load();
    if (ff == 0) return KcPlan();
    if (!ensure_kcluster_ready(dev)) return KcPlan();
    KcPlan kp = plan_kcluster(M, N, K, dev->num_sms, g_force_single.load() ? 0 : dev->pair_workers, dev->kc_clusters,
                              ff == 1, g_force_bn.load(), g_force_ks.load());
    if (kp.ctas > INT32_MAX) kp = KcPlan();
    return kp;
}

template <int kMode>
w8a8_status launch_kcluster(const KcPlan& kp, const uint16_t* A_codes, const uint16_t* Wp, int64_t M, int64_t N,
                            int64_t K, const float* sx, const float* sw, const void* bias, int bias_mode, void* out,
                            uint32_t* status, cudaStream_t stream)
{
    CUtensorMap ta, tb;
    if (!encode_bf16_2d(&ta, A_codes, M, K, w8a8::kBM)) return W8A8_ERR_CUDA;
    if (!encode_bf16_2d(&tb, Wp, N, K, static_cast<uint32_t>(kp.bn))) return W8A8_ERR_CUDA;
    w8a8::KClusterParams p;
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.kb_per_chunk = kMode == w8a8::kModeBf16 ? static_cast<int32_t>((K + w8a8::kBK - 1) / w8a8::kBK)
                                              : w8a8::kMaxKbPerChunk;
    p.tiles_m = static_cast<int32_t>(kp.tiles_m);
    p.bias_mode = bias_mode;
    p.sx = sx;
    p.sw = sw;
    p.bias = bias;
    p.out = out;
    p.status = status;
    p.wait_limit_ns = g_wait_limit_ns.load();
    p.skip_loads = g_skip_loads.load();
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(kp.ks);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(kp.ctas));
    cfg.blockDim = dim3(w8a8::kGemmThreads);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t err;
    if (kp.bn == 64) {
        cfg.dynamicSmemBytes = w8a8::KClusterCfg<64>::kSmemBytes;
        err = cudaLaunchKernelEx(&cfg, w8a8::gemm_kcluster_kernel<kMode, 64>, ta, tb, p);
    } else if (kp.bn == 128) {
        cfg.dynamicSmemBytes = w8a8::KClusterCfg<128>::kSmemBytes;
        err = cudaLaunchKernelEx(&cfg, w8a8::gemm_kcluster_kernel<kMode, 128>, ta, tb, p);
    } else {
        cfg.dynamicSmemBytes = w8a8::KClusterCfg<256>::kSmemBytes;
        err = cudaLaunchKernelEx(&cfg, w8a8::gemm_kcluster_kernel<kMode, 256>, ta, tb, p);
    }
    if (err != cudaSuccess) {
        cudaGetLastError();
        return W8A8_ERR_CUDA;
    }
    return last_launch_status();
}

// The W8A8 linear with its activation quantisation overlapped with the GEMM
// (kModeW8A8Fused): for bf16 X with K = 4096 on the CTA-pair form, when the
// GEMM's first wave of tiles needs fewer rows than there are.  Where the
// weights fit well in L2, the tiles are rasterised row-tile by row-tile
// instead of in groups of 8, so that the first wave touches few row-tiles
// (larger weights keep groups of 8: re-reading them from HBM every few
// row-tiles cost more than the overlap gains).  The first wave's rows (the
// head) are quantised before the GEMM by the row quantiser, the rest by the
// GEMM's own quantiser warps while it runs.  Returns the head's row count,
// or 0 where the fused form does not apply.
int fused_group_m(int64_t N, int64_t K) { return N * K * 2 <= (int64_t(64) << 20) ? 1 : 8; }

int64_t fused_head_rows(const DeviceInfo* dev, int64_t M, int64_t N, int64_t K, int x_dtype, int64_t slots)
{
    if (x_dtype != W8A8_BF16 || K != w8a8::kFusedQuantK || g_force_form.load() >= 0) return 0;
    const GemmPlan g = choose_plan(M, N, K, dev->num_sms, dev->pair_workers, slots);
    if (g.pair != 2) return 0;
    const int tiles_m = static_cast<int>((M + 2 * w8a8::kBM - 1) / (2 * w8a8::kBM));
    const int tiles_n = static_cast<int>((N + w8a8::kBN - 1) / w8a8::kBN);
    const int64_t tiles = static_cast<int64_t>(tiles_m) * tiles_n;
    const int workers = g.grid / 2;
    // Row-tiles of the first wave: the whole tiles its workers start with,
    // and, where the wave reaches the split tail, every tail tile.
    int max_mb = 0;
    const int64_t first = std::min<int64_t>(workers, g.dp_tiles);
    const int group_m = fused_group_m(N, K);
    for (int64_t t = 0; t < first; ++t) {
        const int per_group = group_m * tiles_n;
        const int gi = static_cast<int>(t / per_group);
        const int first_m = gi * group_m;
        const int gsz = std::min(tiles_m - first_m, group_m);
        const int r = static_cast<int>(t - static_cast<int64_t>(gi) * per_group);
        max_mb = std::max(max_mb, first_m + r % gsz);
    }
    if (workers > g.dp_tiles) max_mb = tiles_m - 1;   // the wave reaches the tail tiles
    const int64_t head = std::min<int64_t>(M, static_cast<int64_t>(max_mb + 1) * 2 * w8a8::kBM);
    // The per-tile row counts sit at the top of the header, above the split
    // tiles' counters.
    const int64_t split_counters = (tiles - g.dp_tiles) * 2;
    if (static_cast<int64_t>(kCounterOffWords) + split_counters + tiles_m > w8a8::kHeaderWords) return 0;
    return head < M ? head : 0;
}

template <int kMode>
w8a8_status launch_gemm(DeviceInfo* dev, const uint16_t* A_codes, const uint16_t* Wp, int64_t M, int64_t N,
                        int64_t K, const float* sx, const float* sw, const void* bias, int bias_mode, void* out,
                        uint8_t* ws_aligned, const WsLayout& L, int64_t slots, cudaStream_t stream,
                        uint32_t* row_amax = nullptr, const uint16_t* fused_x = nullptr, int64_t fused_row0 = 0)
{
    if (!ensure_gemm_ready(dev)) return W8A8_ERR_CUDA;
    if constexpr (kMode != w8a8::kModeW8A8RowMax && kMode != w8a8::kModeW8A8Fused) {
        // Few output tiles: the cluster-K form spreads them over the SMs.
        const KcPlan kp = current_kc_plan(dev, M, N, K);
        if (kp.bn != 0)
            return launch_kcluster<kMode>(kp, A_codes, Wp, M, N, K, sx, sw, bias, bias_mode, out,
                                          reinterpret_cast<uint32_t*>(ws_aligned + L.status_off), stream);
    }
    const GemmPlan g = choose_plan(M, N, K, dev->num_sms, dev->pair_workers, slots);
    CUtensorMap ta, tb, ty;
    if (!encode_bf16_2d(&ta, A_codes, M, K, w8a8::kBM)) return W8A8_ERR_CUDA;
    if (!encode_bf16_2d(&tb, Wp, N, K, static_cast<uint32_t>(w8a8::kBN / g.pair))) return W8A8_ERR_CUDA;
    // The pair form stores bf16 Y through TMA in 32-row x 64-column boxes.
    if (kMode != w8a8::kModeS32 && g.pair == 2) {
        if (!encode_bf16_2d(&ty, out, M, N, 32)) return W8A8_ERR_CUDA;
    } else {
        ty = tb;   // not read by these forms
    }
    w8a8::GemmParams p;
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    // INT8 codes: fp32 chunks short enough to be exact integers.  BF16: one
    // fp32 accumulation over the unit's whole K range.
    p.kb_per_chunk = kMode == w8a8::kModeBf16 ? static_cast<int32_t>((K + w8a8::kBK - 1) / w8a8::kBK)
                                              : w8a8::kMaxKbPerChunk;
    p.group_m = kMode == w8a8::kModeW8A8Fused ? fused_group_m(N, K) : 8;
    p.bias_mode = bias_mode;
    p.sx = sx;
    p.sw = sw;
    p.bias = bias;
    p.out = out;
    uint32_t* header = reinterpret_cast<uint32_t*>(ws_aligned + L.status_off);
    p.status = header;
    p.tile_counters = header + kCounterOffWords;
    p.partials = reinterpret_cast<int4*>(ws_aligned + L.slots_off);
    p.wait_limit_ns = g_wait_limit_ns.load();
    p.skip_loads = g_skip_loads.load();
    p.dp_tiles = static_cast<int32_t>(g.dp_tiles);
    p.splits = g.splits;
    p.tail_units = static_cast<int32_t>(g.tail_units);
    p.row_amax = row_amax;
    p.qx = reinterpret_cast<const __nv_bfloat16*>(fused_x);
    p.qcodes = const_cast<uint16_t*>(A_codes);
    p.qsx = const_cast<float*>(sx);
    p.q_row0 = static_cast<int32_t>(fused_row0);
    p.q_ready = header + (w8a8::kHeaderWords - (M + 255) / 256);   // per 256-row tile, in the zeroed header
    // A programmatic dependent of the kernel before it in the stream (the
    // quantiser that writes its codes): its set-up overlaps that kernel's
    // tail, and it waits on the device for its results (griddepcontrol).
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(g.grid));
    cfg.blockDim = dim3(w8a8::gemm_threads(kMode));
    cfg.stream = stream;
    cfg.attrs = attr;
    cudaError_t err;
    if (g.pair == 1) {
        cfg.dynamicSmemBytes = w8a8::GemmCfg<1>::kSmemBytes;
        cfg.numAttrs = 1;
        err = cudaLaunchKernelEx(&cfg, w8a8::gemm_w8a8_tcgen05_kernel<kMode, 1>, ta, tb, ty, p);
    } else {
        cfg.dynamicSmemBytes = w8a8::GemmCfg<2>::kSmemBytes;
        cfg.numAttrs = 2;
        err = cudaLaunchKernelEx(&cfg, w8a8::gemm_w8a8_tcgen05_kernel<kMode, 2>, ta, tb, ty, p);
    }
    if (err != cudaSuccess) {
        cudaGetLastError();
        return W8A8_ERR_CUDA;
    }
    return last_launch_status();
}

// The next layer's codes from rows whose absmax the previous GEMM gathered,
// as a programmatic dependent of that GEMM (it waits on the device for the
// GEMM's Y and row maxima).
w8a8_status launch_codes_known_amax(const uint16_t* H, int64_t M, int64_t F, const uint32_t* amax, uint16_t* codes,
                                    float* sx, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(M));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t err = cudaLaunchKernelEx(&cfg, w8a8::codes_known_amax_kernel<true, 8>,
                                               reinterpret_cast<const __nv_bfloat16*>(H), F, amax,
                                               static_cast<void*>(codes), sx);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return W8A8_ERR_CUDA;
    }
    return last_launch_status();
}

// Workspace of w8a8_mlp, relative to the first 1024-byte boundary:
//   header 1 KB (status word, split-tile counters; both GEMMs use them in turn)
//   sx_x [M], codes_x [M][K] bf16      the up layer's activation
//   amax_h [M] fp32 bits, sx_h [M], codes_h [M][F] bf16   the down layer's
//   slots  INT32 partial tiles, shared by the two GEMMs (one runs at a time)
struct MlpLayout {
    WsLayout up;        // status_off, sx_off, codes_off; slots_off = the shared slots
    size_t amax_off, sxh_off, codesh_off;
};

bool mlp_layout(int64_t M, int64_t K, int64_t F, MlpLayout* L)
{
    if (!ws_layout(M, K, &L->up) || F < 1 || F > INT32_MAX) return false;
    const size_t after_x = L->up.slots_off;
    L->amax_off = after_x;
    L->sxh_off = L->amax_off + align_up(static_cast<size_t>(M) * 4u, kAlign);
    L->codesh_off = L->sxh_off + align_up(static_cast<size_t>(M) * 4u, kAlign);
    L->up.slots_off = L->codesh_off + align_up(static_cast<size_t>(M) * static_cast<size_t>(F) * 2u, kAlign);
    L->up.min_total = kAlign + L->up.slots_off;
    return true;
}

// Copy streams and events of w8a8_linear_host, created once per device (with
// that device current) and kept until the process exits.  Streams and events
// are not device memory; the entry point itself allocates nothing.
constexpr int kMaxHostChunks = 64;
struct HostPipe {
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, end = nullptr;
    cudaEvent_t copied[kMaxHostChunks] = {};
    cudaEvent_t computed[kMaxHostChunks] = {};
};
HostPipe g_pipe[kMaxDevices];
std::mutex g_pipe_mutex;

HostPipe* host_pipe(int dev)
{
    std::lock_guard<std::mutex> lock(g_pipe_mutex);
    HostPipe& hp = g_pipe[dev];
    if (hp.ready) return &hp;
    const unsigned ef = cudaEventDisableTiming;
    bool ok = cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.start, ef) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.end, ef) == cudaSuccess;
    for (int i = 0; ok && i < kMaxHostChunks; ++i)
        ok = cudaEventCreateWithFlags(&hp.copied[i], ef) == cudaSuccess &&
             cudaEventCreateWithFlags(&hp.computed[i], ef) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        return nullptr;   // leaves what was created; a later call retries the rest
    }
    hp.ready = true;
    return &hp;
}

// ---------------------------------------------------------------- norm + modulation + quant

template <bool kBf16Codes, int NV, int kRows, bool kFull, int kNorm>
void launch_norm_cfg(const uint16_t* X, int64_t M, int64_t K, const w8a8::NormParams& np, void* Q, float* S,
                     uint32_t* header, unsigned threads, cudaStream_t stream)
{
    // A CTA per row; the warp form (rows dealt to the CTAs in turn) caps that
    // at the CTAs that fit at once below.  The warp form stages the fp32
    // modulation in shared memory, 8 B per element of a row, and a row buffer
    // per warp, 2 B per element (160 KB at the largest, K = 4096, sixteen
    // warps).
    int64_t blocks = M;
    const size_t smem = kRows > 1 ? static_cast<size_t>(K) * (8u + 2u * kRows) : 0u;
    if constexpr (kRows > 1) {
        // Persistent warps: no more CTAs than fit on the GPU at once.
        static std::atomic<bool> attr_done[kMaxDevices];
        set_dynamic_smem_once(reinterpret_cast<const void*>(
                                  w8a8::norm_quant_rows_kernel<kBf16Codes, NV, kRows, kFull, kNorm>),
                              4096 * (8 + 2 * kRows), attr_done);
        const DeviceInfo* dev = device_info(nullptr);
        int per_sm = 0;
        if (dev != nullptr &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &per_sm, w8a8::norm_quant_rows_kernel<kBf16Codes, NV, kRows, kFull, kNorm>, static_cast<int>(threads),
                smem) == cudaSuccess &&
            per_sm > 0) {
            const int64_t resident = static_cast<int64_t>(per_sm) * dev->num_sms;
            if (blocks > resident) blocks = resident;
        }
        cudaGetLastError();
    }
    w8a8::norm_quant_rows_kernel<kBf16Codes, NV, kRows, kFull, kNorm>
        <<<static_cast<unsigned>(blocks), threads, smem, stream>>>(reinterpret_cast<const __nv_bfloat16*>(X), M, K,
                                                                   np, Q, S, header);
}

// Rows of up to 128 vectors: a warp per row with 4 vectors per lane, CTAs
// of eight warps; up to 512: 16 per lane, CTAs of sixteen warps (one per
// SM); up to 4096 (K <= 32768): a CTA per row, 16 per thread.  Rows of
// exactly 128, 256 or 512 vectors (K = 1024, 2048, 4096) take the warp form
// with 4, 8 or 16 vectors per lane (CTAs of eight, eight and sixteen warps)
// and no range checks.  Sixteen-warp CTAs at K = 4096 measured 10 % faster
// than two CTAs of eight per SM at 6144 rows (one CTA then stages the
// modulation for sixteen warps).
template <bool kBf16Codes, int kNorm>
w8a8_status launch_norm_typed(const uint16_t* X, int64_t M, int64_t K, const w8a8::NormParams& np, void* Q,
                              float* S, uint32_t* header, cudaStream_t stream)
{
    const int64_t V = K / 8;
    if (V == 128)
        launch_norm_cfg<kBf16Codes, 4, 8, true, kNorm>(X, M, K, np, Q, S, header, 256, stream);
    else if (V == 256)
        launch_norm_cfg<kBf16Codes, 8, 8, true, kNorm>(X, M, K, np, Q, S, header, 256, stream);
    else if (V == 512)
        launch_norm_cfg<kBf16Codes, 16, 16, true, kNorm>(X, M, K, np, Q, S, header, 512, stream);
    else if (V <= 128)
        launch_norm_cfg<kBf16Codes, 4, 8, false, kNorm>(X, M, K, np, Q, S, header, 256, stream);
    else if (V <= 512)
        launch_norm_cfg<kBf16Codes, 16, 16, false, kNorm>(X, M, K, np, Q, S, header, 512, stream);
    else {
        const unsigned T = static_cast<unsigned>(((V + 15) / 16 + 31) / 32 * 32);
        launch_norm_cfg<kBf16Codes, 16, 1, false, kNorm>(X, M, K, np, Q, S, header, T, stream);
    }
    return last_launch_status();
}

template <bool kBf16Codes>
w8a8_status launch_norm_quant(const uint16_t* X, int64_t M, int64_t K, int norm, const w8a8::NormParams& np,
                              void* Q, float* S, uint32_t* header, cudaStream_t stream)
{
    if (norm == W8A8_NORM_RMS)
        return launch_norm_typed<kBf16Codes, w8a8::kNormRms>(X, M, K, np, Q, S, header, stream);
    return launch_norm_typed<kBf16Codes, w8a8::kNormLayer>(X, M, K, np, Q, S, header, stream);
}

// Host checks shared by the norm entry points (everything but the outputs).
w8a8_status check_norm_args(const uint16_t* X, int64_t M, int64_t K, int norm, float eps, const void* scale,
                            const void* shift, int mod_dtype, const void* y_mod, w8a8::NormParams* np)
{
    if (!X || M < 0 || K < 0) return W8A8_ERR_INVALID_ARG;
    if (norm != W8A8_NORM_RMS && norm != W8A8_NORM_LAYER) return W8A8_ERR_INVALID_ARG;
    if (!(eps >= 0.0f) || !(eps <= 3.4e38f)) return W8A8_ERR_INVALID_ARG;
    if ((scale || shift) && mod_dtype != W8A8_F32 && mod_dtype != W8A8_BF16) return W8A8_ERR_DTYPE;
    if (M < 1 || M > INT32_MAX || K < 16 || K % 16 != 0 || K > W8A8_NORM_MAX_K) return W8A8_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(X, 16) || (scale && !aligned(scale, 16)) || (shift && !aligned(shift, 16)) ||
        (y_mod && !aligned(y_mod, 16)))
        return W8A8_ERR_ALIGNMENT;
    np->eps = eps;
    np->scale = scale;
    np->shift = shift;
    np->mod_f32 = mod_dtype == W8A8_F32 ? 1 : 0;
    np->y_out = static_cast<uint16_t*>(const_cast<void*>(y_mod));
    return W8A8_OK;
}

// ---------------------------------------------------------------- Query/Key blocks

constexpr int kBlockThreads = 256;   // threads per CTA of the Query/Key block quantiser, at most,
constexpr int kBlockThreadsWide = 512;   // or for blocks of kWideBlockVectors vectors or more
constexpr int64_t kWideBlockVectors = 2048;

template <typename TIn, int NV>
void launch_blocks_cfg(const TIn* X, const w8a8::BlockGeom& g, int64_t blocks, int8_t* Q, float* S,
                       cudaStream_t stream)
{
    const unsigned threads = static_cast<unsigned>((g.tpp * g.vd + 31) / 32 * 32);
    // With the block in registers (NV > 0) the CTAs are persistent, each
    // with NV 16-byte slots per thread for its next block: no more CTAs than
    // fit on the GPU at once.
    const size_t smem = NV > 0 ? static_cast<size_t>(NV) * threads * 16u : 0u;
    int64_t grid = blocks;
    if constexpr (NV > 0) {
        static std::atomic<bool> attr_done[kMaxDevices];
        set_dynamic_smem_once(reinterpret_cast<const void*>(w8a8::quant_blocks_kernel<TIn, NV>),
                              NV * (NV >= 8 ? kBlockThreads : kBlockThreadsWide) * 16, attr_done);
        const DeviceInfo* dev = device_info(nullptr);
        int per_sm = 0;
        if (dev != nullptr &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, w8a8::quant_blocks_kernel<TIn, NV>,
                                                          static_cast<int>(threads), smem) == cudaSuccess &&
            per_sm > 0) {
            const int64_t resident = static_cast<int64_t>(per_sm) * dev->num_sms;
            if (grid > resident) grid = resident;
        }
        cudaGetLastError();
    }
    w8a8::quant_blocks_kernel<TIn, NV><<<static_cast<unsigned>(grid), threads, smem, stream>>>(X, g, blocks, Q, S);
}

template <typename TIn>
w8a8_status launch_blocks_typed(const TIn* X, const w8a8::BlockGeom& g, int64_t blocks, int8_t* Q, float* S,
                                cudaStream_t stream)
{
    // Vectors one thread holds: ceil(block_tokens / tpp).
    const int64_t per = (g.block_tokens + g.tpp - 1) / g.tpp;
    if (per <= 1)
        launch_blocks_cfg<TIn, 1>(X, g, blocks, Q, S, stream);
    else if (per <= 2)
        launch_blocks_cfg<TIn, 2>(X, g, blocks, Q, S, stream);
    else if (per <= 4)
        launch_blocks_cfg<TIn, 4>(X, g, blocks, Q, S, stream);
    else if (per <= 8)
        launch_blocks_cfg<TIn, 8>(X, g, blocks, Q, S, stream);
    else if (per <= 16)
        launch_blocks_cfg<TIn, 16>(X, g, blocks, Q, S, stream);
    else
        launch_blocks_cfg<TIn, 0>(X, g, blocks, Q, S, stream);
    return last_launch_status();
}

}  // namespace

extern "C" {

int w8a8_version(void) { return kVersion; }

const char* w8a8_status_str(int status)
{
    switch (status) {
        case W8A8_OK: return "ok";
        case W8A8_ERR_INVALID_ARG: return "invalid argument (null pointer, negative size or unknown value)";
        case W8A8_ERR_DTYPE: return "dtype not accepted";
        case W8A8_ERR_ALIGNMENT: return "pointer not aligned as required";
        case W8A8_ERR_UNSUPPORTED_SHAPE: return "shape rejected by the W8A8 guard; use the BF16 linear";
        case W8A8_ERR_WORKSPACE: return "workspace missing or too small";
        case W8A8_ERR_CUDA: return "CUDA call or kernel launch failed";
        case W8A8_ERR_TIMEOUT: return "a device-side wait ran out";
        case W8A8_ERR_NO_DEVICE: return "current CUDA device is not sm_103";
        default: return "unknown status";
    }
}

int w8a8_shape_supported(int64_t M, int64_t N, int64_t K, int x_dtype, int bias_dtype, int* reason)
{
    const int r = guard_reasons(M, N, K, x_dtype, bias_dtype);
    if (reason) *reason = r;
    return r == 0 ? 1 : 0;
}

void w8a8_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns < 1000000ull ? 1000000ull : ns); }

void w8a8_debug_skip_loads(int on) { g_skip_loads.store(on ? 1 : 0); }

w8a8_status w8a8_quantize_weight(const void* W, int w_dtype, int64_t N, int64_t K, int8_t* Wq, float* sw,
                                 void* stream)
{
    return quantize_rows_entry(W, w_dtype, N, K, Wq, sw, stream);
}

w8a8_status w8a8_quantize_act(const void* X, int x_dtype, int64_t M, int64_t K, int8_t* Xq, float* sx,
                              void* stream)
{
    return quantize_rows_entry(X, x_dtype, M, K, Xq, sx, stream);
}

w8a8_status w8a8_pack_weight(const int8_t* Wq, int64_t N, int64_t K, uint16_t* Wp, void* stream)
{
    if (!Wq || !Wp || N < 0 || K < 0) return W8A8_ERR_INVALID_ARG;
    if (K % 16 != 0) return W8A8_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(Wq, 16) || !aligned(Wp, 16)) return W8A8_ERR_ALIGNMENT;
    const DeviceInfo* dev = device_info(nullptr);
    if (!dev) return W8A8_ERR_NO_DEVICE;
    if (N == 0 || K == 0) return W8A8_OK;
    return launch_codes_to_bf16(Wq, Wp, N * K, nullptr, dev->num_sms, static_cast<cudaStream_t>(stream));
}

size_t w8a8_linear_workspace_min_bytes(int64_t M, int64_t K)
{
    WsLayout L;
    return ws_layout(M, K, &L) ? L.min_total : 0;
}

size_t w8a8_linear_workspace_bytes(int64_t M, int64_t N, int64_t K)
{
    WsLayout L;
    if (N < 1 || N > INT32_MAX || !ws_layout(M, K, &L)) return 0;
    const GemmPlan g = current_plan(M, N, K, INT64_MAX);
    return L.min_total + static_cast<size_t>(g.tail_units * g.pair) * kSlotBytes;
}

int w8a8_gemm_plan(int64_t M, int64_t N, int64_t K, int num_sms, int64_t max_slots, int64_t* plan)
{
    if (!plan || M < 1 || N < 1 || K < 1 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return 0;
    const int64_t slots = max_slots < 0 ? INT64_MAX : max_slots;
    const GemmPlan g = num_sms > 0 ? choose_plan(M, N, K, num_sms, num_sms / 2, slots) : current_plan(M, N, K, slots);
    plan[0] = g.dp_tiles;
    plan[1] = g.splits;
    plan[2] = g.tail_units;
    plan[3] = g.grid;
    plan[4] = g.pair;
    return 1;
}

void w8a8_debug_force_single_cta(int on) { g_force_single.store(on ? 1 : 0); }

int w8a8_gemm_form(int64_t M, int64_t N, int64_t K, int64_t* form)
{
    if (!form || M < 1 || N < 1 || K < 1 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return 0;
    KcPlan kp;
    int dno = 0;
    DeviceInfo* d = const_cast<DeviceInfo*>(device_info(&dno));
    if (d && ensure_gemm_ready(d)) {
        kp = current_kc_plan(d, M, N, K);
    } else if (g_force_form.load() != 0) {
        int cl[3][4];
        default_kc_clusters(148, cl);
        kp = plan_kcluster(M, N, K, 148, g_force_single.load() ? 0 : 74, cl, g_force_form.load() == 1,
                           g_force_bn.load(), g_force_ks.load());
    }
    form[0] = kp.bn != 0 ? 1 : 0;
    form[1] = kp.bn;
    form[2] = kp.ks;
    form[3] = kp.ctas;
    return 1;
}

void w8a8_debug_force_gemm_form(int form, int bn, int ks)
{
    g_force_form.store(form < 0 ? -1 : (form == 0 ? 0 : 1));
    g_force_bn.store(kc_width_index(bn) >= 0 ? bn : 0);
    g_force_ks.store(kc_size_index(ks) >= 0 ? ks : 0);
}

w8a8_status w8a8_linear_quant_stage(const void* X, int x_dtype, int64_t M, int64_t K, void* ws, size_t ws_bytes,
                                    void* stream)
{
    if (!X || M < 0 || K < 0) return W8A8_ERR_INVALID_ARG;
    if (x_dtype != W8A8_F32 && x_dtype != W8A8_BF16) return W8A8_ERR_DTYPE;
    if (M < 1 || M > INT32_MAX || K < 16 || K % 16 != 0 || K > W8A8_MAX_K) return W8A8_ERR_UNSUPPORTED_SHAPE;
    WsLayout L;
    if (!ws || !ws_layout(M, K, &L) || ws_bytes < L.min_total) return W8A8_ERR_WORKSPACE;
    if (!aligned(X, 16) || !aligned(ws, 16)) return W8A8_ERR_ALIGNMENT;
    if (!device_info(nullptr)) return W8A8_ERR_NO_DEVICE;
    uint8_t* w = ws_base(ws);
    return launch_quant<true>(X, x_dtype, M, K, w + L.codes_off, reinterpret_cast<float*>(w + L.sx_off),
                              reinterpret_cast<uint32_t*>(w + L.status_off), static_cast<cudaStream_t>(stream));
}

w8a8_status w8a8_linear_gemm_stage(int64_t M, int64_t K, const uint16_t* Wp, const float* sw, int64_t N,
                                   const void* bias, int bias_dtype, uint16_t* Y, void* ws, size_t ws_bytes,
                                   void* stream)
{
    if (!Wp || !sw || !Y || M < 0 || N < 0 || K < 0) return W8A8_ERR_INVALID_ARG;
    if (bias && bias_dtype != W8A8_F32 && bias_dtype != W8A8_BF16) return W8A8_ERR_DTYPE;
    if (guard_reasons(M, N, K, W8A8_BF16, bias ? bias_dtype : W8A8_F32) != 0) return W8A8_ERR_UNSUPPORTED_SHAPE;
    WsLayout L;
    if (!ws || !ws_layout(M, K, &L) || ws_bytes < L.min_total) return W8A8_ERR_WORKSPACE;
    if (!aligned(Wp, 16) || !aligned(Y, 16) || !aligned(ws, 16) || !aligned(sw, 16)) return W8A8_ERR_ALIGNMENT;
    if (bias && !aligned(bias, 16)) return W8A8_ERR_ALIGNMENT;
    int devno = 0;
    DeviceInfo* dev = const_cast<DeviceInfo*>(device_info(&devno));
    if (!dev) return W8A8_ERR_NO_DEVICE;
    uint8_t* w = ws_base(ws);
    const int bias_mode = bias ? (bias_dtype == W8A8_F32 ? 1 : 2) : 0;
    return launch_gemm<w8a8::kModeW8A8>(dev, reinterpret_cast<const uint16_t*>(w + L.codes_off), Wp, M, N, K,
                              reinterpret_cast<const float*>(w + L.sx_off), sw, bias, bias_mode, Y, w, L,
                              ws_slots(L, ws_bytes), static_cast<cudaStream_t>(stream));
}

w8a8_status w8a8_linear(const void* X, int x_dtype, int64_t M, int64_t K, const uint16_t* Wp, const float* sw,
                        int64_t N, const void* bias, int bias_dtype, uint16_t* Y, void* ws, size_t ws_bytes,
                        void* stream)
{
    // Validate everything the second stage needs before launching the first.
    if (!X || !Wp || !sw || !Y || M < 0 || N < 0 || K < 0) return W8A8_ERR_INVALID_ARG;
    if (x_dtype != W8A8_F32 && x_dtype != W8A8_BF16) return W8A8_ERR_DTYPE;
    if (bias && bias_dtype != W8A8_F32 && bias_dtype != W8A8_BF16) return W8A8_ERR_DTYPE;
    if (guard_reasons(M, N, K, x_dtype, bias ? bias_dtype : W8A8_F32) != 0) return W8A8_ERR_UNSUPPORTED_SHAPE;
    WsLayout L;
    if (!ws || !ws_layout(M, K, &L) || ws_bytes < L.min_total) return W8A8_ERR_WORKSPACE;
    if (!aligned(X, 16) || !aligned(Wp, 16) || !aligned(Y, 16) || !aligned(ws, 16) || !aligned(sw, 16))
        return W8A8_ERR_ALIGNMENT;
    if (bias && !aligned(bias, 16)) return W8A8_ERR_ALIGNMENT;
    if (M > 0 && N > 0 && K > 0) {
        int devno = 0;
        DeviceInfo* dev = const_cast<DeviceInfo*>(device_info(&devno));
        if (!dev) return W8A8_ERR_NO_DEVICE;
        if (!ensure_gemm_ready(dev)) return W8A8_ERR_CUDA;
        const int64_t head = fused_head_rows(dev, M, N, K, x_dtype, ws_slots(L, ws_bytes));
        if (head > 0) {
            // The head rows now (the launch also clears the workspace header,
            // which holds the row counters), the rest inside the GEMM.
            uint8_t* w = ws_base(ws);
            cudaStream_t s = static_cast<cudaStream_t>(stream);
            w8a8_status st = launch_quant<true>(X, x_dtype, head, K, w + L.codes_off,
                                                reinterpret_cast<float*>(w + L.sx_off),
                                                reinterpret_cast<uint32_t*>(w + L.status_off), s);
            if (st != W8A8_OK) return st;
            const int bias_mode = bias ? (bias_dtype == W8A8_F32 ? 1 : 2) : 0;
            return launch_gemm<w8a8::kModeW8A8Fused>(
                dev, reinterpret_cast<const uint16_t*>(w + L.codes_off), Wp, M, N, K,
                reinterpret_cast<const float*>(w + L.sx_off), sw, bias, bias_mode, Y, w, L, ws_slots(L, ws_bytes), s,
                nullptr, static_cast<const uint16_t*>(X), head);
        }
    }
    w8a8_status st = w8a8_linear_quant_stage(X, x_dtype, M, K, ws, ws_bytes, stream);
    if (st != W8A8_OK) return st;
    return w8a8_linear_gemm_stage(M, K, Wp, sw, N, bias, bias_dtype, Y, ws, ws_bytes, stream);
}

w8a8_status w8a8_gemm_s32(const int8_t* Xq, const uint16_t* Wp, int64_t M, int64_t N, int64_t K, int32_t* acc,
                          void* ws, size_t ws_bytes, void* stream)
{
    if (!Xq || !Wp || !acc || M < 0 || N < 0 || K < 0) return W8A8_ERR_INVALID_ARG;
    if (guard_reasons(M, N, K, W8A8_BF16, W8A8_F32) != 0) return W8A8_ERR_UNSUPPORTED_SHAPE;
    WsLayout L;
    if (!ws || !ws_layout(M, K, &L) || ws_bytes < L.min_total) return W8A8_ERR_WORKSPACE;
    if (!aligned(Xq, 16) || !aligned(Wp, 16) || !aligned(acc, 16) || !aligned(ws, 16))
        return W8A8_ERR_ALIGNMENT;
    int devno = 0;
    DeviceInfo* dev = const_cast<DeviceInfo*>(device_info(&devno));
    if (!dev) return W8A8_ERR_NO_DEVICE;
    uint8_t* w = ws_base(ws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t* status = reinterpret_cast<uint32_t*>(w + L.status_off);
    uint16_t* codes = reinterpret_cast<uint16_t*>(w + L.codes_off);
    w8a8_status st = launch_codes_to_bf16(Xq, codes, M * K, status, dev->num_sms, s);
    if (st != W8A8_OK) return st;
    return launch_gemm<w8a8::kModeS32>(dev, codes, Wp, M, N, K, nullptr, nullptr, nullptr, 0, acc, w, L,
                                       ws_slots(L, ws_bytes),
                             s);
}

w8a8_status w8a8_linear_host(const void* X_host, int x_dtype, int64_t M, int64_t K, const uint16_t* Wp,
                             const float* sw, int64_t N, const void* bias, int bias_dtype, uint16_t* Y_host,
                             void* X_dev, uint16_t* Y_dev, void* ws, size_t ws_bytes, int64_t chunk_rows,
                             void* stream)
{
    if (!X_host || !Y_host || !X_dev || !Y_dev || !Wp || !sw || M < 0 || N < 0 || K < 0 || chunk_rows < 0)
        return W8A8_ERR_INVALID_ARG;
    if (x_dtype != W8A8_F32 && x_dtype != W8A8_BF16) return W8A8_ERR_DTYPE;
    if (bias && bias_dtype != W8A8_F32 && bias_dtype != W8A8_BF16) return W8A8_ERR_DTYPE;
    if (guard_reasons(M, N, K, x_dtype, bias ? bias_dtype : W8A8_F32) != 0) return W8A8_ERR_UNSUPPORTED_SHAPE;
    // Row chunks: the copies of one chunk overlap the other chunks' compute
    // and copies in the other direction.  Default: about eight chunks of
    // whole 256-row tiles, with the first and the last chunk a third of
    // that (whole 128-row tiles): only the first chunk's copy in and the
    // last chunk's compute and copy out run without the other direction's
    // copies beside them.  A nonzero chunk_rows gives equal chunks.
    int64_t rows = chunk_rows;
    int64_t edge = 0;   // rows of the first and last chunk (0: equal chunks)
    if (rows == 0) {
        rows = ((M + 7) / 8 + 255) / 256 * 256;
        edge = rows / 3 / 128 * 128;
        if (edge < 128 || M <= rows + 2 * edge) edge = 0;
    }
    if ((M + rows - 1) / rows + 2 > kMaxHostChunks) {
        rows = (M + kMaxHostChunks - 3) / (kMaxHostChunks - 2);
        edge = 0;
    }
    WsLayout L;
    if (!ws || !ws_layout(rows < M ? rows : M, K, &L) || ws_bytes < L.min_total) return W8A8_ERR_WORKSPACE;
    if (!aligned(X_dev, 16) || !aligned(Y_dev, 16) || !aligned(Wp, 16) || !aligned(sw, 16) || !aligned(ws, 16))
        return W8A8_ERR_ALIGNMENT;
    if (bias && !aligned(bias, 16)) return W8A8_ERR_ALIGNMENT;
    int dev = -1;
    if (!device_info(&dev)) return W8A8_ERR_NO_DEVICE;
    HostPipe* hp = host_pipe(dev);
    if (!hp) return W8A8_ERR_CUDA;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t xe = x_dtype == W8A8_BF16 ? 2u : 4u;
    const size_t x_row = static_cast<size_t>(K) * xe, y_row = static_cast<size_t>(N) * 2u;
    auto fail = [](cudaError_t e) { return e != cudaSuccess; };
    // The copies start after the caller's earlier work on `stream` (which
    // may still use X_dev / Y_dev).
    if (fail(cudaEventRecord(hp->start, s)) || fail(cudaStreamWaitEvent(hp->h2d, hp->start, 0)) ||
        fail(cudaStreamWaitEvent(hp->d2h, hp->start, 0))) {
        cudaGetLastError();
        return W8A8_ERR_CUDA;
    }
    int c = 0;
    for (int64_t r0 = 0, mr = 0; r0 < M; r0 += mr, ++c) {
        const int64_t left = M - r0;
        if (edge > 0 && r0 == 0)
            mr = edge;                                   // first chunk
        else if (edge > 0 && left <= rows + edge && left > edge)
            mr = left - edge;                            // the chunk before the last
        else
            mr = left < rows ? left : rows;              // middle chunks, and the last
        const uint8_t* xh = static_cast<const uint8_t*>(X_host) + static_cast<size_t>(r0) * x_row;
        uint8_t* xd = static_cast<uint8_t*>(X_dev) + static_cast<size_t>(r0) * x_row;
        uint16_t* yd = Y_dev + static_cast<size_t>(r0) * static_cast<size_t>(N);
        uint16_t* yh = Y_host + static_cast<size_t>(r0) * static_cast<size_t>(N);
        if (fail(cudaMemcpyAsync(xd, xh, static_cast<size_t>(mr) * x_row, cudaMemcpyHostToDevice, hp->h2d)) ||
            fail(cudaEventRecord(hp->copied[c], hp->h2d)) || fail(cudaStreamWaitEvent(s, hp->copied[c], 0))) {
            cudaGetLastError();
            return W8A8_ERR_CUDA;
        }
        const w8a8_status st = w8a8_linear(xd, x_dtype, mr, K, Wp, sw, N, bias, bias_dtype, yd, ws, ws_bytes, s);
        if (st != W8A8_OK) return st;
        if (fail(cudaEventRecord(hp->computed[c], s)) || fail(cudaStreamWaitEvent(hp->d2h, hp->computed[c], 0)) ||
            fail(cudaMemcpyAsync(yh, yd, static_cast<size_t>(mr) * y_row, cudaMemcpyDeviceToHost, hp->d2h))) {
            cudaGetLastError();
            return W8A8_ERR_CUDA;
        }
    }
    // Later work on `stream` sees Y_host complete.
    if (fail(cudaEventRecord(hp->end, hp->d2h)) || fail(cudaStreamWaitEvent(s, hp->end, 0))) {
        cudaGetLastError();
        return W8A8_ERR_CUDA;
    }
    return W8A8_OK;
}

size_t w8a8_bf16_linear_workspace_bytes(int64_t M, int64_t N, int64_t K)
{
    if (bf16_guard_reasons(M, N, K, W8A8_BF16) != 0) return 0;
    WsLayout L;
    bf16_ws_layout(&L);
    const GemmPlan g = current_plan(M, N, K, INT64_MAX);
    return L.min_total + static_cast<size_t>(g.tail_units * g.pair) * kSlotBytes;
}

int w8a8_bf16_linear_supported(int64_t M, int64_t N, int64_t K, int bias_dtype, int* reason)
{
    const int r = bf16_guard_reasons(M, N, K, bias_dtype);
    if (reason) *reason = r;
    return r == 0 ? 1 : 0;
}

w8a8_status w8a8_bf16_linear(const uint16_t* X, int64_t M, int64_t K, const uint16_t* W, int64_t N,
                             const void* bias, int bias_dtype, uint16_t* Y, void* ws, size_t ws_bytes, void* stream)
{
    if (!X || !W || !Y || M < 0 || N < 0 || K < 0) return W8A8_ERR_INVALID_ARG;
    if (bias && bias_dtype != W8A8_F32 && bias_dtype != W8A8_BF16) return W8A8_ERR_DTYPE;
    if (bf16_guard_reasons(M, N, K, bias ? bias_dtype : W8A8_F32) != 0) return W8A8_ERR_UNSUPPORTED_SHAPE;
    WsLayout L;
    bf16_ws_layout(&L);
    if (!ws || ws_bytes < L.min_total) return W8A8_ERR_WORKSPACE;
    if (!aligned(X, 16) || !aligned(W, 16) || !aligned(Y, 16) || !aligned(ws, 16)) return W8A8_ERR_ALIGNMENT;
    if (bias && !aligned(bias, 16)) return W8A8_ERR_ALIGNMENT;
    int devno = 0;
    DeviceInfo* dev = const_cast<DeviceInfo*>(device_info(&devno));
    if (!dev) return W8A8_ERR_NO_DEVICE;
    uint8_t* w = ws_base(ws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // No quantiser runs first to clear the header: a one-CTA kernel does,
    // with the GEMM as its programmatic dependent.
    static_assert(w8a8::kHeaderWords * 4 == kAlign, "the header is one alignment unit");
    w8a8::clear_header_kernel<<<1, 256, 0, s>>>(reinterpret_cast<uint32_t*>(w + L.status_off));
    if (cudaGetLastError() != cudaSuccess) return W8A8_ERR_CUDA;
    const int bias_mode = bias ? (bias_dtype == W8A8_F32 ? 1 : 2) : 0;
    return launch_gemm<w8a8::kModeBf16>(dev, X, W, M, N, K, nullptr, nullptr, bias, bias_mode, Y, w, L,
                                        ws_slots(L, ws_bytes), s);
}

w8a8_status w8a8_quantize_qk_blocks(const void* X, int x_dtype, int64_t B, int64_t H, int64_t L, int64_t D,
                                    int layout, int64_t block_tokens, int8_t* Xq, float* scales, void* stream)
{
    if (B < 0 || H < 0 || L < 0 || D < 0 || block_tokens < 0) return W8A8_ERR_INVALID_ARG;
    if (layout != W8A8_LAYOUT_HND && layout != W8A8_LAYOUT_NHD) return W8A8_ERR_INVALID_ARG;
    if (x_dtype != W8A8_F32 && x_dtype != W8A8_BF16) return W8A8_ERR_DTYPE;
    if (B == 0 || H == 0 || L == 0) return W8A8_OK;
    if (!X || !Xq || !scales) return W8A8_ERR_INVALID_ARG;
    const int64_t E = x_dtype == W8A8_BF16 ? 8 : 4;
    if (D < E || D % E != 0 || D / E > 256 || block_tokens < 1 || L > INT32_MAX) return W8A8_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(X, 16) || !aligned(Xq, 16) || !aligned(scales, 4)) return W8A8_ERR_ALIGNMENT;
    w8a8::BlockGeom g;
    g.H = H;
    g.L = L;
    g.block_tokens = block_tokens < L ? block_tokens : L;
    g.nblk = (L + g.block_tokens - 1) / g.block_tokens;
    g.vd = static_cast<int32_t>(D / E);
    // Tokens per pass: as many as 256 threads cover (more warps per SM; a
    // form with up to 16 vectors per thread and fewer threads measured
    // slower at the video attention shape), or 512 threads for blocks of
    // 2048 vectors or more that then take at most 4 vectors a thread (the
    // persistent CTAs work through twice as many blocks, overlapping more of
    // the copies).
    int64_t cap = kBlockThreads / g.vd;
    const int64_t wide = kBlockThreadsWide / g.vd;
    if (g.vd * g.block_tokens >= kWideBlockVectors && (g.block_tokens + wide - 1) / wide <= 4) cap = wide;
    g.tpp = static_cast<int32_t>(cap < g.block_tokens ? cap : g.block_tokens);
    if (layout == W8A8_LAYOUT_HND) {
        g.stride_t = D;
        g.stride_h = L * D;
        g.stride_b = H * L * D;
    } else {
        g.stride_t = H * D;
        g.stride_h = D;
        g.stride_b = L * H * D;
    }
    // The scales follow (b, h, j) for the caller's nblk = ceil(L / block_tokens)
    // also when block_tokens > L (then one block per head).
    const int64_t blocks = B * H * g.nblk;
    if (blocks > INT32_MAX) return W8A8_ERR_UNSUPPORTED_SHAPE;
    const DeviceInfo* dev = device_info(nullptr);
    if (!dev) return W8A8_ERR_NO_DEVICE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (x_dtype == W8A8_BF16)
        return launch_blocks_typed<__nv_bfloat16>(static_cast<const __nv_bfloat16*>(X), g, blocks, Xq, scales, s);
    return launch_blocks_typed<float>(static_cast<const float*>(X), g, blocks, Xq, scales, s);
}

w8a8_status w8a8_norm_quantize_act(const uint16_t* X, int64_t M, int64_t K, int norm, float eps, const void* scale,
                                   const void* shift, int mod_dtype, uint16_t* Y_mod, int8_t* Xq, float* sx,
                                   void* stream)
{
    if (M == 0 && X && K >= 0) return W8A8_OK;
    w8a8::NormParams np;
    w8a8_status st = check_norm_args(X, M, K, norm, eps, scale, shift, mod_dtype, Y_mod, &np);
    if (st != W8A8_OK) return st;
    if (!Xq || !sx) return W8A8_ERR_INVALID_ARG;
    if (!aligned(Xq, 16) || !aligned(sx, 4)) return W8A8_ERR_ALIGNMENT;
    if (!device_info(nullptr)) return W8A8_ERR_NO_DEVICE;
    return launch_norm_quant<false>(X, M, K, norm, np, Xq, sx, nullptr, static_cast<cudaStream_t>(stream));
}

w8a8_status w8a8_norm_linear(const uint16_t* X, int64_t M, int64_t K, int norm, float eps, const void* scale,
                             const void* shift, int mod_dtype, const uint16_t* Wp, const float* sw, int64_t N,
                             const void* bias, int bias_dtype, uint16_t* Y, void* ws, size_t ws_bytes, void* stream)
{
    w8a8::NormParams np;
    w8a8_status st = check_norm_args(X, M, K, norm, eps, scale, shift, mod_dtype, nullptr, &np);
    if (st != W8A8_OK) return st;
    if (!Wp || !sw || !Y || N < 0) return W8A8_ERR_INVALID_ARG;
    if (bias && bias_dtype != W8A8_F32 && bias_dtype != W8A8_BF16) return W8A8_ERR_DTYPE;
    if (guard_reasons(M, N, K, W8A8_BF16, bias ? bias_dtype : W8A8_F32) != 0) return W8A8_ERR_UNSUPPORTED_SHAPE;
    WsLayout L;
    if (!ws || !ws_layout(M, K, &L) || ws_bytes < L.min_total) return W8A8_ERR_WORKSPACE;
    if (!aligned(Wp, 16) || !aligned(Y, 16) || !aligned(ws, 16) || !aligned(sw, 16)) return W8A8_ERR_ALIGNMENT;
    if (bias && !aligned(bias, 16)) return W8A8_ERR_ALIGNMENT;
    int devno = 0;
    DeviceInfo* dev = const_cast<DeviceInfo*>(device_info(&devno));
    if (!dev) return W8A8_ERR_NO_DEVICE;
    uint8_t* w = ws_base(ws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = launch_norm_quant<true>(X, M, K, norm, np, w + L.codes_off, reinterpret_cast<float*>(w + L.sx_off),
                                 reinterpret_cast<uint32_t*>(w + L.status_off), s);
    if (st != W8A8_OK) return st;
    return launch_gemm<w8a8::kModeW8A8>(dev, reinterpret_cast<const uint16_t*>(w + L.codes_off), Wp, M, N, K,
                                        reinterpret_cast<const float*>(w + L.sx_off), sw, bias,
                                        bias ? (bias_dtype == W8A8_F32 ? 1 : 2) : 0, Y, w, L, ws_slots(L, ws_bytes), s);
}

size_t w8a8_mlp_workspace_bytes(int64_t M, int64_t K, int64_t F, int64_t N)
{
    if (guard_reasons(M, F, K, W8A8_BF16, W8A8_BF16) != 0 || guard_reasons(M, N, F, W8A8_BF16, W8A8_BF16) != 0)
        return 0;
    MlpLayout L;
    if (!mlp_layout(M, K, F, &L)) return 0;
    const GemmPlan gu = current_plan(M, F, K, INT64_MAX);
    const GemmPlan gd = current_plan(M, N, F, INT64_MAX);
    const int64_t su = gu.tail_units * gu.pair, sd = gd.tail_units * gd.pair;
    return L.up.min_total + static_cast<size_t>(su > sd ? su : sd) * kSlotBytes;
}

w8a8_status w8a8_mlp(const void* X, int x_dtype, int64_t M, int64_t K, const uint16_t* Wp_up, const float* sw_up,
                     int64_t F, const void* bias_up, int bias_up_dtype, const uint16_t* Wp_down,
                     const float* sw_down, int64_t N, const void* bias_down, int bias_down_dtype, uint16_t* H,
                     uint16_t* Y, void* ws, size_t ws_bytes, void* stream)
{
    if (!X || !Wp_up || !sw_up || !Wp_down || !sw_down || !H || !Y || M < 0 || K < 0 || F < 0 || N < 0)
        return W8A8_ERR_INVALID_ARG;
    if (x_dtype != W8A8_F32 && x_dtype != W8A8_BF16) return W8A8_ERR_DTYPE;
    if (bias_up && bias_up_dtype != W8A8_F32 && bias_up_dtype != W8A8_BF16) return W8A8_ERR_DTYPE;
    if (bias_down && bias_down_dtype != W8A8_F32 && bias_down_dtype != W8A8_BF16) return W8A8_ERR_DTYPE;
    if (guard_reasons(M, F, K, x_dtype, bias_up ? bias_up_dtype : W8A8_F32) != 0 ||
        guard_reasons(M, N, F, W8A8_BF16, bias_down ? bias_down_dtype : W8A8_F32) != 0)
        return W8A8_ERR_UNSUPPORTED_SHAPE;
    MlpLayout L;
    if (!ws || !mlp_layout(M, K, F, &L) || ws_bytes < L.up.min_total) return W8A8_ERR_WORKSPACE;
    if (!aligned(X, 16) || !aligned(Wp_up, 16) || !aligned(sw_up, 16) || !aligned(Wp_down, 16) ||
        !aligned(sw_down, 16) || !aligned(H, 16) || !aligned(Y, 16) || !aligned(ws, 16))
        return W8A8_ERR_ALIGNMENT;
    if ((bias_up && !aligned(bias_up, 16)) || (bias_down && !aligned(bias_down, 16))) return W8A8_ERR_ALIGNMENT;
    int devno = 0;
    DeviceInfo* dev = const_cast<DeviceInfo*>(device_info(&devno));
    if (!dev) return W8A8_ERR_NO_DEVICE;
    uint8_t* w = ws_base(ws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t* header = reinterpret_cast<uint32_t*>(w + L.up.status_off);
    uint32_t* amax = reinterpret_cast<uint32_t*>(w + L.amax_off);
    float* sxh = reinterpret_cast<float*>(w + L.sxh_off);
    uint16_t* codesh = reinterpret_cast<uint16_t*>(w + L.codesh_off);
    const int64_t slots = ws_slots(L.up, ws_bytes);
    // 1. the up layer's activation codes; also clears the header and the
    //    row maxima the up GEMM gathers
    w8a8_status st = launch_quant<true>(X, x_dtype, M, K, w + L.up.codes_off, reinterpret_cast<float*>(w + L.up.sx_off),
                                        header, s, amax);
    if (st != W8A8_OK) return st;
    // 2. H = up layer, with each row's max |H|
    st = launch_gemm<w8a8::kModeW8A8RowMax>(dev, reinterpret_cast<const uint16_t*>(w + L.up.codes_off), Wp_up, M, F, K,
                                      reinterpret_cast<const float*>(w + L.up.sx_off), sw_up, bias_up,
                                      bias_up ? (bias_up_dtype == W8A8_F32 ? 1 : 2) : 0, H, w, L.up, slots, s, amax);
    if (st != W8A8_OK) return st;
    // 3. the down layer's codes from H and the gathered maxima (no reduction)
    st = launch_codes_known_amax(H, M, F, amax, codesh, sxh, s);
    if (st != W8A8_OK) return st;
    // 4. Y = down layer
    return launch_gemm<w8a8::kModeW8A8>(dev, codesh, Wp_down, M, N, F, sxh, sw_down, bias_down,
                                        bias_down ? (bias_down_dtype == W8A8_F32 ? 1 : 2) : 0, Y, w, L.up, slots, s);
}

w8a8_status w8a8_read_status(const void* ws, void* stream, uint32_t* device_bits)
{
    if (!ws || !device_bits) return W8A8_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    if (cudaMemcpyAsync(&v, ws_base(ws), sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return W8A8_ERR_CUDA;
    }
    *device_bits = v;
    return v == 0 ? W8A8_OK : W8A8_ERR_TIMEOUT;
}

}  // extern "C"
