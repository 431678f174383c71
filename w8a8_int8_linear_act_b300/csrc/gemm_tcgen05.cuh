// INT8 x INT8 -> INT32 GEMM with the fused W8A8 epilogue on sm_103a tensor
// cores (zhidx TurboT2VA article, section 01 item 3 "量化策略": INT32
// accumulation, then row scale x channel scale and bias applied once).
//
// sm_103a has no tcgen05 integer MMA (kind::i8 is sm_100a/sm_101a only), so
// the operands are the INT8 codes carried exactly as bf16 values and the MMA
// is tcgen05 kind::f16 with an fp32 accumulator in tensor memory.  Products
// are at most 127^2 = 16129; a K-chunk of at most 1024 keeps every partial sum
// below 1024 * 16129 < 2^24, so every value the accumulator holds is an
// integer that fp32 represents exactly.  After each chunk the epilogue warps
// drain the accumulator (tcgen05.ld), convert it exactly to int32 and add it
// to running INT32 sums in registers; the sums equal the exact INT32
// accumulator.  After the last chunk they apply
//   Y = bf16_rne(((float)acc * sx[m]) * sw[n] + bias[n])
// and store the tile (or store acc itself, for the INT32 test entry point).
//
// Two forms, one persistent CTA per SM either way (10 warps):
//   kPair = 1  a CTA owns a 128 x 256 output tile; per 64-deep k-block it
//              loads A 128 x 64 and B 256 x 64 (48 KB, 4-stage ring) and
//              issues tcgen05.mma.cta_group::1 128x256x16.
//   kPair = 2  a cluster of two CTAs owns a 256 x 256 tile; each CTA loads
//              its 128 rows of A and 128 of the 256 rows of B (32 KB,
//              5-stage ring), and the even CTA issues tcgen05.mma.cta_group::2
//              256x256x16, which reads both CTAs' shared memory and leaves
//              each CTA's 128 rows of the accumulator in its own tensor
//              memory.  Per SM this moves 2/3 of the operand bytes of the
//              single-CTA form for the same MMA work, which is what keeps
//              the tensor pipe fed when every SM streams operands at once.
// Roles: warp 0 TMA producer; warp 1 tensor-memory owner and (in the leader
// CTA) the single MMA-issuing thread; warps 2-9 epilogue, warp w reading
// TMEM lanes 32*(w%4)..+31 (its rows) and one 128-column half of the tile.
// Two 256-column fp32 accumulators let the MMA fill one chunk while the
// epilogue drains the other.  In a pair, both CTAs' copies complete on the
// leader's "full" barrier, which the leader's producer alone arms with the
// bytes of both (the barrier's transaction count may run below zero while
// the peer's bytes land first); the leader's commits arrive on both CTAs'
// barriers, and both CTAs' epilogues release the leader's accumulator.
//
// Work units.  The host plans the tiles as whole-tile units dealt round-robin
// to the workers (CTAs, or CTA pairs), except that when the last wave would
// leave most of them idle (tiles % workers at most half of the workers), its
// tiles are cut along K into `splits` segments, one per worker.  A segment
// writes its INT32 partial (each CTA its own 128 rows) to the workspace,
// fences, and counts itself in on the arrival counter of its (tile, CTA
// rank); the segment that arrives last adds the other partials to its own
// (INT32 addition is exact and associative, so the sum is the exact
// accumulator) and runs the epilogue, then resets the counter.  No CTA ever
// waits for another CTA's segment.
//
// Other modes (kMode below): the INT32 sums themselves (a test entry point);
// bf16 activations and weights with fp32 sums, the native BF16 linear (one
// tensor-memory accumulation per unit, split partials added in segment
// order); and the W8A8 epilogue that also gathers each row's max |Y| for
// the next layer's activation scale (the MLP pair).  The kernel waits for
// the kernel before it (programmatic dependent launch) only after its
// set-up, and lets the kernel after it launch at the same point.
//
// Every mbarrier wait is bounded by a wall-clock limit; a wait that runs out
// sets a bit in the status word and the CTA unwinds (waiting, again with a
// limit, for its own copies and MMAs in flight) and frees its tensor memory.
// A pair meets at a cluster barrier after set-up and before tear-down; every
// path through the kernel reaches both.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "ptx_sm103.cuh"
#include "quant_rows.cuh"

namespace w8a8 {

constexpr int kBM = 128;   // output rows per CTA
constexpr int kBN = 256;   // output columns per tile
constexpr int kBK = 64;    // 64 bf16 = 128 bytes = one swizzle row
constexpr int kEpiWarps = 8;
constexpr int kGemmThreads = 64 + 32 * kEpiWarps;
constexpr int kUmmaK = 16;
constexpr uint32_t kTmemCols = 2 * kBN;  // two fp32 accumulators
constexpr int kMaxKbPerChunk = 16;       // 16 * 64 = 1024: 1024 * 127^2 < 2^24
constexpr int kPartialInt4 = kBM * kBN / 4;  // one CTA's INT32 partial tile, in 16-byte vectors
constexpr int kEpiBarrier = 1;               // named barrier of the epilogue warps

template <int kPair>
struct GemmCfg {
    static constexpr int kTileRows = kBM * kPair;                     // output rows per tile
    static constexpr int kBRows = kBN / kPair;                        // rows of B each CTA loads
    static constexpr uint32_t kAStageBytes = kBM * kBK * 2;
    static constexpr uint32_t kBStageBytes = kBRows * kBK * 2;
    static constexpr uint32_t kStageBytes = kAStageBytes + kBStageBytes;
    static constexpr int kStages = kPair == 2 ? 5 : 4;
    // Pair form: a 5-stage ring (the ring depth is what keeps the tensor
    // pipe fed: 3 stages ran 170 us, 4 stages 150 us, 5 stages 139 us on the
    // 6144 x 4096 x 4096 projection), and the bf16 output staged in shared
    // memory, one 32-row x 64-column 128-byte-swizzled box per epilogue warp
    // at a time, written by TMA stores.
    static constexpr uint32_t kStagingBytes = kPair == 2 ? kEpiWarps * 4096 : 0;
    static constexpr uint32_t kParamBytes = 2 * kBN * 4;            // the tile's sw and bias, fp32
    static constexpr size_t kSmemBytes =
        1024 /* alignment slack */ + kStages * kStageBytes + kStagingBytes + kParamBytes + 512 /* barriers */;
};
static_assert(GemmCfg<1>::kSmemBytes <= 227 * 1024 && GemmCfg<2>::kSmemBytes <= 227 * 1024, "shared memory");
// Split fix-up: each epilogue warp streams its region of the other
// segments' partial tiles through kFixSlots slots of kFixSlotBytes in the
// idle operand ring (and output staging), kFixWarpBytes per warp.
constexpr int kFixSlots = 3;
constexpr uint32_t kFixSlotBytes = 8192;                        // half of a warp's 16 KB region of a partial
constexpr uint32_t kFixWarpBytes = kFixSlots * kFixSlotBytes;
static_assert(kEpiWarps * kFixWarpBytes <= GemmCfg<2>::kStages * GemmCfg<2>::kStageBytes +
                                               GemmCfg<2>::kStagingBytes &&
                  kEpiWarps * kFixWarpBytes <= GemmCfg<1>::kStages * GemmCfg<1>::kStageBytes,
              "fix-up slots fit in the ring and staging");
static_assert((2 * GemmCfg<2>::kStages + 7 + kEpiWarps * kFixSlots) * 8 <= 512 &&
                  (2 * GemmCfg<1>::kStages + 7 + kEpiWarps * kFixSlots) * 8 <= 512,
              "barrier area");
static_assert(GemmCfg<1>::kStages * GemmCfg<1>::kStageBytes >= kPartialInt4 * 16 &&
                  GemmCfg<2>::kStages * GemmCfg<2>::kStageBytes >= kPartialInt4 * 16,
              "a partial tile fits in the operand ring");

// What the kernel computes after the K loop:
//   kModeW8A8  INT8 codes in, exact INT32 sums, Y = bf16(((float)acc*sx)*sw + b)
//   kModeS32   INT8 codes in, the exact INT32 sums themselves
//   kModeBf16  bf16 activations and weights in (the native BF16 linear that
//              guard-rejected shapes and BF16 layers run), fp32 sums (the
//              tensor memory chunks added in fp32), Y = bf16(acc + b)
//   kModeW8A8RowMax  kModeW8A8, and each row's max |Y| gathered into
//              p.row_amax (the next layer's activation scale, MLP pair)
//   kModeW8A8Fused  kModeW8A8 whose own extra warps quantise the activation
//              rows [p.q_row0, M) while the GEMM runs (the rows below q_row0
//              come from the quantiser launched before it); the producers
//              wait for their rows (K = 4096, bf16 X, CTA pairs)
constexpr int kModeW8A8 = 0;
constexpr int kModeS32 = 1;
constexpr int kModeBf16 = 2;
constexpr int kModeW8A8RowMax = 3;
constexpr int kModeW8A8Fused = 4;

// Threads of a GEMM CTA: producer, MMA issuer and the epilogue warps, and in
// kModeW8A8Fused two quantiser warps (12 warps x 32 x 168 registers still
// fit the register file, three warps per sub-partition).
constexpr int kFusedQuantWarps = 2;
__host__ __device__ constexpr int gemm_threads(int mode)
{
    return kGemmThreads + (mode == kModeW8A8Fused ? 32 * kFusedQuantWarps : 0);
}
constexpr int kFusedQuantK = 4096;   // row length the quantiser warps take (16 vectors a lane)

// Status bits (same values as W8A8_DEV_* in the public header).
constexpr uint32_t kDevTimeoutProducer = 0x1;
constexpr uint32_t kDevTimeoutMma = 0x2;
constexpr uint32_t kDevTimeoutEpilogue = 0x4;
constexpr uint32_t kDevTimeoutTeardown = 0x8;

struct GemmParams {
    int32_t M, N, K;
    int32_t kb_per_chunk;      // k-blocks of 64 per TMEM accumulation (INT8 codes: 1..16, exact)
    int32_t group_m;           // tile rasterisation: m-tiles per group
    int32_t bias_mode;         // 0 none, 1 fp32, 2 bf16
    int32_t dp_tiles;          // tiles [0, dp_tiles) are whole-tile units, round-robin over the CTAs
    int32_t splits;            // K-segments per remaining tile (1: no split)
    int32_t tail_units;        // (tiles - dp_tiles) * splits; unit u runs on worker u
    const float* sx;           // [M]
    const float* sw;           // [N]
    const void* bias;          // [N] or nullptr
    void* out;                 // bf16 Y [M][N] or int32 acc [M][N]
    uint32_t* status;          // device status word
    uint32_t* tile_counters;   // [(tiles - dp_tiles) * kPair] arrivals per split (tile, CTA rank)
    int4* partials;            // [tail_units * kPair][kPartialInt4] INT32 partial tiles
    uint32_t* row_amax;        // [M] (kModeW8A8RowMax): each row's max |Y| as fp32 bits, by atomicMax
    uint64_t wait_limit_ns;
    int32_t skip_loads;        // test hook: producer issues no copies
    // kModeW8A8Fused: the bf16 activation, its code and scale buffers (the
    // ones the A tensor map and sx point at), the first row the quantiser
    // warps take (a multiple of 256), and per 256-row tile the number of its
    // rows finished.  status[1] counts rows claimed from q_row0 on.
    const __nv_bfloat16* qx;
    uint16_t* qcodes;
    float* qsx;
    int32_t q_row0;
    uint32_t* q_ready;
};

__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int group_m, int& mb, int& nb)
{
    const int per_group = group_m * tiles_n;
    const int g = t / per_group;
    const int first_m = g * group_m;
    const int gsz = min(tiles_m - first_m, group_m);
    const int r = t - g * per_group;
    mb = first_m + r % gsz;
    nb = r / gsz;
}

// One unit of work: k-blocks [kb0, kb1) of one output tile.  slot < 0 for a
// whole tile; otherwise the tile is split and slot is the unit's partial slot.
struct Unit {
    int tile, kb0, kb1, slot;
};

// The i-th unit of worker `w` of `W` (false once there are no more).
__device__ __forceinline__ bool worker_unit(const GemmParams& p, int num_kb, int w, int W, int i, Unit& u)
{
    const int n_dp = w < p.dp_tiles ? (p.dp_tiles - w + W - 1) / W : 0;
    if (i < n_dp) {
        u.tile = w + i * W;
        u.kb0 = 0;
        u.kb1 = num_kb;
        u.slot = -1;
        return true;
    }
    if (i == n_dp && w < p.tail_units) {
        const int seg = w % p.splits;
        u.tile = p.dp_tiles + w / p.splits;
        u.kb0 = static_cast<int>(static_cast<int64_t>(seg) * num_kb / p.splits);
        u.kb1 = static_cast<int>(static_cast<int64_t>(seg + 1) * num_kb / p.splits);
        u.slot = w;
        return true;
    }
    return false;
}

// kModeW8A8Fused: one quantiser warp.  Rows q_row0 + 0, 1, ... are claimed
// in order (status[1]); a row is held in registers (16 vectors a lane),
// reduced, coded by the row rule of quant_rows.cuh and its scale written,
// then counted into its 256-row tile's q_ready word (a fence, then the
// add: release).  The next claim is taken while the current row is worked
// on.  Any resident CTA makes progress on any row, and no quantiser warp
// waits on another, so the producers that wait for a tile's rows never wait
// on a CTA that is not running.
__device__ __forceinline__ void fused_quant_warp(const GemmParams& p)
{
    constexpr int NV = kFusedQuantK / 8 / 32;
    using IV = InVec<__nv_bfloat16>;
    const int lane = static_cast<int>(threadIdx.x & 31);
    uint32_t* claimed = p.status + 1;
    uint32_t claim = 0;
    if (lane == 0) claim = atomicAdd(claimed, 1u);
    claim = __shfl_sync(0xFFFFFFFFu, claim, 0);
    while (static_cast<int64_t>(p.q_row0) + claim < p.M) {
        const int64_t row = static_cast<int64_t>(p.q_row0) + claim;
        uint32_t next = 0;
        if (lane == 0) next = atomicAdd(claimed, 1u);
        const uint4* src = reinterpret_cast<const uint4*>(p.qx + row * kFusedQuantK);
        uint4 v[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) v[i] = load_stream(src + lane + 32 * i);
        uint32_t m2 = 0;
#pragma unroll
        for (int i = 0; i < NV; ++i) IV::absmax(v[i], m2);
        const RowScale rs = row_scale(warp_max(IV::absmax_value(m2)));
        if (lane == 0) p.qsx[row] = rs.s;
        const int64_t out0 = row * kFusedQuantK;
        if (rs.corr) {
#pragma unroll
            for (int i = 0; i < NV; ++i)
                quantize_vector_corr<true>(v[i], rs, p.qcodes, out0 + static_cast<int64_t>(lane + 32 * i) * 8);
        } else {
            quantize_strided_by_tie_test<__nv_bfloat16, true>(p.qx, out0 + lane * 8, 32 * 8, NV, rs, p.qcodes);
        }
        __syncwarp();
        if (lane == 0) {
            __threadfence();   // this row's codes and scale before its count
            atomicAdd(p.q_ready + (row >> 8), 1u);
        }
        claim = __shfl_sync(0xFFFFFFFFu, next, 0);
    }
}

// kModeW8A8Fused: waits until the 256-row tile `t` (t * 256 >= q_row0) has
// all its rows, with acquire semantics.
__device__ __forceinline__ bool fused_tile_ready(const GemmParams& p, int t, uint64_t limit)
{
    const uint32_t rows = static_cast<uint32_t>(min(256, p.M - t * 256));
    return wait_counter_ge(p.q_ready + t, rows, limit);
}

__device__ __forceinline__ void epi_barrier()
{
    asm volatile("bar.sync %0, %1;" ::"n"(kEpiBarrier), "n"(32 * kEpiWarps) : "memory");
}

template <int kMode, int kPair>
__global__ void __launch_bounds__(gemm_threads(kMode), 1)
    gemm_w8a8_tcgen05_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                             const __grid_constant__ CUtensorMap tmap_y, const GemmParams p)
{
    using C = GemmCfg<kPair>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t* sA = smem;
    uint8_t* sB = smem + S * C::kAStageBytes;
    uint8_t* sOut = smem + S * C::kStageBytes;                      // pair form: output staging
    float* s_sw = reinterpret_cast<float*>(sOut + C::kStagingBytes);  // [kBN] this tile's sw
    float* s_bias = s_sw + kBN;                                      // [kBN] this tile's bias
    uint64_t* bars = reinterpret_cast<uint64_t*>(s_bias + kBN);
    uint64_t* full = bars;                    // [S] TMA -> MMA (the leader's counts both CTAs' bytes)
    uint64_t* empty = bars + S;               // [S] MMA -> TMA
    uint64_t* tfull = bars + 2 * S;           // [2] MMA -> epilogue
    uint64_t* tempty = tfull + 2;             // [2] epilogue -> MMA (the leader's counts both CTAs)
    uint64_t* done = tempty + 2;              // MMA teardown
    uint64_t* peerbar = done + 1;             // pair teardown: the peer's count of issued loads has arrived
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(peerbar + 1);
    uint32_t* peer_issued = tmem_holder + 1;  // pair teardown: loads the peer's producer issued
    uint64_t* fixbars = peerbar + 2;          // [kEpiWarps][kFixSlots] split fix-up: a slot's copy landed
    __shared__ int s_last_arrival;
    __shared__ int s_fix_status;   // split fix-up: 0 every copy landed, 1 a copy timed out
    __shared__ int s_chunk_ready[2];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = kPair == 2 ? cluster_ctarank() : 0u;
    const int worker = kPair == 2 ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
    const int workers = kPair == 2 ? static_cast<int>(cluster_count_x()) : static_cast<int>(gridDim.x);
    const int tiles_m = (p.M + C::kTileRows - 1) / C::kTileRows;
    const int tiles_n = (p.N + kBN - 1) / kBN;
    const int num_kb = (p.K + kBK - 1) / kBK;
    const uint64_t limit = p.wait_limit_ns;
    constexpr uint16_t kBoth = kPair == 2 ? 0x3 : 0x1;
    constexpr bool kOutS32 = kMode == kModeS32;
    constexpr bool kFp32Sums = kMode == kModeBf16;   // sums held as fp32 bit patterns (zero bits = +0.0f)
    constexpr bool kRowMax = kMode == kModeW8A8RowMax;
    constexpr bool kFusedQuant = kMode == kModeW8A8Fused;
    constexpr bool kScaled = kMode == kModeW8A8 || kRowMax || kFusedQuant;   // INT8 codes dequantised by sx and sw

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], kPair * kEpiWarps);
        }
        mbar_init(done, 1);
        mbar_init(peerbar, 1);
        for (int i = 0; i < kEpiWarps * kFixSlots; ++i) mbar_init(&fixbars[i], 1);
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_a);
        tma_prefetch_desc(&tmap_b);
        if constexpr (kPair == 2 && !kOutS32) tma_prefetch_desc(&tmap_y);
    }
    if (warp == 1) {
        tmem_alloc<kPair>(tmem_holder, kTmemCols);
        tmem_relinquish<kPair>();
    }
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (kPair == 2) cluster_sync_all();   // both CTAs' barriers exist before any remote use
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_holder;
    // Launched as a programmatic dependent of the kernel that writes the
    // activation codes, row scales and the workspace header: the set-up
    // above overlaps its tail, nothing below may run before it completes.
    grid_wait_prerequisites();
    // A kernel that consumes this one's output (the row quantiser of the
    // next layer) may be scheduled now; it waits for this grid to finish.
    grid_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t it = 0;
            uint32_t n_issued = 0;   // loads issued, for iterations 0 .. n_issued - 1
            bool ok = true;
            Unit u;
            for (int ui = 0; ok && worker_unit(p, num_kb, worker, workers, ui, u); ++ui) {
                int mb, nb;
                tile_coords(u.tile, tiles_m, tiles_n, p.group_m, mb, nb);
                const int a_row = (mb * kPair + static_cast<int>(rank)) * kBM;
                const int b_row = nb * kBN + static_cast<int>(rank) * C::kBRows;
                if constexpr (kFusedQuant) {
                    // The tile's rows must be quantised first.
                    const int t256 = (mb * kPair * kBM) >> 8;
                    if (t256 * 256 >= p.q_row0) {
                        if (!fused_tile_ready(p, t256, limit)) {
                            atomicOr(p.status, kDevTimeoutProducer);
                            ok = false;
                            break;
                        }
                        fence_proxy_async_global();   // the copies below read what generic stores wrote
                    }
                }
                for (int kb = u.kb0; kb < u.kb1; ++kb, ++it) {
                    const int s = static_cast<int>(it % S);
                    const uint32_t ph = (it / S) & 1u;
                    if (!mbar_wait(&empty[s], ph ^ 1u, limit)) {
                        atomicOr(p.status, kDevTimeoutProducer);
                        ok = false;
                        break;
                    }
                    if (p.skip_loads) continue;
                    if constexpr (kPair == 2) {
                        const uint32_t bar = cluster_map(&full[s], 0);
                        if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * C::kStageBytes);
                        tma_load_2d_pair(sA + s * C::kAStageBytes, &tmap_a, bar, kb * kBK, a_row);
                        tma_load_2d_pair(sB + s * C::kBStageBytes, &tmap_b, bar, kb * kBK, b_row);
                    } else {
                        mbar_arrive_expect_tx(&full[s], C::kStageBytes);
                        tma_load_2d(sA + s * C::kAStageBytes, &tmap_a, &full[s], kb * kBK, a_row);
                        tma_load_2d(sB + s * C::kBStageBytes, &tmap_b, &full[s], kb * kBK, b_row);
                    }
                    n_issued = it + 1;
                }
            }
            // Copies still in flight must land before the CTA exits.  Both
            // producers walk the same sequence of (stage, phase) and issue
            // the loads of iterations 0 .. n - 1, but after a timed-out wait
            // the two counts can differ (by at most S: a producer issues
            // iteration i only after the MMA consumed iteration i - S, which
            // both CTAs had loaded).  In a pair every copy, the peer's too,
            // completes on the leader's "full" barriers, so the peer sends
            // its count to the leader, which then balances each phase the
            // two did not both load:
            //   loaded by the peer alone: armed now with the peer's bytes
            //     (that stage's previous phase is complete: the MMA
            //     consumed it before the peer could reuse the stage);
            //   loaded by the leader alone: the missing peer bytes are
            //     counted as complete;
            // and waits for the last phase of every stage either issued.
            // The peer stays until the closing cluster barrier, which the
            // leader reaches only after these waits.
            uint32_t n_all = n_issued;
            if constexpr (kPair == 2) {
                if (rank != 0) {
                    st_cluster_u32(cluster_map(peer_issued, 0), n_issued);
                    mbar_arrive_release_cluster(cluster_map(peerbar, 0));
                } else {
                    uint32_t n_peer = n_issued;
                    if (mbar_wait_cluster(peerbar, 0, limit))
                        n_peer = *reinterpret_cast<volatile uint32_t*>(peer_issued);
                    else
                        atomicOr(p.status, kDevTimeoutTeardown);
                    for (uint32_t i = n_issued; i < n_peer; ++i)
                        mbar_arrive_expect_tx(&full[i % S], C::kStageBytes);
                    for (uint32_t i = n_peer; i < n_issued; ++i) mbar_complete_tx(&full[i % S], C::kStageBytes);
                    n_all = n_peer > n_issued ? n_peer : n_issued;
                }
            }
            if (rank == 0)
                for (uint32_t i = n_all > static_cast<uint32_t>(S) ? n_all - S : 0u; i < n_all; ++i)
                    if (!mbar_wait(&full[i % S], (i / S) & 1u, limit)) atomicOr(p.status, kDevTimeoutTeardown);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader CTA)
        if (lane == 0 && rank == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(C::kTileRows, kBN);
            uint32_t it = 0, cc = 0;
            bool ok = true;
            Unit u;
            for (int ui = 0; ok && worker_unit(p, num_kb, worker, workers, ui, u); ++ui) {
                for (int kc0 = u.kb0; kc0 < u.kb1 && ok; kc0 += p.kb_per_chunk, ++cc) {
                    const uint32_t b = cc & 1u;
                    const uint32_t bph = (cc >> 1) & 1u;
                    if (!mbar_wait(&tempty[b], bph ^ 1u, limit)) {
                        atomicOr(p.status, kDevTimeoutMma);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t d_tmem = tmem_base + b * kBN;
                    const int kc1 = min(u.kb1, kc0 + p.kb_per_chunk);
                    for (int kb = kc0; kb < kc1; ++kb, ++it) {
                        const int s = static_cast<int>(it % S);
                        const uint32_t ph = (it / S) & 1u;
                        if (!mbar_wait(&full[s], ph, limit)) {
                            atomicOr(p.status, kDevTimeoutMma);
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        const uint32_t a0 = smem_addr(sA + s * C::kAStageBytes);
                        const uint32_t b0 = smem_addr(sB + s * C::kBStageBytes);
#pragma unroll
                        for (int k = 0; k < kBK / kUmmaK; ++k) {
                            mma_bf16<kPair>(d_tmem, smem_desc_k128(a0 + k * kUmmaK * 2),
                                            smem_desc_k128(b0 + k * kUmmaK * 2), idesc,
                                            (kb > kc0 || k > 0) ? 1u : 0u);
                        }
                        mma_commit<kPair>(&empty[s], kBoth);
                    }
                    if (ok) mma_commit<kPair>(&tfull[b], kBoth);
                }
            }
            // Every MMA issued must complete before tensor memory is freed.
            mma_commit<kPair>(done, 0x1);
            if (!mbar_wait(done, 0, limit)) atomicOr(p.status, kDevTimeoutTeardown);
        }
    } else if (kFusedQuant && warp >= 2 + kEpiWarps) {
        // ------------------------------------------------------------ activation rows
        fused_quant_warp(p);
    } else {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;        // TMEM lanes this warp may read
        const int half = (warp - 2) >> 2;    // which 128 columns of the tile
        const int e = warp - 2;              // epilogue warp index, 0..7
        uint32_t cc = 0;
        bool ok = true;
        Unit u;
        for (int ui = 0; ok && worker_unit(p, num_kb, worker, workers, ui, u); ++ui) {
            int mb, nb;
            tile_coords(u.tile, tiles_m, tiles_n, p.group_m, mb, nb);
            const int m = (mb * kPair + static_cast<int>(rank)) * kBM + quarter * 32 + lane;
            const int n0 = nb * kBN + half * 128;
            // The tile's column parameters, one column per epilogue thread,
            // fetched now so that their latency hides behind the K loop.
            epi_barrier();   // the previous unit's epilogue is done reading them
            float sxm = 0.0f;
            if constexpr (!kOutS32) {
                const int i = e * 32 + lane;
                const int n = nb * kBN + i;
                if constexpr (kScaled) s_sw[i] = n < p.N ? p.sw[n] : 0.0f;
                if (p.bias_mode == 1)
                    s_bias[i] = n < p.N ? static_cast<const float*>(p.bias)[n] : 0.0f;
                else if (p.bias_mode == 2)
                    s_bias[i] = n < p.N ? __uint_as_float(static_cast<uint32_t>(
                                              static_cast<const uint16_t*>(p.bias)[n]) << 16)
                                        : 0.0f;
                if constexpr (kFusedQuant) {
                    // The row's scale once the tile's rows are published (the
                    // producer waits for the same rows before the first copy,
                    // so this wait ends before the first chunk is ready).
                    if (m < p.M && m >= p.q_row0 && !fused_tile_ready(p, m >> 8, limit))
                        atomicOr(p.status, kDevTimeoutEpilogue);
                }
                if (kScaled && m < p.M) sxm = p.sx[m];
            }
            int32_t acc[128];
#pragma unroll
            for (int i = 0; i < 128; ++i) acc[i] = 0;
            for (int kc0 = u.kb0; kc0 < u.kb1; kc0 += p.kb_per_chunk, ++cc) {
                const uint32_t b = cc & 1u;
                const uint32_t bph = (cc >> 1) & 1u;
                // One thread takes the bounded wait for the whole epilogue and
                // publishes the outcome, so all eight warps take the same path
                // (their named barriers below could never complete otherwise).
                if (e == 0 && lane == 0) s_chunk_ready[cc & 1u] = mbar_wait(&tfull[b], bph, limit) ? 1 : 0;
                epi_barrier();
                if (!s_chunk_ready[cc & 1u]) {
                    if (e == 0 && lane == 0) atomicOr(p.status, kDevTimeoutEpilogue);
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t taddr =
                    tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + b * kBN + half * 128;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t r[32];
                    tmem_load_32cols(taddr + j * 32, r);
                    tmem_load_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        if constexpr (kFp32Sums)
                            acc[j * 32 + i] =
                                __float_as_int(__fadd_rn(__int_as_float(acc[j * 32 + i]), __uint_as_float(r[i])));
                        else
                            acc[j * 32 + i] += __float2int_rn(__uint_as_float(r[i]));
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (kPair == 2)
                        mbar_arrive_cluster(cluster_map(&tempty[b], 0));
                    else
                        mbar_arrive(&tempty[b]);
                }
            }
            if (!ok) break;

            if (u.slot >= 0) {
                // A K-segment of a split tile: publish this CTA's partial sums,
                // count in, and only the last segment to arrive finishes this
                // CTA's rows of the tile.  Thread (e, lane) always holds the
                // same 128 sums, so the slots use a layout in which each warp
                // access is 512 contiguous bytes, and epilogue warp e's sums
                // fill the 16 KB region e of the slot.
                int4* mine = p.partials + (static_cast<int64_t>(u.slot) * kPair + rank) * kPartialInt4;
#pragma unroll
                for (int g = 0; g < 32; ++g)
                    __stcg(mine + (e * 32 + g) * 32 + lane,
                           make_int4(acc[4 * g], acc[4 * g + 1], acc[4 * g + 2], acc[4 * g + 3]));
                fence_proxy_async_global();   // the last segment reads the slot by bulk copy
                __threadfence();
                // The fix-up below reuses the output staging: the previous
                // tile's stores must have finished reading it.
                if (kPair == 2 && !kOutS32 && lane == 0) bulk_wait_read_all();
                if (e == 0 && lane == 0) s_fix_status = 0;
                epi_barrier();
                const int counter = (u.tile - p.dp_tiles) * kPair + static_cast<int>(rank);
                if (e == 0 && lane == 0)
                    s_last_arrival =
                        (atomicAdd(p.tile_counters + counter, 1u) == static_cast<uint32_t>(p.splits - 1)) ? 1 : 0;
                epi_barrier();
                if (!s_last_arrival) continue;
                __threadfence();
                // This was the CTA's last unit, so its operand ring (and the
                // output staging) is idle.  Each warp streams its own 16 KB
                // region of every other segment's partial (the sums of the
                // rows and columns it holds) through three 8 KB slots of
                // shared memory by asynchronous bulk copies, half a region at
                // a time, and adds each half from shared memory as it lands;
                // the warps do not wait for one another, and up to 192 KB are
                // in flight per CTA.
                // Integer sums may be added in any order.  Floating-point sums
                // are added in segment order, this CTA's own from its slot as
                // well, so the result does not depend on which segment
                // finished last.
                if constexpr (kFp32Sums) {
#pragma unroll
                    for (int i = 0; i < 128; ++i) acc[i] = 0;
                }
                const int first = (u.tile - p.dp_tiles) * p.splits;
                const int n_units = kFp32Sums ? p.splits : p.splits - 1;
                const int n_pieces = 2 * n_units;
                uint8_t* wbuf = smem + e * kFixWarpBytes;
                uint64_t* wbar = fixbars + e * kFixSlots;
                auto piece_src = [&](int j) -> const uint8_t* {
                    int unit = first + (j >> 1);
                    if (!kFp32Sums && unit >= u.slot) ++unit;   // this segment's own partial is in registers
                    const int4* region =
                        p.partials + (static_cast<int64_t>(unit) * kPair + rank) * kPartialInt4 + e * 1024;
                    return reinterpret_cast<const uint8_t*>(region) + (j & 1) * kFixSlotBytes;
                };
                if (lane == 0) {
                    fence_proxy_async_global();
                    for (int j = 0; j < kFixSlots && j < n_pieces; ++j) {
                        mbar_arrive_expect_tx(&wbar[j], kFixSlotBytes);
                        bulk_load(wbuf + j * kFixSlotBytes, piece_src(j), kFixSlotBytes, &wbar[j]);
                    }
                }
                bool fix_ok = true;
                for (int k = 0; k < n_units && fix_ok; ++k) {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int j = 2 * k + hh;
                        const int slot = j % kFixSlots;
                        const bool landed = mbar_wait(&wbar[slot], static_cast<uint32_t>(j / kFixSlots) & 1u, limit);
                        if (!__all_sync(0xFFFFFFFFu, landed)) {
                            fix_ok = false;
                            break;
                        }
                        const int4* sp = reinterpret_cast<const int4*>(wbuf + slot * kFixSlotBytes) + lane;
#pragma unroll
                        for (int g = 0; g < 16; ++g) {
                            const int4 v = sp[g * 32];
                            const int a = 4 * (16 * hh + g);
                            if constexpr (kFp32Sums) {
                                acc[a] = __float_as_int(__fadd_rn(__int_as_float(acc[a]), __int_as_float(v.x)));
                                acc[a + 1] = __float_as_int(__fadd_rn(__int_as_float(acc[a + 1]), __int_as_float(v.y)));
                                acc[a + 2] = __float_as_int(__fadd_rn(__int_as_float(acc[a + 2]), __int_as_float(v.z)));
                                acc[a + 3] = __float_as_int(__fadd_rn(__int_as_float(acc[a + 3]), __int_as_float(v.w)));
                            } else {
                                acc[a] += v.x;
                                acc[a + 1] += v.y;
                                acc[a + 2] += v.z;
                                acc[a + 3] += v.w;
                            }
                        }
                        __syncwarp();   // every lane has read the slot before it is refilled
                        if (lane == 0 && j + kFixSlots < n_pieces) {
                            fence_proxy_async_smem();   // those reads before the copy's writes
                            mbar_arrive_expect_tx(&wbar[slot], kFixSlotBytes);
                            bulk_load(wbuf + slot * kFixSlotBytes, piece_src(j + kFixSlots), kFixSlotBytes,
                                      &wbar[slot]);
                        }
                    }
                }
                if (!fix_ok && lane == 0) s_fix_status = 1;
                epi_barrier();
                if (s_fix_status != 0) {
                    if (e == 0 && lane == 0) atomicOr(p.status, kDevTimeoutEpilogue);
                    ok = false;
                    break;
                }
                if (e == 0 && lane == 0) p.tile_counters[counter] = 0u;   // ready for the next launch
            }

            if constexpr (kOutS32) {
                if (m < p.M) {
                    int32_t* row = static_cast<int32_t*>(p.out) + static_cast<int64_t>(m) * p.N;
#pragma unroll
                    for (int g = 0; g < 32; ++g) {
                        const int n = n0 + g * 4;
                        if (n < p.N)
                            *reinterpret_cast<int4*>(row + n) =
                                make_int4(acc[4 * g], acc[4 * g + 1], acc[4 * g + 2], acc[4 * g + 3]);
                    }
                }
            } else {
                // y = bf16_rne(((float)acc * sx[m]) * sw[n] + bias[n]) (BF16
                // linear: bf16_rne(acc + bias[n])), eight columns at a time,
                // packed as four bf16 pairs.
                const float* swc = s_sw + half * 128;
                const float* bc = s_bias + half * 128;
                auto dequant8 = [&](int g, uint4& out) {
                    float y[8];
                    if constexpr (kFp32Sums) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) y[i] = __int_as_float(acc[8 * g + i]);
                    } else {
                        const float4 w0 = *reinterpret_cast<const float4*>(swc + 8 * g);
                        const float4 w1 = *reinterpret_cast<const float4*>(swc + 8 * g + 4);
                        const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            y[i] = __fmul_rn(__fmul_rn(__int2float_rn(acc[8 * g + i]), sxm), wv[i]);
                    }
                    if (p.bias_mode != 0) {
                        const float4 b0 = *reinterpret_cast<const float4*>(bc + 8 * g);
                        const float4 b1 = *reinterpret_cast<const float4*>(bc + 8 * g + 4);
                        const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                        for (int i = 0; i < 8; ++i) y[i] = __fadd_rn(y[i], bv[i]);
                    }
                    out = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                                     pack_bf16x2(y[6], y[7]));
                };
                // Largest |y| of this thread's row segment (bf16 magnitudes
                // order like unsigned integers), for the next layer's row
                // scale.  Rows past M are skipped below; columns past N are 0.
                uint32_t amax2 = 0;
                auto fold_amax = [&](const uint4& v) {
                    amax2 = __vmaxu2(amax2, v.x & 0x7FFF7FFFu);
                    amax2 = __vmaxu2(amax2, v.y & 0x7FFF7FFFu);
                    amax2 = __vmaxu2(amax2, v.z & 0x7FFF7FFFu);
                    amax2 = __vmaxu2(amax2, v.w & 0x7FFF7FFFu);
                };
                if constexpr (kPair == 2) {
                    // Stage this warp's 32 rows x 128 columns as two 32 x 64
                    // boxes, one after the other in the warp's 4 KB buffer, in
                    // the 128-byte swizzle (16-byte chunk c of row r at chunk
                    // c ^ (r % 8): conflict-free), each TMA-stored as soon as
                    // written; the store clips rows >= M and columns >= N.
                    // Before a box is rewritten, the store that read it last
                    // must have finished reading.
                    uint8_t* buf = sOut + e * 4096;
                    const int row0 = (mb * kPair + static_cast<int>(rank)) * kBM + quarter * 32;
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        if (lane == 0) bulk_wait_read_all();
                        __syncwarp();
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            uint4 v;
                            dequant8(j * 8 + c, v);
                            if constexpr (kRowMax) fold_amax(v);
                            *reinterpret_cast<uint4*>(buf + lane * 128 + ((c ^ (lane & 7)) << 4)) = v;
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            if (row0 < p.M && n0 + 64 * j < p.N) tma_store_2d(&tmap_y, buf, n0 + 64 * j, row0);
                            bulk_commit_group();
                        }
                    }
                } else if (m < p.M) {
                    uint16_t* row = static_cast<uint16_t*>(p.out) + static_cast<int64_t>(m) * p.N;
#pragma unroll
                    for (int g = 0; g < 16; ++g) {
                        const int n = n0 + g * 8;
                        if (n < p.N) {
                            uint4 v;
                            dequant8(g, v);
                            if constexpr (kRowMax) fold_amax(v);
                            *reinterpret_cast<uint4*>(row + n) = v;
                        }
                    }
                }
                if (kRowMax && m < p.M) {
                    const uint32_t a = max(amax2 & 0xFFFFu, amax2 >> 16) << 16;   // fp32 bits of the bf16 max
                    if (a != 0u) atomicMax(p.row_amax + m, a);
                }
            }
        }
        // Output stores still in flight must finish before the CTA exits.
        if (kPair == 2 && !kOutS32 && lane == 0) bulk_wait_all();
    }

    tc_fence_before_sync();
    __syncthreads();
    // A pair leaves together: the leader's MMAs are complete (it waited on
    // `done`) and its copies have landed before either CTA frees tensor
    // memory or exits while the other may still target its shared memory.
    if constexpr (kPair == 2) cluster_sync_all();
    tc_fence_after_sync();
    if (warp == 1) tmem_dealloc<kPair>(tmem_base, kTmemCols);
}

}  // namespace w8a8
