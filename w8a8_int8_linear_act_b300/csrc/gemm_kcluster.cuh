// The W8A8 GEMM for problems with few output tiles (the audio branch's
// 126- and 1001-row activations): the same exact INT32 accumulation and
// fused epilogue as gemm_tcgen05.cuh (zhidx TurboT2VA article, section 01
// item 3 "量化策略": INT32 accumulation, then row scale x channel scale and
// bias applied once after the full sum; the audio and video branches have
// different matrix shapes), cut so that the work spreads over the SMs.
//
// The persistent form gives each SM pair a 256 x 256 tile: at 126 x 2048
// output columns that is 8 tiles for 74 pairs, and each busy pair spends the
// whole tile's MMA time on rows that are mostly past M.  Here an output tile
// is 128 rows x BN columns (BN = 64, 128 or 256) and is computed by a
// thread-block cluster of KS CTAs (KS = 1, 2, 4 or 8), CTA r of the cluster
// taking k-blocks [r * nkb / KS, (r + 1) * nkb / KS).  Each CTA accumulates
// its K range exactly as the persistent form does (codes carried as bf16,
// tcgen05 kind::f16 with fp32 chunks of at most 1024 drained exactly into
// INT32 sums in registers).  Rank r finishes rows [r * 128 / KS, (r + 1) *
// 128 / KS) of the tile: once every CTA of the cluster is done with its
// operand ring (a cluster barrier), each CTA sends its partial sums of those
// rows into rank r's ring with posted stores to distributed shared memory
// (st.shared::cluster); after a second cluster barrier rank r adds the KS
// partials from its own shared memory and runs the epilogue.  INT32 addition
// is exact and associative, so the sum is the exact accumulator; the bf16
// linear's fp32 partials are added in rank order, so its result does not
// depend on timing.  A cluster of one keeps its sums local and needs neither
// barrier.  No global partial slots, counters or fences.
//
// Roles as in the persistent form: warp 0 TMA producer, warp 1 tensor-
// memory owner and MMA issuer (tcgen05.mma.cta_group::1 128 x BN x 16),
// warps 2-9 epilogue (warp w reads TMEM lanes 32 * (w % 4) .. + 31 and one
// half of the BN columns).  While the K loop runs, the epilogue warps stage
// the tile's sw, bias and sx in shared memory.  After the exchange they split
// this CTA's rows into 8-column groups: consecutive threads take consecutive
// groups of a row, so each warp stores whole 128-byte lines of Y, and every
// operand of the epilogue is a shared-memory load.  One tile per cluster
// (not persistent): clusters are independent, so any number of waves is
// correct.  Waits are bounded as in the persistent form; every path through
// the kernel reaches both cluster barriers.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "gemm_tcgen05.cuh"
#include "ptx_sm103.cuh"

namespace w8a8 {

constexpr int kMaxClusterK = 8;   // CTAs of one cluster along K (portable cluster size)

template <int BN>
struct KClusterCfg {
    static_assert(BN == 64 || BN == 128 || BN == 256, "tile width");
    static constexpr uint32_t kAStageBytes = kBM * kBK * 2;             // 128 rows x 64 bf16 codes
    static constexpr uint32_t kBStageBytes = BN * kBK * 2;
    static constexpr uint32_t kStageBytes = kAStageBytes + kBStageBytes;
    static constexpr int kStages = BN == 256 ? 4 : 6;
    static constexpr int kPartStride = BN + 4;                            // int32 words per partial row (padded:
                                                                          // conflict-free 16-byte row writes)
    static constexpr uint32_t kPartBytes = kBM * kPartStride * 4;
    static constexpr uint32_t kTmemCols = 2 * BN;                         // two fp32 accumulators
    static constexpr int kLoadsPerChunk = BN / 64;                        // 32-column TMEM loads per thread
    static constexpr uint32_t kParamBytes = (2 * BN + kBM) * 4;           // the tile's sw, bias (fp32) and sx
    static constexpr size_t kSmemBytes =
        1024 /* alignment */ + kStages * kStageBytes + kParamBytes + 256 /* barriers */;
    static_assert(kStages * kStageBytes >= kPartBytes, "a partial tile fits in the operand ring");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
    static_assert((2 * kStages + 5) * 8 + 4 <= 256, "barrier area");
};

struct KClusterParams {
    int32_t M, N, K;
    int32_t kb_per_chunk;      // k-blocks per TMEM accumulation (INT8 codes: at most 16, exact)
    int32_t tiles_m;           // output tiles along M; tile t is (t % tiles_m, t / tiles_m)
    int32_t bias_mode;         // 0 none, 1 fp32, 2 bf16
    const float* sx;           // [M]
    const float* sw;           // [N]
    const void* bias;          // [N] or nullptr
    void* out;                 // bf16 Y [M][N] or int32 acc [M][N]
    uint32_t* status;          // device status word
    uint64_t wait_limit_ns;
    int32_t skip_loads;        // test hook: producer issues no copies
};

template <int kMode, int BN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kcluster_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                         const KClusterParams p)
{
    using C = KClusterCfg<BN>;
    constexpr int S = C::kStages;
    constexpr bool kOutS32 = kMode == kModeS32;
    constexpr bool kFp32Sums = kMode == kModeBf16;
    static_assert(kMode == kModeW8A8 || kMode == kModeS32 || kMode == kModeBf16, "mode");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t* sA = smem;
    uint8_t* sB = smem + S * C::kAStageBytes;
    int32_t* part = reinterpret_cast<int32_t*>(smem);      // after the K loop: the partial rows this CTA finishes
    float* s_sw = reinterpret_cast<float*>(smem + S * C::kStageBytes);   // [BN] the tile's sw
    float* s_bias = s_sw + BN;                                           // [BN] its bias as fp32 (0: none)
    float* s_sx = s_bias + BN;                                           // [128] its rows' sx
    uint64_t* bars = reinterpret_cast<uint64_t*>(s_sx + kBM);
    uint64_t* full = bars;
    uint64_t* empty = bars + S;
    uint64_t* tfull = bars + 2 * S;
    uint64_t* tempty = tfull + 2;
    uint64_t* done = tempty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(done + 1);
    __shared__ int s_chunk_ready[2];
    // Epilogue threads: this CTA's sums of one row half (row 32 * (warp % 4)
    // + lane, columns (warp - 2) / 4 * BN / 2 ...), kept for the exchange.
    int32_t acc[BN / 2];
#pragma unroll
    for (int i = 0; i < BN / 2; ++i) acc[i] = 0;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t ks = cluster_nctarank();
    const int tile = static_cast<int>(cluster_id_x());
    const int mb = tile % p.tiles_m;
    const int nb = tile / p.tiles_m;
    const int num_kb = (p.K + kBK - 1) / kBK;
    const int kb0 = static_cast<int>(static_cast<int64_t>(rank) * num_kb / ks);
    const int kb1 = static_cast<int>(static_cast<int64_t>(rank + 1) * num_kb / ks);
    const uint64_t limit = p.wait_limit_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], kEpiWarps);
        }
        mbar_init(done, 1);
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_a);
        tma_prefetch_desc(&tmap_b);
    }
    if (warp == 1) {
        tmem_alloc<1>(tmem_holder, C::kTmemCols);
        tmem_relinquish<1>();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_holder;
    // A programmatic dependent of the kernel that writes the codes, row
    // scales and status word: nothing below may run before it completes.
    grid_wait_prerequisites();
    grid_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t it = 0, n_issued = 0;
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const int s = static_cast<int>(it % S);
                const uint32_t ph = (it / S) & 1u;
                if (!mbar_wait(&empty[s], ph ^ 1u, limit)) {
                    atomicOr(p.status, kDevTimeoutProducer);
                    break;
                }
                if (p.skip_loads) continue;
                mbar_arrive_expect_tx(&full[s], C::kStageBytes);
                tma_load_2d(sA + s * C::kAStageBytes, &tmap_a, &full[s], kb * kBK, mb * kBM);
                tma_load_2d(sB + s * C::kBStageBytes, &tmap_b, &full[s], kb * kBK, nb * BN);
                n_issued = it + 1;
            }
            // Copies still in flight land before the ring is reused or the CTA exits.
            for (uint32_t i = n_issued > static_cast<uint32_t>(S) ? n_issued - S : 0u; i < n_issued; ++i)
                if (!mbar_wait(&full[i % S], (i / S) & 1u, limit)) atomicOr(p.status, kDevTimeoutTeardown);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN);
            uint32_t it = 0, cc = 0;
            bool ok = true;
            for (int kc0 = kb0; kc0 < kb1 && ok; kc0 += p.kb_per_chunk, ++cc) {
                const uint32_t b = cc & 1u;
                const uint32_t bph = (cc >> 1) & 1u;
                if (!mbar_wait(&tempty[b], bph ^ 1u, limit)) {
                    atomicOr(p.status, kDevTimeoutMma);
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + b * BN;
                const int kc1 = min(kb1, kc0 + p.kb_per_chunk);
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
                    for (int k = 0; k < kBK / kUmmaK; ++k)
                        mma_bf16<1>(d_tmem, smem_desc_k128(a0 + k * kUmmaK * 2), smem_desc_k128(b0 + k * kUmmaK * 2),
                                    idesc, (kb > kc0 || k > 0) ? 1u : 0u);
                    mma_commit<1>(&empty[s]);
                }
                if (ok) mma_commit<1>(&tfull[b]);
            }
            // Every MMA issued completes before the ring or tensor memory is reused.
            mma_commit<1>(done);
            if (!mbar_wait(done, 0, limit)) atomicOr(p.status, kDevTimeoutTeardown);
        }
    } else {
        // ------------------------------------------------------------ epilogue: drain the K range
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int e = warp - 2;
        // The tile's column and row parameters into shared memory now, so
        // that their latency hides behind the K loop.
        for (int i = e * 32 + lane; i < BN + kBM; i += 32 * kEpiWarps) {
            if (i < BN) {
                const int n = nb * BN + i;
                if constexpr (!kOutS32 && !kFp32Sums) s_sw[i] = n < p.N ? p.sw[n] : 0.0f;
                float bv = 0.0f;
                if (n < p.N && p.bias_mode == 1)
                    bv = static_cast<const float*>(p.bias)[n];
                else if (n < p.N && p.bias_mode == 2)
                    bv = __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(p.bias)[n]) << 16);
                s_bias[i] = bv;
            } else {
                const int m = mb * kBM + (i - BN);
                if constexpr (!kOutS32 && !kFp32Sums) s_sx[i - BN] = m < p.M ? p.sx[m] : 0.0f;
            }
        }
        uint32_t cc = 0;
        for (int kc0 = kb0; kc0 < kb1; kc0 += p.kb_per_chunk, ++cc) {
            const uint32_t b = cc & 1u;
            const uint32_t bph = (cc >> 1) & 1u;
            // One thread takes the bounded wait and publishes the outcome, so
            // all eight warps take the same path.
            if (e == 0 && lane == 0) s_chunk_ready[cc & 1u] = mbar_wait(&tfull[b], bph, limit) ? 1 : 0;
            epi_barrier();
            if (!s_chunk_ready[cc & 1u]) {
                if (e == 0 && lane == 0) atomicOr(p.status, kDevTimeoutEpilogue);
                break;
            }
            tc_fence_after_sync();
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + b * BN + half * (BN / 2);
#pragma unroll
            for (int j = 0; j < C::kLoadsPerChunk; ++j) {
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
            if (lane == 0) mbar_arrive(&tempty[b]);
        }
    }

    // The exchange.  Row r of the tile is finished by rank r / (128 / ks);
    // every CTA sends its partial sums of that row to that rank, which adds
    // the ks partials from its own shared memory.  Partials land in the
    // receiver's operand ring, so every CTA of the cluster must be done with
    // its ring first (barrier A: all MMAs of the cluster are complete, their
    // last accumulators drained), and the sums must have landed before they
    // are read (barrier B).  The sends are posted stores to distributed
    // shared memory; all reads are local.  A cluster of one needs neither.
    const int rows = kBM / static_cast<int>(ks);
    tc_fence_before_sync();
    __syncthreads();
    if (ks > 1) cluster_sync_all();                                     // A
    if (warp >= 2) {
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int r = quarter * 32 + lane;
        const uint32_t owner = static_cast<uint32_t>(r / rows);
        const int lr = r - static_cast<int>(owner) * rows;
        const uint32_t off = static_cast<uint32_t>(((static_cast<int>(rank) * rows + lr) * C::kPartStride +
                                                    half * (BN / 2)) * 4);
        if (owner == rank) {
            int4* dst = reinterpret_cast<int4*>(reinterpret_cast<uint8_t*>(part) + off);
#pragma unroll
            for (int g = 0; g < BN / 8; ++g)
                dst[g] = make_int4(acc[4 * g], acc[4 * g + 1], acc[4 * g + 2], acc[4 * g + 3]);
        } else {
            const uint32_t dst = cluster_map(part, owner) + off;
#pragma unroll
            for (int g = 0; g < BN / 8; ++g)
                st_cluster_v4(dst + 16 * g,
                              make_int4(acc[4 * g], acc[4 * g + 1], acc[4 * g + 2], acc[4 * g + 3]));
        }
    }
    __syncthreads();
    if (ks > 1) cluster_sync_all();                                     // B
    tc_fence_after_sync();

    if (warp >= 2) {
        // ------------------------------------------------------------ epilogue: rows of this rank
        const int t = static_cast<int>(threadIdx.x) - 64;
        const int row0 = static_cast<int>(rank) * rows;
        constexpr int kGroups = BN / 8;   // 8-column groups per row
        const uint8_t* pbytes = reinterpret_cast<const uint8_t*>(part);
        for (int item = t; item < rows * kGroups; item += 32 * kEpiWarps) {
            const int lr = item / kGroups;
            const int cg = item % kGroups;
            const int m = mb * kBM + row0 + lr;
            const int n = nb * BN + cg * 8;
            if (m >= p.M || n >= p.N) continue;
            int4 v0[kMaxClusterK], v1[kMaxClusterK];
#pragma unroll
            for (int j = 0; j < kMaxClusterK; ++j) {
                if (j < static_cast<int>(ks)) {
                    const int4* src = reinterpret_cast<const int4*>(
                        pbytes + ((j * rows + lr) * C::kPartStride + cg * 8) * 4);
                    v0[j] = src[0];
                    v1[j] = src[1];
                } else {
                    v0[j] = make_int4(0, 0, 0, 0);
                    v1[j] = make_int4(0, 0, 0, 0);
                }
            }
            int32_t s8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) s8[i] = 0;
#pragma unroll
            for (int j = 0; j < kMaxClusterK; ++j) {
                if (j >= static_cast<int>(ks)) break;
                const int32_t v[8] = {v0[j].x, v0[j].y, v0[j].z, v0[j].w, v1[j].x, v1[j].y, v1[j].z, v1[j].w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if constexpr (kFp32Sums)
                        s8[i] = __float_as_int(__fadd_rn(__int_as_float(s8[i]), __int_as_float(v[i])));
                    else
                        s8[i] += v[i];
                }
            }
            if constexpr (kOutS32) {
                int4* dst = reinterpret_cast<int4*>(static_cast<int32_t*>(p.out) + static_cast<int64_t>(m) * p.N + n);
                dst[0] = make_int4(s8[0], s8[1], s8[2], s8[3]);
                dst[1] = make_int4(s8[4], s8[5], s8[6], s8[7]);
            } else {
                // y = bf16_rne(((float)acc * sx[m]) * sw[n] + bias[n]) (BF16
                // linear: bf16_rne(acc + bias[n])), each step one fp32 operation.
                float y[8];
                if constexpr (kFp32Sums) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) y[i] = __int_as_float(s8[i]);
                } else {
                    const float sxm = s_sx[row0 + lr];
                    const float4 w0 = *reinterpret_cast<const float4*>(s_sw + cg * 8);
                    const float4 w1 = *reinterpret_cast<const float4*>(s_sw + cg * 8 + 4);
                    const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                    for (int i = 0; i < 8; ++i) y[i] = __fmul_rn(__fmul_rn(__int2float_rn(s8[i]), sxm), wv[i]);
                }
                if (p.bias_mode != 0) {
                    const float4 b0 = *reinterpret_cast<const float4*>(s_bias + cg * 8);
                    const float4 b1 = *reinterpret_cast<const float4*>(s_bias + cg * 8 + 4);
                    const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                    for (int i = 0; i < 8; ++i) y[i] = __fadd_rn(y[i], bv[i]);
                }
                *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + static_cast<int64_t>(m) * p.N + n) =
                    make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                               pack_bf16x2(y[6], y[7]));
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 1) tmem_dealloc<1>(tmem_base, C::kTmemCols);
}


}  // namespace w8a8
