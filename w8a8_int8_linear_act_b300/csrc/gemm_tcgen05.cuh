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
// Kernel shape (one CTA per SM, persistent over 128 x 256 output tiles):
//   warp 0      TMA producer: A (128 x 64) and B (256 x 64) bf16 tiles, 128-byte
//               swizzle, into a 4-stage shared-memory ring (48 KB per stage)
//   warp 1      tensor-memory owner and MMA issuer (one thread): per stage
//               4 x tcgen05.mma 128x256x16 into one of two 256-column fp32
//               accumulators; commits free the stage / publish the chunk
//   warps 2-9   epilogue: warp w reads TMEM lanes 32*(w%4)..+31 (its rows)
//               and one 128-column half of the tile
// Two accumulators let the MMA fill one chunk while the epilogue drains the
// other.  Every mbarrier wait is bounded by a wall-clock limit; a wait that
// runs out sets a bit in the status word and the CTA unwinds (waiting,
// again with a limit, for its own copies and MMAs in flight) and frees its
// tensor memory.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "ptx_sm103.cuh"

namespace w8a8 {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;  // 64 bf16 = 128 bytes = one swizzle row
constexpr int kStages = 4;
constexpr int kEpiWarps = 8;
constexpr int kGemmThreads = 64 + 32 * kEpiWarps;
constexpr int kUmmaK = 16;
constexpr uint32_t kAStageBytes = kBM * kBK * 2;
constexpr uint32_t kBStageBytes = kBN * kBK * 2;
constexpr uint32_t kStageBytes = kAStageBytes + kBStageBytes;
constexpr uint32_t kTmemCols = 2 * kBN;  // two fp32 accumulators
constexpr int kMaxKbPerChunk = 16;       // 16 * 64 = 1024: 1024 * 127^2 < 2^24
constexpr size_t kGemmSmemBytes = 1024 /* alignment slack */ + kStages * kStageBytes + 256 /* barriers */;

// Status bits (same values as W8A8_DEV_* in the public header).
constexpr uint32_t kDevTimeoutProducer = 0x1;
constexpr uint32_t kDevTimeoutMma = 0x2;
constexpr uint32_t kDevTimeoutEpilogue = 0x4;
constexpr uint32_t kDevTimeoutTeardown = 0x8;

struct GemmParams {
    int32_t M, N, K;
    int32_t kb_per_chunk;      // k-blocks of 64 per exact fp32 chunk, 1..16
    int32_t group_m;           // tile rasterisation: m-tiles per group
    int32_t bias_mode;         // 0 none, 1 fp32, 2 bf16
    const float* sx;           // [M]
    const float* sw;           // [N]
    const void* bias;          // [N] or nullptr
    void* out;                 // bf16 Y [M][N] or int32 acc [M][N]
    uint32_t* status;          // device status word
    uint64_t wait_limit_ns;
    int32_t skip_loads;        // test hook: producer issues no copies
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

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
           (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
}

template <bool kOutS32>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_w8a8_tcgen05_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                             const GemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t* sA = smem;
    uint8_t* sB = smem + kStages * kAStageBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    uint64_t* full = bars;                    // [kStages] TMA -> MMA
    uint64_t* empty = bars + kStages;         // [kStages] MMA -> TMA
    uint64_t* tfull = bars + 2 * kStages;     // [2] MMA -> epilogue
    uint64_t* tempty = tfull + 2;             // [2] epilogue -> MMA
    uint64_t* done = tempty + 2;              // MMA teardown
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(done + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tiles_m = (p.M + kBM - 1) / kBM;
    const int tiles_n = (p.N + kBN - 1) / kBN;
    const int num_tiles = tiles_m * tiles_n;
    const int num_kb = (p.K + kBK - 1) / kBK;
    const int chunks = (num_kb + p.kb_per_chunk - 1) / p.kb_per_chunk;
    const uint64_t limit = p.wait_limit_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
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
        tmem_alloc(tmem_holder, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t it = 0;
            uint32_t issued_mask = 0, issued_par = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                int mb, nb;
                tile_coords(t, tiles_m, tiles_n, p.group_m, mb, nb);
                for (int kb = 0; kb < num_kb; ++kb, ++it) {
                    const int s = static_cast<int>(it % kStages);
                    const uint32_t ph = (it / kStages) & 1u;
                    if (!mbar_wait(&empty[s], ph ^ 1u, limit)) {
                        atomicOr(p.status, kDevTimeoutProducer);
                        ok = false;
                        break;
                    }
                    if (p.skip_loads) continue;
                    mbar_arrive_expect_tx(&full[s], kStageBytes);
                    tma_load_2d(sA + s * kAStageBytes, &tmap_a, &full[s], kb * kBK, mb * kBM);
                    tma_load_2d(sB + s * kBStageBytes, &tmap_b, &full[s], kb * kBK, nb * kBN);
                    issued_mask |= 1u << s;
                    issued_par = (issued_par & ~(1u << s)) | (ph << s);
                }
            }
            // Copies still in flight must land before the CTA exits.
            for (int s = 0; s < kStages; ++s)
                if ((issued_mask >> s) & 1u)
                    if (!mbar_wait(&full[s], (issued_par >> s) & 1u, limit)) atomicOr(p.status, kDevTimeoutTeardown);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN);
            uint32_t it = 0, cc = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                for (int c = 0; c < chunks && ok; ++c, ++cc) {
                    const uint32_t b = cc & 1u;
                    const uint32_t bph = (cc >> 1) & 1u;
                    if (!mbar_wait(&tempty[b], bph ^ 1u, limit)) {
                        atomicOr(p.status, kDevTimeoutMma);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t d_tmem = tmem_base + b * kBN;
                    const int kb0 = c * p.kb_per_chunk;
                    const int kb1 = min(num_kb, kb0 + p.kb_per_chunk);
                    for (int kb = kb0; kb < kb1; ++kb, ++it) {
                        const int s = static_cast<int>(it % kStages);
                        const uint32_t ph = (it / kStages) & 1u;
                        if (!mbar_wait(&full[s], ph, limit)) {
                            atomicOr(p.status, kDevTimeoutMma);
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        const uint32_t a0 = smem_addr(sA + s * kAStageBytes);
                        const uint32_t b0 = smem_addr(sB + s * kBStageBytes);
#pragma unroll
                        for (int k = 0; k < kBK / kUmmaK; ++k) {
                            mma_bf16(d_tmem, smem_desc_k128(a0 + k * kUmmaK * 2), smem_desc_k128(b0 + k * kUmmaK * 2),
                                     idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                        }
                        mma_commit(&empty[s]);
                    }
                    if (ok) mma_commit(&tfull[b]);
                }
            }
            // Every MMA issued must complete before tensor memory is freed.
            mma_commit(done);
            if (!mbar_wait(done, 0, limit)) atomicOr(p.status, kDevTimeoutTeardown);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;        // TMEM lanes this warp may read
        const int half = (warp - 2) >> 2;    // which 128 columns of the tile
        uint32_t cc = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            int mb, nb;
            tile_coords(t, tiles_m, tiles_n, p.group_m, mb, nb);
            int32_t acc[128];
#pragma unroll
            for (int i = 0; i < 128; ++i) acc[i] = 0;
            for (int c = 0; c < chunks; ++c, ++cc) {
                const uint32_t b = cc & 1u;
                const uint32_t bph = (cc >> 1) & 1u;
                int got = 1;
                if (lane == 0) got = mbar_wait(&tfull[b], bph, limit) ? 1 : 0;
                got = __shfl_sync(0xFFFFFFFFu, got, 0);
                if (!got) {
                    if (lane == 0) atomicOr(p.status, kDevTimeoutEpilogue);
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
                    for (int i = 0; i < 32; ++i) acc[j * 32 + i] += __float2int_rn(__uint_as_float(r[i]));
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[b]);
            }
            if (!ok) break;

            const int m = mb * kBM + quarter * 32 + lane;
            const int n0 = nb * kBN + half * 128;
            if (m < p.M) {
                if constexpr (kOutS32) {
                    int32_t* row = static_cast<int32_t*>(p.out) + static_cast<int64_t>(m) * p.N;
#pragma unroll
                    for (int g = 0; g < 32; ++g) {
                        const int n = n0 + g * 4;
                        if (n < p.N)
                            *reinterpret_cast<int4*>(row + n) =
                                make_int4(acc[4 * g], acc[4 * g + 1], acc[4 * g + 2], acc[4 * g + 3]);
                    }
                } else {
                    const float sxm = p.sx[m];
                    uint16_t* row = static_cast<uint16_t*>(p.out) + static_cast<int64_t>(m) * p.N;
#pragma unroll
                    for (int g = 0; g < 16; ++g) {
                        const int n = n0 + g * 8;
                        if (n < p.N) {
                            const float4 w0 = __ldg(reinterpret_cast<const float4*>(p.sw + n));
                            const float4 w1 = __ldg(reinterpret_cast<const float4*>(p.sw + n + 4));
                            const float swv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                            float y[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                y[i] = __fmul_rn(__fmul_rn(__int2float_rn(acc[8 * g + i]), sxm), swv[i]);
                            if (p.bias_mode == 1) {
                                const float4 b0 = __ldg(reinterpret_cast<const float4*>(
                                    static_cast<const float*>(p.bias) + n));
                                const float4 b1 = __ldg(reinterpret_cast<const float4*>(
                                    static_cast<const float*>(p.bias) + n + 4));
                                const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                                for (int i = 0; i < 8; ++i) y[i] = __fadd_rn(y[i], bv[i]);
                            } else if (p.bias_mode == 2) {
                                const uint4 bb = __ldg(reinterpret_cast<const uint4*>(
                                    static_cast<const uint16_t*>(p.bias) + n));
                                const uint32_t bw[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    y[2 * i] = __fadd_rn(y[2 * i], __uint_as_float(bw[i] << 16));
                                    y[2 * i + 1] = __fadd_rn(y[2 * i + 1], __uint_as_float(bw[i] & 0xFFFF0000u));
                                }
                            }
                            *reinterpret_cast<uint4*>(row + n) = make_uint4(
                                pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                                pack_bf16x2(y[6], y[7]));
                        }
                    }
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace w8a8
