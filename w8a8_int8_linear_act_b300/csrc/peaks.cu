// Throughput probes for the roofline denominators (declared in
// include/w8a8_peaks.h).  Not part of the layer: they measure how fast this
// GPU runs the warp-level tensor-core MMA (mma.sync) on INT8 and on bf16
// operands, the only integer tensor-core path sm_103a code can use (ptxas
// rejects tcgen05.mma kind::i8 for sm_103a).
//
// Each warp keeps kChains independent accumulators and issues one MMA on
// each per step, so the tensor pipe always has independent work; operands
// stay in registers, so nothing but the MMAs is timed.  The result is
// written only if it equals a value it cannot take (the accumulators start
// from small integers and only grow), which keeps the compiler from
// removing the loop.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/w8a8_peaks.h"

namespace {

constexpr int kChains = 8;

__global__ void __launch_bounds__(256) mma_s8_probe_kernel(int64_t iters, int32_t* sink)
{
    const uint32_t t = threadIdx.x;
    // A: 16 x 32 s8 (4 registers per thread), B: 32 x 8 s8 (2 registers).
    const uint32_t a0 = 0x01010101u * ((t & 3u) + 1u), a1 = a0 ^ 0x02020202u, a2 = a0, a3 = a1;
    const uint32_t b0 = 0x01FF01FFu, b1 = 0xFF01FF01u;
    int32_t d[kChains][4];
#pragma unroll
    for (int c = 0; c < kChains; ++c)
#pragma unroll
        for (int i = 0; i < 4; ++i) d[c][i] = c + i;
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int c = 0; c < kChains; ++c)
            asm volatile(
                "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 "
                "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                : "+r"(d[c][0]), "+r"(d[c][1]), "+r"(d[c][2]), "+r"(d[c][3])
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    int32_t s = 0;
#pragma unroll
    for (int c = 0; c < kChains; ++c) s += d[c][0] ^ d[c][1] ^ d[c][2] ^ d[c][3];
    if (s == 0x7FFFFFFF) sink[blockIdx.x * blockDim.x + t] = s;
}

__global__ void __launch_bounds__(256) mma_bf16_probe_kernel(int64_t iters, int32_t* sink)
{
    const uint32_t t = threadIdx.x;
    // A: 16 x 16 bf16 (4 registers), B: 16 x 8 bf16 (2 registers); values
    // 1.0 and -1.0 so the fp32 sums stay exact small integers.
    const uint32_t one2 = 0x3F803F80u, mix2 = 0xBF803F80u;
    const uint32_t a0 = (t & 1u) ? one2 : mix2, a1 = one2, a2 = mix2, a3 = one2;
    const uint32_t b0 = one2, b1 = mix2;
    float d[kChains][4];
#pragma unroll
    for (int c = 0; c < kChains; ++c)
#pragma unroll
        for (int i = 0; i < 4; ++i) d[c][i] = static_cast<float>(c + i);
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int c = 0; c < kChains; ++c)
            asm volatile(
                "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                : "+f"(d[c][0]), "+f"(d[c][1]), "+f"(d[c][2]), "+f"(d[c][3])
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    float s = 0.0f;
#pragma unroll
    for (int c = 0; c < kChains; ++c) s += d[c][0] + d[c][1] + d[c][2] + d[c][3];
    if (s == -1.0e30f) sink[blockIdx.x * blockDim.x + t] = 1;
}

}  // namespace

extern "C" {

int64_t w8a8_peak_mma_sync_ops(int kind, int blocks, int threads, int64_t iters)
{
    if ((kind != W8A8_PEAK_MMA_S8 && kind != W8A8_PEAK_MMA_BF16) || blocks < 1 || threads < 32 || threads > 256 ||
        threads % 32 != 0 || iters < 1)
        return 0;
    const int64_t per_mma = kind == W8A8_PEAK_MMA_S8 ? 2 * 16 * 8 * 32 : 2 * 16 * 8 * 16;
    return static_cast<int64_t>(blocks) * (threads / 32) * iters * kChains * per_mma;
}

int w8a8_peak_mma_sync(int kind, int blocks, int threads, int64_t iters, int32_t* sink, void* stream)
{
    if (w8a8_peak_mma_sync_ops(kind, blocks, threads, iters) == 0 || sink == nullptr) return 1;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (kind == W8A8_PEAK_MMA_S8)
        mma_s8_probe_kernel<<<static_cast<unsigned>(blocks), static_cast<unsigned>(threads), 0, s>>>(iters, sink);
    else
        mma_bf16_probe_kernel<<<static_cast<unsigned>(blocks), static_cast<unsigned>(threads), 0, s>>>(iters, sink);
    return cudaGetLastError() == cudaSuccess ? 0 : 6;
}

}  // extern "C"
