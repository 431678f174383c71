// Per-row symmetric INT8 quantisation (zhidx TurboT2VA article, section 01
// item 3 "量化策略": activations per row, dynamically; weights per output
// channel, statically — both are rows of the operand as stored).
//
//   s    = absmax / 127            (IEEE division, __fdiv_rn)
//   s==0 -> zero row: scale 1, codes 0
//   q    = clamp(rint_half_even(x / s), -127, 127)
//
// One CTA per row.  The row is read once from HBM with 16-byte vector loads
// (thread t takes vectors t, t + T, t + 2T, ... so every warp instruction
// covers 512 contiguous bytes), held in registers while the absmax is
// reduced (warp shuffles, then one shared-memory step across warps), then
// quantised and written with 4/8/16-byte vector stores.  Rows too long for
// the register budget take a second pass over the row instead (served from
// L2).  The codes go out either as int8 (the API's codes) or as bf16 values
// of the same integers (the tensor-core GEMM's operand).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

namespace w8a8 {

template <typename TIn>
struct InVec;

template <>
struct InVec<__nv_bfloat16> {
    static constexpr int kElems = 8;  // per 16-byte vector
    __device__ static __forceinline__ void unpack(const uint4& v, float (&f)[8])
    {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
};

template <>
struct InVec<float> {
    static constexpr int kElems = 4;
    __device__ static __forceinline__ void unpack(const uint4& v, float (&f)[4])
    {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
};

__device__ __forceinline__ int quant_code(float x, float s)
{
    const int r = __float2int_rn(__fdiv_rn(x, s));  // round to nearest, ties to even
    return min(127, max(-127, r));
}

// Writes E codes (E = 8 or 4) starting at element offset `e0` of row `row`.
template <bool kBf16Codes, int E>
__device__ __forceinline__ void store_codes(void* Q, int64_t off, const int (&q)[E])
{
    if constexpr (kBf16Codes) {
        uint32_t w[E / 2];
#pragma unroll
        for (int i = 0; i < E / 2; ++i) {
            const uint32_t lo = __bfloat16_as_ushort(__int2bfloat16_rn(q[2 * i]));
            const uint32_t hi = __bfloat16_as_ushort(__int2bfloat16_rn(q[2 * i + 1]));
            w[i] = lo | (hi << 16);
        }
        uint16_t* dst = static_cast<uint16_t*>(Q) + off;
        if constexpr (E == 8)
            *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
        else
            *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    } else {
        uint32_t w[E / 4];
#pragma unroll
        for (int i = 0; i < E / 4; ++i)
            w[i] = (static_cast<uint32_t>(q[4 * i]) & 0xFFu) | ((static_cast<uint32_t>(q[4 * i + 1]) & 0xFFu) << 8) |
                   ((static_cast<uint32_t>(q[4 * i + 2]) & 0xFFu) << 16) |
                   ((static_cast<uint32_t>(q[4 * i + 3]) & 0xFFu) << 24);
        int8_t* dst = static_cast<int8_t*>(Q) + off;
        if constexpr (E == 8)
            *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
        else
            *reinterpret_cast<uint32_t*>(dst) = w[0];
    }
}

__device__ __forceinline__ uint4 load_stream(const uint4* p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Block-wide max of non-negative values; every thread gets the result.
__device__ __forceinline__ float block_max(float v, float* red /* >= 32 floats */)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    const int nwarps = blockDim.x >> 5;
    if (nwarps == 1) return v;
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float m = 0.0f;
    for (int w = 0; w < nwarps; ++w) m = fmaxf(m, red[w]);
    return m;
}

// NV > 0: each thread keeps up to NV vectors of the row in registers (single
// HBM read).  NV == 0: two passes over the row (for very long rows).
// `status`, when not NULL, is cleared by block 0 (start of a linear call).
template <typename TIn, bool kBf16Codes, int NV>
__global__ void __launch_bounds__(1024) quant_rows_kernel(const TIn* __restrict__ A, int64_t K,
                                                          void* __restrict__ Q, float* __restrict__ S,
                                                          uint32_t* __restrict__ status)
{
    using IV = InVec<TIn>;
    constexpr int E = IV::kElems;
    __shared__ float red[32];

    const int64_t row = blockIdx.x;
    const int V = static_cast<int>(K / E);  // 16-byte vectors in the row (K % 16 == 0)
    const uint4* src = reinterpret_cast<const uint4*>(A + row * K);
    const int64_t out0 = row * K;
    const int T = blockDim.x;

    if (status != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *status = 0u;

    float amax = 0.0f;
    if constexpr (NV > 0) {
        uint4 v[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int idx = threadIdx.x + i * T;
            if (idx < V) v[i] = load_stream(src + idx);
        }
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int idx = threadIdx.x + i * T;
            if (idx < V) {
                float f[E];
                IV::unpack(v[i], f);
#pragma unroll
                for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(f[e]));
            }
        }
        amax = block_max(amax, red);
        const float s = __fdiv_rn(amax, 127.0f);
        const bool zero_row = (s == 0.0f);
        if (threadIdx.x == 0) S[row] = zero_row ? 1.0f : s;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int idx = threadIdx.x + i * T;
            if (idx < V) {
                float f[E];
                IV::unpack(v[i], f);
                int q[E];
#pragma unroll
                for (int e = 0; e < E; ++e) q[e] = zero_row ? 0 : quant_code(f[e], s);
                store_codes<kBf16Codes, E>(Q, out0 + static_cast<int64_t>(idx) * E, q);
            }
        }
    } else {
        for (int idx = threadIdx.x; idx < V; idx += T) {
            float f[E];
            IV::unpack(load_stream(src + idx), f);
#pragma unroll
            for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(f[e]));
        }
        amax = block_max(amax, red);
        const float s = __fdiv_rn(amax, 127.0f);
        const bool zero_row = (s == 0.0f);
        if (threadIdx.x == 0) S[row] = zero_row ? 1.0f : s;
        for (int idx = threadIdx.x; idx < V; idx += T) {
            float f[E];
            IV::unpack(src[idx], f);
            int q[E];
#pragma unroll
            for (int e = 0; e < E; ++e) q[e] = zero_row ? 0 : quant_code(f[e], s);
            store_codes<kBf16Codes, E>(Q, out0 + static_cast<int64_t>(idx) * E, q);
        }
    }
}

// int8 codes -> the same integers as bf16 (exact), 16 codes per thread step.
// `status`, when not NULL, is cleared by thread 0 of block 0.
__global__ void codes_to_bf16_kernel(const int8_t* __restrict__ Qi, uint16_t* __restrict__ Qb, int64_t n16,
                                     uint32_t* __restrict__ status)
{
    if (status != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *status = 0u;
    const uint4* src = reinterpret_cast<const uint4*>(Qi);
    uint4* dst = reinterpret_cast<uint4*>(Qb);
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n16;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint4 v = src[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int lo = static_cast<int8_t>((w[j] >> (16 * h)) & 0xFFu);
                const int hi = static_cast<int8_t>((w[j] >> (16 * h + 8)) & 0xFFu);
                o[2 * j + h] = static_cast<uint32_t>(__bfloat16_as_ushort(__int2bfloat16_rn(lo))) |
                               (static_cast<uint32_t>(__bfloat16_as_ushort(__int2bfloat16_rn(hi))) << 16);
            }
        }
        dst[2 * i] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[2 * i + 1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

}  // namespace w8a8
