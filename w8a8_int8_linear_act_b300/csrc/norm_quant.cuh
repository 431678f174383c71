// Normalisation and modulation fused into the per-row activation
// quantisation, the prologue of a linear layer in the joint Transformer
// (zhidx TurboT2VA article, section 01: normalisation, modulation, gated
// residual and rotary embedding are fused to cut intermediate reads and
// writes; arXiv paper, appendix C "Fused Multimodal Transformer
// Operations").  Per row x of K bf16 values:
//
//   RMS norm:   mu = 0
//   LayerNorm:  mu = fp32(sum_k x_k / K)
//   v   = fp32(sum_k (x_k - mu)^2 / K)
//   r   = 1 / sqrt(v + eps)                     (correctly rounded fp32)
//   y_k = bf16_rne(fma((x_k - mu) * r, 1 + scale_k, shift_k))
//
// each step one fp32 operation rounded to nearest, the last multiply and add
// fused into one (the sums in any order);
// scale and shift are optional [K] vectors (adaLN-style modulation shared by
// all rows).  y is then quantised by the row rule of quant_rows.cuh, and
// optionally also written out.  The unfused form would write y (2 B per
// element) and read it back for the quantiser; here the row is read once.
//
// Structure: as the quantiser (a warp per row, up to 16 vectors per lane,
// for K <= 4096; a CTA per row up to 32768), with the row held in registers
// through three reductions: the sum (LayerNorm), the sum of squared
// deviations, and the absmax of y.  The warp form is persistent: CTAs of
// eight or sixteen warps, as many as fit on the GPU at once (at most one per
// row), each preparing the modulation once in shared memory as fp32
// (1 + scale, shift); the rows are dealt to the CTAs in turn, so that every
// SM gets rows even when there are few, and each warp works through its
// rows grid-stride, copying its next row into a buffer of its own in shared
// memory while the current row's arithmetic runs, so that HBM keeps
// streaming during the arithmetic.  The per-element arithmetic
// runs on packed pairs of fp32 (f32x2), one instruction for two elements.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "quant_rows.cuh"

namespace w8a8 {

constexpr int kNormRms = 1;
constexpr int kNormLayer = 2;

struct NormParams {
    float eps;
    const void* scale;     // [K] or nullptr
    const void* shift;     // [K] or nullptr
    int32_t mod_f32;       // scale/shift dtype: 1 fp32, 0 bf16
    uint16_t* y_out;       // [R][K] bf16 y, or nullptr
};

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// Block-wide sum; every thread gets the result.  `red` is used by this
// reduction alone (the callers give each reduction its own array).
__device__ __forceinline__ float block_sum(float v, float* red)
{
    v = warp_sum(v);
    const int nwarps = blockDim.x >> 5;
    if (nwarps == 1) return v;
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float s = 0.0f;
    for (int w = 0; w < nwarps; ++w) s = __fadd_rn(s, red[w]);
    return s;
}

// Pairwise sum of eight partial sums.
__device__ __forceinline__ float sum8(const float (&p)[8])
{
    return __fadd_rn(__fadd_rn(__fadd_rn(p[0], p[1]), __fadd_rn(p[2], p[3])),
                     __fadd_rn(__fadd_rn(p[4], p[5]), __fadd_rn(p[6], p[7])));
}

// The eight modulation values of vector idx (elements 8 idx .. 8 idx + 7)
// as loaded: one 16-byte vector for bf16, two for fp32.
struct ModVec {
    uint4 a, b;
};

__device__ __forceinline__ ModVec load_mod(const void* p, int32_t f32, int idx)
{
    ModVec m;
    if (f32) {
        const uint4* q = static_cast<const uint4*>(p) + 2 * idx;
        m.a = __ldg(q);
        m.b = __ldg(q + 1);
    } else {
        m.a = __ldg(static_cast<const uint4*>(p) + idx);
        m.b = make_uint4(0, 0, 0, 0);
    }
    return m;
}

__device__ __forceinline__ void unpack_mod(const ModVec& m, int32_t f32, float (&out)[8])
{
    if (f32) {
        out[0] = __uint_as_float(m.a.x); out[1] = __uint_as_float(m.a.y);
        out[2] = __uint_as_float(m.a.z); out[3] = __uint_as_float(m.a.w);
        out[4] = __uint_as_float(m.b.x); out[5] = __uint_as_float(m.b.y);
        out[6] = __uint_as_float(m.b.z); out[7] = __uint_as_float(m.b.w);
    } else {
        InVec<__nv_bfloat16>::unpack(m.a, out);
    }
}

// Hides the packed row from the compiler between passes, so that each pass
// unpacks it again (two bf16 per register) instead of keeping all K/32
// unpacked floats of a lane live across the reductions.
template <int NV>
__device__ __forceinline__ void keep_packed(uint4 (&v)[NV])
{
#pragma unroll
    for (int i = 0; i < NV; ++i) asm volatile("" : "+r"(v[i].x), "+r"(v[i].y), "+r"(v[i].z), "+r"(v[i].w));
}

// Copies lane t's vectors t, t + 32, ... of row `row` into the warp's
// buffer in shared memory (one commit group).
template <int NV, bool kFull>
__device__ __forceinline__ void copy_row_async(const __nv_bfloat16* __restrict__ A, int64_t row, int64_t K,
                                               uint4* buf, int t)
{
    const int V = static_cast<int>(K / 8);
    const uint4* src = reinterpret_cast<const uint4*>(A + row * K);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int idx = t + i * 32;
        if (kFull || idx < V) cp_async_16(buf + idx, src + idx);
    }
    cp_async_commit();
}

// One row: thread t of T holds vectors t, t + T, ... of the row.
// kWarp: the row belongs to one warp (T = 32).  Its vectors are already on
// their way into the warp's shared-memory buffer `buf` (copy_row_async);
// once the first pass has taken them into registers, the copy of `next`
// (when not negative), the warp's following row, is started into the same
// buffer, so that it streams in while this row's arithmetic runs.  The
// modulation is staged in s_mod.
// Otherwise the row belongs to the whole CTA, is loaded straight into
// registers, reduces block-wide, and reads the modulation per vector.
// kFull: the row is exactly NV vectors per lane of the warp (K = 256 NV),
// so no lane has a vector out of range.
template <bool kBf16Codes, int NV, bool kWarp, bool kFull, int kNorm>
__device__ __forceinline__ void norm_quant_row(const __nv_bfloat16* __restrict__ A, int64_t row, int64_t next,
                                               int64_t K, const NormParams& np, void* __restrict__ Q,
                                               float* __restrict__ S, int t, int T, const float4* s_mod,
                                               uint4* buf, float* red_sum, float* red_sq, float* red_max)
{
    using IV = InVec<__nv_bfloat16>;
    const int V = static_cast<int>(K / 8);
    const uint4* src = reinterpret_cast<const uint4*>(A + row * K);
    const int64_t out0 = row * K;
    const float kf = static_cast<float>(K);

    uint4 v[NV];
    if constexpr (kWarp) {
        cp_async_wait_all();   // this lane's own copies: no exchange between lanes
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int idx = t + i * T;
            v[i] = (kFull || idx < V) ? buf[idx] : make_uint4(0, 0, 0, 0);
        }
    } else {
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int idx = t + i * T;
            v[i] = (kFull || idx < V) ? load_stream(src + idx) : make_uint4(0, 0, 0, 0);
        }
    }
    // The first pass below reads every v[i], so this lane's shared-memory
    // reads have returned before its copies of the next row overwrite them.
    auto start_next = [&]() {
        if constexpr (kWarp) {
            if (next >= 0) copy_row_async<NV, kFull>(A, next, K, buf, t);
        }
    };

    // Each sum runs in eight independent partial sums per thread (one per
    // element position of a vector), so the adds do not form one long
    // dependent chain; the partials are then added pairwise.
    float mu = 0.0f;
    if constexpr (kNorm == kNormLayer) {
        float2 p2[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                        make_float2(0.0f, 0.0f)};
#pragma unroll
        for (int i = 0; i < NV; ++i) {   // padding vectors are zero
            p2[0] = add2(p2[0], bf16x2_to_f2(v[i].x));
            p2[1] = add2(p2[1], bf16x2_to_f2(v[i].y));
            p2[2] = add2(p2[2], bf16x2_to_f2(v[i].z));
            p2[3] = add2(p2[3], bf16x2_to_f2(v[i].w));
        }
        const float p8[8] = {p2[0].x, p2[0].y, p2[1].x, p2[1].y, p2[2].x, p2[2].y, p2[3].x, p2[3].y};
        start_next();
        float s = sum8(p8);
        s = kWarp ? warp_sum(s) : block_sum(s, red_sum);
        mu = __fdiv_rn(s, kf);
        keep_packed(v);
    }
    float2 q2[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                    make_float2(0.0f, 0.0f)};
    const float2 mu2 = make_float2(mu, mu);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        if (kFull || t + i * T < V) {
            const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float2 d = bf16x2_to_f2(w[j]);
                if constexpr (kNorm == kNormLayer) d = sub2(d, mu2);
                q2[j] = fma2(d, d, q2[j]);
            }
        }
    }
    const float q8[8] = {q2[0].x, q2[0].y, q2[1].x, q2[1].y, q2[2].x, q2[2].y, q2[3].x, q2[3].y};
    if constexpr (kNorm != kNormLayer) start_next();
    float q = sum8(q8);
    q = kWarp ? warp_sum(q) : block_sum(q, red_sq);
    keep_packed(v);
    const float r = __frsqrt_rn(__fadd_rn(__fdiv_rn(q, kf), np.eps));

    // y, rounded to bf16, replaces x in the registers.
    const bool has_sc = np.scale != nullptr, has_sh = np.shift != nullptr;
    uint32_t m2 = 0;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int idx = t + i * T;
        if (kFull || idx < V) {
            float x[8], a[8], b[8];
            IV::unpack(v[i], x);
            if constexpr (kWarp) {
                const float4 a0 = s_mod[idx], a1 = s_mod[V + idx];
                const float4 b0 = s_mod[2 * V + idx], b1 = s_mod[3 * V + idx];
                a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
                a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
                b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
                b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
            } else {
                float sc[8], sh[8];
                if (has_sc) unpack_mod(load_mod(np.scale, np.mod_f32, idx), np.mod_f32, sc);
                if (has_sh) unpack_mod(load_mod(np.shift, np.mod_f32, idx), np.mod_f32, sh);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    a[e] = has_sc ? __fadd_rn(1.0f, sc[e]) : 1.0f;
                    b[e] = has_sh ? sh[e] : -0.0f;
                }
            }
            uint32_t yw[4];
            const float2 r2 = make_float2(r, r);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float2 d = make_float2(x[2 * j], x[2 * j + 1]);
                if constexpr (kNorm == kNormLayer) d = sub2(d, mu2);
                const float2 y = fma2(mul2(d, r2), make_float2(a[2 * j], a[2 * j + 1]),
                                      make_float2(b[2 * j], b[2 * j + 1]));
                yw[j] = pack_bf16x2(y.x, y.y);
            }
            v[i] = make_uint4(yw[0], yw[1], yw[2], yw[3]);
            if (np.y_out != nullptr)
                *reinterpret_cast<uint4*>(np.y_out + out0 + static_cast<int64_t>(idx) * 8) = v[i];
            IV::absmax(v[i], m2);
        }
    }
    const float amax = kWarp ? warp_max(IV::absmax_value(m2)) : block_max(IV::absmax_value(m2), red_max);
    const RowScale rs = row_scale(amax);
    if (t == 0) S[row] = rs.s;
    if (rs.corr) {
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int idx = t + i * T;
            if (kFull || idx < V) quantize_vector_corr<kBf16Codes>(v[i], rs, Q, out0 + static_cast<int64_t>(idx) * 8);
        }
    } else {
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int idx = t + i * T;
            if (kFull || idx < V)
                quantize_vector<__nv_bfloat16, kBf16Codes>(v[i], rs, Q, out0 + static_cast<int64_t>(idx) * 8);
        }
    }
}

// kRowsPerCta > 1 (warp form): a CTA of kRowsPerCta warps stages the
// modulation once, then warp w of CTA c takes rows w * gridDim.x + c,
// + stride, ... (stride = gridDim.x * kRowsPerCta: consecutive rows go to
// consecutive CTAs); the launcher sizes the grid to the CTAs that fit on
// the GPU at once (and at most one per row), so that every warp works
// through several rows, its next row streaming into its shared-memory
// buffer while it computes on the current one.  Dynamic shared memory:
// the modulation (8 B per element of a row), then a row buffer per warp
// (2 B per element).  kRowsPerCta == 1: a CTA per row (long rows).
// kFull (warp form only): K = 256 NV.
template <bool kBf16Codes, int NV, int kRowsPerCta, bool kFull, int kNorm>
__global__ void __launch_bounds__(kRowsPerCta > 1 ? 32 * kRowsPerCta : 256, kRowsPerCta > 1 && kRowsPerCta < 16 ? 2 : 1)
    norm_quant_rows_kernel(const __nv_bfloat16* __restrict__ A, int64_t R, int64_t K, NormParams np,
                           void* __restrict__ Q, float* __restrict__ S, uint32_t* __restrict__ header)
{
    __shared__ float red_sum[32], red_sq[32], red_max[32];

    grid_launch_dependents();
    if (header != nullptr && blockIdx.x == 0)
        for (int i = threadIdx.x; i < kHeaderWords; i += blockDim.x) header[i] = 0u;

    // Warp form: the CTA first turns the modulation into fp32 a = 1 + scale
    // (1 without scale) and b = shift (-0 without shift, which leaves every
    // sum unchanged) in shared memory, as four float4 arrays of V entries
    // (elements 0-3 and 4-7 of each vector apart, so that lanes reading
    // neighbouring vectors hit distinct banks).  fma(x r, 1, -0) and
    // fma(x r, a, -0) equal x r and (x r) a exactly, so y = fma(x r, a, b)
    // takes the same roundings as the steps it stands for.
    extern __shared__ float4 s_mod[];
    if constexpr (kRowsPerCta > 1) {
        const bool has_sc = np.scale != nullptr, has_sh = np.shift != nullptr;
        const int V = static_cast<int>(K / 8);
        for (int k8 = threadIdx.x; k8 < V; k8 += blockDim.x) {
            float a[8], b[8];
            if (has_sc) {
                unpack_mod(load_mod(np.scale, np.mod_f32, k8), np.mod_f32, a);
#pragma unroll
                for (int e = 0; e < 8; ++e) a[e] = __fadd_rn(1.0f, a[e]);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) a[e] = 1.0f;
            }
            if (has_sh) {
                unpack_mod(load_mod(np.shift, np.mod_f32, k8), np.mod_f32, b);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) b[e] = -0.0f;
            }
            s_mod[k8] = make_float4(a[0], a[1], a[2], a[3]);
            s_mod[V + k8] = make_float4(a[4], a[5], a[6], a[7]);
            s_mod[2 * V + k8] = make_float4(b[0], b[1], b[2], b[3]);
            s_mod[3 * V + k8] = make_float4(b[4], b[5], b[6], b[7]);
        }
        const int64_t stride = static_cast<int64_t>(gridDim.x) * kRowsPerCta;
        const int lane = static_cast<int>(threadIdx.x & 31);
        int64_t row = static_cast<int64_t>(threadIdx.x >> 5) * gridDim.x + blockIdx.x;
        uint4* buf = reinterpret_cast<uint4*>(s_mod + 4 * V) + (threadIdx.x >> 5) * V;
        if (row < R) copy_row_async<NV, kFull>(A, row, K, buf, lane);
        __syncthreads();
        for (; row < R; row += stride)
            norm_quant_row<kBf16Codes, NV, true, kFull, kNorm>(A, row, row + stride < R ? row + stride : -1, K, np,
                                                               Q, S, lane, 32, s_mod, buf, red_sum, red_sq,
                                                               red_max);
    } else {
        norm_quant_row<kBf16Codes, NV, false, false, kNorm>(A, static_cast<int64_t>(blockIdx.x), -1, K, np, Q, S,
                                                            static_cast<int>(threadIdx.x),
                                                            static_cast<int>(blockDim.x), s_mod, nullptr, red_sum,
                                                            red_sq, red_max);
    }
}

}  // namespace w8a8
