// Per-row symmetric INT8 quantisation (zhidx TurboT2VA article, section 01
// item 3 "量化策略": activations per row, dynamically; weights per output
// channel, statically — both are rows of the operand as stored).
//
//   s    = fp32(absmax / 127)      (IEEE division)
//   s==0 -> zero row: scale 1, codes 0
//   q    = clamp(round_half_even(fp32(x / s)), -127, 127)
//
// Structure.  A row is read once from HBM with 16-byte vector loads (thread
// t of the row's T threads takes vectors t, t + T, t + 2T, ..., so every warp
// instruction covers 512 contiguous bytes) and held in registers while its
// absmax is reduced, then quantised and written with 8/16-byte vector
// stores.  Rows of up to 512 vectors (K <= 4096 for bf16, 2048 for fp32) take
// one warp each, four rows per CTA, reduced with warp shuffles alone; rows of
// up to 4096 vectors take a CTA of up to 256 threads with 16 vectors each
// (shuffles, then one shared-memory step).  Longer rows take a second pass
// over the row instead of holding it (served from L2).  The codes go out either as int8 (the API's
// codes) or as bf16 values of the same integers (the tensor-core GEMM's
// operand).
//
// Exact codes without a division per element.  With r = fp32(1/s)
// (correctly rounded) and p = x * r the exact product, |p - x/s| <=
// |x/s| * 2^-24 < 2^-17 for |x/s| <= 127.5, and the fp32 quotient fp32(x/s)
// is within 2^-18 of x/s, so |p - fp32(x/s)| < 2^-16.  One fused multiply-add
// t = fma(x, r, 1.5 * 2^23) rounds p + 1.5 * 2^23 once; for |p| < 2^22 that
// sum has a unit in the last place of exactly 1, so q = t - 1.5 * 2^23 is
// round_half_even(p) (the classic magic-number rounding, with the product
// never rounded on its own).  A second fma gives d = fp32(p - q) (relative
// error 2^-24).  Whenever |d| <= 1/2 - 2^-14, p lies more than
// 2^-14 - 2^-24 > 2^-16 inside (q - 1/2, q + 1/2), so fp32(x/s) lies strictly
// inside it too and rounds to the same q.  Only elements closer than that
// to a tie (about one in 8000 for smooth data), and rows whose reciprocal
// overflows (s below 2^-128), take the IEEE division.  The test is made
// once per 16-byte vector (the largest |d| of its elements), and the
// division sits behind that one branch in an out-of-line function.  In the
// fast path |p| <= 127 * (1 + 2^-22), so no clamp is needed there.
//
// bf16 inputs take neither the test nor the division (quantize_vector_corr):
// one more fused multiply-add turns fp32(x r) into the correctly rounded
// quotient fp32(x / s) itself (Markstein's correction step), and that rounds
// to the code directly.  bf16 data with a round absmax puts many elements
// exactly on a tie of x r (0.3 % of a Gaussian Query tensor), where the test
// above would send most vectors to the division; fp32 inputs keep the test.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "ptx_sm103.cuh"

namespace w8a8 {

constexpr float kRoundMagic = 12582912.0f;            // 1.5 * 2^23
constexpr uint32_t kRoundMagicBits = 0x4B400000u;
constexpr float kNearHalf = 0.5f - 0.00006103515625f; // 0.5 - 2^-14
constexpr int kHeaderWords = 256;                     // workspace header: 1 KB of 32-bit words

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
    // Largest |x| of the vector folded into a running maximum kept as two
    // bf16 magnitudes (bit patterns of non-negative floats order like the
    // values, so an unsigned 16-bit max is exact).
    __device__ static __forceinline__ void absmax(const uint4& v, uint32_t& m2)
    {
        m2 = __vmaxu2(m2, v.x & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, v.y & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, v.z & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, v.w & 0x7FFF7FFFu);
    }
    __device__ static __forceinline__ float absmax_value(uint32_t m2)
    {
        return fmaxf(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xFFFF0000u));
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
    __device__ static __forceinline__ void absmax(const uint4& v, uint32_t& m)
    {
        m = max(m, v.x & 0x7FFFFFFFu);
        m = max(m, v.y & 0x7FFFFFFFu);
        m = max(m, v.z & 0x7FFFFFFFu);
        m = max(m, v.w & 0x7FFFFFFFu);
    }
    __device__ static __forceinline__ float absmax_value(uint32_t m) { return __uint_as_float(m); }
};

// Row constants shared by every element of a row.
struct RowScale {
    float s;        // scale (1 for a zero row)
    float r;        // fp32(1 / s)
    bool exact;     // reciprocal overflowed: every element takes the division
    bool corr;      // bf16 elements may take quantize_vector_corr (s >= 2^-100, r finite)
};

// A zero row (amax / 127 == 0, including an fp32 amax that underflows) gets
// s = 1; its elements are all zero or so small that x * 1 rounds to code 0.
__device__ __forceinline__ RowScale row_scale(float amax)
{
    RowScale rs;
    const float s = __fdiv_rn(amax, 127.0f);
    rs.s = (s == 0.0f) ? 1.0f : s;
    rs.r = __frcp_rn(rs.s);
    rs.exact = !(fabsf(rs.r) <= 3.402823466e38f);
    rs.corr = !rs.exact && rs.s >= 7.888609052210118e-31f;   // 2^-100
    return rs;
}

// Writes E codes at element offset `off`: for bf16 codes q holds the codes
// as integer-valued floats, for int8 codes it holds kRoundMagic + code.
template <bool kBf16Codes, int E>
__device__ __forceinline__ void store_codes(void* Q, int64_t off, const float (&q)[E])
{
    if constexpr (kBf16Codes) {
        // bf16 of the integer q is the top half of fp32(q): |q| <= 127 needs
        // at most 8 significant bits, so the truncation is exact.
        uint32_t w[E / 2];
#pragma unroll
        for (int i = 0; i < E / 2; ++i) w[i] = __byte_perm(__float_as_uint(q[2 * i]), __float_as_uint(q[2 * i + 1]), 0x7632);
        uint16_t* dst = static_cast<uint16_t*>(Q) + off;
        if constexpr (E == 8)
            *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
        else
            *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    } else {
        // q here holds kRoundMagic + code (see quantize_vector): the low
        // byte of its bits is the code's two's-complement byte
        // (kRoundMagicBits has a zero low byte and |code| < 2^22).
        uint32_t b[E];
#pragma unroll
        for (int i = 0; i < E; ++i) b[i] = __float_as_uint(q[i]);
        uint32_t w[E / 4];
#pragma unroll
        for (int i = 0; i < E / 4; ++i) {
            const uint32_t p01 = __byte_perm(b[4 * i], b[4 * i + 1], 0x0040);
            const uint32_t p23 = __byte_perm(b[4 * i + 2], b[4 * i + 3], 0x0040);
            w[i] = __byte_perm(p01, p23, 0x5410);
        }
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

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// Block-wide max of non-negative values; every thread gets the result.
__device__ __forceinline__ float block_max(float v, float* red /* >= 32 floats */)
{
    v = warp_max(v);
    const int nwarps = blockDim.x >> 5;
    if (nwarps == 1) return v;
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    // Every warp folds the per-warp maxima with shuffles (max is exact and
    // order-free, so every thread gets the same value).
    const int lane = static_cast<int>(threadIdx.x & 31);
    return warp_max(lane < nwarps ? red[lane] : 0.0f);
}

// round_half_even(clamp(fp32(x / s), -127, 127)) by IEEE division.  Out of
// line: it runs only for elements within 2^-14 of a tie, and inlining its
// code at every element would crowd the instruction cache.
__device__ __noinline__ float code_by_division(float x, float s)
{
    const float d = fminf(fmaxf(__fdiv_rn(x, s), -127.0f), 127.0f);
    return __fsub_rn(__fadd_rn(d, kRoundMagic), kRoundMagic);
}

// Codes of one 16-byte vector.  Fast path: x * r rounded half-to-even by one
// fused multiply-add with the magic constant; if any element of the vector
// lies within 2^-14 of a tie (or the row needs exact division), that element
// is redone with the IEEE quotient fp32(x / s), clamped to [-127, 127].
template <typename TIn, bool kBf16Codes>
__device__ __forceinline__ void quantize_vector(const uint4& vec, const RowScale& rs, void* Q, int64_t off)
{
    using IV = InVec<TIn>;
    constexpr int E = IV::kElems;
    float x[E];
    IV::unpack(vec, x);
    // t = kRoundMagic + code; the int8 store takes t as it is, the bf16 one
    // the code q = t - kRoundMagic.
    float t[E], q[E];
    float dmax = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        t[e] = __fmaf_rn(x[e], rs.r, kRoundMagic);
        q[e] = __fsub_rn(t[e], kRoundMagic);
        dmax = fmaxf(dmax, fabsf(__fmaf_rn(x[e], rs.r, -q[e])));
    }
    if (dmax > kNearHalf || rs.exact) {
#pragma unroll
        for (int e = 0; e < E; ++e)
            if (rs.exact || fabsf(__fmaf_rn(x[e], rs.r, -q[e])) > kNearHalf) {
                q[e] = code_by_division(x[e], rs.s);
                t[e] = __fadd_rn(q[e], kRoundMagic);
            }
    }
    if constexpr (kBf16Codes)
        store_codes<true, E>(Q, off, q);
    else
        store_codes<false, E>(Q, off, t);
}

// Two independent fp32 operations in one instruction (sm_100 and later);
// each half is rounded exactly as the scalar operation would round it, so
// the packed forms change no result, only the instruction count.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 add2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 sub2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// Both bf16 of a 32-bit word as fp32 (low half first).
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w)
{
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// Codes of one vector of bf16, without a tie test or a division, for a row
// with rs.corr.  Per element, in packed pairs of fp32:
//   q0  = fp32(x r)
//   rem = fma(-q0, s, x)      the remainder x - q0 s, exact
//   q1  = fma(rem, r, q0)     = fp32(x / s), the correctly rounded quotient
//   t   = q1 + 1.5 2^23       rounds q1 to an integer, half to even
// The last FMA is Markstein's correction step (P. Markstein, IBM J. Res.
// Dev. 34(1), 1990; the FMA-based division theorems in Muller et al.,
// Handbook of Floating-Point Arithmetic, ch. 5): with r the correctly rounded
// reciprocal it yields the correctly rounded quotient, so rounding q1 to an
// integer gives exactly round_half_even(fp32(x / s)) -- the codes of the
// division form, ties included, which the fast path of quantize_vector has
// to refer to the division.  For bf16 x and s = fp32(amax / 127) with amax
// bf16 this was checked against exact rational arithmetic for every pair of
// significands and 40 binary orders of magnitude of x below amax, both
// signs; the steps scale exactly by powers of two, which covers every row
// whose values stay normal (s >= 2^-100; other rows use quantize_vector).
// |fp32(x / s)| <= 127 (1 + 2^-23) here, so no clamp is needed.
template <bool kBf16Codes>
__device__ __forceinline__ void quantize_vector_corr(const uint4& vec, const RowScale& rs, void* Q, int64_t off)
{
    const uint32_t w[4] = {vec.x, vec.y, vec.z, vec.w};
    const float2 rr = make_float2(rs.r, rs.r), ns = make_float2(-rs.s, -rs.s);
    const float2 mm = make_float2(kRoundMagic, kRoundMagic);
    float t[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 x = bf16x2_to_f2(w[i]);
        const float2 q0 = mul2(x, rr);
        const float2 rem = fma2(q0, ns, x);
        const float2 q1 = fma2(rem, rr, q0);
        const float2 tt = add2(q1, mm);
        t[2 * i] = tt.x;
        t[2 * i + 1] = tt.y;
    }
    if constexpr (kBf16Codes) {
        // q = t - M, +0 for a zero code.
        float q[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 qq = sub2(make_float2(t[2 * i], t[2 * i + 1]), mm);
            q[2 * i] = qq.x;
            q[2 * i + 1] = qq.y;
        }
        store_codes<true, 8>(Q, off, q);
    } else {
        store_codes<false, 8>(Q, off, t);
    }
}

// Codes, by quantize_vector, of `count` 16-byte vectors of A at element
// offsets base, base + stride, ... (the codes at the same offsets of Q).  For
// the rare bf16 rows without rs.corr (scales below 2^-100, or a reciprocal
// that overflows): out of line and reading the vectors again from memory, so
// that the common path keeps neither its registers nor its code.
template <typename TIn, bool kBf16Codes>
__device__ __noinline__ void quantize_strided_by_tie_test(const TIn* __restrict__ A, int64_t base, int64_t stride,
                                                          int count, RowScale rs, void* __restrict__ Q)
{
    for (int j = 0; j < count; ++j) {
        const int64_t off = base + j * stride;
        quantize_vector<TIn, kBf16Codes>(*reinterpret_cast<const uint4*>(A + off), rs, Q, off);
    }
}

// Rows of A [R][K] -> codes Q [R][K] and scales S [R].
//   kRowsPerCta > 0: blockDim.x == 32 * kRowsPerCta, warp w takes row
//                    blockIdx.x * kRowsPerCta + w (rows past R do nothing);
//                    registers are capped so that 21 warps fit on an SM;
//   kRowsPerCta == 0: the whole CTA takes row blockIdx.x.
// NV > 0: each thread keeps up to NV vectors of the row in registers (single
// HBM read).  NV == 0: two passes over the row (for very long rows).
// `header`, when not NULL, is the workspace header (status word and the
// GEMM's split-tile counters), cleared by block 0 at the start of a call.
// `zero_rows`, when not NULL, is a per-row word cleared with the row's scale
// (the row absmax that the following GEMM gathers for the next layer).
constexpr int kQuantWarpsPerSm = 21;

template <typename TIn, bool kBf16Codes, int NV, int kRowsPerCta>
__global__ void __launch_bounds__(kRowsPerCta > 0 ? 32 * kRowsPerCta : (NV > 0 ? 256 : 1024),
                                  kRowsPerCta > 0 ? kQuantWarpsPerSm / (kRowsPerCta > 0 ? kRowsPerCta : 1)
                                                  : (NV > 0 && NV <= 2 ? 8 : 1))
    quant_rows_kernel(const TIn* __restrict__ A, int64_t R, int64_t K,
                                                          void* __restrict__ Q, float* __restrict__ S,
                                                          uint32_t* __restrict__ header,
                                                          uint32_t* __restrict__ zero_rows)
{
    using IV = InVec<TIn>;
    constexpr int E = IV::kElems;
    __shared__ float red[32];

    // The GEMM that follows may be scheduled as soon as every CTA of this
    // grid is resident; it waits for this grid's results before reading.
    grid_launch_dependents();
    if (header != nullptr && blockIdx.x == 0)
        for (int i = threadIdx.x; i < kHeaderWords; i += blockDim.x) header[i] = 0u;

    const int64_t row = kRowsPerCta > 0 ? static_cast<int64_t>(blockIdx.x) * kRowsPerCta + (threadIdx.x >> 5)
                                        : static_cast<int64_t>(blockIdx.x);
    if (kRowsPerCta > 0 && row >= R) return;   // warp-uniform; no block-wide barrier follows
    const int T = kRowsPerCta > 0 ? 32 : static_cast<int>(blockDim.x);
    const int t = kRowsPerCta > 0 ? static_cast<int>(threadIdx.x & 31) : static_cast<int>(threadIdx.x);
    const int V = static_cast<int>(K / E);  // 16-byte vectors in the row (K % 16 == 0)
    const uint4* src = reinterpret_cast<const uint4*>(A + row * K);
    const int64_t out0 = row * K;

    uint32_t m2 = 0;
    if constexpr (NV > 0) {
        uint4 v[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int idx = t + i * T;
            v[i] = (idx < V) ? load_stream(src + idx) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < NV; ++i) IV::absmax(v[i], m2);
        const float amax = kRowsPerCta > 0 ? warp_max(IV::absmax_value(m2)) : block_max(IV::absmax_value(m2), red);
        const RowScale rs = row_scale(amax);
        if (t == 0) {
            S[row] = rs.s;
            if (zero_rows != nullptr) zero_rows[row] = 0u;
        }
        if constexpr (E == 8) {
            if (rs.corr) {
#pragma unroll
                for (int i = 0; i < NV; ++i) {
                    const int idx = t + i * T;
                    if (idx < V)
                        quantize_vector_corr<kBf16Codes>(v[i], rs, Q, out0 + static_cast<int64_t>(idx) * E);
                }
            } else if (t < V) {
                quantize_strided_by_tie_test<TIn, kBf16Codes>(A, out0 + static_cast<int64_t>(t) * E,
                                                              static_cast<int64_t>(T) * E, (V - t + T - 1) / T, rs, Q);
            }
        } else {
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int idx = t + i * T;
                if (idx < V) quantize_vector<TIn, kBf16Codes>(v[i], rs, Q, out0 + static_cast<int64_t>(idx) * E);
            }
        }
    } else {
        for (int idx = t; idx < V; idx += T) IV::absmax(load_stream(src + idx), m2);
        const float amax = kRowsPerCta > 0 ? warp_max(IV::absmax_value(m2)) : block_max(IV::absmax_value(m2), red);
        const RowScale rs = row_scale(amax);
        if (t == 0) {
            S[row] = rs.s;
            if (zero_rows != nullptr) zero_rows[row] = 0u;
        }
        if (E == 8 && rs.corr) {
            for (int idx = t; idx < V; idx += T)
                quantize_vector_corr<kBf16Codes>(src[idx], rs, Q, out0 + static_cast<int64_t>(idx) * E);
        } else if (t < V) {
            quantize_strided_by_tie_test<TIn, kBf16Codes>(A, out0 + static_cast<int64_t>(t) * E,
                                                          static_cast<int64_t>(T) * E, (V - t + T - 1) / T, rs, Q);
        }
    }
}

// Codes of bf16 rows whose absmax is already known: the row rule without the
// reduction, for the layer after a GEMM that gathered each row's max |Y|
// while writing Y (amax_bits: fp32 bits, 0 for an all-zero row).  One CTA
// per row; a thread loads up to kU vectors before quantising any, so every
// warp keeps 16 * kU bytes per lane in flight.  Launched as a programmatic
// dependent of that GEMM: it waits for the GEMM's results before reading.
template <bool kBf16Codes, int kU>
__global__ void __launch_bounds__(256) codes_known_amax_kernel(const __nv_bfloat16* __restrict__ A, int64_t K,
                                                               const uint32_t* __restrict__ amax_bits,
                                                               void* __restrict__ Q, float* __restrict__ S)
{
    grid_launch_dependents();
    grid_wait_prerequisites();
    const int64_t row = blockIdx.x;
    const RowScale rs = row_scale(__uint_as_float(amax_bits[row]));
    if (threadIdx.x == 0) S[row] = rs.s;
    const int V = static_cast<int>(K / 8);
    const uint4* src = reinterpret_cast<const uint4*>(A + row * K);
    const int64_t out0 = row * K;
    for (int base = static_cast<int>(threadIdx.x); base < V; base += kU * static_cast<int>(blockDim.x)) {
        uint4 v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int idx = base + u * static_cast<int>(blockDim.x);
            v[u] = idx < V ? load_stream(src + idx) : make_uint4(0, 0, 0, 0);
        }
        if (rs.corr) {
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int idx = base + u * static_cast<int>(blockDim.x);
                if (idx < V) quantize_vector_corr<kBf16Codes>(v[u], rs, Q, out0 + static_cast<int64_t>(idx) * 8);
            }
        } else {
            const int n = (V - base + static_cast<int>(blockDim.x) - 1) / static_cast<int>(blockDim.x);
            quantize_strided_by_tie_test<__nv_bfloat16, kBf16Codes>(A, out0 + static_cast<int64_t>(base) * 8,
                                                                    static_cast<int64_t>(blockDim.x) * 8,
                                                                    n < kU ? n : kU, rs, Q);
        }
    }
}

// Clears the workspace header (status word and split-tile counters) for a
// GEMM that no quantiser precedes (the BF16 linear).  It releases its
// dependents at entry, so the GEMM, launched as its programmatic dependent,
// runs its set-up meanwhile and waits on the device for these stores.
__global__ void __launch_bounds__(256) clear_header_kernel(uint32_t* __restrict__ header)
{
    grid_launch_dependents();
    for (int i = threadIdx.x; i < kHeaderWords; i += blockDim.x) header[i] = 0u;
}

// int8 codes -> the same integers as bf16 (exact), 16 codes per thread step.
// `header`, when not NULL, is the workspace header, cleared by block 0.
__global__ void codes_to_bf16_kernel(const int8_t* __restrict__ Qi, uint16_t* __restrict__ Qb, int64_t n16,
                                     uint32_t* __restrict__ header)
{
    grid_launch_dependents();
    if (header != nullptr && blockIdx.x == 0)
        for (int i = threadIdx.x; i < kHeaderWords; i += blockDim.x) header[i] = 0u;
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
