// Per-block symmetric INT8 quantisation of attention Query and Key (zhidx
// TurboT2VA article, section 01 item 4: on the H20 path SageSLA quantises
// Query and Key to INT8).  A block is `block_tokens` consecutive tokens of one
// (batch, head); its scale is the block's absmax / 127 and its codes follow
// the same rule as the linear layer's rows:
//
//   s    = fp32(absmax / 127)      (IEEE division; zero block -> s = 1)
//   q    = clamp(round_half_even(fp32(x / s)), -127, 127)
//
// Layouts: the tensor is [B][H][L][D] ("HND") or [B][L][H][D] ("NHD"), D
// contiguous; the codes have the same shape and strides, the scales are
// [B][H][ceil(L / block_tokens)].
//
// Structure.  One CTA per block.  A token's D elements are VD = D / E
// 16-byte vectors; thread t takes vector t % VD of tokens t / VD, t / VD +
// TPP, ... (TPP tokens per pass), so its column in the token is fixed and no
// index is divided per vector, and every warp instruction covers whole
// 16-byte vectors of neighbouring tokens.  A CTA has up to 256 threads (a
// 128-token block of D = 128: 8 vectors per thread).  The block is held in
// registers while its absmax is reduced (shuffles, then one shared-memory
// step) and then quantised with the row quantiser's vector routine; blocks
// too long for the registers are read twice (the second time from L2).
#pragma once

#include <cstdint>

#include "quant_rows.cuh"

namespace w8a8 {

struct BlockGeom {
    int64_t H;             // heads
    int64_t L;             // tokens
    int64_t block_tokens;  // tokens per block
    int64_t nblk;          // blocks per (batch, head): ceil(L / block_tokens)
    int64_t stride_b;      // element strides of batch, head and token (codes share them)
    int64_t stride_h;
    int64_t stride_t;
    int32_t vd;            // 16-byte vectors per token: D / E, 1..256
    int32_t tpp;           // tokens per pass, 1 <= tpp * vd <= 256
};

// Up to 8 vectors a thread: at most 64 registers, four 256-thread CTAs per
// SM (79 registers gave three); 16 vectors keep their registers.
template <typename TIn, int NV>
__global__ void __launch_bounds__(256, NV >= 16 ? 2 : 4) quant_blocks_kernel(const TIn* __restrict__ A, BlockGeom g,
                                                           int8_t* __restrict__ Q, float* __restrict__ S)
{
    using IV = InVec<TIn>;
    constexpr int E = IV::kElems;
    __shared__ float red[32];

    const int64_t blk = blockIdx.x;          // ((b * H) + h) * nblk + j
    const int64_t j = blk % g.nblk;
    const int64_t bh = blk / g.nblk;
    const int64_t b = bh / g.H;
    const int64_t h = bh - b * g.H;
    const int64_t t0 = j * g.block_tokens;
    const int ntok = static_cast<int>(min(g.block_tokens, g.L - t0));
    const int t = static_cast<int>(threadIdx.x);
    const bool active = t < g.tpp * g.vd;    // the CTA is rounded up to whole warps
    const int col = active ? t % g.vd : 0;
    const int tok0 = active ? t / g.vd : ntok;
    const int64_t base = b * g.stride_b + h * g.stride_h + t0 * g.stride_t + static_cast<int64_t>(col) * E;
    const int64_t step = static_cast<int64_t>(g.tpp) * g.stride_t;   // elements between a thread's vectors

    uint32_t m2 = 0;
    if constexpr (NV > 0) {
        uint4 v[NV];
        const int64_t first = base + tok0 * g.stride_t;
#pragma unroll
        for (int i = 0; i < NV; ++i)
            v[i] = tok0 + i * g.tpp < ntok ? load_stream(reinterpret_cast<const uint4*>(A + first + i * step))
                                           : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int i = 0; i < NV; ++i) IV::absmax(v[i], m2);
        const RowScale rs = row_scale(block_max(IV::absmax_value(m2), red));
        if (t == 0) S[blk] = rs.s;
#pragma unroll
        for (int i = 0; i < NV; ++i)
            if (tok0 + i * g.tpp < ntok) quantize_vector<TIn, false>(v[i], rs, Q, first + i * step);
    } else {
        for (int tok = tok0; tok < ntok; tok += g.tpp)
            IV::absmax(load_stream(reinterpret_cast<const uint4*>(A + base + tok * g.stride_t)), m2);
        const RowScale rs = row_scale(block_max(IV::absmax_value(m2), red));
        if (t == 0) S[blk] = rs.s;
        for (int tok = tok0; tok < ntok; tok += g.tpp)
            quantize_vector<TIn, false>(*reinterpret_cast<const uint4*>(A + base + tok * g.stride_t), rs, Q,
                                        base + tok * g.stride_t);
    }
}

}  // namespace w8a8
