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
// Structure.  A CTA per block at a time.  A token's D elements are VD = D / E
// 16-byte vectors; thread t takes vector t % VD of tokens t / VD, t / VD +
// TPP, ... (TPP tokens per pass), so its column in the token is fixed and no
// index is divided per vector, and every warp instruction covers whole
// 16-byte vectors of neighbouring tokens.  A CTA has up to 256 threads, or
// 512 for blocks of 2048 vectors or more (a 128-token block of D = 128: 512
// threads of 4 vectors), so that a persistent CTA works through more,
// smaller blocks' worth of copies.  The block is held in
// registers while its absmax is reduced (shuffles, then one shared-memory
// step) and then quantised with the row quantiser's vector routine; blocks
// too long for the registers are read twice (the second time from L2).
// With the block in registers the CTAs are persistent and each thread's
// vectors of the CTA's next block stream into shared memory meanwhile.
#pragma once

#include <cstdint>
#include <type_traits>

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

// Up to 8 vectors a thread: at most 64 registers, 1024 threads per SM (79
// registers gave 768); 16 vectors keep their registers.  CTAs of up to 512
// threads take up to 4 vectors a thread, 256 threads more.
//
// NV > 0: persistent.  The grid holds the CTAs that fit on the GPU at once;
// CTA c takes blocks c, c + gridDim.x, ...  Each thread copies its own
// vectors of its next block into shared memory (cp.async, NV * blockDim.x
// 16-byte slots of dynamic shared memory, slot i * blockDim.x + t for its
// vector i) while it reduces and quantises the current one, so that HBM
// keeps streaming during the arithmetic; no thread reads another's slots.
// NV == 0: a CTA per block (gridDim.x == number of blocks).
template <typename TIn, int NV>
__global__ void __launch_bounds__(NV >= 8 ? 256 : 512, NV >= 16 ? 2 : (NV >= 8 ? 4 : 2)) quant_blocks_kernel(const TIn* __restrict__ A, BlockGeom g,
                                                                             int64_t nblocks, int8_t* __restrict__ Q,
                                                                             float* __restrict__ S)
{
    using IV = InVec<TIn>;
    constexpr int E = IV::kElems;
    // Two reduction arrays, used alternately by consecutive blocks of a CTA:
    // a warp writing one for block n + 2 has passed block n + 1's barrier,
    // which every warp reaches only after its last read of block n's.
    __shared__ float red[2][32];

    const int t = static_cast<int>(threadIdx.x);
    const bool active = t < g.tpp * g.vd;    // the CTA is rounded up to whole warps
    const int col = active ? t % g.vd : 0;
    const int tok0 = active ? t / g.vd : static_cast<int>(g.block_tokens);
    const int64_t step = static_cast<int64_t>(g.tpp) * g.stride_t;   // elements between a thread's vectors

    // Element offset of this thread's first vector in block blk, and the
    // block's token count.  Block, head and block counts are below 2^31
    // (checked by the host), so the index split runs in 32 bits.
    auto locate = [&](int64_t blk, int& ntok) -> int64_t {
        const uint32_t nb = static_cast<uint32_t>(g.nblk), hh = static_cast<uint32_t>(g.H);
        const uint32_t bk = static_cast<uint32_t>(blk);   // blk = ((b * H) + h) * nblk + j
        const uint32_t bh = bk / nb;
        const uint32_t j = bk - bh * nb;
        const uint32_t b = bh / hh;
        const uint32_t h = bh - b * hh;
        const int64_t t0 = static_cast<int64_t>(j) * g.block_tokens;
        ntok = static_cast<int>(min(g.block_tokens, g.L - t0));
        return static_cast<int64_t>(b) * g.stride_b + static_cast<int64_t>(h) * g.stride_h +
               (t0 + tok0) * g.stride_t + static_cast<int64_t>(col) * E;
    };

    if constexpr (NV > 0) {
        extern __shared__ uint4 s_slots[];
        const int T = static_cast<int>(blockDim.x);
        // Blocks of exactly NV passes of every thread (the common case: whole
        // blocks, every thread active) skip the per-vector range checks.
        const bool whole_geom = g.tpp * NV == g.block_tokens && g.tpp * g.vd == T;
        auto copy_block = [&](int64_t first, int ntok, auto whole_c) {
            constexpr bool kWhole = decltype(whole_c)::value;
#pragma unroll
            for (int i = 0; i < NV; ++i)
                if (kWhole || tok0 + i * g.tpp < ntok) cp_async_16(&s_slots[i * T + t], A + first + i * step);
            cp_async_commit();
        };
        // One block: its vectors from the slots, the absmax, the next block's
        // copies (once every slot has been read), the scale, the codes.
        auto run_block = [&](int64_t blk, int it, int64_t first, int ntok, int64_t next_first, int next_ntok,
                             auto whole_c) {
            constexpr bool kWhole = decltype(whole_c)::value;
            cp_async_wait_all();
            uint4 v[NV];
#pragma unroll
            for (int i = 0; i < NV; ++i)
                v[i] = (kWhole || tok0 + i * g.tpp < ntok) ? s_slots[i * T + t] : make_uint4(0, 0, 0, 0);
            uint32_t m2 = 0;
#pragma unroll
            for (int i = 0; i < NV; ++i) IV::absmax(v[i], m2);
            if (next_first >= 0) {
                if (whole_geom && next_ntok == g.block_tokens)
                    copy_block(next_first, next_ntok, std::true_type{});
                else
                    copy_block(next_first, next_ntok, std::false_type{});
            }
            const RowScale rs = row_scale(block_max(IV::absmax_value(m2), red[it & 1]));
            if (t == 0) S[blk] = rs.s;
            if constexpr (E == 8) {
                if (rs.corr) {
#pragma unroll
                    for (int i = 0; i < NV; ++i)
                        if (kWhole || tok0 + i * g.tpp < ntok) quantize_vector_corr<false>(v[i], rs, Q, first + i * step);
                } else if (tok0 < ntok) {
                    quantize_strided_by_tie_test<TIn, false>(A, first, step, (ntok - tok0 + g.tpp - 1) / g.tpp, rs,
                                                             Q);
                }
            } else {
#pragma unroll
                for (int i = 0; i < NV; ++i)
                    if (kWhole || tok0 + i * g.tpp < ntok) quantize_vector<TIn, false>(v[i], rs, Q, first + i * step);
            }
        };
        int64_t blk = blockIdx.x;
        int ntok = 0;
        int64_t first = 0;
        if (blk < nblocks) {
            first = locate(blk, ntok);
            if (whole_geom && ntok == g.block_tokens)
                copy_block(first, ntok, std::true_type{});
            else
                copy_block(first, ntok, std::false_type{});
        }
        for (int it = 0; blk < nblocks; blk += gridDim.x, ++it) {
            int next_ntok = 0;
            int64_t next_first = -1;
            if (blk + gridDim.x < nblocks) next_first = locate(blk + gridDim.x, next_ntok);
            if (whole_geom && ntok == g.block_tokens)
                run_block(blk, it, first, ntok, next_first, next_ntok, std::true_type{});
            else
                run_block(blk, it, first, ntok, next_first, next_ntok, std::false_type{});
            first = next_first;
            ntok = next_ntok;
        }
    } else {
        const int64_t blk = blockIdx.x;
        int ntok;
        const int64_t base = locate(blk, ntok);
        uint32_t m2 = 0;
        for (int tok = tok0; tok < ntok; tok += g.tpp)
            IV::absmax(load_stream(reinterpret_cast<const uint4*>(A + base + (tok - tok0) * g.stride_t)), m2);
        const RowScale rs = row_scale(block_max(IV::absmax_value(m2), red[0]));
        if (t == 0) S[blk] = rs.s;
        for (int tok = tok0; tok < ntok; tok += g.tpp) {
            const int64_t off = base + (tok - tok0) * g.stride_t;
            if (E == 8 && rs.corr)
                quantize_vector_corr<false>(*reinterpret_cast<const uint4*>(A + off), rs, Q, off);
            else
                quantize_vector<TIn, false>(*reinterpret_cast<const uint4*>(A + off), rs, Q, off);
        }
    }
}

}  // namespace w8a8
