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

template <typename TIn, int NV>
__global__ void __launch_bounds__(256) quant_blocks_kernel(const TIn* __restrict__ A, BlockGeom g,
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

// Persistent form, for blocks that one TMA box covers (D <= 256 elements,
// block_tokens <= 256, a block of at most 48 KB).  The input is described to
// TMA as a 4-D tensor with the layout's strides, innermost first: (d, token,
// head, batch) head-major, (d, head, token, batch) token-major, so a block of
// one (batch, head) is a box of D x block_tokens elements (the head and
// batch extents 1) that lands in shared memory as [block_tokens][D] in both
// layouts; tokens past L are filled with zeros by the copy (they do not
// change the absmax and are not stored).  Each CTA walks blocks blockIdx.x, + gridDim.x, ... with a ring of
// `stages` shared-memory buffers: the copies of its next blocks are in
// flight while it quantises the current one, so every SM keeps several
// blocks' bytes moving instead of waiting a full DRAM latency per block.
// A block is read twice from shared memory (absmax, then codes): thread t
// takes the 16-byte vector t % VD of tokens t / VD, t / VD + TPP, ...
// (consecutive threads read consecutive vectors: no bank conflicts; the
// int8 codes go to global memory as coalesced 8- or 4-byte stores).
constexpr int kQkRingThreads = 256;
constexpr int kQkMaxStages = 6;
constexpr uint32_t kQkRingBytes = 96 * 1024;

struct BlockRing {
    int64_t nblocks;        // B * H * nblk
    int32_t stage_bytes;    // one block's buffer, a multiple of 1024
    int32_t stages;         // 2 .. kQkMaxStages
    uint32_t box_bytes;     // bytes one block's copy delivers (block_tokens x D elements)
    int32_t head_major;     // tensor map dims: 1 (d, token, head, batch), 0 (d, head, token, batch)
    uint64_t wait_limit_ns;
};

template <typename TIn>
__global__ void __launch_bounds__(kQkRingThreads) quant_blocks_ring_kernel(const __grid_constant__ CUtensorMap tmap,
                                                                           BlockGeom g, BlockRing rg,
                                                                           int8_t* __restrict__ Q, float* __restrict__ S)
{
    using IV = InVec<TIn>;
    constexpr int E = IV::kElems;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full[kQkMaxStages];
    __shared__ float red[32];
    __shared__ int s_ok;
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t* ring = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const int t = static_cast<int>(threadIdx.x);
    const int G = static_cast<int>(gridDim.x);

    // Block index -> (batch, head, block in head); the copy of block blk into slot.
    auto coords = [&](int64_t blk, int64_t& b, int64_t& h, int64_t& j) {
        j = blk % g.nblk;
        const int64_t bh = blk / g.nblk;
        b = bh / g.H;
        h = bh - b * g.H;
    };
    auto issue = [&](int64_t blk, int slot) {
        int64_t b, h, j;
        coords(blk, b, h, j);
        const int32_t tok = static_cast<int32_t>(j * g.block_tokens);
        mbar_arrive_expect_tx(&full[slot], rg.box_bytes);
        tma_load_4d(ring + slot * rg.stage_bytes, &tmap, &full[slot], 0, rg.head_major ? tok : static_cast<int32_t>(h),
                    rg.head_major ? static_cast<int32_t>(h) : tok, static_cast<int32_t>(b));
    };
    if (t == 0) {
        for (int s = 0; s < rg.stages; ++s) mbar_init(&full[s], 1);
        mbar_fence_init();
        tma_prefetch_desc(&tmap);
        for (int s = 0; s < rg.stages; ++s) {
            const int64_t blk = blockIdx.x + static_cast<int64_t>(s) * G;
            if (blk < rg.nblocks) issue(blk, s);
        }
    }
    __syncthreads();

    const bool active = t < g.tpp * g.vd;
    const int col = active ? t % g.vd : 0;
    const int tok0 = active ? t / g.vd : static_cast<int>(g.block_tokens);
    int64_t i = 0;
    int64_t blk = blockIdx.x;
    for (; blk < rg.nblocks; blk += G, ++i) {
        const int slot = static_cast<int>(i % rg.stages);
        const uint32_t ph = static_cast<uint32_t>(i / rg.stages) & 1u;
        // One thread takes the bounded wait; all follow its outcome.
        if (t == 0) s_ok = mbar_wait(&full[slot], ph, rg.wait_limit_ns) ? 1 : 0;
        __syncthreads();
        if (!s_ok) break;
        int64_t b, h, j;
        coords(blk, b, h, j);
        const int64_t t0 = j * g.block_tokens;
        const int ntok = static_cast<int>(min(g.block_tokens, g.L - t0));
        const uint4* src = reinterpret_cast<const uint4*>(ring + slot * rg.stage_bytes);
        uint32_t m2 = 0;
        for (int tok = tok0; tok < ntok; tok += g.tpp) IV::absmax(src[tok * g.vd + col], m2);
        const RowScale rs = row_scale(block_max(IV::absmax_value(m2), red));
        if (t == 0) S[blk] = rs.s;
        const int64_t base = b * g.stride_b + h * g.stride_h + t0 * g.stride_t + static_cast<int64_t>(col) * E;
        for (int tok = tok0; tok < ntok; tok += g.tpp)
            quantize_vector<TIn, false>(src[tok * g.vd + col], rs, Q, base + tok * g.stride_t);
        __syncthreads();   // the slot is read out (and `red` is free again)
        const int64_t next = blk + static_cast<int64_t>(rg.stages) * G;
        if (t == 0 && next < rg.nblocks) issue(next, slot);
    }
    if (blk < rg.nblocks) {
        // A copy did not arrive within the limit: the blocks this CTA did
        // not finish get a NaN scale, and copies still in flight land (again
        // with the limit) before the CTA exits.
        if (t == 0) {
            for (int64_t k = blk; k < rg.nblocks; k += G) S[k] = __int_as_float(0x7FC00000);
            for (int s = 0; s < rg.stages; ++s) {
                const int64_t ii = i + s;
                const int64_t kb = blockIdx.x + ii * G;
                if (kb < rg.nblocks)
                    mbar_wait(&full[ii % rg.stages], static_cast<uint32_t>(ii / rg.stages) & 1u, rg.wait_limit_ns);
            }
        }
    }
}

}  // namespace w8a8
