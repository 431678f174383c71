/*
 * w8a8_peaks.h — throughput probes of libw8a8_peaks.so, used to measure the
 * roofline denominators of the W8A8 linear on this GPU.
 *
 * Not part of the layer and without counterpart on the pages.  The layer's
 * contraction is exact INT8 x INT8 -> INT32 arithmetic.  sm_103a has no
 * integer form of the 5th-generation tensor-core MMA (ptxas rejects
 * tcgen05.mma kind::i8 for sm_103a), so the candidate INT8 rates are the
 * warp-level MMA (mma.sync, s8 operands, s32 accumulator) and library
 * kernels; the layer itself carries the codes as bf16 on tcgen05 kind::f16.
 * These probes time the warp-level MMA so that the benchmark can compare
 * the rates on the same GPU and say which one a "% of INT8 peak" uses.
 *
 * Conventions as in w8a8.h: `sink` is caller-owned device memory, `stream`
 * a cudaStream_t passed as void*, nothing is allocated or synchronised.
 */
#ifndef W8A8_PEAKS_H
#define W8A8_PEAKS_H

#include <stdint.h>

#if defined(__GNUC__)
#define W8A8_PEAKS_API __attribute__((visibility("default")))
#else
#define W8A8_PEAKS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define W8A8_PEAK_MMA_S8 0    /* mma.sync m16n8k32, s8 x s8 -> s32: 8192 ops per warp MMA */
#define W8A8_PEAK_MMA_BF16 1  /* mma.sync m16n8k16, bf16 x bf16 -> f32: 4096 ops per warp MMA */

/* Operations (2 per multiply-add) one w8a8_peak_mma_sync launch performs:
 * blocks x (threads / 32) warps x iters steps x 8 independent MMAs per step.
 * Returns 0 for arguments that launch would refuse.  Host only. */
W8A8_PEAKS_API int64_t w8a8_peak_mma_sync_ops(int kind, int blocks, int threads, int64_t iters);

/* Launches the probe of `kind` on `stream`: `blocks` CTAs of `threads`
 * threads (a multiple of 32, at most 256), each warp issuing `iters` steps
 * of 8 independent register-operand MMAs.  `sink` (device, at least
 * blocks * threads int32) is written only in a case that cannot occur; it
 * keeps the work from being optimised away.  Time the launch with events
 * on `stream`.  Returns 0, 1 for invalid arguments (nothing launched) or 6
 * when the launch failed. */
W8A8_PEAKS_API int w8a8_peak_mma_sync(int kind, int blocks, int threads, int64_t iters, int32_t* sink,
                                      void* stream);

#ifdef __cplusplus
}
#endif

#endif /* W8A8_PEAKS_H */
