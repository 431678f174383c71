/*
 * w8a8.h — C ABI of the guarded W8A8 linear layer on B300 (sm_103a).
 *
 * The operation.  The zhidx article "音视频生成提速54倍！浙大等团队开源联合蒸馏方案
 * TurboT2VA", section 01 item 3 ("量化策略"), gives the linear layers of the
 * video/audio transformer branches as W8A8: the weight is quantised once,
 * offline, to INT8 with one scale per output channel; the activation is
 * quantised on every call to INT8 with one scale per row (token); the product
 * accumulates in INT32; the scales and the bias are applied once, after the
 * whole accumulation.  Shapes the fast operator cannot take fall back to the
 * native BF16 linear.  The paperlayer summary of arXiv 2608.24674, section
 * "C. Fused Multimodal Transformer Operations", calls this guarded
 * acceleration by shape with a safe fallback.
 *
 * Arithmetic, identical to the CPU oracle the tests compare against:
 *   s[r]    = fp32(absmax_k |A[r][k]| / 127)            IEEE division
 *             a row with s == 0 (all zeros, or an fp32 absmax that underflows)
 *             gets s = 1 and zero codes
 *   q[r][k] = clamp(round_half_even(fp32(A[r][k] / s[r])), -127, 127)
 *   acc[m][n] = sum_k Xq[m][k] * Wq[n][k]                exact, INT32
 *   Y[m][n]   = bf16_rne(((float)acc * sx[m]) * sw[n] + bias[n])
 *               (each step an fp32 operation rounded to nearest even)
 *
 * Conventions for every entry point below.
 *  - Matrices are row-major with the K dimension contiguous: X [M][K],
 *    W / Wq / Wp [N][K] (one row per output channel, as in a linear layer's
 *    weight), Y [M][N].
 *  - Every pointer argument is DEVICE memory owned by the caller, unless a
 *    comment says otherwise.  The library allocates nothing, frees nothing
 *    and never synchronises the stream or the device (except
 *    w8a8_read_status, which says so).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Work is enqueued on it asynchronously; results are ready when
 *    the stream reaches that point.  The current CUDA device must be the one
 *    that owns the pointers.
 *  - `dtype` arguments take a w8a8_dtype value.
 *  - Errors are returned as w8a8_status.  On any error other than
 *    W8A8_ERR_CUDA nothing has been launched.  The library never throws,
 *    exits, traps or asserts on the device.  Device-side waits are bounded:
 *    a wait that runs out records W8A8_DEV_* bits in the workspace's status
 *    word (see w8a8_read_status) and the kernel returns.
 *  - Alignment: X, W, Wq, Wp, Y, acc, sw, bias and workspace 16-byte
 *    aligned; sx 4-byte aligned (allocations from cudaMalloc or the PyTorch
 *    caching allocator satisfy all of these).
 */
#ifndef W8A8_H
#define W8A8_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define W8A8_API __attribute__((visibility("default")))
#else
#define W8A8_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    W8A8_OK = 0,
    W8A8_ERR_INVALID_ARG = 1,       /* NULL pointer, negative size, unknown dtype value */
    W8A8_ERR_DTYPE = 2,             /* dtype not accepted by this entry point */
    W8A8_ERR_ALIGNMENT = 3,         /* a pointer misses the alignment stated above */
    W8A8_ERR_UNSUPPORTED_SHAPE = 4, /* the shape guard rejects (M, N, K); run the BF16 linear instead */
    W8A8_ERR_WORKSPACE = 5,         /* workspace NULL or smaller than *_workspace_bytes() */
    W8A8_ERR_CUDA = 6,              /* a CUDA runtime call or kernel launch failed */
    W8A8_ERR_TIMEOUT = 7,           /* a device-side wait ran out (from w8a8_read_status) */
    W8A8_ERR_NO_DEVICE = 8          /* no sm_103 device current */
} w8a8_status;

typedef enum {
    W8A8_F32 = 0,
    W8A8_BF16 = 1
} w8a8_dtype;

/* Reasons reported by w8a8_shape_supported (bitwise OR). */
#define W8A8_REASON_M          0x01  /* M < 1 or M > 2^30 */
#define W8A8_REASON_N          0x02  /* N < 8, N % 8 != 0 or N > 2^30 */
#define W8A8_REASON_K          0x04  /* K < 16 or K % 16 != 0 */
#define W8A8_REASON_K_RANGE    0x08  /* K > 133144: K * 127^2 could leave INT32 */
#define W8A8_REASON_X_DTYPE    0x10  /* activation dtype is not F32 or BF16 */
#define W8A8_REASON_BIAS_DTYPE 0x20  /* bias dtype is not F32 or BF16 */

/* Bits of the device status word (w8a8_read_status). */
#define W8A8_DEV_TIMEOUT_PRODUCER 0x1  /* TMA producer waited too long for a free stage (or, in
                                          w8a8_linear's in-GEMM quantisation, for a tile's rows) */
#define W8A8_DEV_TIMEOUT_MMA      0x2  /* MMA issuer waited too long for data or accumulator space */
#define W8A8_DEV_TIMEOUT_EPILOGUE 0x4  /* epilogue waited too long for a finished accumulator */
#define W8A8_DEV_TIMEOUT_TEARDOWN 0x8  /* in-flight copies or MMAs did not finish at exit */

/* Largest K whose worst case |acc| = K * 127 * 127 still fits INT32. */
#define W8A8_MAX_K 133144

/* ---------------------------------------------------------------------------
 * Shape guard ("guarded W8A8").  Returns 1 when (M, N, K) with these dtypes
 * runs on the INT8 path, 0 otherwise; `reason` (may be NULL) receives the
 * W8A8_REASON_* bits of every failed condition (0 when supported).  Pure host
 * function: no CUDA call, callable without a GPU.  The conditions are the
 * kernels' own needs: 16-byte row pitches for the TMA copies of int8 and
 * bf16 rows (K % 16), 16-byte output vectors (N % 8), an INT32 accumulator
 * that cannot overflow (K <= W8A8_MAX_K).  The pages name no criteria.
 * ------------------------------------------------------------------------- */
W8A8_API int w8a8_shape_supported(int64_t M, int64_t N, int64_t K, int x_dtype, int bias_dtype, int* reason);

/* ---------------------------------------------------------------------------
 * Static per-output-channel weight quantisation (offline, once per layer).
 *   W  [N][K] of `w_dtype` (F32 or BF16)       in
 *   Wq [N][K] int8 codes                        out
 *   sw [N]    fp32 scales                       out
 * Needs K % 16 == 0, 1 <= K <= W8A8_MAX_K, N >= 1.
 * ------------------------------------------------------------------------- */
W8A8_API w8a8_status w8a8_quantize_weight(const void* W, int w_dtype, int64_t N, int64_t K,
                                 int8_t* Wq, float* sw, void* stream);

/* ---------------------------------------------------------------------------
 * Dynamic per-row activation quantisation.
 *   X  [M][K] of `x_dtype` (F32 or BF16)       in
 *   Xq [M][K] int8 codes                        out
 *   sx [M]    fp32 scales                       out
 * Same arithmetic and limits as w8a8_quantize_weight.  M == 0 (or N == 0
 * for the weight) is a no-op that returns W8A8_OK; the pointers may then be NULL.
 * ------------------------------------------------------------------------- */
W8A8_API w8a8_status w8a8_quantize_act(const void* X, int x_dtype, int64_t M, int64_t K,
                              int8_t* Xq, float* sx, void* stream);

/* ---------------------------------------------------------------------------
 * Weight operand for the tensor-core GEMM.  B300 (sm_103a) has no tcgen05
 * integer MMA, so the GEMM multiplies the INT8 codes carried exactly in bf16
 * (every integer in [-127, 127] is a bf16 value) and keeps every partial sum
 * an exact integer (see w8a8_linear).  This converts the static codes once:
 *   Wq [N][K] int8                              in
 *   Wp [N][K] bf16 bit patterns (uint16)        out, Wp[n][k] == (bf16)Wq[n][k]
 * Needs K % 16 == 0.  Wp takes 2 * N * K bytes.
 * ------------------------------------------------------------------------- */
W8A8_API w8a8_status w8a8_pack_weight(const int8_t* Wq, int64_t N, int64_t K, uint16_t* Wp, void* stream);

/* Workspace sizes for w8a8_linear, w8a8_linear_gemm_stage and w8a8_gemm_s32.
 *
 * w8a8_linear_workspace_min_bytes(M, K): the smallest workspace accepted:
 * 1024 bytes of alignment slack, a 1024-byte header (status word and the
 * GEMM's split-tile counters), M fp32 row scales and the M x K activation
 * codes (as bf16), each on a 1024-byte boundary inside the buffer.
 *
 * w8a8_linear_workspace_bytes(M, N, K): the minimum plus room for the INT32
 * partial tiles (128 KB each) of the GEMM's K-split last wave, as planned
 * for the current device (for a 148-SM device when no device is current).
 * When the tiles do not fill the SMs evenly, the GEMM cuts the tiles of the
 * last, partly filled wave along K so that every SM works on it, and adds
 * the INT32 partials exactly.  A workspace between the two sizes is
 * accepted; the GEMM then splits only as far as the room allows (results
 * are identical either way, only the time differs).
 *
 * Both return 0 for invalid sizes. */
W8A8_API size_t w8a8_linear_workspace_min_bytes(int64_t M, int64_t K);
W8A8_API size_t w8a8_linear_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* How the GEMM deals its output tiles to the device's SMs, for a workspace
 * with room for `max_slots` partial tiles of 128 x 256 INT32 (< 0:
 * unlimited).  A tile is 256 x 256 and runs on a pair of CTAs on two SMs
 * (one tcgen05 MMA of cta_group::2 for both), for any M; where pairs cannot
 * be resident, or under w8a8_debug_force_single_cta, a tile is 128 x 256 on
 * one CTA.  `num_sms` > 0 plans for that many SMs (pairs:
 * num_sms / 2); <= 0 plans for the current device as the launch will (148
 * SMs when none is current).  Writes plan[0] = whole tiles (dealt
 * round-robin to the workers), plan[1] = K-segments per remaining tile (1 =
 * no split), plan[2] = K-segment units (remaining tiles x segments, one per
 * worker), plan[3] = CTAs launched, plan[4] = CTAs per tile (1 or 2).
 * Returns 1, or 0 for invalid sizes.  Pure host function apart from the
 * device query; exposed for inspection and tests. */
W8A8_API int w8a8_gemm_plan(int64_t M, int64_t N, int64_t K, int num_sms, int64_t max_slots, int64_t* plan);

/* ---------------------------------------------------------------------------
 * Which GEMM kernel the INT8 linear, the INT32 test export and the BF16
 * linear launch for (M, N, K) (the MLP pair's up layer always takes the
 * persistent form).  Host only; uses the current device's SM count and
 * cluster occupancy (a 148-SM device when none is current).
 *   form[0]  0: the persistent form whose tile schedule w8a8_gemm_plan gives;
 *            1: the cluster-K form, for problems with few output tiles:
 *            each 128-row x form[1]-column output tile is computed by a
 *            thread-block cluster of form[2] CTAs that split K and add their
 *            exact INT32 partial sums through distributed shared memory
 *   form[1]  tile width of the cluster-K form (64, 128 or 256), else 0
 *   form[2]  CTAs per cluster (1, 2, 4 or 8), else 0
 *   form[3]  CTAs launched by the cluster-K form, else 0
 * The form is chosen by estimated kernel time: the cluster-K form only for
 * problems that leave the persistent form's single wave of 256 x 256 tiles
 * mostly idle (the audio branch's 126- and 1001-row shapes).  Both forms
 * compute the same exact INT32 sums and the same epilogue (identical
 * bytes).  Returns 1, or 0 for invalid sizes.  form: int64_t[4].
 * ------------------------------------------------------------------------- */
W8A8_API int w8a8_gemm_form(int64_t M, int64_t N, int64_t K, int64_t* form);

/* ---------------------------------------------------------------------------
 * The guarded W8A8 linear: Y = dequant(quant(X) * Wq^T) + bias, in two
 * kernels on `stream`: (1) per-row activation quantisation into the
 * workspace, (2) the tcgen05 GEMM with the fused epilogue.  For bf16 X with
 * K = 4096 on the CTA-pair form, (1) quantises only the rows the GEMM's
 * first wave of tiles reads, and two extra warps of every GEMM CTA quantise
 * the rest while it runs (each tile waits on the device until its rows are
 * published); codes, scales and Y are the same bytes either way.
 *   X    [M][K] of `x_dtype` (F32 or BF16)               in
 *   Wp   [N][K] packed weight codes (w8a8_pack_weight)   in
 *   sw   [N]    fp32 weight scales                       in
 *   bias [N]    of `bias_dtype`, or NULL for no bias     in
 *   Y    [M][N] bf16 bit patterns                        out
 *   ws   workspace of >= w8a8_linear_workspace_min_bytes(M, K) bytes,
 *        w8a8_linear_workspace_bytes(M, N, K) for full speed; its contents
 *        on entry do not matter; on return (stream-ordered) it holds the
 *        status word, sx and the activation codes.
 * Shapes the guard rejects return W8A8_ERR_UNSUPPORTED_SHAPE with nothing
 * launched: the caller runs its BF16 linear for them.
 * The GEMM accumulates in fp32 tensor memory over K-chunks of at most 1024
 * (1024 * 127^2 < 2^24, so every partial sum is an exactly representable
 * integer) and drains each chunk into INT32 registers; the result equals the
 * exact INT32 accumulator.  Calls sharing one workspace must not overlap.
 * ------------------------------------------------------------------------- */
W8A8_API w8a8_status w8a8_linear(const void* X, int x_dtype, int64_t M, int64_t K,
                        const uint16_t* Wp, const float* sw, int64_t N,
                        const void* bias, int bias_dtype,
                        uint16_t* Y, void* ws, size_t ws_bytes, void* stream);

/* The two halves of w8a8_linear, exposed so that each can be timed or
 * reused alone.  quant_stage(...) then gemm_stage(...) with the same
 * workspace gives w8a8_linear's results (the same bytes; w8a8_linear may
 * overlap the two, as described above). */
W8A8_API w8a8_status w8a8_linear_quant_stage(const void* X, int x_dtype, int64_t M, int64_t K,
                                    void* ws, size_t ws_bytes, void* stream);
W8A8_API w8a8_status w8a8_linear_gemm_stage(int64_t M, int64_t K, const uint16_t* Wp, const float* sw,
                                   int64_t N, const void* bias, int bias_dtype,
                                   uint16_t* Y, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * INT32 accumulators alone (for checking them bit for bit):
 *   Xq  [M][K] int8 activation codes            in
 *   Wp  [N][K] packed weight codes              in
 *   acc [M][N] int32                            out, acc = Xq * Wq^T exactly
 *   ws  >= w8a8_linear_workspace_min_bytes(M, K) (see w8a8_linear)
 * Same guard as w8a8_linear (with x_dtype = BF16, no bias).
 * ------------------------------------------------------------------------- */
W8A8_API w8a8_status w8a8_gemm_s32(const int8_t* Xq, const uint16_t* Wp, int64_t M, int64_t N, int64_t K,
                          int32_t* acc, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * w8a8_linear for callers that cannot allocate device memory.  The paper has
 * no counterpart: this entry point exists for this library's users only.
 *
 * Who needs it: code that has no way to obtain a device buffer where it calls
 * the layer — for example a plugin inside an inference runtime that owns the
 * whole device memory budget and gives its plugins no scratch space, or a
 * latency-critical path that must not call cudaMalloc (which can synchronise
 * the device) and has no memory pool to draw from.  Such a caller still owns
 * X, Wp, sw, bias and Y; only the workspace is taken care of here.
 *
 * The workspace is a scratch array built into the library: a file-scope
 * device array of W8A8_NOALLOC_SCRATCH_BYTES (64 MiB) that every GPU which
 * loads the library keeps until the process exits.
 *  - Arguments, results and the arithmetic are those of w8a8_linear.
 *  - No cudaMalloc, cudaFree or other allocating call is made.
 *  - Shapes whose smallest workspace does not fit in the array,
 *    w8a8_linear_workspace_min_bytes(M, K) > W8A8_NOALLOC_SCRATCH_BYTES
 *    (M * K above about 33.5 million), return W8A8_ERR_WORKSPACE with
 *    nothing launched.  What the array has beyond that minimum holds the
 *    GEMM's split partial tiles.
 *  - The array is defined in a translation unit of its own, so a process
 *    that never calls the two entry points here does not load it (the
 *    CUDA runtime loads modules lazily by default).
 *  - The first call on a device looks up the array's device address
 *    (once per device, with that device current) and keeps it with the
 *    device's context; after cudaDeviceReset the next call looks it up
 *    again.  Make that first call before any stream capture.
 *  - All calls on a device share the one array, and it keeps the previous
 *    call's contents; what must start at zero is cleared by each call.
 *    Calls that can overlap on the GPU (different streams, or threads that
 *    do not order their launches) race on the array: serialise them.
 *  - The device status word lives in the built-in array: read it with
 *    w8a8_noalloc_read_status, not w8a8_read_status.
 * ------------------------------------------------------------------------- */
#define W8A8_NOALLOC_SCRATCH_BYTES (64ull << 20)
W8A8_API w8a8_status w8a8_linear_noalloc(const void* X, int x_dtype, int64_t M, int64_t K,
                                         const uint16_t* Wp, const float* sw, int64_t N,
                                         const void* bias, int bias_dtype, uint16_t* Y, void* stream);

/* ---------------------------------------------------------------------------
 * The device status word of w8a8_linear_noalloc's built-in workspace, as
 * w8a8_read_status gives it for a caller-owned one (no paper counterpart
 * either): waits for `stream` (synchronises it), copies the word to the host
 * into *device_bits (W8A8_DEV_* bits), and returns W8A8_OK when it is 0,
 * W8A8_ERR_TIMEOUT when a device-side wait of the last w8a8_linear_noalloc
 * call on this device ran out.  Like that entry point it allocates nothing;
 * its first call on a device looks up the array's address.
 * ------------------------------------------------------------------------- */
W8A8_API w8a8_status w8a8_noalloc_read_status(void* stream, uint32_t* device_bits);

/* ---------------------------------------------------------------------------
 * w8a8_linear from and to HOST memory, pipelined over row chunks.
 *   X_host [M][K] of `x_dtype`, host memory                 in
 *   Y_host [M][N] bf16 bit patterns, host memory            out
 *   X_dev  [M][K] of `x_dtype`, device staging               (caller-owned)
 *   Y_dev  [M][N] bf16, device staging                       (caller-owned)
 *   ws     >= w8a8_linear_workspace_min_bytes(chunk, K) for the chunk size
 *          used (w8a8_linear_workspace_bytes(chunk, N, K) for full speed)
 *   chunk_rows  rows per chunk (equal chunks, at most 64); 0 = about M / 8
 *          rounded up to 256 rows, with the first and the last chunk a
 *          third as long (whole 128-row tiles) when M is large enough
 * Wp, sw, bias as in w8a8_linear.  For each chunk of rows: the host-to-device
 * copy of X on a copy stream, then w8a8_linear on `stream`, then the
 * device-to-host copy of Y on a second copy stream, so the copies of one
 * chunk overlap the other chunks' compute and the copies in the other
 * direction.  The whole call is ordered on `stream` like any other entry
 * point: it starts after earlier work on `stream`, and later work on
 * `stream` sees Y_host written.  Host buffers should be page-locked
 * (cudaHostAlloc / cudaHostRegister) for the copies to run asynchronously.
 * The library creates two copy streams and a set of events per device on
 * the first call (no device memory) and keeps them until the process exits;
 * make that first call before any stream capture.  Calls on one device must
 * not overlap (they share those streams and events).  The status word in
 * `ws` reflects the last chunk only.
 * ------------------------------------------------------------------------- */
W8A8_API w8a8_status w8a8_linear_host(const void* X_host, int x_dtype, int64_t M, int64_t K,
                                      const uint16_t* Wp, const float* sw, int64_t N,
                                      const void* bias, int bias_dtype, uint16_t* Y_host,
                                      void* X_dev, uint16_t* Y_dev, void* ws, size_t ws_bytes,
                                      int64_t chunk_rows, void* stream);

/* ---------------------------------------------------------------------------
 * The native BF16 linear, for the branches the guarded W8A8 path does not
 * take.  The zhidx TurboT2VA article (section 01 item 3, "量化策略") has branches
 * whose shapes the optimised operator cannot take fall back to native BF16,
 * and the paperlayer summary of arXiv 2608.24674 (section "C. Fused
 * Multimodal Transformer Operations") guards the acceleration by
 * architectural role as well as by shape.  Same tcgen05 GEMM, with the bf16
 * operands loaded as they are and fp32 accumulation:
 *   Y[m][n] = bf16_rne(sum_k X[m][k] * W[n][k] + bias[n])
 * (the products are exact in fp32; the tensor cores accumulate the sum in
 * fp32 over each tile's K range, and a tile whose K range the schedule cuts
 * into segments adds the segments' fp32 sums in segment order, so the
 * result is within fp32 rounding of the exact sum and the same on every
 * call, but not bit-identical to another summation order).
 *   X    [M][K] bf16                                    in
 *   W    [N][K] bf16                                    in
 *   bias [N] of `bias_dtype` (F32 or BF16), or NULL     in
 *   Y    [M][N] bf16                                    out
 *   ws   >= 2048 bytes; w8a8_bf16_linear_workspace_bytes(M, N, K) for full
 *        speed (adds the K-split partial tiles, as for w8a8_linear)
 * Shapes: 1 <= M <= 2^30, 8 <= N <= 2^30 with N % 8 == 0, 8 <= K <= 2^30
 * with K % 8 == 0 (16-byte rows for the tensor copies).  Others return
 * W8A8_ERR_UNSUPPORTED_SHAPE with nothing launched; w8a8_bf16_linear_supported
 * reports which (W8A8_REASON_* bits).
 * ------------------------------------------------------------------------- */
W8A8_API int w8a8_bf16_linear_supported(int64_t M, int64_t N, int64_t K, int bias_dtype, int* reason);
W8A8_API size_t w8a8_bf16_linear_workspace_bytes(int64_t M, int64_t N, int64_t K);
W8A8_API w8a8_status w8a8_bf16_linear(const uint16_t* X, int64_t M, int64_t K, const uint16_t* W, int64_t N,
                                      const void* bias, int bias_dtype, uint16_t* Y, void* ws, size_t ws_bytes,
                                      void* stream);

/* ---------------------------------------------------------------------------
 * Normalisation and modulation fused into the activation quantisation, the
 * prologue of a linear layer (zhidx TurboT2VA article, section 01: the
 * inference stack fuses normalisation and modulation to cut intermediate
 * reads and writes; arXiv paper, appendix C).  Per row x of X [M][K] bf16:
 *   mu = 0 (W8A8_NORM_RMS) or fp32(sum x / K) (W8A8_NORM_LAYER)
 *   r  = 1 / sqrt(fp32(sum (x - mu)^2 / K) + eps)   (correctly rounded)
 *   y  = bf16_rne(fma((x - mu) * r, 1 + scale, shift))   (fp32 steps)
 * then y is quantised by the row rule (as w8a8_quantize_act).  scale and
 * shift are optional [K] vectors of `mod_dtype` (F32 or BF16, 16-byte
 * aligned), shared by all rows; NULL omits that step.  The fp32 sums run
 * in an order of the kernel's choosing.  K % 16 == 0, K <= W8A8_NORM_MAX_K.
 *
 * w8a8_norm_quantize_act: codes Xq [M][K] int8 and scales sx [M]; Y_mod
 *   (nullable) also receives y [M][K] bf16.
 * w8a8_norm_linear: the same prologue feeding the W8A8 GEMM, with the
 *   arguments, workspace and errors of w8a8_linear (X bf16).
 * ------------------------------------------------------------------------- */
#define W8A8_NORM_RMS 1
#define W8A8_NORM_LAYER 2
#define W8A8_NORM_MAX_K 32768
W8A8_API w8a8_status w8a8_norm_quantize_act(const uint16_t* X, int64_t M, int64_t K, int norm, float eps,
                                            const void* scale, const void* shift, int mod_dtype, uint16_t* Y_mod,
                                            int8_t* Xq, float* sx, void* stream);
W8A8_API w8a8_status w8a8_norm_linear(const uint16_t* X, int64_t M, int64_t K, int norm, float eps,
                                      const void* scale, const void* shift, int mod_dtype, const uint16_t* Wp,
                                      const float* sw, int64_t N, const void* bias, int bias_dtype, uint16_t* Y,
                                      void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * MLP pair: Y = down(up(X)), both layers on the W8A8 path, with the down
 * layer's per-row activation quantisation fed by the up layer's epilogue.
 * Each layer is the linear above (zhidx TurboT2VA article, section 01 item
 * 3); between them nothing is applied (no activation function: the pages
 * name none).  The up GEMM's epilogue gathers each row's max |H| over the
 * bf16 values it writes (an exact integer max on the bit patterns, by
 * atomicMax), so the down layer's codes come from one streaming pass over
 * H with no reduction.  H, the codes and the scales are bit-identical to
 * w8a8_linear(X) followed by w8a8_linear(H).
 *   X      [M][K] F32 or BF16                           in
 *   Wp_up  [F][K] packed codes, sw_up [F], bias_up [F]  in (bias nullable)
 *   Wp_down[N][F] packed codes, sw_down [N], bias_down [N]  in
 *   H      [M][F] bf16, the up layer's output           out
 *   Y      [M][N] bf16                                  out
 *   ws     >= w8a8_mlp_workspace_bytes(M, K, F, N) for full speed (the
 *          smallest accepted holds both layers' codes and scales and no
 *          split-tile slots); caller-owned, 16-byte aligned.
 * Both (M, F, K) and (M, N, F) must pass w8a8_shape_supported; errors as for
 * w8a8_linear, nothing launched on an error.  Four launches on `stream`:
 * quantiser, up GEMM, codes pass, down GEMM, each after the first a
 * programmatic dependent of the one before.
 * ------------------------------------------------------------------------- */
W8A8_API size_t w8a8_mlp_workspace_bytes(int64_t M, int64_t K, int64_t F, int64_t N);
W8A8_API w8a8_status w8a8_mlp(const void* X, int x_dtype, int64_t M, int64_t K, const uint16_t* Wp_up,
                              const float* sw_up, int64_t F, const void* bias_up, int bias_up_dtype,
                              const uint16_t* Wp_down, const float* sw_down, int64_t N, const void* bias_down,
                              int bias_down_dtype, uint16_t* H, uint16_t* Y, void* ws, size_t ws_bytes,
                              void* stream);

/* ---------------------------------------------------------------------------
 * Per-block INT8 quantisation of attention Query or Key (zhidx TurboT2VA
 * article, section 01 item 4: the SageSLA self-attention path quantises
 * Query and Key to INT8).  A block is `block_tokens` consecutive tokens of
 * one (batch, head), the last block of a head possibly shorter; each block
 * gets one scale and the linear layer's row rule:
 *   s = fp32(absmax / 127) (zero block: 1), q = clamp(rne(fp32(x / s)), +-127).
 *   X      [B][H][L][D] (layout W8A8_LAYOUT_HND) or [B][L][H][D]
 *          (W8A8_LAYOUT_NHD) of `x_dtype` (F32 or BF16), D contiguous   in
 *   Xq     int8 codes, same shape and layout as X                       out
 *   scales [B][H][ceil(L / block_tokens)] fp32                         out
 * Needs D % 8 == 0 and D <= 2048 for BF16 (D % 4 == 0 and D <= 1024 for
 * F32), block_tokens >= 1, L <= 2^31 - 1; X and Xq 16-byte aligned.  Any of B, H, L == 0
 * is a no-op returning W8A8_OK.  Errors: W8A8_ERR_INVALID_ARG (NULL
 * pointer, negative size, unknown layout), W8A8_ERR_DTYPE,
 * W8A8_ERR_UNSUPPORTED_SHAPE (D or block_tokens), W8A8_ERR_ALIGNMENT; nothing
 * is launched on an error.  Asynchronous on `stream`.
 * ------------------------------------------------------------------------- */
#define W8A8_LAYOUT_HND 0
#define W8A8_LAYOUT_NHD 1
W8A8_API w8a8_status w8a8_quantize_qk_blocks(const void* X, int x_dtype, int64_t B, int64_t H, int64_t L, int64_t D,
                                             int layout, int64_t block_tokens, int8_t* Xq, float* scales,
                                             void* stream);

/* ---------------------------------------------------------------------------
 * Device status of the last call that used `ws`: synchronises `stream`,
 * copies the workspace's status word to *device_bits (host pointer) and
 * returns W8A8_OK when it is 0, W8A8_ERR_TIMEOUT when a bounded device wait
 * ran out (bits W8A8_DEV_*), W8A8_ERR_CUDA if the copy failed.
 * ------------------------------------------------------------------------- */
W8A8_API w8a8_status w8a8_read_status(const void* ws, void* stream, uint32_t* device_bits);

/* Limit, in nanoseconds, for every device-side wait of later launches from
 * this process (default 2e9 = 2 s).  Values below 1e6 are raised to 1e6. */
W8A8_API void w8a8_set_wait_limit_ns(uint64_t ns);

/* Test hook: when `on` is nonzero, later GEMM launches issue no operand
 * copies, so the MMA and epilogue waits run out after the wait limit and
 * the status word reports it.  Used only by the failure-detection test. */
W8A8_API void w8a8_debug_skip_loads(int on);

/* Test hook: when `on` is nonzero, later GEMM launches (and plans) use the
 * single-CTA form for every M, so that tests can compare both forms on the
 * same inputs.  Results are identical either way. */
W8A8_API void w8a8_debug_force_single_cta(int on);

/* Test switch: which GEMM form every later launch takes.  form -1: chosen
 * per shape (the default); 0: always the persistent form; 1: always the
 * cluster-K form, with tile width bn (64, 128, 256; 0 = chosen) and cluster
 * size ks (1, 2, 4, 8; 0 = chosen).  Used by the tests to compare the forms
 * on the same shapes; not thread-safe with concurrent launches. */
W8A8_API void w8a8_debug_force_gemm_form(int form, int bn, int ks);

/* Static text for a status value. */
W8A8_API const char* w8a8_status_str(int status);

/* Library version, for the binding's load check. */
W8A8_API int w8a8_version(void);

#ifdef __cplusplus
}
#endif

#endif /* W8A8_H */
