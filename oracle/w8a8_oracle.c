/*
 * CPU oracle for the guarded W8A8 linear layer.  TEST INFRASTRUCTURE ONLY:
 * it is built and called by the tests, by the bench's CPU-baseline leg and by
 * the smoke check, never by the product library.  It shares no code, header,
 * table or helper with the CUDA path.
 *
 * What it computes comes from the quantisation-strategy passage of the
 * zhidx article "音视频生成提速54倍！浙大等团队开源联合蒸馏方案TurboT2VA",
 * section 01, item 3 ("量化策略"): linear layers use W8A8; weights are
 * quantised statically to INT8 per output channel, activations dynamically to
 * INT8 per row; the matrix product accumulates in INT32; the scales and the
 * bias are applied once, after the whole accumulation has finished.
 *
 * The pages fix no arithmetic detail beyond that.  The readings taken here
 * (each one restated where it is used):
 *   - symmetric absmax scale, s = fp32(amax / 127), IEEE division;
 *   - a row whose scale comes out as 0 (amax == 0, or an fp32 absmax so small
 *     that amax/127 underflows) is a zero row: s = 1 and every code is 0;
 *   - code q = clamp(round_half_even(fp32(x / s)), -127, 127), IEEE division;
 *   - INT32 accumulator = exact integer dot product (computed in int64 and
 *     checked to fit INT32);
 *   - epilogue y32 = ((float)acc * sx[m]) * sw[n] + bias[n], each step one
 *     fp32 operation rounded to nearest-even, in that order, no fused
 *     multiply-add; Y = bf16 round-to-nearest-even of y32.
 *
 * Everything is scalar, in the order the definition states.  Rows are
 * independent, so the outer loops over rows run on OpenMP threads; nothing
 * else is reordered or blocked.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fopenmp
 *        -shared -fPIC  (see build_oracle.py beside this file).
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- bf16 <-> fp32, written out from the bf16 format definition ---------
 * bf16 is the upper 16 bits of an IEEE binary32.  Widening is exact. */
static float bf16_bits_to_float(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Narrowing with round-to-nearest, ties to even, on the 16 dropped bits.
 * NaN is kept a (quiet) NaN; infinities and overflow to infinity follow from
 * the same rounding rule. */
uint16_t oracle_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);          /* quiet NaN */
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xffffu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;                                     /* carries into the exponent when needed */
    return (uint16_t)upper;
}

/* The same rounding over an array (one call instead of one per value). */
void oracle_bf16_rne_array(const float* x, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_rne(x[i]);
}

float oracle_bf16_to_float(uint16_t h) { return bf16_bits_to_float(h); }

/* ---- round half to even, written out ------------------------------------
 * For |v| < 2^23 the value v - floor(v) is exact in fp32, so the comparison
 * with one half is exact. */
static float round_half_even(float v)
{
    if (!(fabsf(v) < 8388608.0f))      /* already an integer, inf or NaN */
        return v;
    float f = floorf(v);
    float d = v - f;
    if (d > 0.5f) return f + 1.0f;
    if (d < 0.5f) return f;
    /* exact tie: pick the even neighbour */
    return (fmodf(f, 2.0f) == 0.0f) ? f : f + 1.0f;
}

static int8_t clamp_code(float r)
{
    if (r > 127.0f) return 127;
    if (r < -127.0f) return -127;
    return (int8_t)r;
}

/* One row: absmax, scale, codes.  `get(k)` is the row's k-th value in fp32. */
#define QUANTIZE_ROW(GET)                                              \
    do {                                                               \
        float amax = 0.0f;                                             \
        for (int64_t k = 0; k < K; ++k) {                              \
            float a = fabsf(GET(k));                                   \
            if (a > amax) amax = a;                                    \
        }                                                              \
        volatile float sv = amax / 127.0f;                             \
        float s = sv;                                                  \
        if (s == 0.0f) {                                               \
            scale[r] = 1.0f;                                           \
            for (int64_t k = 0; k < K; ++k) q[r * K + k] = 0;          \
        } else {                                                       \
            scale[r] = s;                                              \
            for (int64_t k = 0; k < K; ++k) {                          \
                volatile float v = GET(k) / s;                         \
                q[r * K + k] = clamp_code(round_half_even(v));         \
            }                                                          \
        }                                                              \
    } while (0)

/* Per-row symmetric INT8 quantisation of an fp32 matrix A[R][K] (row-major).
 * Used for activations (rows = tokens, dynamic) and for weights (rows =
 * output channels, static): the article gives both as INT8 with one scale per
 * row of the operand as it is stored.  Returns 0, or -1 on a non-finite
 * input (the method is not defined there). */
int oracle_quantize_rows_f32(const float* A, int64_t R, int64_t K, int8_t* q, float* scale)
{
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t r = 0; r < R; ++r) {
        const float* row = A + r * K;
        for (int64_t k = 0; k < K; ++k)
            if (!isfinite(row[k])) bad = 1;
#define GET_F32(k) (row[(k)])
        QUANTIZE_ROW(GET_F32);
#undef GET_F32
    }
    return bad ? -1 : 0;
}

/* Same, for a bf16 matrix given as raw 16-bit patterns. */
int oracle_quantize_rows_bf16(const uint16_t* A, int64_t R, int64_t K, int8_t* q, float* scale)
{
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t r = 0; r < R; ++r) {
        const uint16_t* row = A + r * K;
        for (int64_t k = 0; k < K; ++k)
            if (!isfinite(bf16_bits_to_float(row[k]))) bad = 1;
#define GET_BF16(k) (bf16_bits_to_float(row[(k)]))
        QUANTIZE_ROW(GET_BF16);
#undef GET_BF16
    }
    return bad ? -1 : 0;
}

/* INT32 accumulators of the INT8 product for a chosen set of rows:
 *   acc[i][n] = sum_k Xq[rows[i]][k] * Wq[n][k]
 * Xq is [M][K], Wq is [N][K] (both K-contiguous; Wq holds one output channel
 * per row, like a linear layer's weight).  The sum runs in int64; the return
 * value counts accumulators that do not fit INT32 (0 means all fit). */
int64_t oracle_gemm_s32(const int8_t* Xq, const int8_t* Wq, int64_t M, int64_t N, int64_t K,
                        const int64_t* rows, int64_t nrows, int32_t* acc)
{
    int64_t overflow = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : overflow)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows[i];
        if (m < 0 || m >= M) { overflow += N; continue; }
        const int8_t* x = Xq + m * K;
        for (int64_t n = 0; n < N; ++n) {
            const int8_t* w = Wq + n * K;
            int64_t sum = 0;
            for (int64_t k = 0; k < K; ++k)
                sum += (int64_t)x[k] * (int64_t)w[k];
            if (sum > INT32_MAX || sum < INT32_MIN) { overflow += 1; sum = 0; }
            acc[i * N + n] = (int32_t)sum;
        }
    }
    return overflow;
}

/* Epilogue, applied once to finished accumulators:
 *   y32[i][n] = ((float)acc[i][n] * sx[i]) * sw[n] + bias[n]
 *   Y[i][n]   = bf16_rne(y32[i][n])
 * sx holds the scales of the same rows as acc (row i of acc uses sx[i]).
 * bias may be NULL: the add is then skipped (a layer without bias).  Every
 * step is a separate fp32 operation; volatile keeps the compiler from
 * contracting them into a fused multiply-add. */
void oracle_epilogue(const int32_t* acc, int64_t nrows, int64_t N, const float* sx,
                     const float* sw, const float* bias, float* y32, uint16_t* y_bf16)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < nrows; ++i) {
        for (int64_t n = 0; n < N; ++n) {
            volatile float a = (float)acc[i * N + n];
            volatile float t = a * sx[i];
            volatile float u = t * sw[n];
            float y = u;
            if (bias) {
                volatile float b = u + bias[n];
                y = b;
            }
            if (y32) y32[i * N + n] = y;
            if (y_bf16) y_bf16[i * N + n] = oracle_bf16_rne(y);
        }
    }
}

/* Threads the OpenMP loops above will use (reported beside CPU timings). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
