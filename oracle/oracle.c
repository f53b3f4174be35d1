/*
 * CPU oracle for the FP8 (E4M3) block-scaled GEMM library.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the bench's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * What it computes, and where the definition comes from:
 *   - E4M3 ("fn" variant, dtype float8_e4m3fn) decode from the bit pattern:
 *     the format named in "Optimizing FP8 GEMM kernels in JAX with Triton for
 *     Blackwell GPUs" (format paragraph: E4M3 preferred for its range /
 *     precision balance) and the dtype in "Triton FP8 CUTLASS-named kernel
 *     benchmarking" (parameter list: torch.float8_e4m3fn).
 *   - E5M2 (the other FP8 format the JAX/Blackwell page's format paragraph
 *     weighs against E4M3; the Triton tutorial ch. 12, section 12.6.1 lists
 *     FP8 among the fifth-generation tensor core's types): 1 sign, 5 exponent
 *     bits (bias 15), 2 mantissa bits, with infinities and NaNs in the top
 *     binade (the IEEE-style layout); largest finite 57344.  Operands of a
 *     GEMM may mix the formats.
 *   - E2M1 (FP4, the microscaling element format of the MXFP4 variant the
 *     Triton tutorial ch. 12 lists beside MXFP8): 1 sign, 2 exponent bits
 *     (bias 1), 1 mantissa bit, values 0, 0.5, 1, 1.5, 2, 3, 4, 6; no
 *     infinities or NaNs.  Held one code per byte (low four bits).
 *   - E2M3 and E3M2 (FP6: the Triton tutorial ch. 12 lists FP6 among the
 *     fifth-generation tensor core's types in its 12.6.1 hardware table and
 *     an FP6 GEMM in its 12.6.4 stability table; it prints no layout, so the
 *     microscaling element formats are taken): 1 sign bit and 2 exponent
 *     bits (bias 1) + 3 mantissa bits, largest 7.5, or 3 exponent bits (bias
 *     3) + 2 mantissa bits, largest 28; exponent field 0 subnormal; no
 *     infinities or NaNs.  Held one code per byte (low six bits).
 *   - Quantisation x -> RNE_satfinite(fl32(x / s)) with a per-tensor scale
 *     s = fl32(amax / 448) or a 1x32 block scale along K equal to the smallest
 *     power of two >= amax / 448 (the microscaling paragraph of the JAX/Blackwell
 *     page; "2nd-gen Transformer Engine integrates micro-scaling (MXFP8)" in the
 *     Triton tutorial ch. 12, section 12.6.1).
 *   - GEMM C = (sA A)(sB B)^T with A[M,K], B[N,K] row-major: the pseudo-kernel
 *     of the JAX/Blackwell page (fp32 accumulate, down-converting store), with
 *     B held K-contiguous.
 *   - The grouped (MoE) variant: per expert e, rows [off_e, off_e + M_e) of A
 *     multiply B[e] (MoE paragraph of the JAX/Blackwell page).
 *   - The grouped raster order of output tiles ("GROUP_M" swizzle of the
 *     persistent matmul in the Triton tutorial ch. 12, section 12.7).
 *   - NVFP4 (the other FP4 micro-scaling format the Triton tutorial ch. 12,
 *     section 12.6.1 names, beside MXFP8 / MXFP4): E2M1 elements, one E4M3
 *     block scale per 16 elements along K, one fp32 scale per tensor.  The
 *     pages print no recipe; the reading taken is stated at
 *     oracle_quantize_nvfp4.  GEMM: the 1x16 block-scaled sum times
 *     alpha = fl32(gA gB), rounded once: fl32(alpha * sum).
 *   - A fused epilogue after the GEMM value v: act(v + bias[j]) with act none,
 *     ReLU or GELU (the bias_add_relu case in the benchmark list of the Triton
 *     FP8 benchmarking page; GELU in its erf form x * Phi(x)), in fp64.
 *
 * All arithmetic is fp64.  Per-block inner sums are exact for E4M3: each
 * product of two E4M3 values is an integer multiple of 2^-18 with magnitude
 * <= 448^2 < 2^18, so any sum of fewer than 2^17 of them fits in the 53-bit
 * significand.  With E5M2 operands products span 2^-32 .. 2^32 and a sum may
 * round (relative error <= K 2^-53, far inside the tolerance).  E2M1, E2M3
 * and E3M2 values are multiples of 2^-1, 2^-3 and 2^-4 below 28, so their
 * products with each other or with E4M3 are exact in the same way.
 * Steps the pages fix in fp32 (fl32(amax/448), fl32(x/s), fl32(sA*sB),
 * fl32(alpha*acc)) are done in fp32 here too.
 *
 * Parity unpinned: the rounding order of the tensor core's fp32 accumulation.
 * Only the stated tolerance bounds it.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_EXPORT __attribute__((visibility("default")))

/* ------------------------------------------------------------------ */
/* E4M3 decode                                                         */
/* ------------------------------------------------------------------ */

/* Value of an E4M3 ("fn") bit pattern: 1 sign bit, 4 exponent bits with bias
 * 7, 3 mantissa bits.  Exponent field 0 is subnormal (m * 2^-9).  There are no
 * infinities; only S.1111.111 is NaN, so the largest finite value is
 * 1.75 * 2^8 = 448. */
ORACLE_EXPORT double oracle_e4m3_decode(uint8_t code) {
    int s = (code >> 7) & 1;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

ORACLE_EXPORT void oracle_e4m3_table(double *out256) {
    for (int c = 0; c < 256; ++c) out256[c] = oracle_e4m3_decode((uint8_t)c);
}

/* Value of an E5M2 bit pattern: 1 sign bit, 5 exponent bits with bias 15, 2
 * mantissa bits.  Exponent field 0 is subnormal (m * 2^-16); exponent field 31
 * is infinity (m = 0) or NaN (m != 0); the largest finite value is
 * 1.75 * 2^15 = 57344. */
ORACLE_EXPORT double oracle_e5m2_decode(uint8_t code) {
    int s = (code >> 7) & 1;
    int e = (code >> 2) & 31;
    int m = code & 3;
    double mag;
    if (e == 31) {
        if (m != 0) return NAN;
        mag = INFINITY;
    } else if (e == 0) {
        mag = ldexp((double)m, -16);
    } else {
        mag = ldexp(1.0 + (double)m / 4.0, e - 15);
    }
    return s ? -mag : mag;
}

ORACLE_EXPORT void oracle_e5m2_table(double *out256) {
    for (int c = 0; c < 256; ++c) out256[c] = oracle_e5m2_decode((uint8_t)c);
}

/* Value of an E2M1 code in the low four bits of a byte (the high four bits
 * are ignored): 1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit.
 * Exponent field 0 is subnormal (m * 0.5); largest value 1.5 * 2^2 = 6. */
ORACLE_EXPORT double oracle_e2m1_decode(uint8_t code) {
    int s = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double mag = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

ORACLE_EXPORT void oracle_e2m1_table(double *out256) {
    for (int c = 0; c < 256; ++c) out256[c] = oracle_e2m1_decode((uint8_t)c);
}

/* Value of an FP6 code in the low six bits of a byte (the high two bits are
 * ignored): sign bit 5, then `ebits` exponent bits with bias `bias` and
 * 5 - ebits mantissa bits.  Exponent field 0 is subnormal. */
static double fp6_decode(uint8_t code, int ebits, int bias) {
    const int mbits = 5 - ebits;
    int s = (code >> 5) & 1;
    int e = (code >> mbits) & ((1 << ebits) - 1);
    int m = code & ((1 << mbits) - 1);
    double mag = e == 0 ? ldexp((double)m, 1 - bias - mbits)
                        : ldexp(1.0 + (double)m / (double)(1 << mbits), e - bias);
    return s ? -mag : mag;
}

/* E2M3: bias 1, values k/8 below 2, up to 1.875 * 2^2 = 7.5. */
ORACLE_EXPORT double oracle_e2m3_decode(uint8_t code) { return fp6_decode(code, 2, 1); }
/* E3M2: bias 3, subnormals m/16, up to 1.75 * 2^4 = 28. */
ORACLE_EXPORT double oracle_e3m2_decode(uint8_t code) { return fp6_decode(code, 3, 3); }

ORACLE_EXPORT void oracle_e2m3_table(double *out256) {
    for (int c = 0; c < 256; ++c) out256[c] = oracle_e2m3_decode((uint8_t)c);
}
ORACLE_EXPORT void oracle_e3m2_table(double *out256) {
    for (int c = 0; c < 256; ++c) out256[c] = oracle_e3m2_decode((uint8_t)c);
}

/* Round a finite, non-negative real y to the grid of an FP8 format with
 * `mbits` mantissa bits and exponent bias `bias` (normal binades from 2^(1 -
 * bias) up; below that the subnormal quantum 2^(1 - bias - mbits)), with
 * round-to-nearest, ties to even mantissa, then saturate to `maxv`.  Works on
 * the magnitude; the caller supplies the sign.  Returns the 7-bit magnitude
 * code. */
static uint8_t fp8_mag_code(double y, int mbits, int bias, double maxv) {
    if (y == 0.0) return 0;
    const int emin = 1 - bias;
    int E = ilogb(y); /* exponent of the leading bit */
    if (E < emin) E = emin;
    double quantum = ldexp(1.0, E - mbits);
    double n = y / quantum; /* exact: power-of-two division */
    double fl = floor(n);
    double frac = n - fl;
    double r;
    if (frac > 0.5)
        r = fl + 1.0;
    else if (frac < 0.5)
        r = fl;
    else
        r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    double v = r * quantum; /* rounded magnitude, may carry into next binade */
    if (v > maxv) v = maxv; /* satfinite */
    /* encode v exactly */
    if (v < ldexp(1.0, emin)) return (uint8_t)(int)(v / ldexp(1.0, emin - mbits));
    int e = ilogb(v);
    int m = (int)((v / ldexp(1.0, e) - 1.0) * (double)(1 << mbits));
    return (uint8_t)(((e + bias) << mbits) | m);
}

static uint8_t e4m3_mag_code(double y) { return fp8_mag_code(y, 3, 7, 448.0); }

/* E4M3 code of the fp32 value y: RNE, satfinite, NaN -> 0x7F, -0 -> 0x80. */
ORACLE_EXPORT uint8_t oracle_e4m3_encode(float y) {
    if (isnan(y)) return 0x7F;
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs((double)y);
    if (isinf(a)) return (uint8_t)(sign | 0x7E);
    return (uint8_t)(sign | e4m3_mag_code(a));
}

/* E5M2 code of the fp32 value y: RNE, satfinite (infinities saturate to the
 * largest finite 57344 as well), NaN -> 0x7F, -0 -> 0x80. */
ORACLE_EXPORT uint8_t oracle_e5m2_encode(float y) {
    if (isnan(y)) return 0x7F;
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs((double)y);
    if (isinf(a)) return (uint8_t)(sign | 0x7B);
    return (uint8_t)(sign | fp8_mag_code(a, 2, 15, 57344.0));
}

/* E2M1 code of the fp32 value y: RNE, satfinite (to +-6, infinities too),
 * NaN -> 0x07 (E2M1 has no NaN; the library's quantiser does the same), -0 ->
 * 0x08.  One code per byte, high four bits zero. */
ORACLE_EXPORT uint8_t oracle_e2m1_encode(float y) {
    if (isnan(y)) return 0x07;
    uint8_t sign = signbit(y) ? 0x08 : 0x00;
    double a = fabs((double)y);
    if (isinf(a)) return (uint8_t)(sign | 0x07);
    return (uint8_t)(sign | fp8_mag_code(a, 1, 1, 6.0));
}

/* E2M3 / E3M2 codes of the fp32 value y: RNE, satfinite (to the largest
 * value, infinities too), NaN -> 0x1F (the largest positive value: FP6 has
 * no NaN; the library's quantiser does the same), -0 -> 0x20.  One code per
 * byte, high two bits zero. */
ORACLE_EXPORT uint8_t oracle_e2m3_encode(float y) {
    if (isnan(y)) return 0x1F;
    uint8_t sign = signbit(y) ? 0x20 : 0x00;
    double a = fabs((double)y);
    if (isinf(a)) return (uint8_t)(sign | 0x1F);
    return (uint8_t)(sign | fp8_mag_code(a, 3, 1, 7.5));
}
ORACLE_EXPORT uint8_t oracle_e3m2_encode(float y) {
    if (isnan(y)) return 0x1F;
    uint8_t sign = signbit(y) ? 0x20 : 0x00;
    double a = fabs((double)y);
    if (isinf(a)) return (uint8_t)(sign | 0x1F);
    return (uint8_t)(sign | fp8_mag_code(a, 2, 3, 28.0));
}

/* Element formats of the quantisers and GEMM operands */
enum { ORACLE_E4M3 = 0, ORACLE_E5M2 = 1, ORACLE_E2M1 = 2, ORACLE_E2M3 = 3, ORACLE_E3M2 = 4 };

static uint8_t encode_fmt(float y, int fmt) {
    switch (fmt) {
    case ORACLE_E2M1: return oracle_e2m1_encode(y);
    case ORACLE_E2M3: return oracle_e2m3_encode(y);
    case ORACLE_E3M2: return oracle_e3m2_encode(y);
    case ORACLE_E5M2: return oracle_e5m2_encode(y);
    default: return oracle_e4m3_encode(y);
    }
}
static double fmt_max(int fmt) {
    switch (fmt) {
    case ORACLE_E2M1: return 6.0;
    case ORACLE_E2M3: return 7.5;
    case ORACLE_E3M2: return 28.0;
    case ORACLE_E5M2: return 57344.0;
    default: return 448.0;
    }
}

/* ------------------------------------------------------------------ */
/* bf16 rounding                                                       */
/* ------------------------------------------------------------------ */

/* Round a real value (given in fp64) directly to bf16 (8 significant bits,
 * fp32 exponent range) with round-to-nearest-even, returned as a float. */
ORACLE_EXPORT float oracle_bf16_round(double x) {
    if (isnan(x)) return NAN;
    if (isinf(x) || x == 0.0) return (float)x;
    double a = fabs(x);
    int E = ilogb(a);
    if (E < -126) E = -126; /* bf16 subnormals share fp32's quantum 2^-133 */
    double quantum = ldexp(1.0, E - 7);
    double n = a / quantum;
    double fl = floor(n);
    double frac = n - fl;
    double r;
    if (frac > 0.5)
        r = fl + 1.0;
    else if (frac < 0.5)
        r = fl;
    else
        r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    double v = r * quantum;
    /* largest finite bf16 is (2 - 2^-7) * 2^127; the RNE overflow threshold
     * is halfway to 2^128 */
    if (v >= ldexp(1.0, 128)) v = INFINITY;
    return (float)(x < 0 ? -v : v);
}

/* Size of one bf16 unit in the last place at |x|: 2^(floor(log2|x|) - 7) for
 * normal values, 2^-133 for zero and subnormals. */
ORACLE_EXPORT double oracle_bf16_ulp(double x) {
    double a = fabs(x);
    if (a == 0.0 || a < ldexp(1.0, -126)) return ldexp(1.0, -133);
    if (isinf(a) || isnan(a)) return INFINITY;
    return ldexp(1.0, ilogb(a) - 7);
}

/* ------------------------------------------------------------------ */
/* Quantisation                                                        */
/* ------------------------------------------------------------------ */

/* max |x| over non-NaN entries */
static float amax_of(const float *x, int64_t n, int64_t stride) {
    float m = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float v = fabsf(x[i * stride]);
        if (!isnan(v) && v > m) m = v;
    }
    return m;
}

/* Per-tensor quantisation: s = fl32(amax / fmax) (fmax = 448 for E4M3, 57344
 * for E5M2), q = RNE_satfinite(fl32(x / s)).  When s comes out as 0 (amax = 0,
 * or amax so small that the quotient underflows) s = 1 is used instead, so no
 * division by zero happens. */
ORACLE_EXPORT void oracle_quantize_tensor_fmt(const float *x, int64_t rows, int64_t cols,
                                              int fmt, uint8_t *q, float *scale_out) {
    float amax = amax_of(x, rows * cols, 1);
    float s = amax / (float)fmt_max(fmt);
    if (s == 0.0f) s = 1.0f;
    for (int64_t i = 0; i < rows * cols; ++i) q[i] = encode_fmt(x[i] / s, fmt);
    *scale_out = s;
}

ORACLE_EXPORT void oracle_quantize_tensor(const float *x, int64_t rows, int64_t cols,
                                          uint8_t *q, float *scale_out) {
    oracle_quantize_tensor_fmt(x, rows, cols, ORACLE_E4M3, q, scale_out);
}

/* The power-of-two block scale: the smallest 2^e with 2^e * fmax >= amax,
 * clamped to e in [-126, 127]; amax = 0 gives 1. */
ORACLE_EXPORT float oracle_pow2_scale_fmt(float amax, int fmt) {
    if (amax == 0.0f || isnan(amax)) return 1.0f;
    if (isinf(amax)) return ldexpf(1.0f, 127);
    int e = -126;
    /* linear search is fine: at most 254 steps, exact comparisons in fp64 */
    while (e < 127 && ldexp(fmt_max(fmt), e) < (double)amax) ++e;
    return ldexpf(1.0f, e);
}

ORACLE_EXPORT float oracle_pow2_scale(float amax) { return oracle_pow2_scale_fmt(amax, ORACLE_E4M3); }

typedef struct {
    const float *x;
    uint8_t *q;
    float *scales;
    int64_t cols, r0, r1;
    int fmt;
    int literal; /* block scale fl32(amax / fmax) instead of the power of two */
} quant_job;

static void *quant_block32_rows(void *arg);

/* 1x32 block quantisation along the contiguous (K) axis.  cols % 32 == 0.
 * scales: [rows, cols/32] fp32, each a power of two.  Rows are independent, so
 * they are split across up to 64 threads (no effect on the result). */
/* 1x32 block quantisation with the literal block scale s = fl32(amax / fmax)
 * (1 when that is 0): the "fp32 scale = block amax/448" wording of the
 * workloads, taken literally rather than rounded up to a power of two. */
static void quantize_block32_impl(const float *x, int64_t rows, int64_t cols, int fmt,
                                  int literal, uint8_t *q, float *scales);

ORACLE_EXPORT void oracle_quantize_block32_literal(const float *x, int64_t rows, int64_t cols,
                                                   int fmt, uint8_t *q, float *scales) {
    quantize_block32_impl(x, rows, cols, fmt, 1, q, scales);
}

ORACLE_EXPORT void oracle_quantize_block32_fmt(const float *x, int64_t rows, int64_t cols,
                                               int fmt, uint8_t *q, float *scales) {
    quantize_block32_impl(x, rows, cols, fmt, 0, q, scales);
}

static void quantize_block32_impl(const float *x, int64_t rows, int64_t cols, int fmt,
                                  int literal, uint8_t *q, float *scales) {
    int nt = (int)(rows * cols / (1 << 20));
    if (nt < 1) nt = 1;
    if (nt > 64) nt = 64;
    if (nt > rows) nt = (int)rows;
    pthread_t tid[64];
    quant_job jobs[64];
    int64_t per = (rows + nt - 1) / nt;
    for (int t = 0; t < nt; ++t) {
        jobs[t].x = x; jobs[t].q = q; jobs[t].scales = scales; jobs[t].cols = cols;
        jobs[t].fmt = fmt;
        jobs[t].literal = literal;
        jobs[t].r0 = t * per < rows ? t * per : rows;
        jobs[t].r1 = (t + 1) * per < rows ? (t + 1) * per : rows;
        if (nt == 1 || pthread_create(&tid[t], NULL, quant_block32_rows, &jobs[t]) != 0) {
            quant_block32_rows(&jobs[t]);
            tid[t] = 0;
        }
    }
    for (int t = 0; t < nt; ++t)
        if (nt > 1 && tid[t]) pthread_join(tid[t], NULL);
}

ORACLE_EXPORT void oracle_quantize_block32(const float *x, int64_t rows, int64_t cols,
                                           uint8_t *q, float *scales) {
    oracle_quantize_block32_fmt(x, rows, cols, ORACLE_E4M3, q, scales);
}

static void *quant_block32_rows(void *arg) {
    quant_job *j = (quant_job *)arg;
    const float *x = j->x;
    uint8_t *q = j->q;
    float *scales = j->scales;
    int64_t cols = j->cols;
    int64_t nb = cols / 32;
    for (int64_t r = j->r0; r < j->r1; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const float *blk = x + r * cols + b * 32;
            float s;
            if (j->literal) {
                s = amax_of(blk, 32, 1) / (float)fmt_max(j->fmt);
                if (s == 0.0f) s = 1.0f;
            } else {
                s = oracle_pow2_scale_fmt(amax_of(blk, 32, 1), j->fmt);
            }
            scales[r * nb + b] = s;
            for (int k = 0; k < 32; ++k) q[r * cols + b * 32 + k] = encode_fmt(blk[k] / s, j->fmt);
        }
    }
    return NULL;
}

/* ------------------------------------------------------------------ */
/* GEMM                                                                */
/* ------------------------------------------------------------------ */

enum { ORACLE_OUT_BF16 = 0, ORACLE_OUT_F32 = 1 };
enum { ORACLE_ACT_NONE = 0, ORACLE_ACT_RELU = 1, ORACLE_ACT_GELU = 2 };

/* Activation in fp64.  ReLU: y < 0 ? 0 : y (NaN stays NaN).  GELU:
 * y * Phi(y) = 0.5 y (1 + erf(y / sqrt 2)). */
ORACLE_EXPORT double oracle_act(double y, int act) {
    if (act == ORACLE_ACT_RELU) return y < 0.0 ? 0.0 : y;
    if (act == ORACLE_ACT_GELU) return 0.5 * y * (1.0 + erf(y / sqrt(2.0)));
    return y;
}

typedef struct {
    const uint8_t *A, *B;
    const float *sfa, *sfb; /* block: [M,K/32], [N,K/32]; tensor: 1 value each */
    int block;
    const double *ta, *tb; /* decode tables of A's and B's format */
    int64_t M, N, K;
    int out_kind;
    float *C;        /* rounded output (bf16 values held in float, or fp32) */
    double *exact;   /* nullable: the value before the output rounding */
    double *bound;   /* nullable: tolerance per element */
    int64_t row_begin, row_end;
    const int64_t *pi, *pj; /* sampled mode: element list (nullable) */
    int64_t n_samples;
    const float *bias;      /* fused epilogue: [N] (nullable) */
    int act;
    int use_alpha;          /* block mode: v = fl32(alpha * sum) (NVFP4's global scales) */
    float alpha;
} gemm_job;

static double dec_e4m3[256], dec_e5m2[256], dec_e2m1[256], dec_e2m3[256], dec_e3m2[256];
static pthread_once_t dec_once = PTHREAD_ONCE_INIT;
static void fill_tables(void) {
    oracle_e4m3_table(dec_e4m3);
    oracle_e5m2_table(dec_e5m2);
    oracle_e2m1_table(dec_e2m1);
    oracle_e2m3_table(dec_e2m3);
    oracle_e3m2_table(dec_e3m2);
}
static const double *table_of(int fmt) {
    pthread_once(&dec_once, fill_tables);
    switch (fmt) {
    case ORACLE_E2M1: return dec_e2m1;
    case ORACLE_E2M3: return dec_e2m3;
    case ORACLE_E3M2: return dec_e3m2;
    case ORACLE_E5M2: return dec_e5m2;
    default: return dec_e4m3;
    }
}

/* One output element.  Block mode (block = 16: 1x16 blocks, scales
 * [M,K/16], [N,K/16]; any other nonzero value: 1x32 blocks):
 *   v = sum_kb sfa[i,kb] * sfb[j,kb] * (sum_{k in kb} dec(a_ik) dec(b_jk))
 * and with use_alpha v = fl32(alpha * v).
 * Tensor mode:
 *   acc = sum_k dec(a_ik) dec(b_jk), alpha = fl32(sA * sB), v = fl32(alpha * acc)
 * The tolerance bound is 2^-8 * sum_k |sA a_ik| |sB b_jk| + 1 bf16 ulp of the
 * rounded reference. */
static void one_element(const gemm_job *g, int64_t i, int64_t j, float *out, double *exact,
                        double *bound) {
    const uint8_t *a = g->A + i * g->K;
    const uint8_t *b = g->B + j * g->K;
    double v, absum = 0.0;
    if (g->block) {
        const int64_t bs = g->block == 16 ? 16 : 32;
        int64_t nb = g->K / bs;
        double total = 0.0;
        for (int64_t kb = 0; kb < nb; ++kb) {
            double part = 0.0, apart = 0.0;
            for (int64_t k = kb * bs; k < kb * bs + bs; ++k) {
                double p = g->ta[a[k]] * g->tb[b[k]];
                part += p;
                apart += fabs(p);
            }
            double sc = (double)g->sfa[i * nb + kb] * (double)g->sfb[j * nb + kb];
            total += sc * part;
            absum += fabs(sc) * apart;
        }
        v = total;
        if (g->use_alpha) {
            v = (double)(float)((double)g->alpha * total);
            absum *= fabs((double)g->alpha);
        }
    } else {
        double acc = 0.0, aacc = 0.0;
        for (int64_t k = 0; k < g->K; ++k) {
            double p = g->ta[a[k]] * g->tb[b[k]];
            acc += p;
            aacc += fabs(p);
        }
        float alpha = g->sfa[0] * g->sfb[0];
        v = (double)(float)((double)alpha * acc);
        absum = fabs((double)g->sfa[0] * (double)g->sfb[0]) * aacc;
    }
    double lip = 1.0, extra = 0.0;
    if (g->bias != NULL || g->act != ORACLE_ACT_NONE) {
        /* epilogue: y = act(v + bias[j]); |GELU'| <= 1.13; the GPU adds the
         * bias and evaluates the activation in fp32 (2^-20 relative covers it) */
        double b = g->bias != NULL ? (double)g->bias[j] : 0.0;
        extra = ldexp(fabs(v) + fabs(b), -20);
        v = oracle_act(v + b, g->act);
        if (g->act == ORACLE_ACT_GELU) lip = 1.13;
    }
    float r = (g->out_kind == ORACLE_OUT_BF16) ? oracle_bf16_round(v) : (float)v;
    *out = r;
    if (exact) *exact = v;
    if (bound) *bound = lip * ldexp(absum, -8) + extra + oracle_bf16_ulp((double)r);
}

static void *gemm_worker(void *arg) {
    gemm_job *g = (gemm_job *)arg;
    if (g->pi) {
        for (int64_t s = g->row_begin; s < g->row_end; ++s)
            one_element(g, g->pi[s], g->pj[s], &g->C[s], g->exact ? &g->exact[s] : NULL,
                        g->bound ? &g->bound[s] : NULL);
        return NULL;
    }
    for (int64_t i = g->row_begin; i < g->row_end; ++i)
        for (int64_t j = 0; j < g->N; ++j) {
            int64_t o = i * g->N + j;
            one_element(g, i, j, &g->C[o], g->exact ? &g->exact[o] : NULL,
                        g->bound ? &g->bound[o] : NULL);
        }
    return NULL;
}

static void run_jobs(gemm_job proto, int64_t n_items, int threads) {
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    if (n_items < threads) threads = (int)(n_items > 0 ? n_items : 1);
    pthread_t tid[256];
    gemm_job jobs[256];
    int64_t per = (n_items + threads - 1) / threads;
    int started = 0;
    for (int t = 0; t < threads; ++t) {
        jobs[t] = proto;
        jobs[t].row_begin = t * per;
        jobs[t].row_end = (t + 1) * per < n_items ? (t + 1) * per : n_items;
        if (jobs[t].row_begin >= jobs[t].row_end) continue;
        if (threads == 1 || pthread_create(&tid[t], NULL, gemm_worker, &jobs[t]) != 0) {
            gemm_worker(&jobs[t]);
            tid[t] = 0;
        } else {
            ++started;
        }
    }
    for (int t = 0; t < threads; ++t)
        if (threads > 1 && jobs[t].row_begin < jobs[t].row_end && tid[t]) pthread_join(tid[t], NULL);
}

/* Full GEMM.  block = 0: sfa, sfb each point to one fp32 per-tensor scale.
 * block = 1: sfa [M, K/32], sfb [N, K/32].  a_fmt, b_fmt: ORACLE_E4M3,
 * ORACLE_E5M2, ORACLE_E2M1, ORACLE_E2M3 or ORACLE_E3M2.  C, exact, bound:
 * [M, N]. */
/* GEMM with operand formats and the fused epilogue (bias [N] nullable, act). */
ORACLE_EXPORT void oracle_gemm_ex(const uint8_t *A, const uint8_t *B, const float *sfa,
                                  const float *sfb, int block, int a_fmt, int b_fmt,
                                  const float *bias, int act, int64_t M, int64_t N, int64_t K,
                                  int out_kind, float *C, double *exact, double *bound,
                                  int threads) {
    gemm_job g;
    memset(&g, 0, sizeof g);
    g.A = A; g.B = B; g.sfa = sfa; g.sfb = sfb; g.block = block;
    g.ta = table_of(a_fmt); g.tb = table_of(b_fmt);
    g.bias = bias; g.act = act;
    g.M = M; g.N = N; g.K = K; g.out_kind = out_kind;
    g.C = C; g.exact = exact; g.bound = bound;
    run_jobs(g, M, threads);
}

ORACLE_EXPORT void oracle_gemm_fmt(const uint8_t *A, const uint8_t *B, const float *sfa,
                                   const float *sfb, int block, int a_fmt, int b_fmt, int64_t M,
                                   int64_t N, int64_t K, int out_kind, float *C, double *exact,
                                   double *bound, int threads) {
    gemm_job g;
    memset(&g, 0, sizeof g);
    g.A = A; g.B = B; g.sfa = sfa; g.sfb = sfb; g.block = block;
    g.ta = table_of(a_fmt); g.tb = table_of(b_fmt);
    g.M = M; g.N = N; g.K = K; g.out_kind = out_kind;
    g.C = C; g.exact = exact; g.bound = bound;
    run_jobs(g, M, threads);
}

ORACLE_EXPORT void oracle_gemm(const uint8_t *A, const uint8_t *B, const float *sfa,
                               const float *sfb, int block, int64_t M, int64_t N, int64_t K,
                               int out_kind, float *C, double *exact, double *bound,
                               int threads) {
    oracle_gemm_fmt(A, B, sfa, sfb, block, ORACLE_E4M3, ORACLE_E4M3, M, N, K, out_kind, C, exact,
                    bound, threads);
}

/* Sampled GEMM: only the n elements (pi[s], pj[s]). Outputs are length n. */
ORACLE_EXPORT void oracle_gemm_sample_ex(const uint8_t *A, const uint8_t *B, const float *sfa,
                                         const float *sfb, int block, int a_fmt, int b_fmt,
                                         const float *bias, int act, int64_t M, int64_t N,
                                         int64_t K, int out_kind, const int64_t *pi,
                                         const int64_t *pj, int64_t n, float *C, double *exact,
                                         double *bound, int threads) {
    gemm_job g;
    memset(&g, 0, sizeof g);
    g.A = A; g.B = B; g.sfa = sfa; g.sfb = sfb; g.block = block;
    g.ta = table_of(a_fmt); g.tb = table_of(b_fmt);
    g.bias = bias; g.act = act;
    g.M = M; g.N = N; g.K = K; g.out_kind = out_kind;
    g.C = C; g.exact = exact; g.bound = bound;
    g.pi = pi; g.pj = pj; g.n_samples = n;
    run_jobs(g, n, threads);
}

ORACLE_EXPORT void oracle_gemm_sample_fmt(const uint8_t *A, const uint8_t *B, const float *sfa,
                                          const float *sfb, int block, int a_fmt, int b_fmt,
                                          int64_t M, int64_t N, int64_t K, int out_kind,
                                          const int64_t *pi, const int64_t *pj, int64_t n,
                                          float *C, double *exact, double *bound, int threads) {
    gemm_job g;
    memset(&g, 0, sizeof g);
    g.A = A; g.B = B; g.sfa = sfa; g.sfb = sfb; g.block = block;
    g.ta = table_of(a_fmt); g.tb = table_of(b_fmt);
    g.M = M; g.N = N; g.K = K; g.out_kind = out_kind;
    g.C = C; g.exact = exact; g.bound = bound;
    g.pi = pi; g.pj = pj; g.n_samples = n;
    run_jobs(g, n, threads);
}

ORACLE_EXPORT void oracle_gemm_sample(const uint8_t *A, const uint8_t *B, const float *sfa,
                                      const float *sfb, int block, int64_t M, int64_t N,
                                      int64_t K, int out_kind, const int64_t *pi,
                                      const int64_t *pj, int64_t n, float *C, double *exact,
                                      double *bound, int threads) {
    oracle_gemm_sample_fmt(A, B, sfa, sfb, block, ORACLE_E4M3, ORACLE_E4M3, M, N, K, out_kind, pi,
                           pj, n, C, exact, bound, threads);
}

/* NVFP4 GEMM: A, B E2M1 codes (one per byte) [M,K], [N,K]; sfa, sfb the
 * decoded block scales [M,K/16], [N,K/16] (exact in fp32); ga, gb the
 * tensors' fp32 scales; bias (nullable) / act the fused epilogue.
 * C = out(act(fl32(fl32(ga gb) * sum) + bias[j])).  K % 16 == 0. */
ORACLE_EXPORT void oracle_gemm_nvfp4(const uint8_t *A, const uint8_t *B, const float *sfa,
                                     const float *sfb, float ga, float gb, const float *bias,
                                     int act, int64_t M, int64_t N, int64_t K, int out_kind,
                                     float *C, double *exact, double *bound, int threads) {
    gemm_job g;
    memset(&g, 0, sizeof g);
    g.A = A; g.B = B; g.sfa = sfa; g.sfb = sfb; g.block = 16;
    g.ta = table_of(ORACLE_E2M1); g.tb = table_of(ORACLE_E2M1);
    g.use_alpha = 1; g.alpha = ga * gb;
    g.bias = bias; g.act = act;
    g.M = M; g.N = N; g.K = K; g.out_kind = out_kind;
    g.C = C; g.exact = exact; g.bound = bound;
    run_jobs(g, M, threads);
}

ORACLE_EXPORT void oracle_gemm_nvfp4_sample(const uint8_t *A, const uint8_t *B, const float *sfa,
                                            const float *sfb, float ga, float gb,
                                            const float *bias, int act, int64_t M, int64_t N,
                                            int64_t K, int out_kind, const int64_t *pi,
                                            const int64_t *pj, int64_t n, float *C, double *exact,
                                            double *bound, int threads) {
    gemm_job g;
    memset(&g, 0, sizeof g);
    g.A = A; g.B = B; g.sfa = sfa; g.sfb = sfb; g.block = 16;
    g.ta = table_of(ORACLE_E2M1); g.tb = table_of(ORACLE_E2M1);
    g.use_alpha = 1; g.alpha = ga * gb;
    g.bias = bias; g.act = act;
    g.M = M; g.N = N; g.K = K; g.out_kind = out_kind;
    g.C = C; g.exact = exact; g.bound = bound;
    g.pi = pi; g.pj = pj; g.n_samples = n;
    run_jobs(g, n, threads);
}

/* NVFP4 quantisation of x [rows, cols] (cols % 16 == 0), the reading taken
 * (the pages name the format and print no recipe):
 *   g = fl32(amax / 2688) over the non-NaN |x| (2688 = 6 x 448, the largest
 *       E2M1 value times the largest E4M3 scale), 1 when that is 0;
 *   per 1x16 block along cols: t = fl32(amax_b / fl32(6 g)),
 *       s = the E4M3 code of t, round to nearest even, saturating (t >= 0);
 *   elements: d = fl32(dec(s) * g); q = the E2M1 code of fl32(x / d), round
 *       to nearest even, saturating, NaN -> +6; all codes 0 when d is 0.
 * q: one E2M1 code per byte [rows, cols]; sf: E4M3 codes [rows, cols/16];
 * g_out: g. */
ORACLE_EXPORT void oracle_quantize_nvfp4(const float *x, int64_t rows, int64_t cols, uint8_t *q,
                                         uint8_t *sf, float *g_out) {
    const float amax = amax_of(x, rows * cols, 1);
    float g = amax / 2688.0f;
    if (g == 0.0f) g = 1.0f;
    const float g6 = 6.0f * g;
    const int64_t nb = cols / 16;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const float *xb = x + r * cols + b * 16;
            uint8_t *qb = q + r * cols + b * 16;
            const float t = amax_of(xb, 16, 1) / g6;
            const uint8_t s = oracle_e4m3_encode(t);
            const float d = (float)oracle_e4m3_decode(s) * g;
            for (int k = 0; k < 16; ++k) qb[k] = d > 0.0f ? oracle_e2m1_encode(xb[k] / d) : 0;
            sf[r * nb + b] = s;
        }
    *g_out = g;
}

/* ------------------------------------------------------------------ */
/* Grouped (MoE) problem list and raster order                         */
/* ------------------------------------------------------------------ */

/* offsets[0] = 0, offsets[e+1] = offsets[e] + counts[e] */
ORACLE_EXPORT void oracle_grouped_offsets(const int32_t *counts, int32_t E, int32_t *offsets) {
    offsets[0] = 0;
    for (int32_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
}

/* Grouped raster order of one problem's npm x npn tile grid, group height G:
 * tiles are walked in bands of G tile-rows; inside a band, down the rows of
 * one tile-column first, then on to the next column. */
ORACLE_EXPORT void oracle_raster(int64_t t, int64_t npm, int64_t npn, int64_t G, int64_t *pid_m,
                                 int64_t *pid_n) {
    int64_t band = G * npn;
    int64_t grp = t / band;
    int64_t first_m = grp * G;
    int64_t rows_here = npm - first_m < G ? npm - first_m : G;
    int64_t in_band = t % band;
    *pid_m = first_m + in_band % rows_here;
    *pid_n = in_band / rows_here;
}

/* Tile list of a single GEMM in launch order: out[2t] = pid_m, out[2t+1] = pid_n. */
ORACLE_EXPORT int64_t oracle_tile_map(int64_t M, int64_t N, int64_t BM, int64_t BN, int64_t G,
                                      int64_t *out, int64_t cap) {
    int64_t npm = (M + BM - 1) / BM, npn = (N + BN - 1) / BN, T = npm * npn;
    for (int64_t t = 0; t < T && t < cap; ++t) oracle_raster(t, npm, npn, G, &out[2 * t], &out[2 * t + 1]);
    return T;
}

/* Tile list of a grouped GEMM: experts in index order, expert e owning
 * ceil(M_e/BM) * ceil(N/BN) consecutive tiles (none when M_e = 0), each
 * expert's tiles in the grouped raster order above.
 * out[4t..4t+3] = (expert, m_tile, n_tile, 0).  Returns the tile count. */
ORACLE_EXPORT int64_t oracle_grouped_tile_map(const int32_t *counts, int32_t E, int64_t N,
                                              int64_t BM, int64_t BN, int64_t G, int32_t *out,
                                              int64_t cap) {
    int64_t npn = (N + BN - 1) / BN, t = 0;
    for (int32_t e = 0; e < E; ++e) {
        int64_t npm = (counts[e] + BM - 1) / BM;
        for (int64_t l = 0; l < npm * npn; ++l, ++t) {
            int64_t pm, pn;
            oracle_raster(l, npm, npn, G, &pm, &pn);
            if (t < cap) {
                out[4 * t + 0] = e;
                out[4 * t + 1] = (int32_t)pm;
                out[4 * t + 2] = (int32_t)pn;
                out[4 * t + 3] = 0;
            }
        }
    }
    return t;
}

/* Grouped GEMM: A [sum M_e, K] with expert e's rows at [off_e, off_e + M_e),
 * B [E, N, K], sfa [sum M_e, K/32], sfb [E, N, K/32]; C [sum M_e, N].
 * Each expert is an independent block-scaled GEMM. */
ORACLE_EXPORT void oracle_grouped_gemm(const uint8_t *A, const uint8_t *B, const float *sfa,
                                       const float *sfb, const int32_t *counts, int32_t E,
                                       int64_t N, int64_t K, int out_kind, float *C,
                                       double *exact, double *bound, int threads) {
    int64_t off = 0, nb = K / 32;
    for (int32_t e = 0; e < E; ++e) {
        int64_t Me = counts[e];
        if (Me > 0)
            oracle_gemm(A + off * K, B + (int64_t)e * N * K, sfa + off * nb,
                        sfb + (int64_t)e * N * nb, 1, Me, N, K, out_kind, C + off * N,
                        exact ? exact + off * N : NULL, bound ? bound + off * N : NULL, threads);
        off += Me;
    }
}

/* Algorithmic FLOP count of C = A B^T: 2 M N K ("TFLOPS = 2*M*N*K/(t*1e12)"
 * in the monitoring checklist of the Triton FP8 benchmarking page). */
ORACLE_EXPORT double oracle_gemm_flops(int64_t M, int64_t N, int64_t K) {
    return 2.0 * (double)M * (double)N * (double)K;
}
