/*
 * qlin_oracle.c -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.
 *
 * A plain, slow, CPU-only restatement of what the quantized linear layer
 * computes.  Only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark may load this library.  It shares no code, header, table or
 * helper with the CUDA path; every function below is written from the pages'
 * statement of the method, with no blocking, fusion or reordering beyond what
 * that statement implies.
 *
 * Sources (web pages; titles as printed, section names in brackets):
 *   [QDC]  "量化、蒸馏与模型压缩" (Quantization, distillation and model
 *          compression), llm-knowledge-atlas notes 03-05.
 *   [L19]  "十九：模型压缩：量化、ZeroQuant、LLM.int8() 与 SmoothQuant".
 *   [CH11] "第11章 模型量化与压缩" (Chapter 11, model quantization and
 *          compression), ai-infra-guide.
 *   [CSDN] "大模型压缩：从研究到生产的完整攻略（1）" (Model compression:
 *          a complete guide from research to production, part 1).
 *
 * Floating point: compiled without fast-math and without FP contraction, so
 * every float operation below is one IEEE-754 binary32 operation, correctly
 * rounded to nearest-even (x86-64 SSE arithmetic).
 *
 * Readings of points the pages leave open (each is also listed in the design
 * notes of the repository):
 *   - round() is round-half-to-even, applied to the correctly rounded binary32
 *     quotient fl(x/s); the zero point is added after rounding ([QDC] core
 *     formula; [L19] section 3; [CH11] 11.1.1).
 *   - symmetric codes use [-qmax, qmax] with s = fl(absmax/qmax) ([CH11]
 *     11.1.2, [CSDN] symmetric quantization).
 *   - asymmetric range is widened to contain 0 (rmin = min(min x, 0),
 *     rmax = max(max x, 0)) so that 0 is represented exactly ([CSDN]
 *     asymmetric quantization; [CH11] 11.1.2), s = fl(fl(rmax-rmin)/(qmax-qmin))
 *     and z = clip(qmin + rne(fl(-rmin/s)), qmin, qmax), which is the page's
 *     round(-min/s) for unsigned codes.
 *   - a scope whose scale comes out as 0 (all-zero data, or an fp16 scale
 *     that underflows) stores s = 1.
 *   - fp16 scales are rounded to nearest-even binary16, saturating at 65504,
 *     and the stored (rounded) scale is the one used to quantize.
 *   - percentile clipping: T = the ceil(n*p/100)-th smallest |x| of the scope
 *     (nearest rank, p in percent, computed in binary64), s = fl(T/qmax);
 *     values beyond T clip ([CH11] 11.1.5; [CSDN] solution strategies).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_PER_TENSOR = 0, ORC_PER_ROW = 1, ORC_PER_COL = 2, ORC_PER_GROUP = 3 };
enum { ORC_SMOOTH_NONE = 0, ORC_SMOOTH_DIVIDE = 1, ORC_SMOOTH_MULTIPLY = 2 };

/* ------------------------------------------------------------------------ */
/* Number formats                                                           */
/* ------------------------------------------------------------------------ */

/* bf16 -> binary32: the bf16 pattern is the upper half of the binary32. */
float orc_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary32 -> bf16, round to nearest, ties to even (NaN kept quiet). */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep_lsb = (u >> 16) & 1u;
    u += 0x7fffu + keep_lsb;
    return (uint16_t)(u >> 16);
}

/* Value of f after rounding to bf16 (returned as binary32). */
float orc_round_bf16(float f)
{
    return orc_bf16_to_f32(orc_f32_to_bf16(f));
}

/* Array forms, for comparing many values at once. */
void orc_round_bf16_n(const float *x, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_round_bf16(x[i]);
}

/* binary32 -> binary16 -> binary32, nearest-even, saturating at +-65504. */
float orc_round_f16(float f)
{
    _Float16 h = (_Float16)f;
    float r = (float)h;
    if (isinf(r) && !isinf(f))
        r = (f > 0.0f) ? 65504.0f : -65504.0f;
    return r;
}

void orc_round_f16_n(const float *x, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_round_f16(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Scopes: which scale/zero point an element (r, c) uses                    */
/* ([L19] section 4 granularity; [CH11] 11.1.3 table 11-1; [QDC] 1.1 groups) */
/* ------------------------------------------------------------------------ */

int64_t orc_num_scopes(int gran, int64_t rows, int64_t cols, int64_t group)
{
    switch (gran) {
    case ORC_PER_TENSOR: return 1;
    case ORC_PER_ROW:    return rows;
    case ORC_PER_COL:    return cols;
    case ORC_PER_GROUP:  return (group > 0) ? rows * (cols / group) : -1;
    default:             return -1;
    }
}

static int64_t scope_of(int gran, int64_t r, int64_t c, int64_t cols, int64_t group)
{
    switch (gran) {
    case ORC_PER_TENSOR: return 0;
    case ORC_PER_ROW:    return r;
    case ORC_PER_COL:    return c;
    default:             return r * (cols / group) + c / group;
    }
}

/* Optional smoothing of element (r, c): x / s_c or x * s_c in binary32
 * ([QDC] 2.3 SmoothQuant; [CH11] 11.4.2 -- X diag(s)^-1). */
static float smooth_one(float v, const float *smooth, int mode, int64_t c)
{
    if (mode == ORC_SMOOTH_DIVIDE)
        return v / smooth[c];
    if (mode == ORC_SMOOTH_MULTIPLY)
        return v * smooth[c];
    return v;
}

static int cmp_float(const void *a, const void *b)
{
    float x = *(const float *)a, y = *(const float *)b;
    return (x < y) ? -1 : (x > y) ? 1 : 0;
}

/* Nearest-rank position (1-based) of the p-th percentile among n values. */
int64_t orc_percentile_rank(int64_t n, double p)
{
    double k = ceil((double)n * p / 100.0);
    if (k < 1.0) k = 1.0;
    if (k > (double)n) k = (double)n;
    return (int64_t)k;
}

/*
 * Affine quantizer ([QDC] core formula; [L19] section 3; [CH11] 11.1.1-11.1.5;
 * [CSDN] linear quantization).
 *
 *   x      : rows x cols binary32, row-major, already widened from its storage.
 *   smooth : NULL or cols factors, applied as smooth_mode says.
 *   q      : rows x cols codes (int32 holding the integer code).
 *   s, z   : one per scope; read when static_scale != 0, written otherwise.
 * Returns 0, or -1 on an argument the method does not define.
 */
int orc_quantize(const float *x, int64_t rows, int64_t cols,
                 const float *smooth, int smooth_mode,
                 int qmin, int qmax, int symmetric, int gran, int64_t group,
                 double percentile, int scale_f16, int static_scale,
                 int32_t *q, float *s, int32_t *z)
{
    if (rows < 0 || cols < 0 || qmax <= qmin) return -1;
    if (symmetric && qmin != -qmax) return -1;
    if (gran == ORC_PER_GROUP && (group <= 0 || cols % group != 0)) return -1;
    if (percentile > 0.0 && !symmetric) return -1;
    int64_t nsc = orc_num_scopes(gran, rows, cols, group);
    if (nsc < 0) return -1;
    int64_t n = rows * cols;

    /* Step 1: widen + optional smoothing. */
    float *xs = (float *)malloc((size_t)(n > 0 ? n : 1) * sizeof(float));
    if (!xs) return -2;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            xs[r * cols + c] = smooth_one(x[r * cols + c], smooth, smooth_mode, c);

    if (!static_scale) {
        /* Step 2: range statistics of every scope. */
        float *lo = (float *)calloc((size_t)(nsc > 0 ? nsc : 1), sizeof(float));
        float *hi = (float *)calloc((size_t)(nsc > 0 ? nsc : 1), sizeof(float));
        if (!lo || !hi) { free(xs); free(lo); free(hi); return -2; }
        if (percentile > 0.0) {
            /* Percentile clipping: gather |x| of each scope, sort, take the
             * nearest-rank element. */
            int64_t *cnt = (int64_t *)calloc((size_t)(nsc > 0 ? nsc : 1), sizeof(int64_t));
            for (int64_t r = 0; r < rows; ++r)
                for (int64_t c = 0; c < cols; ++c)
                    cnt[scope_of(gran, r, c, cols, group)]++;
            for (int64_t sc = 0; sc < nsc; ++sc) {
                float *buf = (float *)malloc((size_t)(cnt[sc] > 0 ? cnt[sc] : 1) * sizeof(float));
                int64_t m = 0;
                for (int64_t r = 0; r < rows; ++r)
                    for (int64_t c = 0; c < cols; ++c)
                        if (scope_of(gran, r, c, cols, group) == sc)
                            buf[m++] = fabsf(xs[r * cols + c]);
                if (m > 0) {
                    qsort(buf, (size_t)m, sizeof(float), cmp_float);
                    hi[sc] = buf[orc_percentile_rank(m, percentile) - 1];
                }
                free(buf);
            }
            free(cnt);
        } else {
            /* Min-max: lo/hi start at 0, so the range always contains 0. */
            for (int64_t r = 0; r < rows; ++r)
                for (int64_t c = 0; c < cols; ++c) {
                    int64_t sc = scope_of(gran, r, c, cols, group);
                    float v = xs[r * cols + c];
                    if (symmetric) {
                        float a = fabsf(v);
                        if (a > hi[sc]) hi[sc] = a;
                    } else {
                        if (v < lo[sc]) lo[sc] = v;
                        if (v > hi[sc]) hi[sc] = v;
                    }
                }
        }
        /* Step 3: scale and zero point of every scope. */
        for (int64_t sc = 0; sc < nsc; ++sc) {
            float scale;
            if (symmetric)
                scale = hi[sc] / (float)qmax;
            else
                scale = (hi[sc] - lo[sc]) / (float)(qmax - qmin);
            if (scale_f16)
                scale = orc_round_f16(scale);
            if (scale == 0.0f)
                scale = 1.0f;
            s[sc] = scale;
            if (symmetric) {
                z[sc] = 0;
            } else {
                float t = (-lo[sc]) / scale;
                long zz = (long)qmin + (long)nearbyintf(t);
                if (zz < qmin) zz = qmin;
                if (zz > qmax) zz = qmax;
                z[sc] = (int32_t)zz;
            }
        }
        free(lo);
        free(hi);
    }

    /* Step 4: codes. q = clip(rne(fl(x/s)) + z, qmin, qmax). */
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            int64_t sc = scope_of(gran, r, c, cols, group);
            float t = xs[r * cols + c] / s[sc];
            double v = (double)nearbyintf(t) + (double)z[sc];
            if (v < (double)qmin) v = (double)qmin;
            if (v > (double)qmax) v = (double)qmax;
            q[r * cols + c] = (int32_t)v;
        }
    free(xs);
    return 0;
}

/* Dequantization x^ = fl(s * (q - z)) ([QDC] core formula; [CSDN]
 * asymmetric dequantization formula). */
int orc_dequantize(const int32_t *q, const float *s, const int32_t *z,
                   int64_t rows, int64_t cols, int gran, int64_t group, float *y)
{
    if (gran == ORC_PER_GROUP && (group <= 0 || cols % group != 0)) return -1;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            int64_t sc = scope_of(gran, r, c, cols, group);
            int32_t zz = z ? z[sc] : 0;
            y[r * cols + c] = s[sc] * (float)(q[r * cols + c] - zz);
        }
    return 0;
}

/* max |x| over each scope (the statistic of the symmetric scale; also the
 * per-channel maxima that SmoothQuant's factors are built from, [CH11]
 * 11.4.5 step 1). */
int orc_absmax(const float *x, int64_t rows, int64_t cols, int gran, int64_t group, float *out)
{
    int64_t nsc = orc_num_scopes(gran, rows, cols, group);
    if (nsc < 0 || (gran == ORC_PER_GROUP && cols % group != 0)) return -1;
    for (int64_t sc = 0; sc < nsc; ++sc) out[sc] = 0.0f;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            int64_t sc = scope_of(gran, r, c, cols, group);
            float a = fabsf(x[r * cols + c]);
            if (a > out[sc]) out[sc] = a;
        }
    return 0;
}

/* SmoothQuant factors s_j = max|X_j|^alpha / max|W_j|^(1-alpha)
 * ([QDC] 2.3 eq. 1; [CH11] 11.4.3).  alpha = 0.5 is evaluated as
 * fl(fl(sqrt(mx)) / fl(sqrt(mw))) in binary32; other alphas in binary64 and
 * rounded once.  A channel with a zero maximum gets s_j = 1. */
void orc_smooth_factors(const float *xmax, const float *wmax, int64_t K, float alpha, float *s)
{
    for (int64_t j = 0; j < K; ++j) {
        float mx = xmax[j], mw = wmax[j];
        if (mx == 0.0f || mw == 0.0f) {
            s[j] = 1.0f;
        } else if (alpha == 0.5f) {
            s[j] = sqrtf(mx) / sqrtf(mw);
        } else {
            double v = pow((double)mx, (double)alpha) / pow((double)mw, 1.0 - (double)alpha);
            s[j] = (float)v;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Code storage                                                             */
/* ------------------------------------------------------------------------ */

/* Two 4-bit codes per byte, element 2i in the low nibble; signed codes are
 * stored in two's complement ([CSDN] INT4 "0.5 bytes"). */
void orc_pack_nibbles(const int32_t *q, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; i += 2) {
        uint32_t lo = (uint32_t)q[i] & 0xFu;
        uint32_t hi = (i + 1 < n) ? ((uint32_t)q[i + 1] & 0xFu) : 0u;
        out[i / 2] = (uint8_t)(lo | (hi << 4));
    }
}

void orc_unpack_nibbles(const uint8_t *in, int64_t n, int is_signed, int32_t *q)
{
    for (int64_t i = 0; i < n; ++i) {
        int32_t v = (in[i / 2] >> ((i & 1) ? 4 : 0)) & 0xF;
        if (is_signed && v >= 8) v -= 16;
        q[i] = v;
    }
}

/* ------------------------------------------------------------------------ */
/* W8A8 linear layer ([L19] section 6; [CH11] 11.1.4, 11.4.5 step 6)          */
/* ------------------------------------------------------------------------ */

/* INT8 x INT8 -> exact integer sums, acc[m,n] = sum_k qx[m,k] * qw[n,k]
 * (both operands K-contiguous).  int64 so that any overflow of the int32
 * range is visible to the caller. */
void orc_w8a8_acc(const int8_t *qx, const int8_t *qw, int64_t M, int64_t N, int64_t K, int64_t *acc)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            int64_t sum = 0;
            for (int64_t k = 0; k < K; ++k)
                sum += (int64_t)qx[m * K + k] * (int64_t)qw[n * K + k];
            acc[m * N + n] = sum;
        }
}

/* Dequant epilogue in binary64: y[m,n] = acc[m,n] * sx[m] * sw[n]
 * (per-token scale x per-output-channel scale). */
void orc_w8a8_out(const int64_t *acc, const float *sx, const float *sw, int64_t M, int64_t N, double *y)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            y[m * N + n] = (double)acc[m * N + n] * (double)sx[m] * (double)sw[n];
}

/* ------------------------------------------------------------------------ */
/* W4A16 linear layer ([CH11] 11.1.6 worked case: dequantize to a 16-bit     */
/* weight, then a 16-bit matmul)                                             */
/* ------------------------------------------------------------------------ */

/* w^[n,k] = bf16( fl(s[n, k/g] * (q[n,k] - z[n, k/g])) ); s already holds the
 * stored (fp16-rounded) scale; z may be NULL for symmetric codes. */
void orc_w4_dequant(const int32_t *q, const float *s, const int32_t *z,
                    int64_t N, int64_t K, int64_t g, float *what)
{
    int64_t ng = K / g;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            int64_t sc = n * ng + k / g;
            int32_t zz = z ? z[sc] : 0;
            what[n * K + k] = orc_round_bf16(s[sc] * (float)(q[n * K + k] - zz));
        }
}

/* Plain binary64 matmul y[m,n] = sum_k x[m,k] * w[n,k]. */
void orc_matmul_f64(const float *x, const float *w, int64_t M, int64_t N, int64_t K, double *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double sum = 0.0;
            for (int64_t k = 0; k < K; ++k)
                sum += (double)x[m * K + k] * (double)w[n * K + k];
            y[m * N + n] = sum;
        }
}

/* ------------------------------------------------------------------------ */
/* W4A8 linear layer: group-wise INT4 weights x per-token INT8 activations   */
/* ([CH11] 11.4.5 step 6 and 11.9.7: AWQ-style INT4 weights with             */
/* SmoothQuant INT8 activations; integer products summed exactly, then the   */
/* scales).  Each weight group g (g consecutive k of a row) has its own      */
/* scale s[n,g] and zero point z[n,g], so the integer sums are kept per      */
/* group and the scales are applied afterwards:                              */
/*   acc[g][m][n] = sum_{k in group g} qx[m,k] * (q[n,k] - z[n,g])           */
/*   y[m][n]      = sx[m] * sum_g s[n,g] * acc[g][m][n]     (binary64)        */
/* which is the product of the dequantized operands x^ = sx*qx and           */
/* w^ = s*(q - z).                                                           */
/* ------------------------------------------------------------------------ */

/* qx: M x K int8 codes; q: N x K int32 weight codes; z: N x K/g or NULL
 * (symmetric codes, z = 0); acc: (K/g) x M x N int64. */
void orc_w4a8_acc(const int8_t *qx, const int32_t *q, const int32_t *z, int64_t M, int64_t N, int64_t K,
                  int64_t g, int64_t *acc)
{
    int64_t ng = K / g;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            for (int64_t gi = 0; gi < ng; ++gi) {
                int64_t zz = z ? z[n * ng + gi] : 0;
                int64_t sum = 0;
                for (int64_t k = gi * g; k < (gi + 1) * g; ++k)
                    sum += (int64_t)qx[m * K + k] * ((int64_t)q[n * K + k] - zz);
                acc[(gi * M + m) * N + n] = sum;
            }
}

/* y[m][n] = sx[m] * sum_g s[n,g] * acc[g][m][n] in binary64; s holds the
 * stored (binary16-rounded) scales, N x K/g. */
void orc_w4a8_out(const int64_t *acc, const float *sx, const float *s, int64_t M, int64_t N, int64_t ng, double *y)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double t = 0.0;
            for (int64_t gi = 0; gi < ng; ++gi)
                t += (double)s[n * ng + gi] * (double)acc[(gi * M + m) * N + n];
            y[m * N + n] = (double)sx[m] * t;
        }
}

/* ------------------------------------------------------------------------ */
/* SmoothQuant calibration ([CH11] 11.4.3 table 11-4, 11.4.4, 11.4.5 steps   */
/* 1-3; [QDC] 2.3)                                                           */
/* ------------------------------------------------------------------------ */

/* Running per-channel maxima over calibration batches:
 * running[j] = max(running[j], max_i |x[i][j]|). */
void orc_channel_absmax_update(const float *x, int64_t rows, int64_t cols, float *running)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            float a = fabsf(x[r * cols + c]);
            if (a > running[c]) running[c] = a;
        }
}

/* Folding diag(s)^-1 into the LayerNorm that produces X: LN(x) diag(s)^-1 is
 * a LayerNorm with gamma'_j = gamma_j / s_j and beta'_j = beta_j / s_j
 * (binary32 divisions).  beta may be NULL. */
void orc_fold_layernorm(const float *gamma, const float *beta, const float *s, int64_t K,
                        float *gamma_out, float *beta_out)
{
    for (int64_t j = 0; j < K; ++j) {
        gamma_out[j] = gamma[j] / s[j];
        if (beta && beta_out) beta_out[j] = beta[j] / s[j];
    }
}

/* Quantization error of a tensor against its (smoothed) original:
 * x'[r][c] = x[r][c] / smooth[c] (divide mode, binary32) or x[r][c] * smooth[c]
 * (multiply mode) or x itself; xhat = fl(s * (q - z)) of the scope.
 * out[0] = sum (x' - xhat)^2, out[1] = sum x'^2, out[2] = max |x' - xhat|,
 * the sums in binary64 in row-major order. */
void orc_quant_error(const float *x, int64_t rows, int64_t cols, const float *smooth, int smooth_mode,
                     const int32_t *q, const float *s, const int32_t *z, int gran, int64_t group, double *out)
{
    double se = 0.0, sx = 0.0, mx = 0.0;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            int64_t sc = scope_of(gran, r, c, cols, group);
            float v = smooth_one(x[r * cols + c], smooth, smooth_mode, c);
            float xh = s[sc] * (float)(q[r * cols + c] - (z ? z[sc] : 0));
            double d = (double)v - (double)xh;
            se += d * d;
            sx += (double)v * (double)v;
            if (fabs(d) > mx) mx = fabs(d);
        }
    out[0] = se;
    out[1] = sx;
    out[2] = mx;
}

/* ------------------------------------------------------------------------ */
/* LLM.int8() mixed-precision decomposition ([L19] sections 9-11):           */
/*   XW = X_normal W_normal (INT8, vector-wise scales) + X_outlier W_outlier   */
/* (16-bit).  Outlier dimensions are the input channels j with               */
/* max_m |x[m][j]| > threshold.  The weight is stored once in INT8 (per      */
/* output channel, scales sw); its outlier columns take part in the 16-bit   */
/* product dequantized, w^[n][j] = sw[n] * qw[n][j].                         */
/* ------------------------------------------------------------------------ */

/* Ascending list of the outlier channels of x (rows x cols); returns their
 * number. */
int64_t orc_llmint8_outlier_cols(const float *x, int64_t rows, int64_t cols, float threshold, int32_t *cols_out)
{
    int64_t n = 0;
    for (int64_t c = 0; c < cols; ++c) {
        int outlier = 0;
        for (int64_t r = 0; r < rows; ++r)
            if (fabsf(x[r * cols + c]) > threshold) outlier = 1;
        if (outlier) cols_out[n++] = (int32_t)c;
    }
    return n;
}

/* y[m][n] = sw[n] * (sx[m] * acc[m][n] + sum_{j in cols} x[m][j] * qw[n][j])
 * in binary64: acc holds the INT8 sums over the normal channels (the
 * outlier channels' activation codes are 0), the second term is the 16-bit
 * product of the outlier channels with the dequantized weight (the factor
 * sw[n] taken out of the sum). */
void orc_llmint8_out(const float *x, const int8_t *qw, const float *sw, const float *sx, const int64_t *acc,
                     const int32_t *cols, int64_t n_out, int64_t M, int64_t N, int64_t K, double *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double o = 0.0;
            for (int64_t i = 0; i < n_out; ++i)
                o += (double)x[m * K + cols[i]] * (double)qw[n * K + cols[i]];
            y[m * N + n] = (double)sw[n] * ((double)sx[m] * (double)acc[m * N + n] + o);
        }
}

/* ------------------------------------------------------------------------ */
/* Threads used by the OpenMP loops above (1 when built without OpenMP).     */
/* ------------------------------------------------------------------------ */
int orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}
