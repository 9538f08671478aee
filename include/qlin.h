/*
 * qlin.h -- C ABI of libqlin.so, a quantized linear layer for NVIDIA B300
 * (sm_103a).
 *
 * The method (affine quantizer, its granularities, and the two quantized
 * linear-layer paths) is the one stated on these pages:
 *   [QDC]  "量化、蒸馏与模型压缩" (Quantization, distillation and model
 *          compression), llm-knowledge-atlas notes 03-05: core formula,
 *          section 1 (error of y = Wx), 1.1 (groups), 2.3 (SmoothQuant).
 *   [L19]  "十九：模型压缩：量化、ZeroQuant、LLM.int8() 与 SmoothQuant":
 *          section 3 (basic formula), 4 (granularity), 6 (W8A8).
 *   [CH11] "第11章 模型量化与压缩" (ai-infra-guide chapter 11): 11.1.1-11.1.6
 *          (affine quantization, symmetric/asymmetric, granularity, dynamic vs
 *          static, calibration, INT4 worked case), 11.4.2-11.4.5 (SmoothQuant).
 *   [CSDN] "大模型压缩：从研究到生产的完整攻略（1）": symmetric and
 *          asymmetric quantization sections, outliers.
 *
 * Conventions for every entry point:
 *   - Pointers named as device pointers must be CUDA device (or managed)
 *     memory on the current device; the caller owns every buffer.  The library
 *     allocates no memory except where an entry point says so.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and returns without synchronizing.
 *   - Arguments are validated on the host before any launch.  On a bad
 *     argument the call returns a negative qlin_status and launches nothing.
 *     A failed launch returns QLIN_ERR_CUDA.  No C++ exception crosses the ABI.
 *   - Inputs must be finite; results for NaN/Inf inputs are unspecified (but
 *     never out-of-bounds accesses).
 *   - Rounding: codes are round-half-to-even of the correctly rounded binary32
 *     quotient fl(x/s), and the zero point is added after rounding.
 */
#ifndef QLIN_H
#define QLIN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QLIN_OK = 0,
    QLIN_ERR_ARG = -1,          /* invalid argument (shape, pointer, range) */
    QLIN_ERR_UNSUPPORTED = -2,  /* valid for the method, not implemented    */
    QLIN_ERR_CUDA = -3,         /* a CUDA runtime call or launch failed      */
    QLIN_ERR_TIMEOUT = -4,      /* a bounded device-side wait gave up        */
    QLIN_ERR_WORKSPACE = -5,    /* workspace missing or too small            */
    QLIN_ERR_LAYOUT = -6        /* packed-weight header does not match       */
} qlin_status;

/* Granularity: which elements share one scale / zero point
 * ([L19] section 4; [CH11] 11.1.3 table 11-1; [QDC] 1.1). */
typedef enum {
    QLIN_PER_TENSOR = 0,  /* one scope                                          */
    QLIN_PER_ROW = 1,     /* one per row: per-token (activations) or per-output-
                             channel (weights stored [out x in])                */
    QLIN_PER_COL = 2,     /* one per column: per-input-channel                  */
    QLIN_PER_GROUP = 3    /* one per g contiguous elements of a row             */
} qlin_gran;

typedef enum {
    QLIN_F32 = 0, QLIN_BF16 = 1, QLIN_F16 = 2,
    QLIN_S8 = 3, QLIN_U8 = 4, QLIN_S4 = 5, QLIN_U4 = 6, QLIN_S32 = 7
} qlin_dtype;

typedef enum {
    QLIN_SMOOTH_NONE = 0,
    QLIN_SMOOTH_DIVIDE = 1,   /* x' = fl(x / smooth[c])  -- X diag(s)^-1 ([QDC] 2.3) */
    QLIN_SMOOTH_MULTIPLY = 2  /* x' = fl(x * smooth[c])  -- diag(s) W (weights)      */
} qlin_smooth;

/* Quantization parameters: the pages' (s, z, qmin/qmax, g, granularity)
 * statement of the problem ([QDC] symbol table; [CH11] 11.1.1-11.1.5). */
typedef struct {
    qlin_dtype code;         /* code storage: QLIN_S8, QLIN_U8, QLIN_S4, QLIN_U4      */
    int qmin, qmax;          /* integer range, must fit `code`; e.g. [-127,127]      */
    int symmetric;           /* 1: z = 0, s = absmax/qmax, needs qmin == -qmax        */
    qlin_gran gran;
    int group;               /* g for QLIN_PER_GROUP (must divide cols), else ignored */
    double clip_percentile;  /* 0: min-max; else p in (0,100]: symmetric per-tensor
                                nearest-rank percentile of |x| replaces max|x|        */
    qlin_dtype scale_dtype;  /* QLIN_F32 or QLIN_F16 (stored scale is what quantizes) */
    int static_scale;        /* 1: read caller's s (and z); 0: compute them (dynamic) */
    int smooth_mode;         /* qlin_smooth                                           */
} qlin_qparams;

/* Operation ids for qlin_workspace_size. */
enum { QLIN_OP_QUANTIZE = 0, QLIN_OP_ABSMAX = 1, QLIN_OP_GEMM_W8A8 = 2, QLIN_OP_GEMM_W4A16 = 3,
       QLIN_OP_GEMM_W4A8 = 4, QLIN_OP_QUANT_ERROR = 5 };

/* Library version (major*10000 + minor*100 + patch). */
int qlin_version(void);

/* Human-readable text of a qlin_status (static string, never NULL). */
const char *qlin_status_string(int status);

/*
 * Bytes of device workspace an operation needs (0 = none; pass ws = NULL).
 * For QLIN_OP_QUANTIZE and QLIN_OP_ABSMAX, M = rows, N = cols, K ignored
 * (for ABSMAX, p->gran selects the granularity); per-row and per-group scopes
 * and static scales need none.  The workspace is scratch
 * owned by the caller; it may be reused once the call's work on `stream`
 * has completed.
 */
size_t qlin_workspace_size(int op, int64_t M, int64_t N, int64_t K, const qlin_qparams *p);

/*
 * qlin_quantize -- affine quantizer q = clip(round(x/s) + z, qmin, qmax)
 * ([QDC] core formula; [L19] section 3; [CH11] 11.1.1-11.1.5; [CSDN] linear
 * quantization), with optional per-column smoothing first ([QDC] 2.3;
 * [CH11] 11.4.2).
 *
 *   x      device, rows x cols elements of type xt (F32, BF16 or F16), row
 *          stride ld elements (ld >= cols).
 *   smooth device, cols binary32 factors, or NULL when p->smooth_mode is NONE.
 *   q      device output codes, dense row-major: S8/U8 one byte per code
 *          (rows*cols bytes); S4/U4 two codes per byte, element 2i in the low
 *          nibble, S4 in two's complement (rows*cols/2 bytes; cols even).
 *   s      device scales, one per scope (1, rows, cols or rows*cols/g), binary32
 *          or binary16 as p->scale_dtype says; written (dynamic) or read
 *          (p->static_scale).
 *   z      device int32 zero points, one per scope; written or read like s.
 *          May be NULL for symmetric parameters.
 *   ws     device workspace of qlin_workspace_size(QLIN_OP_QUANTIZE, rows,
 *          cols, 0, p) bytes (NULL when that is 0).
 * Dynamic scales: symmetric s = fl(max|x| / qmax); asymmetric
 * s = fl(fl(rmax - rmin) / (qmax - qmin)) with rmin = min(min x, 0),
 * rmax = max(max x, 0), z = clip(qmin + rne(fl(-rmin / s)), qmin, qmax).
 * A scale that comes out as 0 is stored as 1; an F16 scale is rounded to
 * nearest-even binary16, saturating at 65504.
 * Percentile clipping (p->clip_percentile > 0) is supported for symmetric
 * QLIN_PER_TENSOR only (else QLIN_ERR_UNSUPPORTED); its rank is
 * k = ceil(n * p / 100) computed in binary64, clamped to [1, n].
 */
int qlin_quantize(const void *x, qlin_dtype xt, int64_t rows, int64_t cols, int64_t ld,
                  const float *smooth, const qlin_qparams *p,
                  void *q, void *s, int32_t *z, void *ws, size_t ws_bytes, void *stream);

/*
 * qlin_dequantize -- x^ = s * (q - z) ([QDC] core formula; [CSDN] asymmetric
 * dequantization), evaluated as one binary32 product and then rounded to yt
 * (F32, BF16 or F16, nearest-even).
 *   q, s, z  device, in the layouts qlin_quantize writes for p (z may be NULL
 *            for symmetric parameters).
 *   y        device output, rows x cols dense row-major of type yt.
 */
int qlin_dequantize(const void *q, const void *s, const int32_t *z, const qlin_qparams *p,
                    int64_t rows, int64_t cols, void *y, qlin_dtype yt, void *stream);

/*
 * qlin_absmax -- max|x| of every scope of the given granularity (the
 * symmetric-scale statistic; with QLIN_PER_COL on X and on W it gives the
 * channel maxima SmoothQuant's factors are built from, [CH11] 11.4.5 step 1).
 *   x    device, rows x cols of type xt, row stride ld.
 *   out  device binary32, one value per scope.
 *   ws   device workspace of qlin_workspace_size(QLIN_OP_ABSMAX, rows, cols,
 *        0, p) bytes where p->gran = gran.
 */
int qlin_absmax(const void *x, qlin_dtype xt, int64_t rows, int64_t cols, int64_t ld,
                qlin_gran gran, int group, float *out, void *ws, size_t ws_bytes, void *stream);

/*
 * qlin_smooth_factors -- s_j = max|X_j|^alpha / max|W_j|^(1-alpha)
 * ([QDC] 2.3 eq. 1; [CH11] 11.4.3), j < K.  alpha = 0.5 is evaluated as
 * fl(sqrt(mx) / sqrt(mw)) with correctly rounded binary32 operations; other
 * alphas with binary32 pow (a few ulp).  A channel with a zero maximum gets
 * s_j = 1.  xmax, wmax, s: device binary32 arrays of K values.
 */
int qlin_smooth_factors(const float *xmax, const float *wmax, int64_t K, float alpha,
                        float *s, void *stream);

/*
 * qlin_absmax_update -- SmoothQuant calibration ([CH11] 11.4.5 steps 1-2):
 * running[j] = max(running[j], max_i |x[i][j]|) over one calibration batch,
 * so that after all batches running holds max|X_j| over the calibration data.
 *   x        device, rows x cols of type xt, row stride ld.
 *   running  device binary32 [cols], non-negative (start from zeros); updated
 *            in place.  The result does not depend on the order of the
 *            updates.
 */
int qlin_absmax_update(const void *x, qlin_dtype xt, int64_t rows, int64_t cols, int64_t ld, float *running,
                       void *stream);

/*
 * qlin_fold_layernorm -- absorbs X diag(s)^-1 into the LayerNorm that
 * produces X ([CH11] 11.4.4: LayerNorm(X) diag(s)^-1 = LayerNorm'(X) with
 * gamma' = gamma / s; the bias likewise): gamma_out[j] = fl(gamma[j] / s[j]),
 * beta_out[j] = fl(beta[j] / s[j]) (correctly rounded binary32 divisions).
 * beta and beta_out are both NULL for a LayerNorm without bias (RMSNorm).
 * All pointers device binary32 arrays of K values.
 */
int qlin_fold_layernorm(const float *gamma, const float *beta, const float *s, int64_t K, float *gamma_out,
                        float *beta_out, void *stream);

/*
 * qlin_quant_error -- quantization-error statistics of a tensor, the measure
 * behind the choice of the migration strength alpha ([CH11] 11.4.3 table
 * 11-4: activation and weight INT8 error per alpha).  For every element,
 * x' = x (smoothed by `smooth` as p->smooth_mode says, the binary32 value the
 * quantizer sees) and x^ = fl(s * (q - z)) of its scope; writes
 *   out[0] = sum (x' - x^)^2,  out[1] = sum x'^2,  out[2] = max |x' - x^|
 * in binary64 to the device array out.  q, s, z are in the layouts
 * qlin_quantize writes for p.  The sums are taken in a fixed order, so the
 * result is reproducible.
 *   ws  device workspace of qlin_workspace_size(QLIN_OP_QUANT_ERROR, ...)
 *       bytes.
 */
int qlin_quant_error(const void *x, qlin_dtype xt, int64_t rows, int64_t cols, int64_t ld, const float *smooth,
                     const qlin_qparams *p, const void *q, const void *s, const int32_t *z, double *out, void *ws,
                     size_t ws_bytes, void *stream);

/* Header at the start of a packed INT4 weight blob (layout version 1). */
#define QLIN_W4_MAGIC 0x34574C51u  /* "QLW4" */
#define QLIN_W4_VERSION 1u
typedef struct {
    uint32_t magic, version;
    int64_t N, K;            /* weight is N (output channels) x K (input)     */
    int32_t group, asym;     /* g in {32, 64, 128}; asym: per-group zero point */
    uint64_t codes_off, scales_off, zeros_off, total_bytes;  /* byte offsets  */
} qlin_w4_header;

/* Bytes of the packed blob qlin_pack_w4 writes for these sizes. */
size_t qlin_pack_w4_size(int64_t N, int64_t K, int group, int asym);

/*
 * qlin_pack_w4 -- rearrange group-wise INT4 weights ([CH11] 11.1.6: W [N x K]
 * in row-wise groups of g, 4-bit codes, fp16 per-group scales) into the
 * layout qlin_gemm_w4a16 streams.
 *   q      device canonical codes from qlin_quantize: N x K nibbles, two per
 *          byte (S4 two's complement when z == NULL, else U4).
 *   s_f16  device binary16 scales, N x K/g, row-major.
 *   z      device int32 zero points in [0, 15], N x K/g, or NULL (symmetric).
 *   packed device output of capacity packed_cap >= qlin_pack_w4_size(...).
 *   hdr    host output (may be NULL): a copy of the blob's header, which
 *          qlin_gemm_w4a16 takes to describe the blob.
 * Requirements: K % g == 0, g in {32, 64, 128}, N % 16 == 0, K % 64 == 0.
 */
int qlin_pack_w4(const void *q, const void *s_f16, const int32_t *z, int64_t N, int64_t K,
                 int group, void *packed, size_t packed_cap, qlin_w4_header *hdr, void *stream);

/*
 * qlin_gemm_w8a8 -- W8A8 linear layer ([L19] section 6; [CH11] 11.1.4,
 * 11.4.5 step 6): acc[m,n] = sum_k qx[m,k] * qw[n,k] exactly in int32, then
 * y[m,n] = (float(acc) * sx[m]) * sw[n] in binary32, rounded once to yt.
 *   qx     device int8 [M x K], row-major (per-token codes).
 *   sx     device binary32 [M] per-token scales.
 *   qw     device int8 [N x K], row-major (per-output-channel codes).
 *   sw     device binary32 [N] per-channel scales.
 *   y      device output [M x N] of type yt (F32 or BF16), row-major.
 *   acc_out device int32 [M x N] exact sums, or NULL.
 *   ws     device workspace of qlin_workspace_size(QLIN_OP_GEMM_W8A8, M, N, K)
 *          bytes, 16-byte aligned: an INT32 [M x N] tile that the kernel only
 *          touches when the exact accumulation must be drained (rows whose
 *          sum of |code| over a run of K would reach 2^24 / 128), followed by
 *          the INT32 partial sums of the output tiles whose K range is split
 *          across CTAs (the tiles of a last, partial wave over the device's
 *          SMs).  No initialisation is needed.  The size depends on the SM
 *          count of the current device.
 * Requirements: K % 16 == 0; qx, qw 16-byte aligned.  The exact sums must fit
 * int32 (always true for codes in [-127,127] when K < 133,144).
 */
int qlin_gemm_w8a8(const int8_t *qx, const float *sx, const int8_t *qw, const float *sw,
                   int64_t M, int64_t N, int64_t K, void *y, qlin_dtype yt,
                   int32_t *acc_out, void *ws, size_t ws_bytes, void *stream);

/*
 * qlin_gemm_w4a16 -- W4A16 linear layer ([CH11] 11.1.6 step 5: dequantize,
 * then a 16-bit matmul): w^[n,k] = bf16(fl(s[n,k/g] * (q[n,k] - z[n,k/g]))),
 * y[m,n] = sum_k x[m,k] * w^[n,k] accumulated in binary32, rounded once to
 * bf16.
 *   x      device bf16 [M x K], row-major, 16-byte aligned.
 *   packed device blob written by qlin_pack_w4; hdr its header (host copy).
 *   y      device bf16 [M x N], row-major, 16-byte aligned.
 *   ws     device workspace of qlin_workspace_size(QLIN_OP_GEMM_W4A16, M, N, K)
 *          bytes, 16-byte aligned (fp32 partial sums of the K split used for
 *          M > 16; none for M <= 16).
 * M <= 16 runs a split-K GEMV; larger M runs the tensor-core GEMM, whose
 * split-K partial sums are added in a fixed order (results are reproducible).
 */
int qlin_gemm_w4a16(const void *x, const void *packed, const qlin_w4_header *hdr, int64_t M,
                    void *y, void *ws, size_t ws_bytes, void *stream);

/*
 * qlin_gemm_w4a8 -- W4A8 linear layer: group-wise INT4 weights (the packed
 * blob of qlin_pack_w4) x per-token INT8 activations ([CH11] 11.4.5 step 6,
 * integer products summed exactly, then the scales; [CH11] 11.9.7 and
 * 11.10.2: AWQ INT4 weights combined with SmoothQuant INT8 activations).
 * Every weight group g has its own scale, so the exact integer sums are kept
 * per group:
 *   acc_g[m,n] = sum_{k in g} qx[m,k] * (q[n,k] - z[n,g])   (exact, int32)
 *   y[m,n]     = sx[m] * sum_g s[n,g] * acc_g[m,n]          (binary32, one
 *                rounding to yt at the end)
 * with z = 0 for symmetric INT4 codes.
 *   qx     device int8 [M x K] per-token codes, row-major, 16-byte aligned.
 *   sx     device binary32 [M] per-token scales.
 *   packed device blob written by qlin_pack_w4; hdr its header (host copy).
 *   y      device [M x N] of type yt (F32 or BF16), row-major.
 *   acc_out NULL, or device int32 [K/g][M][N]: the exact per-group sums
 *          acc_g (a test aid; the call zeroes it first).
 *   ws     device workspace of qlin_workspace_size(QLIN_OP_GEMM_W4A8, M, N, K)
 *          bytes (NULL when 0).
 * Results are reproducible: partial sums are added in a fixed order.
 */
int qlin_gemm_w4a8(const int8_t *qx, const float *sx, const void *packed, const qlin_w4_header *hdr, int64_t M,
                   void *y, qlin_dtype yt, int32_t *acc_out, void *ws, size_t ws_bytes, void *stream);

/*
 * qlin_gemm_llmint8 -- LLM.int8() mixed-precision decomposition of the W8A8
 * layer ([L19] sections 9-11): XW = X_normal W_normal + X_outlier W_outlier.
 * The outlier dimensions are the input channels j with max_m |x[m][j]| >
 * threshold.  They are taken out of the INT8 product: the per-token INT8
 * codes of x are computed with those channels set to 0 (vector-wise scale
 * sx[m] = max over the normal channels / 127), and the outlier channels are
 * multiplied in 16-bit with the weight's own columns dequantized:
 *   y[m,n] = sw[n] * (sx[m] * acc[m,n] + sum_{j outlier} x[m,j] * qw[n,j])
 * acc being the exact INT32 sums over the normal channels; one rounding to yt.
 *   x       device bf16 [M x K], row stride ld (16-byte aligned rows); the
 *           outlier channels are multiplied in bf16 with fp32 accumulation.
 *   qw, sw  the weight in INT8 per output channel: device int8 [N x K]
 *           (16-byte aligned) and binary32 [N] scales (qlin_quantize,
 *           QLIN_PER_ROW, symmetric [-127, 127]).
 *   threshold  finite, >= 0 (LLM.int8() uses 6.0 on activations).
 *   max_outliers  the most outlier channels the workspace is sized for (0..K).
 *           More outlier channels than that make qlin_device_error report
 *           QLIN_ERR_WORKSPACE; y is then unspecified.
 *   y       device [M x N] of type yt (F32 or BF16).
 *   outliers NULL, or device int32 [1 + K]: the number of outlier channels,
 *           then their indices in ascending order.
 *   ws      device workspace of qlin_llmint8_workspace_size(M, N, K,
 *           max_outliers) bytes, 256-byte aligned.
 * Requirements: K % 16 == 0, K < 133,144.
 */
size_t qlin_llmint8_workspace_size(int64_t M, int64_t N, int64_t K, int64_t max_outliers);
int qlin_gemm_llmint8(const void *x, qlin_dtype xt, int64_t M, int64_t K, int64_t ld, const int8_t *qw,
                      const float *sw, int64_t N, float threshold, int64_t max_outliers, void *y, qlin_dtype yt,
                      int32_t *outliers, void *ws, size_t ws_bytes, void *stream);

/*
 * KV-cache quantization in token groups outside a recent window ([CH11]
 * 11.6.3 granularity, 11.6.4 K/V sensitivity, 11.6.5 KIVI's grouped
 * on-demand quantization).  K is quantized per channel -- one scale and zero
 * point per channel over each group of `group` tokens -- and V per token --
 * one per token and head over head_dim channels; codes are asymmetric,
 * [0, 2^bits - 1], with qlin_quantize's arithmetic (range widened to
 * contain 0, round-half-even of the correctly rounded binary32 quotient, zero
 * point added after rounding; binary32 scales, int32 zero points).  The
 * `residual` most recent tokens stay in bf16; a group is quantized once all
 * of its tokens have left that window, so after every append
 *   quantized = group * floor(max(length - residual, 0) / group).
 * The caller owns one device block of qlin_kv_cache_bytes(...) bytes, which
 * qlin_kv_cache_init carves into the buffers below; the struct lives in host
 * memory and qlin_kv_append keeps its counters.
 */
typedef struct {
    int64_t capacity;        /* tokens the cache can hold (a multiple of group)       */
    int32_t channels;        /* C = heads * head_dim values per token (C % 16 == 0)   */
    int32_t head_dim;        /* D: V's scope; D % 8 == 0, C % D == 0                  */
    int32_t group;           /* G tokens per K scope and per quantization step        */
    int32_t residual;        /* R most recent tokens kept in bf16                     */
    int32_t bits;            /* 8 or 4                                                */
    int32_t reserved;
    int64_t length;          /* tokens appended so far                                */
    int64_t quantized;       /* tokens in the quantized store                         */
    void *k_codes, *v_codes; /* device [capacity x C] codes (4-bit: two per byte,    */
                             /* element 2i in the low nibble)                         */
    float *k_scale;          /* device [capacity / G x C]                             */
    int32_t *k_zero;         /* device [capacity / G x C]                             */
    float *v_scale;          /* device [capacity x C / D]                             */
    int32_t *v_zero;         /* device [capacity x C / D]                             */
    void *k_recent, *v_recent; /* device bf16 rings of (R + G) x C: token t of      */
                             /* [quantized, length) in slot t mod (R + G)             */
} qlin_kv_cache;

/* Device bytes one cache of these parameters needs (0 for invalid ones). */
size_t qlin_kv_cache_bytes(int64_t capacity, int channels, int head_dim, int group, int residual, int bits);

/* Host only: fill *c for an empty cache whose buffers live in the device
 * block mem (256-byte aligned, mem_bytes >= qlin_kv_cache_bytes(...)).  The
 * block needs no initialisation. */
int qlin_kv_cache_init(qlin_kv_cache *c, void *mem, size_t mem_bytes, int64_t capacity, int channels, int head_dim,
                       int group, int residual, int bits);

/* Append n tokens: k_new, v_new device bf16 [n x C] (16-byte aligned).  Groups
 * that leave the recent window are quantized (from the ring or straight from
 * k_new / v_new), the new tokens that stay in 16-bit go to the ring, and
 * c->length / c->quantized are updated (host side).  length + n must not
 * exceed capacity.  The launches are ordered on `stream`; calls on one cache
 * must be issued in order on one stream. */
int qlin_kv_append(qlin_kv_cache *c, const void *k_new, const void *v_new, int64_t n, void *stream);

/* The cache as attention reads it: k_out, v_out device bf16 [length x C]
 * (16-byte aligned) receive bf16(fl(s * (q - z))) for tokens below
 * c->quantized and the stored bf16 values for the others. */
int qlin_kv_read(const qlin_kv_cache *c, void *k_out, void *v_out, void *stream);

/*
 * qlin_quantize_noalloc -- qlin_quantize for callers that cannot allocate
 * device memory.  The pages have no counterpart: this is a deployment
 * convenience, not part of the method.
 *
 * Some callers cannot call cudaMalloc or any allocating routine (a plug-in
 * whose host owns all device memory, code running under an allocator's lock,
 * a loop with a fixed memory plan), so they cannot provide the workspace that
 * the per-tensor, per-column and percentile scopes of qlin_quantize need.
 * This entry point takes qlin_quantize's arguments without ws / ws_bytes and
 * uses a fixed scratch array of QLIN_NOALLOC_SCRATCH_BYTES in the library's
 * own device memory instead, held on every GPU that loads the library until
 * the process exits.  It allocates nothing.
 *   - Limit: an operation whose workspace (qlin_workspace_size with
 *     QLIN_OP_QUANTIZE) exceeds QLIN_NOALLOC_SCRATCH_BYTES returns
 *     QLIN_ERR_WORKSPACE and launches nothing (e.g. per-column statistics of
 *     more than 65,536 columns).  Per-row and per-group scopes and static
 *     scales need no scratch at any size.  Argument errors are reported
 *     before the limit is checked, exactly as qlin_quantize reports them.
 *   - A call that needs the scratch looks up the array's device address with
 *     cudaGetSymbolAddress (with the call's device current).  Outside stream
 *     capture it does so on every call; during a capture it uses the address
 *     an earlier call on that device found, so make one call on each device
 *     before capturing (a first call during a capture returns QLIN_ERR_CUDA).
 *   - Every call on a device shares the one array, and the array keeps the
 *     last call's contents; each call clears what it needs zeroed on its own
 *     stream.  Calls whose work overlaps on the GPU (other streams, other host
 *     threads) race on the array and must be serialized by the caller.
 * All other arguments, results and errors are those of qlin_quantize.
 */
#define QLIN_NOALLOC_SCRATCH_BYTES (512u * 1024u)
int qlin_quantize_noalloc(const void *x, qlin_dtype xt, int64_t rows, int64_t cols, int64_t ld,
                          const float *smooth, const qlin_qparams *p,
                          void *q, void *s, int32_t *z, void *stream);

/*
 * qlin_device_error -- synchronizes `stream`, then returns and clears the
 * library's device-side error word: QLIN_OK, or QLIN_ERR_TIMEOUT when a
 * bounded wait inside a kernel gave up (that kernel's outputs are then
 * unspecified).  Returns QLIN_ERR_CUDA if the synchronization itself fails.
 */
int qlin_device_error(void *stream);

/*
 * qlin_debug_stall_producers -- failure-detection test hook (not part of the
 * method).  With enable = 1, the producer roles of the pipelined kernels
 * (the TMA / bulk-copy issuers of the W8A8 and W4A16 tensor-core GEMMs and of
 * the streamed per-token quantizer) issue no copies, and every bounded
 * device-side wait gives up after wait_limit_cycles (> 0) SM clock cycles.
 * The waiting roles then time out, record QLIN_ERR_TIMEOUT in the device error
 * word (qlin_device_error), wait (bounded) for the MMAs they issued, free
 * their TMEM and return; their outputs are unspecified.  enable = 0 restores
 * normal operation and the default limit (4e9 cycles, about 2 s).  Applies to
 * the current device; synchronizes it before and after.  Returns QLIN_OK,
 * QLIN_ERR_ARG (enable with a non-positive limit) or QLIN_ERR_CUDA.
 */
int qlin_debug_stall_producers(int enable, long long wait_limit_cycles);

#ifdef __cplusplus
}
#endif

#endif /* QLIN_H */
