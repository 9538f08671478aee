// api.cu -- the extern "C" entry points of libqlin.so: argument validation on
// the host, then a launch on the caller's stream.  Nothing here allocates.
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "qlin_common.cuh"
#include "qlin_internal.h"

using namespace qlin;

namespace {

inline bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// QLIN_ERR_CUDA for a failed runtime call; with QLIN_DEBUG set in the
// environment the CUDA error text is also printed to stderr.
inline int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return QLIN_OK;
    if (getenv("QLIN_DEBUG")) fprintf(stderr, "qlin: CUDA error %d: %s\n", (int)e, cudaGetErrorString(e));
    return QLIN_ERR_CUDA;
}

inline bool is_float_type(int t) { return t == QLIN_F32 || t == QLIN_BF16 || t == QLIN_F16; }

inline int type_bytes(int t) { return t == QLIN_F32 ? 4 : 2; }

// The code storage must hold [qmin, qmax].
bool code_range_ok(const qlin_qparams* p) {
    if (p->qmax <= p->qmin) return false;
    switch (p->code) {
    case QLIN_S8: return p->qmin >= -128 && p->qmax <= 127;
    case QLIN_U8: return p->qmin >= 0 && p->qmax <= 255;
    case QLIN_S4: return p->qmin >= -8 && p->qmax <= 7;
    case QLIN_U4: return p->qmin >= 0 && p->qmax <= 15;
    default: return false;
    }
}

int64_t scopes(const qlin_qparams* p, int64_t rows, int64_t cols) {
    switch (p->gran) {
    case QLIN_PER_TENSOR: return 1;
    case QLIN_PER_ROW: return rows;
    case QLIN_PER_COL: return cols;
    case QLIN_PER_GROUP: return rows * (cols / p->group);
    default: return -1;
    }
}

int check_qparams(const qlin_qparams* p, int64_t rows, int64_t cols) {
    if (!p) return QLIN_ERR_ARG;
    if (!code_range_ok(p)) return QLIN_ERR_ARG;
    if (p->symmetric && p->qmin != -p->qmax) return QLIN_ERR_ARG;
    if (p->gran < QLIN_PER_TENSOR || p->gran > QLIN_PER_GROUP) return QLIN_ERR_ARG;
    if (p->gran == QLIN_PER_GROUP && (p->group <= 0 || cols % p->group != 0)) return QLIN_ERR_ARG;
    if (p->scale_dtype != QLIN_F32 && p->scale_dtype != QLIN_F16) return QLIN_ERR_ARG;
    if (p->smooth_mode < QLIN_SMOOTH_NONE || p->smooth_mode > QLIN_SMOOTH_MULTIPLY) return QLIN_ERR_ARG;
    if (!(p->clip_percentile >= 0.0) || p->clip_percentile > 100.0) return QLIN_ERR_ARG;
    if ((p->code == QLIN_S4 || p->code == QLIN_U4) && (cols % 2 != 0)) return QLIN_ERR_ARG;
    if (rows < 0 || cols < 0) return QLIN_ERR_ARG;
    return QLIN_OK;
}

// A packed W4 header must describe a layout-1 blob this library writes.
int check_w4_header(const qlin_w4_header* hdr) {
    if (hdr->magic != QLIN_W4_MAGIC || hdr->version != QLIN_W4_VERSION) return QLIN_ERR_LAYOUT;
    if (hdr->N <= 0 || hdr->K <= 0 || (hdr->group != 32 && hdr->group != 64 && hdr->group != 128))
        return QLIN_ERR_LAYOUT;
    if (hdr->K % 64 != 0 || hdr->N % 16 != 0) return QLIN_ERR_LAYOUT;
    qlin_w4_header ref;
    w4_layout(hdr->N, hdr->K, hdr->group, hdr->asym ? 1 : 0, &ref);
    if (ref.codes_off != hdr->codes_off || ref.scales_off != hdr->scales_off || ref.zeros_off != hdr->zeros_off ||
        ref.total_bytes != hdr->total_bytes)
        return QLIN_ERR_LAYOUT;
    return QLIN_OK;
}

}  // namespace

namespace qlin {

// Every argument check of qlin_quantize except the workspace: QLIN_OK,
// QLIN_NOTHING_TO_DO (valid, empty input) or a negative qlin_status.
int quantize_check(const void* x, int xt, int64_t rows, int64_t cols, int64_t ld, const float* smooth,
                   const qlin_qparams* p, const void* q, const void* s, const int32_t* z) {
    int rc = check_qparams(p, rows, cols);
    if (rc != QLIN_OK) return rc;
    if (!is_float_type(xt) || ld < cols) return QLIN_ERR_ARG;
    if (rows == 0 || cols == 0) return QLIN_NOTHING_TO_DO;
    if (!x || !q || !s) return QLIN_ERR_ARG;
    if (!p->symmetric && !z) return QLIN_ERR_ARG;
    if (p->smooth_mode != QLIN_SMOOTH_NONE && !smooth) return QLIN_ERR_ARG;
    if (!aligned(x, type_bytes(xt)) || !aligned(s, p->scale_dtype == QLIN_F16 ? 2 : 4) || (z && !aligned(z, 4)))
        return QLIN_ERR_ARG;
    if (p->clip_percentile > 0.0 && (!p->symmetric || p->gran != QLIN_PER_TENSOR)) return QLIN_ERR_UNSUPPORTED;
    if (p->static_scale && p->clip_percentile > 0.0) return QLIN_ERR_ARG;
    return QLIN_OK;
}

}  // namespace qlin

extern "C" {

int qlin_version(void) { return 10000; }

const char* qlin_status_string(int status) {
    switch (status) {
    case QLIN_OK: return "ok";
    case QLIN_ERR_ARG: return "invalid argument";
    case QLIN_ERR_UNSUPPORTED: return "unsupported combination";
    case QLIN_ERR_CUDA: return "CUDA error";
    case QLIN_ERR_TIMEOUT: return "device-side wait timed out";
    case QLIN_ERR_WORKSPACE: return "workspace missing or too small";
    case QLIN_ERR_LAYOUT: return "packed weight layout mismatch";
    default: return "unknown status";
    }
}

size_t qlin_workspace_size(int op, int64_t M, int64_t N, int64_t K, const qlin_qparams* p) {
    switch (op) {
    case QLIN_OP_QUANTIZE:
        if (!p || M < 0 || N < 0) return 0;
        return quantize_ws_bytes(M, N, p);
    case QLIN_OP_ABSMAX: {
        if (!p) return 0;
        qlin_qparams q = *p;
        q.static_scale = 0;
        q.clip_percentile = 0.0;
        return quantize_ws_bytes(M, N, &q);
    }
    case QLIN_OP_GEMM_W8A8: return w8a8_ws_bytes(M, N, K);
    case QLIN_OP_GEMM_W4A16: return w4a16_ws_bytes(M, N, K);
    case QLIN_OP_GEMM_W4A8: return w4a8_ws_bytes(M, N, K);
    case QLIN_OP_QUANT_ERROR: return quant_error_ws_bytes();
    default: return 0;
    }
}

int qlin_quantize(const void* x, qlin_dtype xt, int64_t rows, int64_t cols, int64_t ld, const float* smooth,
                  const qlin_qparams* p, void* q, void* s, int32_t* z, void* ws, size_t ws_bytes, void* stream) {
    int rc = quantize_check(x, xt, rows, cols, ld, smooth, p, q, s, z);
    if (rc == QLIN_NOTHING_TO_DO) return QLIN_OK;
    if (rc != QLIN_OK) return rc;
    size_t need = quantize_ws_bytes(rows, cols, p);
    if (need > 0 && (!ws || ws_bytes < need || !aligned(ws, 16))) return QLIN_ERR_WORKSPACE;
    return cuda_status(run_quantize(x, xt, rows, cols, ld, smooth, p, q, s, z, ws, (cudaStream_t)stream));
}

int qlin_dequantize(const void* q, const void* s, const int32_t* z, const qlin_qparams* p, int64_t rows, int64_t cols,
                    void* y, qlin_dtype yt, void* stream) {
    int rc = check_qparams(p, rows, cols);
    if (rc != QLIN_OK) return rc;
    if (!is_float_type(yt)) return QLIN_ERR_ARG;
    if (rows == 0 || cols == 0) return QLIN_OK;
    if (!q || !s || !y) return QLIN_ERR_ARG;
    if (!aligned(y, type_bytes(yt)) || !aligned(s, p->scale_dtype == QLIN_F16 ? 2 : 4) || (z && !aligned(z, 4)))
        return QLIN_ERR_ARG;
    return cuda_status(run_dequantize(q, s, p->symmetric ? nullptr : z, p, rows, cols, y, yt, (cudaStream_t)stream));
}

int qlin_absmax(const void* x, qlin_dtype xt, int64_t rows, int64_t cols, int64_t ld, qlin_gran gran, int group,
                float* out, void* ws, size_t ws_bytes, void* stream) {
    if (!is_float_type(xt) || rows < 0 || cols < 0 || ld < cols) return QLIN_ERR_ARG;
    if (gran < QLIN_PER_TENSOR || gran > QLIN_PER_GROUP) return QLIN_ERR_ARG;
    if (gran == QLIN_PER_GROUP && (group <= 0 || cols % group != 0)) return QLIN_ERR_ARG;
    if (rows == 0 || cols == 0) return QLIN_OK;
    if (!x || !out || !aligned(x, type_bytes(xt)) || !aligned(out, 4)) return QLIN_ERR_ARG;
    qlin_qparams p{};
    p.code = QLIN_S8;
    p.qmin = -127;
    p.qmax = 127;
    p.symmetric = 1;
    p.gran = gran;
    p.group = group;
    p.scale_dtype = QLIN_F32;
    size_t need = quantize_ws_bytes(rows, cols, &p);
    if (need > 0 && (!ws || ws_bytes < need || !aligned(ws, 16))) return QLIN_ERR_WORKSPACE;
    return cuda_status(run_absmax(x, xt, rows, cols, ld, gran, group, out, ws, (cudaStream_t)stream));
}

int qlin_smooth_factors(const float* xmax, const float* wmax, int64_t K, float alpha, float* s, void* stream) {
    if (K < 0 || !(alpha >= 0.0f && alpha <= 1.0f)) return QLIN_ERR_ARG;
    if (K == 0) return QLIN_OK;
    if (!xmax || !wmax || !s) return QLIN_ERR_ARG;
    return cuda_status(run_smooth_factors(xmax, wmax, K, alpha, s, (cudaStream_t)stream));
}

size_t qlin_pack_w4_size(int64_t N, int64_t K, int group, int asym) {
    if (N <= 0 || K <= 0 || group <= 0 || K % group != 0) return 0;
    qlin_w4_header h;
    w4_layout(N, K, group, asym ? 1 : 0, &h);
    return (size_t)h.total_bytes;
}

int qlin_pack_w4(const void* q, const void* s_f16, const int32_t* z, int64_t N, int64_t K, int group, void* packed,
                 size_t packed_cap, qlin_w4_header* hdr, void* stream) {
    if (N <= 0 || K <= 0) return QLIN_ERR_ARG;
    if (group != 32 && group != 64 && group != 128) return QLIN_ERR_UNSUPPORTED;
    if (K % group != 0 || K % 64 != 0 || N % 16 != 0) return QLIN_ERR_UNSUPPORTED;
    if (!q || !s_f16 || !packed) return QLIN_ERR_ARG;
    if (!aligned(packed, 256) || !aligned(s_f16, 2) || (z && !aligned(z, 4))) return QLIN_ERR_ARG;
    qlin_w4_header h;
    w4_layout(N, K, group, z ? 1 : 0, &h);
    if (packed_cap < h.total_bytes) return QLIN_ERR_WORKSPACE;
    if (hdr) *hdr = h;
    return cuda_status(run_pack_w4(q, s_f16, z, &h, packed, (cudaStream_t)stream));
}

int qlin_gemm_w8a8(const int8_t* qx, const float* sx, const int8_t* qw, const float* sw, int64_t M, int64_t N,
                   int64_t K, void* y, qlin_dtype yt, int32_t* acc_out, void* ws, size_t ws_bytes, void* stream) {
    if (M < 0 || N < 0 || K < 0) return QLIN_ERR_ARG;
    if (yt != QLIN_F32 && yt != QLIN_BF16) return QLIN_ERR_ARG;
    if (K % 16 != 0 || K >= 133144) return QLIN_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return QLIN_OK;
    if (!qx || !sx || !qw || !sw || !y) return QLIN_ERR_ARG;
    if (!aligned(qx, 16) || !aligned(qw, 16) || !aligned(sx, 4) || !aligned(sw, 4) || !aligned(y, type_bytes(yt)) ||
        (acc_out && !aligned(acc_out, 4)))
        return QLIN_ERR_ARG;
    size_t need = w8a8_ws_bytes(M, N, K);
    if (need > 0 && (!ws || ws_bytes < need || !aligned(ws, 16))) return QLIN_ERR_WORKSPACE;
    if (K == 0) return QLIN_ERR_UNSUPPORTED;
    return cuda_status(run_gemm_w8a8(qx, sx, qw, sw, M, N, K, y, yt, acc_out, ws, (cudaStream_t)stream));
}

int qlin_gemm_w4a16(const void* x, const void* packed, const qlin_w4_header* hdr, int64_t M, void* y, void* ws,
                    size_t ws_bytes, void* stream) {
    if (!hdr || M < 0) return QLIN_ERR_ARG;
    int rc = check_w4_header(hdr);
    if (rc != QLIN_OK) return rc;
    if (M == 0) return QLIN_OK;
    if (!x || !packed || !y) return QLIN_ERR_ARG;
    if (!aligned(x, 16) || !aligned(packed, 256) || !aligned(y, 16)) return QLIN_ERR_ARG;
    size_t need = w4a16_ws_bytes(M, hdr->N, hdr->K);
    if (need > 0 && (!ws || ws_bytes < need || !aligned(ws, 16))) return QLIN_ERR_WORKSPACE;
    return cuda_status(run_gemm_w4a16(x, packed, hdr, M, y, ws, (cudaStream_t)stream));
}

int qlin_debug_stall_producers(int enable, long long wait_limit_cycles) {
    if (enable && wait_limit_cycles <= 0) return QLIN_ERR_ARG;
    const int stall = enable ? 1 : 0;
    const long long limit = enable ? wait_limit_cycles : kDefaultWaitLimitCycles;
    if (cudaDeviceSynchronize() != cudaSuccess) return QLIN_ERR_CUDA;
    if (cudaMemcpyToSymbol(g_wait_limit_cycles, &limit, sizeof limit) != cudaSuccess) return QLIN_ERR_CUDA;
    if (cudaMemcpyToSymbol(g_stall_producers, &stall, sizeof stall) != cudaSuccess) return QLIN_ERR_CUDA;
    return cudaDeviceSynchronize() == cudaSuccess ? QLIN_OK : QLIN_ERR_CUDA;
}

int qlin_gemm_w4a8(const int8_t* qx, const float* sx, const void* packed, const qlin_w4_header* hdr, int64_t M,
                   void* y, qlin_dtype yt, int32_t* acc_out, void* ws, size_t ws_bytes, void* stream) {
    if (!hdr || M < 0) return QLIN_ERR_ARG;
    if (yt != QLIN_F32 && yt != QLIN_BF16) return QLIN_ERR_ARG;
    int rc = check_w4_header(hdr);
    if (rc != QLIN_OK) return rc;
    if (M == 0) return QLIN_OK;
    if (!qx || !sx || !packed || !y) return QLIN_ERR_ARG;
    if (!aligned(qx, 16) || !aligned(sx, 4) || !aligned(packed, 256) || !aligned(y, type_bytes(yt)) ||
        (acc_out && !aligned(acc_out, 4)))
        return QLIN_ERR_ARG;
    size_t need = w4a8_ws_bytes(M, hdr->N, hdr->K);
    if (need > 0 && (!ws || ws_bytes < need || !aligned(ws, 16))) return QLIN_ERR_WORKSPACE;
    return cuda_status(run_gemm_w4a8(qx, sx, packed, hdr, M, y, yt, acc_out, ws, (cudaStream_t)stream));
}

int qlin_absmax_update(const void* x, qlin_dtype xt, int64_t rows, int64_t cols, int64_t ld, float* running,
                       void* stream) {
    if (!is_float_type(xt) || rows < 0 || cols < 0 || ld < cols) return QLIN_ERR_ARG;
    if (rows == 0 || cols == 0) return QLIN_OK;
    if (!x || !running || !aligned(x, type_bytes(xt)) || !aligned(running, 4)) return QLIN_ERR_ARG;
    return cuda_status(run_absmax_update(x, xt, rows, cols, ld, running, (cudaStream_t)stream));
}

int qlin_fold_layernorm(const float* gamma, const float* beta, const float* s, int64_t K, float* gamma_out,
                        float* beta_out, void* stream) {
    if (K < 0 || (beta && !beta_out) || (!beta && beta_out)) return QLIN_ERR_ARG;
    if (K == 0) return QLIN_OK;
    if (!gamma || !s || !gamma_out) return QLIN_ERR_ARG;
    return cuda_status(run_fold_layernorm(gamma, beta, s, K, gamma_out, beta_out, (cudaStream_t)stream));
}

int qlin_quant_error(const void* x, qlin_dtype xt, int64_t rows, int64_t cols, int64_t ld, const float* smooth,
                     const qlin_qparams* p, const void* q, const void* s, const int32_t* z, double* out, void* ws,
                     size_t ws_bytes, void* stream) {
    int rc = check_qparams(p, rows, cols);
    if (rc != QLIN_OK) return rc;
    if (!is_float_type(xt) || ld < cols || !out) return QLIN_ERR_ARG;
    if (!x && rows * cols > 0) return QLIN_ERR_ARG;
    if (!q || !s || (!p->symmetric && !z)) return QLIN_ERR_ARG;
    if (p->smooth_mode != QLIN_SMOOTH_NONE && !smooth) return QLIN_ERR_ARG;
    if (!aligned(out, 8)) return QLIN_ERR_ARG;
    if (!ws || ws_bytes < quant_error_ws_bytes() || !aligned(ws, 16)) return QLIN_ERR_WORKSPACE;
    return cuda_status(run_quant_error(x, xt, rows, cols, ld, smooth, p, q, s, z, out, ws, (cudaStream_t)stream));
}

size_t qlin_llmint8_workspace_size(int64_t M, int64_t N, int64_t K, int64_t max_outliers) {
    if (M < 0 || N < 0 || K < 0 || max_outliers < 0 || max_outliers > K) return 0;
    return llmint8_ws_bytes(M, N, K, max_outliers);
}

int qlin_gemm_llmint8(const void* x, qlin_dtype xt, int64_t M, int64_t K, int64_t ld, const int8_t* qw,
                      const float* sw, int64_t N, float threshold, int64_t max_outliers, void* y, qlin_dtype yt,
                      int32_t* outliers, void* ws, size_t ws_bytes, void* stream) {
    if (M < 0 || N < 0 || K < 0 || ld < K || max_outliers < 0 || max_outliers > K) return QLIN_ERR_ARG;
    if (xt != QLIN_BF16) return QLIN_ERR_ARG;
    if (yt != QLIN_F32 && yt != QLIN_BF16) return QLIN_ERR_ARG;
    if (!(threshold >= 0.0f) || isinf(threshold)) return QLIN_ERR_ARG;
    if (K % 16 != 0 || K >= 133144 || K == 0) return QLIN_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return QLIN_OK;
    if (!x || !qw || !sw || !y) return QLIN_ERR_ARG;
    if (!aligned(x, 16) || (ld * 2) % 16 != 0 || !aligned(qw, 16) || !aligned(sw, 4) ||
        !aligned(y, type_bytes(yt)) || (outliers && !aligned(outliers, 4)))
        return QLIN_ERR_ARG;
    const size_t need = llmint8_ws_bytes(M, N, K, max_outliers);
    if (!ws || ws_bytes < need || !aligned(ws, 256)) return QLIN_ERR_WORKSPACE;
    return cuda_status(run_gemm_llmint8(x, xt, M, K, ld, qw, sw, N, threshold, max_outliers, y, yt, outliers, ws,
                                        (cudaStream_t)stream));
}

static bool kv_params_ok(int64_t capacity, int C, int D, int G, int R, int bits) {
    if (capacity < 0 || C <= 0 || D <= 0 || G <= 0 || R < 0) return false;
    if (C % 16 != 0 || D % 8 != 0 || C % D != 0 || capacity % G != 0) return false;
    return bits == 4 || bits == 8;
}

size_t qlin_kv_cache_bytes(int64_t capacity, int channels, int head_dim, int group, int residual, int bits) {
    if (!kv_params_ok(capacity, channels, head_dim, group, residual, bits)) return 0;
    size_t off[8], total = 0;
    kv_layout(capacity, channels, head_dim, group, residual, bits, off, &total);
    return total;
}

int qlin_kv_cache_init(qlin_kv_cache* c, void* mem, size_t mem_bytes, int64_t capacity, int channels, int head_dim,
                       int group, int residual, int bits) {
    if (!c || !kv_params_ok(capacity, channels, head_dim, group, residual, bits)) return QLIN_ERR_ARG;
    size_t off[8], total = 0;
    kv_layout(capacity, channels, head_dim, group, residual, bits, off, &total);
    if (!mem || !aligned(mem, 256)) return QLIN_ERR_ARG;
    if (mem_bytes < total) return QLIN_ERR_WORKSPACE;
    uint8_t* b = reinterpret_cast<uint8_t*>(mem);
    c->capacity = capacity;
    c->channels = channels;
    c->head_dim = head_dim;
    c->group = group;
    c->residual = residual;
    c->bits = bits;
    c->reserved = 0;
    c->length = 0;
    c->quantized = 0;
    c->k_codes = b + off[0];
    c->v_codes = b + off[1];
    c->k_scale = reinterpret_cast<float*>(b + off[2]);
    c->k_zero = reinterpret_cast<int32_t*>(b + off[3]);
    c->v_scale = reinterpret_cast<float*>(b + off[4]);
    c->v_zero = reinterpret_cast<int32_t*>(b + off[5]);
    c->k_recent = b + off[6];
    c->v_recent = b + off[7];
    return QLIN_OK;
}

int qlin_kv_append(qlin_kv_cache* c, const void* k_new, const void* v_new, int64_t n, void* stream) {
    if (!c || n < 0) return QLIN_ERR_ARG;
    if (!kv_params_ok(c->capacity, c->channels, c->head_dim, c->group, c->residual, c->bits)) return QLIN_ERR_ARG;
    if (c->length < 0 || c->length + n > c->capacity) return QLIN_ERR_ARG;
    if (n == 0) return QLIN_OK;
    if (!k_new || !v_new || !aligned(k_new, 16) || !aligned(v_new, 16)) return QLIN_ERR_ARG;
    const int64_t T2 = c->length + n;
    const int64_t over = T2 - c->residual;
    const int64_t q_new = over > 0 ? (over / c->group) * c->group : 0;
    int rc = cuda_status(run_kv_append(c, k_new, v_new, n, q_new, (cudaStream_t)stream));
    if (rc != QLIN_OK) return rc;
    c->length = T2;
    c->quantized = q_new;
    return QLIN_OK;
}

int qlin_kv_read(const qlin_kv_cache* c, void* k_out, void* v_out, void* stream) {
    if (!c) return QLIN_ERR_ARG;
    if (!kv_params_ok(c->capacity, c->channels, c->head_dim, c->group, c->residual, c->bits)) return QLIN_ERR_ARG;
    if (c->length == 0) return QLIN_OK;
    if (!k_out || !v_out || !aligned(k_out, 16) || !aligned(v_out, 16)) return QLIN_ERR_ARG;
    return cuda_status(run_kv_read(c, k_out, v_out, (cudaStream_t)stream));
}

int qlin_device_error(void* stream) {
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return QLIN_ERR_CUDA;
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return QLIN_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return QLIN_ERR_CUDA;
    return v == 0 ? QLIN_OK : v;
}

}  // extern "C"
