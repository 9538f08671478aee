// qlin_internal.h -- host-side launchers shared between the entry points
// (api.cu) and the kernel files.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/qlin.h"

namespace qlin {

int num_sms();
int64_t percentile_rank(int64_t n, double p);
// Raise a kernel's dynamic shared-memory limit on the current device to at
// least `bytes`, calling the runtime only the first time a (kernel, device)
// pair needs a larger limit (the call costs host time on every launch).
cudaError_t ensure_smem(const void* kernel, int bytes);

size_t quantize_ws_bytes(int64_t rows, int64_t cols, const qlin_qparams* p);
// Argument checks of qlin_quantize (all but the workspace); returns QLIN_OK,
// QLIN_NOTHING_TO_DO for a valid empty input, or a negative qlin_status.
constexpr int QLIN_NOTHING_TO_DO = 1;
int quantize_check(const void* x, int xt, int64_t rows, int64_t cols, int64_t ld, const float* smooth,
                   const qlin_qparams* p, const void* q, const void* s, const int32_t* z);
cudaError_t run_quantize(const void* x, int xt, int64_t rows, int64_t cols, int64_t ld, const float* smooth,
                         const qlin_qparams* p, void* q, void* s, int32_t* z, void* ws, cudaStream_t st);
cudaError_t run_absmax(const void* x, int xt, int64_t rows, int64_t cols, int64_t ld, int gran, int group,
                       float* out, void* ws, cudaStream_t st);
cudaError_t run_dequantize(const void* q, const void* s, const int32_t* z, const qlin_qparams* p, int64_t rows,
                           int64_t cols, void* y, int yt, cudaStream_t st);
cudaError_t run_smooth_factors(const float* xmax, const float* wmax, int64_t K, float alpha, float* s,
                               cudaStream_t st);

// W8A8 (gemm_w8a8.cu)
size_t w8a8_ws_bytes(int64_t M, int64_t N, int64_t K);
cudaError_t run_gemm_w8a8(const int8_t* qx, const float* sx, const int8_t* qw, const float* sw, int64_t M,
                          int64_t N, int64_t K, void* y, int yt, int32_t* acc_out, void* ws, cudaStream_t st,
                          const float* add = nullptr);

// W4A16 (gemm_w4a16.cu)
void w4_layout(int64_t N, int64_t K, int group, int asym, qlin_w4_header* h);
cudaError_t run_pack_w4(const void* q, const void* s_f16, const int32_t* z, const qlin_w4_header* h, void* packed,
                        cudaStream_t st);
size_t w4a16_ws_bytes(int64_t M, int64_t N, int64_t K);
cudaError_t run_gemm_w4a16(const void* x, const void* packed, const qlin_w4_header* h, int64_t M, void* y,
                           void* ws, cudaStream_t st);

// W4A8 (gemm_w4a8.cu)
size_t w4a8_ws_bytes(int64_t M, int64_t N, int64_t K);
cudaError_t run_gemm_w4a8(const int8_t* qx, const float* sx, const void* packed, const qlin_w4_header* h, int64_t M,
                          void* y, int yt, int32_t* acc_out, void* ws, cudaStream_t st);

// SmoothQuant calibration (calib.cu)
cudaError_t run_absmax_update(const void* x, int xt, int64_t rows, int64_t cols, int64_t ld, float* running,
                              cudaStream_t st);
cudaError_t run_fold_layernorm(const float* gamma, const float* beta, const float* s, int64_t K, float* gamma_out,
                               float* beta_out, cudaStream_t st);
size_t quant_error_ws_bytes();
cudaError_t run_quant_error(const void* x, int xt, int64_t rows, int64_t cols, int64_t ld, const float* smooth,
                            const qlin_qparams* p, const void* q, const void* s, const int32_t* z, double* out,
                            void* ws, cudaStream_t st);

// LLM.int8() decomposition (llmint8.cu)
size_t llmint8_ws_bytes(int64_t M, int64_t N, int64_t K, int64_t max_outliers);
cudaError_t run_gemm_llmint8(const void* x, int xt, int64_t M, int64_t K, int64_t ld, const int8_t* qw,
                             const float* sw, int64_t N, float threshold, int64_t max_outliers, void* y, int yt,
                             int32_t* report, void* ws, cudaStream_t st);

// KV-cache quantization (kvcache.cu)
void kv_layout(int64_t capacity, int C, int D, int G, int R, int bits, size_t off[8], size_t* total);
cudaError_t run_kv_append(const qlin_kv_cache* c, const void* k_new, const void* v_new, int64_t n, int64_t q_new,
                          cudaStream_t st);
cudaError_t run_kv_read(const qlin_kv_cache* c, void* k_out, void* v_out, cudaStream_t st);

}  // namespace qlin
