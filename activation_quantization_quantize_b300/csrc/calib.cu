// calib.cu -- SmoothQuant calibration: running channel maxima over
// calibration batches, folding 1/s into the previous LayerNorm, and the
// quantization-error statistics that compare migration strengths.
//
// Method ("第11章 模型量化与压缩" 11.4.3 table 11-4 and 11.4.4; "量化、蒸馏与
// 模型压缩" 2.3): s_j = max|X_j|^alpha / max|W_j|^(1-alpha) from maxima
// collected over calibration data; X diag(s)^-1 is absorbed by the LayerNorm
// that produces X (gamma' = gamma / s, beta' = beta / s) and W' = diag(s) W is
// quantized offline; alpha trades activation error for weight error.
#include "qlin_common.cuh"
#include "qlin_internal.h"

namespace qlin {

// running[j] = max(running[j], max_i |x[i][j]|).  A thread keeps the maxima of
// 8 columns over a slab of rows, then raises the running values with an
// atomic max on their binary32 bit patterns (non-negative, so the pattern
// order is the value order; the result does not depend on the order).
template <typename T>
__global__ void __launch_bounds__(256) k_colmax_update(const T* __restrict__ x, int64_t rows, int64_t cols, int64_t ld,
                                                       int rows_per_block, uint32_t* __restrict__ running) {
    const int64_t nchunks = cols / 8;
    const int64_t c8 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // chunk column
    if (c8 >= nchunks) return;
    const int64_t r0 = (int64_t)blockIdx.y * rows_per_block;
    int64_t r1 = r0 + rows_per_block;
    if (r1 > rows) r1 = rows;
    float m[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int64_t r = r0; r < r1; ++r) {
        float v[8];
        load8<T>(x + r * ld + c8 * 8, v);
#pragma unroll
        for (int j = 0; j < 8; ++j) m[j] = fmaxf(m[j], fabsf(v[j]));
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
        if (m[j] > 0.0f) atomicMax(running + c8 * 8 + j, __float_as_uint(m[j]));
}

// Scalar form for columns that do not come in aligned chunks of 8.
template <typename T>
__global__ void k_colmax_update_generic(const T* __restrict__ x, int64_t rows, int64_t cols, int64_t ld,
                                        uint32_t* __restrict__ running) {
    for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < cols; c += (int64_t)gridDim.x * blockDim.x) {
        float m = 0.0f;
        for (int64_t r = 0; r < rows; ++r) m = fmaxf(m, fabsf(to_f32<T>(x[r * ld + c])));
        if (m > 0.0f) atomicMax(running + c, __float_as_uint(m));
    }
}

__global__ void k_fold_layernorm(const float* __restrict__ gamma, const float* __restrict__ beta,
                                 const float* __restrict__ s, int64_t K, float* __restrict__ gamma_out,
                                 float* __restrict__ beta_out) {
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < K; j += (int64_t)gridDim.x * blockDim.x) {
        gamma_out[j] = __fdiv_rn(gamma[j], s[j]);
        if (beta) beta_out[j] = __fdiv_rn(beta[j], s[j]);
    }
}

// ------------------------------------------------------------------ quantization error
struct ErrArgs {
    const void* x;
    int64_t rows, cols, ld;
    const float* smooth;
    int smooth_mode;
    const void* q;
    const void* s;
    const int32_t* z;
    int gran, group, scale_f16, code4, code_signed;
};

constexpr int kErrBlocks = 296;  // partial sums: a fixed count, so the reduction order is fixed

template <typename T>
__device__ __forceinline__ float err_load(const ErrArgs& a, int64_t r, int64_t c) {
    float v = to_f32<T>(reinterpret_cast<const T*>(a.x)[r * a.ld + c]);
    if (a.smooth_mode == QLIN_SMOOTH_DIVIDE) return __fdiv_rn(v, a.smooth[c]);
    if (a.smooth_mode == QLIN_SMOOTH_MULTIPLY) return __fmul_rn(v, a.smooth[c]);
    return v;
}

__device__ __forceinline__ int err_code(const ErrArgs& a, int64_t r, int64_t c) {
    if (a.code4) {
        const uint8_t b = reinterpret_cast<const uint8_t*>(a.q)[r * (a.cols / 2) + c / 2];
        int v = (c & 1) ? (b >> 4) : (b & 0xF);
        if (a.code_signed && v >= 8) v -= 16;
        return v;
    }
    if (a.code_signed) return reinterpret_cast<const int8_t*>(a.q)[r * a.cols + c];
    return reinterpret_cast<const uint8_t*>(a.q)[r * a.cols + c];
}

// Block b takes elements [b * n / B, (b + 1) * n / B) of the row-major order;
// each thread sums its elements in binary64, the block reduces in a fixed
// tree, and writes (sum d^2, sum x'^2, max |d|) to part[b].
template <typename T>
__global__ void __launch_bounds__(256) k_quant_error(ErrArgs a, double* __restrict__ part) {
    const int64_t n = a.rows * a.cols;
    const int64_t e0 = n * blockIdx.x / gridDim.x, e1 = n * (blockIdx.x + 1) / gridDim.x;
    double se = 0.0, sx = 0.0, mx = 0.0;
    for (int64_t e = e0 + threadIdx.x; e < e1; e += blockDim.x) {
        const int64_t r = e / a.cols, c = e - r * a.cols;
        int64_t sc;
        switch (a.gran) {
        case QLIN_PER_TENSOR: sc = 0; break;
        case QLIN_PER_ROW: sc = r; break;
        case QLIN_PER_COL: sc = c; break;
        default: sc = r * (a.cols / a.group) + c / a.group;
        }
        const float s = a.scale_f16 ? __half2float(reinterpret_cast<const __half*>(a.s)[sc])
                                    : reinterpret_cast<const float*>(a.s)[sc];
        const int z = a.z ? a.z[sc] : 0;
        const float xh = __fmul_rn(s, (float)(err_code(a, r, c) - z));
        const float v = err_load<T>(a, r, c);
        const double d = (double)v - (double)xh;
        se = fma(d, d, se);
        sx = fma((double)v, (double)v, sx);
        mx = fmax(mx, fabs(d));
    }
    __shared__ double red[3][256];
    red[0][threadIdx.x] = se;
    red[1][threadIdx.x] = sx;
    red[2][threadIdx.x] = mx;
    __syncthreads();
    for (int o = blockDim.x / 2; o > 0; o >>= 1) {
        if ((int)threadIdx.x < o) {
            red[0][threadIdx.x] += red[0][threadIdx.x + o];
            red[1][threadIdx.x] += red[1][threadIdx.x + o];
            red[2][threadIdx.x] = fmax(red[2][threadIdx.x], red[2][threadIdx.x + o]);
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        part[3 * blockIdx.x] = red[0][0];
        part[3 * blockIdx.x + 1] = red[1][0];
        part[3 * blockIdx.x + 2] = red[2][0];
    }
}

__global__ void k_quant_error_final(const double* __restrict__ part, int nparts, double* __restrict__ out) {
    if (threadIdx.x != 0) return;
    double se = 0.0, sx = 0.0, mx = 0.0;
    for (int b = 0; b < nparts; ++b) {
        se += part[3 * b];
        sx += part[3 * b + 1];
        mx = fmax(mx, part[3 * b + 2]);
    }
    out[0] = se;
    out[1] = sx;
    out[2] = mx;
}

// ------------------------------------------------------------------ launchers
cudaError_t run_absmax_update(const void* x, int xt, int64_t rows, int64_t cols, int64_t ld, float* running,
                              cudaStream_t st) {
    uint32_t* run = reinterpret_cast<uint32_t*>(running);
    const int es = xt == QLIN_F32 ? 4 : 2;
    const bool vec = cols % 8 == 0 && ((uintptr_t)x % 16 == 0) && ((ld * es) % 16 == 0);
    if (vec) {
        // a thread keeps 8 columns over a slab of at least 64 rows, so each
        // column takes few atomics; enough slabs to fill the SMs
        const int64_t nchunks = cols / 8;
        const int64_t gx = ceil_div(nchunks, 256);
        int64_t gy = ceil_div((int64_t)num_sms() * 8, gx);
        if (gy > ceil_div(rows, 64)) gy = ceil_div(rows, 64);
        if (gy < 1) gy = 1;
        const int rpb = (int)ceil_div(rows, gy);
        gy = ceil_div(rows, rpb);
        dim3 grid((unsigned)gx, (unsigned)gy);
        switch (xt) {
        case QLIN_BF16:
            k_colmax_update<__nv_bfloat16><<<grid, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(x), rows, cols,
                                                                 ld, rpb, run);
            break;
        case QLIN_F16:
            k_colmax_update<__half><<<grid, 256, 0, st>>>(reinterpret_cast<const __half*>(x), rows, cols, ld, rpb, run);
            break;
        default:
            k_colmax_update<float><<<grid, 256, 0, st>>>(reinterpret_cast<const float*>(x), rows, cols, ld, rpb, run);
        }
    } else {
        const unsigned grid = (unsigned)ceil_div(cols, 256);
        switch (xt) {
        case QLIN_BF16:
            k_colmax_update_generic<__nv_bfloat16><<<grid, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(x),
                                                                         rows, cols, ld, run);
            break;
        case QLIN_F16:
            k_colmax_update_generic<__half><<<grid, 256, 0, st>>>(reinterpret_cast<const __half*>(x), rows, cols, ld,
                                                                  run);
            break;
        default:
            k_colmax_update_generic<float><<<grid, 256, 0, st>>>(reinterpret_cast<const float*>(x), rows, cols, ld, run);
        }
    }
    return cudaGetLastError();
}

cudaError_t run_fold_layernorm(const float* gamma, const float* beta, const float* s, int64_t K, float* gamma_out,
                               float* beta_out, cudaStream_t st) {
    int64_t grid = ceil_div(K, 256);
    if (grid > 4096) grid = 4096;
    k_fold_layernorm<<<(unsigned)grid, 256, 0, st>>>(gamma, beta, s, K, gamma_out, beta_out);
    return cudaGetLastError();
}

size_t quant_error_ws_bytes() { return (size_t)kErrBlocks * 3 * sizeof(double); }

cudaError_t run_quant_error(const void* x, int xt, int64_t rows, int64_t cols, int64_t ld, const float* smooth,
                            const qlin_qparams* p, const void* q, const void* s, const int32_t* z, double* out,
                            void* ws, cudaStream_t st) {
    ErrArgs a;
    a.x = x;
    a.rows = rows;
    a.cols = cols;
    a.ld = ld;
    a.smooth = smooth;
    a.smooth_mode = p->smooth_mode;
    a.q = q;
    a.s = s;
    a.z = p->symmetric ? nullptr : z;
    a.gran = p->gran;
    a.group = p->group;
    a.scale_f16 = p->scale_dtype == QLIN_F16;
    a.code4 = p->code == QLIN_S4 || p->code == QLIN_U4;
    a.code_signed = p->code == QLIN_S8 || p->code == QLIN_S4;
    double* part = reinterpret_cast<double*>(ws);
    switch (xt) {
    case QLIN_BF16: k_quant_error<__nv_bfloat16><<<kErrBlocks, 256, 0, st>>>(a, part); break;
    case QLIN_F16: k_quant_error<__half><<<kErrBlocks, 256, 0, st>>>(a, part); break;
    default: k_quant_error<float><<<kErrBlocks, 256, 0, st>>>(a, part);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    k_quant_error_final<<<1, 32, 0, st>>>(part, kErrBlocks, out);
    return cudaGetLastError();
}

}  // namespace qlin
