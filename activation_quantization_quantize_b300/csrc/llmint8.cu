// llmint8.cu -- LLM.int8() mixed-precision decomposition of the W8A8 layer.
//
// Method ("十九：模型压缩：量化、ZeroQuant、LLM.int8() 与 SmoothQuant"
// sections 9-11): XW = X_normal W_normal + X_outlier W_outlier.  The few
// input channels that carry outliers (any |x| above a threshold) are taken
// out of the INT8 product and multiplied in 16-bit; the rest run through the
// INT8 GEMM with vector-wise (per-token x per-output-channel) scales.  The
// weight is stored once in INT8 (per output channel); its outlier columns are
// dequantized for the 16-bit product, so
//     y[m,n] = sw[n] * (sx[m] * acc[m,n] + sum_{j outlier} x[m,j] * qw[n,j])
// with acc the exact INT32 sums over the normal channels.
//
// Kernels, in launch order:
//   colmax (calib.cu)   max |x| of every channel
//   k_outlier_cols      ascending list of the channels above the threshold
//   k_llmint8_xquant    per-token INT8 codes with the outlier channels zeroed
//                       (they neither widen the scale nor enter the INT8
//                       sums), and the outlier channels gathered as bf16
//   k_gather_wcols      the weight's outlier columns as bf16 codes
//   k_outlier_gemm      o = X_outlier qw_outlier^T in binary32 (bf16 MMAs)
//   k_w8a8_tc           INT8 GEMM whose epilogue adds o before the scale sw,
//                       so the output is rounded once
#include "qlin_common.cuh"
#include "qlin_internal.h"

namespace qlin {

namespace li8 {
constexpr int SCAN_THREADS = 1024;
constexpr int GBM = 128, GBN = 128, GBK = 16;  // outlier GEMM tile
constexpr int GPAD = 8;                        // bf16 padding per smem row (bank spread)
}  // namespace li8

// One CTA: flags[j] = (colmax[j] > tau); cols = ascending list of flagged j;
// count[0] = how many, count[1] = min(count, max_out).  More than max_out
// outlier channels record QLIN_ERR_WORKSPACE in the device error word (the
// later kernels use the first max_out).
__global__ void __launch_bounds__(li8::SCAN_THREADS) k_outlier_cols(const float* __restrict__ colmax, int64_t K,
                                                                   float tau, int max_out, uint8_t* __restrict__ flags,
                                                                   int32_t* __restrict__ cols,
                                                                   int32_t* __restrict__ count,
                                                                   int32_t* __restrict__ report) {
    __shared__ int part[li8::SCAN_THREADS];
    const int t = threadIdx.x;
    const int64_t per = ceil_div(K, (int64_t)li8::SCAN_THREADS);
    const int64_t j0 = t * per, j1 = (j0 + per < K) ? j0 + per : K;
    int n = 0;
    for (int64_t j = j0; j < j1; ++j) {
        const bool f = colmax[j] > tau;
        flags[j] = f ? 1 : 0;
        n += f ? 1 : 0;
    }
    part[t] = n;
    __syncthreads();
    // inclusive scan (Hillis-Steele)
    for (int o = 1; o < li8::SCAN_THREADS; o <<= 1) {
        const int v = t >= o ? part[t - o] : 0;
        __syncthreads();
        part[t] += v;
        __syncthreads();
    }
    int pos = part[t] - n;
    for (int64_t j = j0; j < j1; ++j)
        if (flags[j]) {
            cols[pos] = (int32_t)j;
            if (report) report[1 + pos] = (int32_t)j;
            ++pos;
        }
    if (t == li8::SCAN_THREADS - 1) {
        const int total = part[t];
        count[0] = total;
        count[1] = total < max_out ? total : max_out;
        if (report) report[0] = total;
        if (total > max_out) raise_device_error(QLIN_ERR_WORKSPACE);
    }
}

// One CTA per row (grid-stride): masked max|x| -> sx, codes (zeros in the
// outlier channels), and the gathered outlier values xo[m][0..Kp).
template <typename T>
__global__ void __launch_bounds__(256) k_llmint8_xquant(const T* __restrict__ x, int64_t M, int64_t K, int64_t ld,
                                                        const uint8_t* __restrict__ flags,
                                                        const int32_t* __restrict__ cols,
                                                        const int32_t* __restrict__ count, int Kp,
                                                        int8_t* __restrict__ qx, float* __restrict__ sx,
                                                        __nv_bfloat16* __restrict__ xo) {
    __shared__ float red[8];
    const int tid = threadIdx.x;
    const int64_t nchunks = K / 8;
    const int n_out = count[1];
    const CodeRange cr = make_range(-127, 127);
    for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
        const T* xr = x + m * ld;
        float hi = 0.0f;
        for (int64_t c = tid; c < nchunks; c += 256) {
            float v[8];
            load8<T>(xr + c * 8, v);
            const uint2 f = __ldg(reinterpret_cast<const uint2*>(flags) + c);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t fb = ((j < 4 ? f.x : f.y) >> (8 * (j & 3))) & 0xFFu;
                if (!fb) hi = fmaxf(hi, fabsf(v[j]));
            }
        }
        hi = warp_max(hi);
        if ((tid & 31) == 0) red[tid >> 5] = hi;
        __syncthreads();
        hi = red[0];
#pragma unroll
        for (int w = 1; w < 8; ++w) hi = fmaxf(hi, red[w]);
        float s;
        int z;
        scale_zero(0.0f, hi, -127, 127, true, false, s, z);
        if (tid == 0) sx[m] = s;
        const ScopeParams sp = make_scope(s, 0);
        for (int64_t c = tid; c < nchunks; c += 256) {
            float v[8];
            load8<T>(xr + c * 8, v);
            const uint2 f = __ldg(reinterpret_cast<const uint2*>(flags) + c);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t fb = ((j < 4 ? f.x : f.y) >> (8 * (j & 3))) & 0xFFu;
                if (fb) v[j] = 0.0f;
            }
            uint32_t cb[8];
            code_bits8<true, false>(v, sp, cr, cb);
            uint2 w;
            w.x = pack_bytes4(cb[0], cb[1], cb[2], cb[3]);
            w.y = pack_bytes4(cb[4], cb[5], cb[6], cb[7]);
            reinterpret_cast<uint2*>(qx + m * K)[c] = w;
        }
        for (int i = tid; i < Kp; i += 256) {
            const float v = i < n_out ? to_f32<T>(xr[cols[i]]) : 0.0f;
            xo[m * Kp + i] = __float2bfloat16_rn(v);  // a bf16 value: exact
        }
        __syncthreads();  // red is reused by the next row
    }
}

__global__ void k_gather_wcols(const int8_t* __restrict__ qw, int64_t N, int64_t K, const int32_t* __restrict__ cols,
                               const int32_t* __restrict__ count, int Kp, __nv_bfloat16* __restrict__ wo) {
    const int n_out = count[1];
    const int64_t total = N * Kp;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = e / Kp;
        const int i = (int)(e - n * Kp);
        wo[e] = __float2bfloat16_rn(i < n_out ? (float)qw[n * K + cols[i]] : 0.0f);  // |code| <= 128: exact
    }
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816_acc(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// o[m][n] = sum_{i < n_out} xo[m][i] * wo[n][i] in binary32.  CTA tile
// 128 x 128, 8 warps of 64 (m) x 32 (n); k steps of 16 over the outlier
// channels (the zero padding past n_out is skipped).
__global__ void __launch_bounds__(256) k_outlier_gemm(const __nv_bfloat16* __restrict__ xo,
                                                      const __nv_bfloat16* __restrict__ wo, int64_t M, int64_t N,
                                                      int Kp, const int32_t* __restrict__ count,
                                                      float* __restrict__ o) {
    using namespace li8;
    __shared__ __align__(16) __nv_bfloat16 sa[GBM][GBK + GPAD];
    __shared__ __align__(16) __nv_bfloat16 sb[GBN][GBK + GPAD];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wm = warp >> 2, wn = warp & 3;
    const int64_t m0 = (int64_t)blockIdx.y * GBM, n0 = (int64_t)blockIdx.x * GBN;
    const int ksteps = (count[1] + GBK - 1) / GBK;
    float acc[4][4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.0f;
    for (int ks = 0; ks < ksteps; ++ks) {
        {   // 128 rows x 16 bf16 = 2 x 16 B per row; one piece per thread per operand
            const int row = tid >> 1, half = tid & 1;
            const int64_t ma = m0 + row, nb = n0 + row;
            const int kk = ks * GBK + half * 8;
            uint4 va = make_uint4(0, 0, 0, 0), vb = make_uint4(0, 0, 0, 0);
            if (ma < M) va = __ldg(reinterpret_cast<const uint4*>(xo + ma * Kp + kk));
            if (nb < N) vb = __ldg(reinterpret_cast<const uint4*>(wo + nb * Kp + kk));
            *reinterpret_cast<uint4*>(&sa[row][half * 8]) = va;
            *reinterpret_cast<uint4*>(&sb[row][half * 8]) = vb;
        }
        __syncthreads();
        uint32_t af[4][4], bf[4][2];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = wm * 64 + i * 16 + (lane & 15);
            const int c = (lane >> 4) * 8;
            ldsm_x4(static_cast<uint32_t>(__cvta_generic_to_shared(&sa[r][c])), af[i][0], af[i][1], af[i][2], af[i][3]);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            // two n8 tiles: matrices (n 0-7, k 0-7), (n 0-7, k 8-15), (n 8-15, k 0-7), (n 8-15, k 8-15)
            const int r = wn * 32 + j * 16 + (lane & 7) + ((lane >> 4) << 3);
            const int c = ((lane >> 3) & 1) * 8;
            uint32_t r0, r1, r2, r3;
            ldsm_x4(static_cast<uint32_t>(__cvta_generic_to_shared(&sb[r][c])), r0, r1, r2, r3);
            bf[2 * j][0] = r0;
            bf[2 * j][1] = r1;
            bf[2 * j + 1][0] = r2;
            bf[2 * j + 1][1] = r3;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) mma_bf16_16816_acc(acc[i][j], af[i], bf[j][0], bf[j][1]);
        __syncthreads();
    }
    const int gq = lane >> 2, t = lane & 3;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t m = m0 + wm * 64 + i * 16 + gq + 8 * h;
            if (m >= M) continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t n = n0 + wn * 32 + j * 8 + 2 * t;
                if (n + 1 < N && (N & 1) == 0) {
                    *reinterpret_cast<float2*>(o + m * N + n) = make_float2(acc[i][j][2 * h], acc[i][j][2 * h + 1]);
                } else {
                    if (n < N) o[m * N + n] = acc[i][j][2 * h];
                    if (n + 1 < N) o[m * N + n + 1] = acc[i][j][2 * h + 1];
                }
            }
        }
}

// ------------------------------------------------------------------ workspace and launch
struct Li8Layout {
    size_t colmax, flags, cols, count, qx, sx, xo, wo, o, w8, total;
    int Kp;
};

static Li8Layout li8_layout(int64_t M, int64_t N, int64_t K, int64_t max_outliers) {
    auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
    Li8Layout l;
    l.Kp = (int)(((max_outliers + 15) / 16) * 16);
    size_t off = 0;
    l.colmax = off; off = up(off + (size_t)K * 4);
    l.flags = off;  off = up(off + (size_t)K);
    l.cols = off;   off = up(off + (size_t)K * 4);
    l.count = off;  off = up(off + 16);
    l.qx = off;     off = up(off + (size_t)M * K);
    l.sx = off;     off = up(off + (size_t)M * 4);
    l.xo = off;     off = up(off + (size_t)M * l.Kp * 2);
    l.wo = off;     off = up(off + (size_t)N * l.Kp * 2);
    l.o = off;      off = up(off + (size_t)M * N * 4);
    l.w8 = off;     off = up(off + w8a8_ws_bytes(M, N, K));
    l.total = off;
    return l;
}

size_t llmint8_ws_bytes(int64_t M, int64_t N, int64_t K, int64_t max_outliers) {
    return li8_layout(M, N, K, max_outliers).total;
}

cudaError_t run_gemm_llmint8(const void* x, int xt, int64_t M, int64_t K, int64_t ld, const int8_t* qw,
                             const float* sw, int64_t N, float threshold, int64_t max_outliers, void* y, int yt,
                             int32_t* report, void* ws, cudaStream_t st) {
    const Li8Layout l = li8_layout(M, N, K, max_outliers);
    uint8_t* base = reinterpret_cast<uint8_t*>(ws);
    float* colmax = reinterpret_cast<float*>(base + l.colmax);
    uint8_t* flags = base + l.flags;
    int32_t* cols = reinterpret_cast<int32_t*>(base + l.cols);
    int32_t* count = reinterpret_cast<int32_t*>(base + l.count);
    int8_t* qx = reinterpret_cast<int8_t*>(base + l.qx);
    float* sx = reinterpret_cast<float*>(base + l.sx);
    __nv_bfloat16* xo = reinterpret_cast<__nv_bfloat16*>(base + l.xo);
    __nv_bfloat16* wo = reinterpret_cast<__nv_bfloat16*>(base + l.wo);
    float* o = reinterpret_cast<float*>(base + l.o);
    cudaError_t e = cudaMemsetAsync(colmax, 0, (size_t)K * 4, st);
    if (e != cudaSuccess) return e;
    if ((e = run_absmax_update(x, xt, M, K, ld, colmax, st)) != cudaSuccess) return e;
    k_outlier_cols<<<1, li8::SCAN_THREADS, 0, st>>>(colmax, K, threshold, (int)max_outliers, flags, cols, count,
                                                    report);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    int64_t grid = M < (int64_t)num_sms() * 8 ? M : (int64_t)num_sms() * 8;
    (void)xt;  // bf16 activations (the outlier product is a bf16 product)
    k_llmint8_xquant<__nv_bfloat16><<<(unsigned)grid, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(x), M, K,
                                                                    ld, flags, cols, count, l.Kp, qx, sx, xo);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (l.Kp > 0) {
        k_gather_wcols<<<num_sms() * 4, 256, 0, st>>>(qw, N, K, cols, count, l.Kp, wo);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    dim3 g((unsigned)ceil_div(N, li8::GBN), (unsigned)ceil_div(M, li8::GBM));
    k_outlier_gemm<<<g, 256, 0, st>>>(xo, wo, M, N, l.Kp, count, o);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return run_gemm_w8a8(qx, sx, qw, sw, M, N, K, y, yt, nullptr, base + l.w8, st, o);
}

}  // namespace qlin
