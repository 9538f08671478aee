// gemm_w8a8.cu -- INT8 x INT8 -> exact INT32 linear layer with the
// per-token x per-output-channel dequantization epilogue.
//
// Method ("十九：模型压缩：量化、ZeroQuant、LLM.int8() 与 SmoothQuant" section 6;
// "第11章 模型量化与压缩" 11.1.4 and 11.4.5 step 6): activations are quantized
// per token, weights per output channel, the contraction runs on integers with
// INT32 accumulation, and y[m,n] = acc[m,n] * sx[m] * sw[n].
//
// Kernel here: the legacy warp-level tensor path (mma.sync m16n8k32 s8,
// native INT32 accumulation).  CTA tile 128 x 128 x 64, 8 warps (2 x 4), a
// 4-stage cp.async pipeline, XOR-swizzled 64-byte smem rows read by ldmatrix.
#include "qlin_common.cuh"
#include "qlin_internal.h"

namespace qlin {

namespace w8 {
constexpr int BM = 128, BN = 128, BK = 64, STAGES = 4, THREADS = 256;
constexpr int TILE_BYTES = BM * BK;  // == BN * BK
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte cp.async with zero fill when !pred.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
    int n = pred ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

// byte offset of (row, 16-byte chunk) inside a [rows x 64 B] tile
__device__ __forceinline__ uint32_t sw_off(int row, int chunk) {
    return (uint32_t)(row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_s8_16832(int c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(w8::THREADS) k_w8a8_mma(const int8_t* __restrict__ qx, const float* __restrict__ sx,
                                                          const int8_t* __restrict__ qw, const float* __restrict__ sw,
                                                          int64_t M, int64_t N, int64_t K, void* __restrict__ y,
                                                          int yt, int32_t* __restrict__ acc_out) {
    using namespace w8;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * TILE_BYTES;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wm = warp >> 2, wn = warp & 3;  // warp tile 64 (m) x 32 (n)
    const int64_t m0 = (int64_t)blockIdx.y * BM, n0 = (int64_t)blockIdx.x * BN;
    const int64_t ktiles = ceil_div(K, BK);

    auto load_stage = [&](int stage, int64_t kt) {
        const int64_t k0 = kt * BK;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            int piece = tid + THREADS * i;  // 512 pieces of 16 B per operand tile
            int row = piece >> 2, ch = piece & 3;
            int64_t kk = k0 + ch * 16;
            bool kin = kk < K;
            int64_t ma = m0 + row, nb = n0 + row;
            bool pa = kin && ma < M, pb = kin && nb < N;
            const int8_t* ga = qx + (pa ? ma * K + kk : 0);
            const int8_t* gb = qw + (pb ? nb * K + kk : 0);
            cp_async16(smem_u32(sA + stage * TILE_BYTES + sw_off(row, ch)), ga, pa);
            cp_async16(smem_u32(sB + stage * TILE_BYTES + sw_off(row, ch)), gb, pb);
        }
    };

    int acc[4][4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][j][e] = 0;

#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < ktiles) load_stage(s, s);
        cp_async_commit();
    }

    for (int64_t kt = 0; kt < ktiles; ++kt) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();
        int64_t nk = kt + STAGES - 1;
        if (nk < ktiles) load_stage((int)(nk % STAGES), nk);
        cp_async_commit();

        const int stage = (int)(kt % STAGES);
        const uint8_t* tA = sA + stage * TILE_BYTES;
        const uint8_t* tB = sB + stage * TILE_BYTES;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {  // two k32 steps per 64-byte tile
            uint32_t af[4][4], bf[4][2];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                // A 16x32 fragment: matrices (rows 0-7,k0-15),(rows 8-15,k0-15),(rows 0-7,k16-31),(rows 8-15,k16-31)
                int row = wm * 64 + i * 16 + (lane & 15);
                int ch = ks * 2 + (lane >> 4);
                ldmatrix_x4(smem_u32(tA + sw_off(row, ch)), af[i][0], af[i][1], af[i][2], af[i][3]);
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                // B: two n8 tiles; matrices (n0-7,k0-15),(n0-7,k16-31),(n8-15,k0-15),(n8-15,k16-31)
                int nrow = wn * 32 + j * 16 + (lane & 7) + ((lane >> 4) << 3);
                int ch = ks * 2 + ((lane >> 3) & 1);
                uint32_t r0, r1, r2, r3;
                ldmatrix_x4(smem_u32(tB + sw_off(nrow, ch)), r0, r1, r2, r3);
                bf[2 * j][0] = r0;
                bf[2 * j][1] = r1;
                bf[2 * j + 1][0] = r2;
                bf[2 * j + 1][1] = r3;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) mma_s8_16832(acc[i][j], af[i], bf[j][0], bf[j][1]);
        }
    }
    cp_async_wait<0>();

    // Epilogue: y = (float(acc) * sx[m]) * sw[n], one rounding to the output type.
    const int gq = lane >> 2, t = lane & 3;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            int64_t m = m0 + wm * 64 + i * 16 + gq + 8 * h;
            if (m >= M) continue;
            float smv = sx[m];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                int64_t n = n0 + wn * 32 + j * 8 + 2 * t;
                int a0 = acc[i][j][2 * h], a1 = acc[i][j][2 * h + 1];
                if (acc_out) {
                    if (n < N) acc_out[m * N + n] = a0;
                    if (n + 1 < N) acc_out[m * N + n + 1] = a1;
                }
                float v0 = 0.0f, v1 = 0.0f;
                if (n < N) v0 = ((float)a0 * smv) * sw[n];
                if (n + 1 < N) v1 = ((float)a1 * smv) * sw[n + 1];
                if (yt == QLIN_BF16) {
                    __nv_bfloat16* yb = reinterpret_cast<__nv_bfloat16*>(y);
                    if (n < N) yb[m * N + n] = __float2bfloat16_rn(v0);
                    if (n + 1 < N) yb[m * N + n + 1] = __float2bfloat16_rn(v1);
                } else {
                    float* yf = reinterpret_cast<float*>(y);
                    if (n < N) yf[m * N + n] = v0;
                    if (n + 1 < N) yf[m * N + n + 1] = v1;
                }
            }
        }
    }
}

size_t w8a8_ws_bytes(int64_t, int64_t, int64_t) { return 0; }

cudaError_t run_gemm_w8a8(const int8_t* qx, const float* sx, const int8_t* qw, const float* sw, int64_t M, int64_t N,
                          int64_t K, void* y, int yt, int32_t* acc_out, void*, cudaStream_t st) {
    using namespace w8;
    size_t smem = (size_t)2 * STAGES * TILE_BYTES;
    cudaError_t e = cudaFuncSetAttribute(k_w8a8_mma, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)ceil_div(N, BN), (unsigned)ceil_div(M, BM));
    k_w8a8_mma<<<grid, THREADS, smem, st>>>(qx, sx, qw, sw, M, N, K, y, yt, acc_out);
    return cudaGetLastError();
}

}  // namespace qlin
