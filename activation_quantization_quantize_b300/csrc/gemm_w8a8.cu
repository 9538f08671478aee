// gemm_w8a8.cu -- INT8 x INT8 -> exact INT32 linear layer with the
// per-token x per-output-channel dequantization epilogue.
//
// Method ("十九：模型压缩：量化、ZeroQuant、LLM.int8() 与 SmoothQuant" section 6;
// "第11章 模型量化与压缩" 11.1.4 and 11.4.5 step 6): activations are quantized
// per token, weights per output channel, the contraction runs on integers with
// INT32 accumulation, and y[m,n] = acc[m,n] * sx[m] * sw[n].
//
// sm_103a has no INT8 tcgen05 MMA, and its legacy INT8 path (mma.sync s8,
// cuBLASLt INT8) runs at roughly a tenth of the 16-bit tensor rate.  The main
// kernel (k_w8a8_tc) therefore computes the exact integer contraction on the
// fp16 tensor cores: codes in [-128, 127] are exact in fp16, every product
// (<= 2^14) is exact in fp32, and a sum of integers stays exact while its
// magnitude is below 2^24.  The converter warps report, per activation row and
// k-block of 64, the sum of |code|; the MMA warp accumulates it since the
// accumulator was last emptied.  Before a k-block could push any partial sum
// to 2^24 (sum|qx| * 128 >= 2^24), the accumulators are drained into an INT32
// workspace tile and restarted.  The INT32 result is therefore bit-exact for
// every input.
//
// k_w8a8_mma (warp-level mma.sync s8, native INT32 accumulation) is the
// legacy-path kernel, kept for comparison (QLIN_W8A8_KERNEL=mma).
#include <stdlib.h>
#include <string.h>

#include "qlin_common.cuh"
#include "qlin_internal.h"
#include "tc_ptx.cuh"
#include "tma_map.h"

namespace qlin {

namespace w8 {
constexpr int BM = 128, BN = 128, BK = 64, STAGES = 4, THREADS = 256;
constexpr int TILE_BYTES = BM * BK;  // == BN * BK
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}


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
            cp_async16_zfill(smem_u32(sA + stage * TILE_BYTES + sw_off(row, ch)), ga, pa);
            cp_async16_zfill(smem_u32(sB + stage * TILE_BYTES + sw_off(row, ch)), gb, pb);
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

// ====================================================================== tcgen05 kernel
namespace w8tc {
constexpr int BM = 256;                   // rows of qx per CTA: two M=128 MMAs (TMEM lanes)
constexpr int BN = 256;                   // max rows of qw per CTA (TMEM columns); the launch picks bn <= BN
constexpr int BK = 64;                    // k per stage (one 128-byte fp16 row)
constexpr int S16 = 2;                    // fp16 operand stages (converter -> MMA)
constexpr int S8 = 3;                     // int8 staging stages (TMA -> converter)
constexpr int A_BYTES = BM * BK * 2;      // 32 KB fp16 tile (two 16 KB halves)
constexpr int A_HALF = A_BYTES / 2;
constexpr int B_BYTES = BN * BK * 2;      // 32 KB fp16 tile
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int A8_BYTES = BM * BK;         // 16 KB int8 tile (rows of 64 bytes)
constexpr int B8_BYTES = BN * BK;         // 16 KB
constexpr int STAGE8_BYTES = A8_BYTES + B8_BYTES;
constexpr int NCONV_WARPS = 16;           // warps 0-15: int8 -> fp16 converters
constexpr int NCONV = NCONV_WARPS * 32;
constexpr int EPI_WARP0 = 16;             // warps 16-19: drains + epilogue (one per TMEM lane quarter)
constexpr int MMA_WARP = 20;              // warp 20: TMEM owner, MMA issuer
constexpr int TMA_WARP = 21;              // warp 21: int8 tile loads
constexpr int THREADS = 22 * 32;
constexpr int PIECES = (BM + BN) * BK / 16;   // max 16-byte int8 pieces per k-block (2048)
constexpr int PPT = PIECES / NCONV;           // max pieces per converter thread (4)
constexpr int A_PIECES = BM * BK / 16;        // 1024
constexpr uint32_t ROWSUM_LIMIT = 131071;     // sum|qx| * 128 < 2^24
constexpr uint32_t TMEM_COLS = 512;           // [0,256): rows 0-127, [256,512): rows 128-255 (fp32)
constexpr uint32_t EV_DRAIN = 1, EV_FINAL = 2;
constexpr size_t CTRL_BYTES = 2048;
constexpr size_t SMEM_BYTES = 1024 + (size_t)S16 * STAGE_BYTES + (size_t)S8 * STAGE8_BYTES + CTRL_BYTES;
// Longest sleep between polls of a warp idle until a tile event: none; the
// suspending try_wait already frees the warp's issue slots and wakes it as
// soon as the phase completes (a sleep would delay every drain).
constexpr uint32_t kIdleSleepNs = 0;
}  // namespace w8tc

// int8 x4 -> two fp16x2 words, exact: bias to unsigned, place each byte in the
// low mantissa of fp16 1024 (0x64xx = 1024 + u), subtract 1152.
__device__ __forceinline__ void s8x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
    uint32_t u = w ^ 0x80808080u;
    uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
    uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
}

// acc + sum of |b| over the four signed int8 codes b of w, exactly: prmt in
// sign-replicate mode makes 0xFF in every negative byte and 0x00 elsewhere;
// with 0x01 or-ed in, each byte is the sign (+1 / -1) of its code, and the
// signed dot product of codes and signs is the sum of |b| (|-128| = 128).
__device__ __forceinline__ int abs_sum4(uint32_t w, int acc) {
    uint32_t m;
    asm("prmt.b32 %0, %1, 0, 0xBA98;" : "=r"(m) : "r"(w));
    return __dp4a((int)w, (int)(m | 0x01010101u), acc);
}

// Epilogue of W (16 or 32) consecutive outputs of row m starting at column nb:
// acc_out (exact sums) and y = (float(acc) * sx[m]) * sw[n], one rounding.
template <int W>
__device__ __forceinline__ void store_row(const int (&tot)[W], int64_t m, int64_t nb, int64_t N, float sxm,
                                            const float* __restrict__ sw, void* __restrict__ y, int yt,
                                            int32_t* __restrict__ acc_out, const float* __restrict__ add) {
    const bool full = (nb + W <= N) && (N % 8 == 0);
    if (acc_out) {
        int32_t* ap = acc_out + m * N + nb;
        if (full) {
#pragma unroll
            for (int j = 0; j < W; j += 4) *reinterpret_cast<int4*>(ap + j) = make_int4(tot[j], tot[j + 1], tot[j + 2], tot[j + 3]);
        } else {
            for (int j = 0; j < W; ++j)
                if (nb + j < N) ap[j] = tot[j];
        }
    }
    float f[W];
#pragma unroll
    for (int j = 0; j < W; ++j) {
        float swn = (nb + j < N) ? __ldg(sw + nb + j) : 0.0f;
        f[j] = ((float)tot[j] * sxm) * swn;
    }
    if (add) {  // y = (acc * sx + add) * sw, the addend's row segment read as 16-byte vectors
        const float* ap = add + m * N + nb;
        if (full) {
#pragma unroll
            for (int j = 0; j < W; j += 4) {
                const float4 v = __ldg(reinterpret_cast<const float4*>(ap + j));
                f[j] = fmaf(v.x, __ldg(sw + nb + j), f[j]);
                f[j + 1] = fmaf(v.y, __ldg(sw + nb + j + 1), f[j + 1]);
                f[j + 2] = fmaf(v.z, __ldg(sw + nb + j + 2), f[j + 2]);
                f[j + 3] = fmaf(v.w, __ldg(sw + nb + j + 3), f[j + 3]);
            }
        } else {
            for (int j = 0; j < W; ++j)
                if (nb + j < N) f[j] = fmaf(__ldg(ap + j), __ldg(sw + nb + j), f[j]);
        }
    }
    if (yt == QLIN_BF16) {
        __nv_bfloat16* yp = reinterpret_cast<__nv_bfloat16*>(y) + m * N + nb;
        if (full) {
#pragma unroll
            for (int j = 0; j < W; j += 8) {
                __nv_bfloat162 p0 = __floats2bfloat162_rn(f[j], f[j + 1]);
                __nv_bfloat162 p1 = __floats2bfloat162_rn(f[j + 2], f[j + 3]);
                __nv_bfloat162 p2 = __floats2bfloat162_rn(f[j + 4], f[j + 5]);
                __nv_bfloat162 p3 = __floats2bfloat162_rn(f[j + 6], f[j + 7]);
                uint4 u;
                u.x = *reinterpret_cast<uint32_t*>(&p0);
                u.y = *reinterpret_cast<uint32_t*>(&p1);
                u.z = *reinterpret_cast<uint32_t*>(&p2);
                u.w = *reinterpret_cast<uint32_t*>(&p3);
                *reinterpret_cast<uint4*>(yp + j) = u;
            }
        } else {
            for (int j = 0; j < W; ++j)
                if (nb + j < N) yp[j] = __float2bfloat16_rn(f[j]);
        }
    } else {
        float* yp = reinterpret_cast<float*>(y) + m * N + nb;
        if (full) {
#pragma unroll
            for (int j = 0; j < W; j += 4) *reinterpret_cast<float4*>(yp + j) = make_float4(f[j], f[j + 1], f[j + 2], f[j + 3]);
        } else {
            for (int j = 0; j < W; ++j)
                if (nb + j < N) yp[j] = f[j];
        }
    }
}

struct W8TcArgs {
    const float* sx;
    const float* sw;
    int64_t M, N, K;
    void* y;
    int yt;
    int32_t* acc_out;
    int32_t* drain;   // [M][N] INT32 partial sums, written only when a drain occurs
    int32_t* part;    // [tail tiles][tail_split][BM][BN] INT32 sums of the split tail tiles
    const float* add; // NULL, or [M][N] binary32 terms added before the output scale: y = (acc*sx + add)*sw
    int64_t full_tiles;  // CTAs [0, full_tiles) own whole tiles
    int tail_split;      // K parts of each later tile (one CTA per part)
    int num_m_tiles;
    int bn;           // weight rows per CTA (multiple of 32, <= 256)
    uint32_t idesc;   // MMA instruction descriptor (M = 128, N = bn)
};

// A CTA owns a 256 x 256 output tile: two M=128 MMAs per k-step share the
// converted weight tile, so widening (and shared-memory traffic) per FLOP is a
// third lower than with a 128-row tile.  int8 tiles arrive by TMA (zero-filled
// past M, N and K) into a staging ring; converter warps widen them to fp16 in
// the 128B-swizzled layout the MMA reads; one thread issues tcgen05.mma
// (kind::f16, fp32 in TMEM).  Drains (rare) add the accumulators into an INT32
// tile in global memory.
__global__ void __launch_bounds__(w8tc::THREADS, 1)
    k_w8a8_tc(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b, W8TcArgs p) {
    using namespace w8tc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* tiles = smem;                                   // S16 x (A fp16 | B fp16)
    uint8_t* stage8 = smem + S16 * STAGE_BYTES;              // S8 x (A int8 | B int8)
    uint64_t* bars = reinterpret_cast<uint64_t*>(stage8 + S8 * STAGE8_BYTES);
    // bars: full16[S16], empty16[S16], full8[S8], empty8[S8], acc_full, acc_empty, ev, done
    uint16_t* rowsum = reinterpret_cast<uint16_t*>(bars + 2 * S16 + 2 * S8 + 4);  // [S16][BM]
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(rowsum + S16 * BM);  // tmem, event, abort
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bn = p.bn;
    // Tile and k-block range of this CTA: whole tiles first; each tile of the
    // last, partial wave is cut into tail_split K parts whose exact INT32 sums
    // go to their own slice of `part` (summed by k_w8a8_tail).
    int64_t tile = blockIdx.x;
    int kpart = 0, nparts = 1;
    if (tile >= p.full_tiles) {
        const int64_t u = tile - p.full_tiles;
        tile = p.full_tiles + u / p.tail_split;
        kpart = (int)(u % p.tail_split);
        nparts = p.tail_split;
    }
    const int64_t m0 = (tile % p.num_m_tiles) * BM;
    const int64_t n0 = (tile / p.num_m_tiles) * bn;
    const int nkb_all = (int)ceil_div(p.K, BK);
    const int kb0 = (int)((int64_t)nkb_all * kpart / nparts);
    const int nkb = (int)((int64_t)nkb_all * (kpart + 1) / nparts) - kb0;
    const bool split = nparts > 1;
    // INT32 target of drains (and, for split tiles, of the final sums)
    int32_t* const dtile = split ? p.part + ((tile - p.full_tiles) * nparts + kpart) * (int64_t)BM * BN
                                 : p.drain + m0 * p.N + n0;
    const int64_t dld = split ? BN : p.N;
    const int npieces = (BM + bn) * BK / 16;

    const uint32_t bar0 = tc::smem_addr(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S16 + s); };
    auto full8_bar = [&](int s) { return bar0 + 8u * (2 * S16 + s); };
    auto empty8_bar = [&](int s) { return bar0 + 8u * (2 * S16 + S8 + s); };
    const uint32_t acc_full = bar0 + 8u * (2 * S16 + 2 * S8);
    const uint32_t acc_empty = acc_full + 8u;
    const uint32_t ev_bar = acc_full + 16u;
    const uint32_t done_bar = acc_full + 24u;

    if (threadIdx.x == 0) {
        // converter warps arrive once per warp (an elected lane after __syncwarp)
        for (int s = 0; s < S16; ++s) {
            tc::mbar_init(full_bar(s), NCONV_WARPS);
            tc::mbar_init(empty_bar(s), 1);
        }
        for (int s = 0; s < S8; ++s) {
            tc::mbar_init(full8_bar(s), 1);
            tc::mbar_init(empty8_bar(s), NCONV_WARPS);
        }
        tc::mbar_init(acc_full, 1);
        tc::mbar_init(acc_empty, 4);  // one arrival per epilogue warp
        tc::mbar_init(ev_bar, 1);
        tc::mbar_init(done_bar, 1);
        misc[2] = 0;
        tc::mbar_init_fence();
    }
    if (warp == MMA_WARP) {
        tc::tmem_alloc(tc::smem_addr((const void*)&misc[0]), TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp < NCONV_WARPS) {
        // ---------------------------------------------------------- converters
        const int tid = threadIdx.x;
        // swizzled byte offsets (within a stage) of each piece's first 16-byte
        // chunk; the second chunk is at offset ^ 16.  Pieces j < 4 are
        // activation rows tid/4 + 64 j, the rest weight rows.
        uint32_t soff[PPT];
#pragma unroll
        for (int j = 0; j < PPT; ++j) {
            const int piece = tid + NCONV * j;
            const bool is_a = j < A_PIECES / NCONV;
            const int pr = is_a ? piece : piece - A_PIECES;
            soff[j] = (is_a ? 0u : (uint32_t)A_BYTES) + tc::sw128_off((uint32_t)(pr >> 2), 2u * (uint32_t)(pr & 3));
        }
        const uint32_t rs_row = (uint32_t)(tid >> 2);
        const bool rs_leader = (tid & 3) == 0;
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % S16, s8 = kb % S8;
            const uint32_t ph = (uint32_t)(kb / S16) & 1u, ph8 = (uint32_t)(kb / S8) & 1u;
            if (!tc::mbar_wait_warp(full8_bar(s8), ph8, abort_flag)) break;
            const uint8_t* a8 = stage8 + (size_t)s8 * STAGE8_BYTES;
            uint4 cur[PPT];
#pragma unroll
            for (int j = 0; j < PPT; ++j)
                cur[j] = (tid + NCONV * j < npieces) ? *reinterpret_cast<const uint4*>(a8 + (size_t)(tid + NCONV * j) * 16)
                                                    : make_uint4(0, 0, 0, 0);
            int rs[A_PIECES / NCONV];
#pragma unroll
            for (int j = 0; j < A_PIECES / NCONV; ++j) {
                int a = abs_sum4(cur[j].x, 0);
                a = abs_sum4(cur[j].y, a);
                a = abs_sum4(cur[j].z, a);
                a = abs_sum4(cur[j].w, a);
                a += __shfl_xor_sync(0xffffffffu, a, 1);
                a += __shfl_xor_sync(0xffffffffu, a, 2);
                rs[j] = a;  // sum |q| of the row's 64 codes of this k-block (<= 8192)
            }
            uint32_t hbuf[PPT][8];
#pragma unroll
            for (int j = 0; j < PPT; ++j) {
                s8x4_to_f16(cur[j].x, hbuf[j][0], hbuf[j][1]);
                s8x4_to_f16(cur[j].y, hbuf[j][2], hbuf[j][3]);
                s8x4_to_f16(cur[j].z, hbuf[j][4], hbuf[j][5]);
                s8x4_to_f16(cur[j].w, hbuf[j][6], hbuf[j][7]);
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(empty8_bar(s8));  // the staging slot may be refilled
            if (!tc::mbar_wait_warp(empty_bar(s), ph ^ 1u, abort_flag)) break;
            uint8_t* tS = tiles + (size_t)s * STAGE_BYTES;
#pragma unroll
            for (int j = 0; j < PPT; ++j) {
                if (tid + NCONV * j >= npieces) continue;
                *reinterpret_cast<uint4*>(tS + soff[j]) = make_uint4(hbuf[j][0], hbuf[j][1], hbuf[j][2], hbuf[j][3]);
                *reinterpret_cast<uint4*>(tS + (soff[j] ^ 16u)) =
                    make_uint4(hbuf[j][4], hbuf[j][5], hbuf[j][6], hbuf[j][7]);
            }
            if (rs_leader) {
#pragma unroll
                for (int j = 0; j < A_PIECES / NCONV; ++j) rowsum[s * BM + rs_row + (NCONV / 4) * j] = (uint16_t)rs[j];
            }
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(full_bar(s));
        }
    } else if (warp == TMA_WARP) {
        // ---------------------------------------------------------- int8 tile loads
        if (lane == 0 && !tc::producers_stalled()) {
            for (int kb = 0; kb < nkb; ++kb) {
                const int s8 = kb % S8;
                const uint32_t ph8 = (uint32_t)(kb / S8) & 1u;
                if (!tc::mbar_wait(empty8_bar(s8), ph8 ^ 1u, abort_flag)) break;
                tc::mbar_arrive_expect_tx(full8_bar(s8), (uint32_t)(BM + bn) * BK);
                const uint32_t dst = tc::smem_addr(stage8 + (size_t)s8 * STAGE8_BYTES);
                tc::tma_load_2d(dst, &tm_a, (kb0 + kb) * BK, (int)m0, full8_bar(s8));
                tc::tma_load_2d(dst + A8_BYTES, &tm_b, (kb0 + kb) * BK, (int)n0, full8_bar(s8));
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ---------------------------------------------------------- MMA issuer
        const uint32_t IDESC = p.idesc;
        const uint32_t tiles_addr = tc::smem_addr(tiles);
        uint32_t S[8] = {0, 0, 0, 0, 0, 0, 0, 0};  // running sum|qx| of rows 8 lane .. 8 lane + 7
        bool started = false;
        uint32_t ndrain = 0;
        bool ok = true;
        for (int kb = 0; kb < nkb && ok; ++kb) {
            const int s = kb % S16;
            const uint32_t ph = (uint32_t)(kb / S16) & 1u;
            if (!tc::mbar_wait_warp(full_bar(s), ph, abort_flag)) {
                ok = false;
                break;
            }
            uint32_t B[8], mx = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                B[i] = rowsum[s * BM + lane * 8 + i];
                mx = max(mx, S[i] + B[i]);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (started && mx > ROWSUM_LIMIT) {
                // drain the accumulators into the INT32 tile before adding this k-block
                if (tc::elect_one()) {
                    misc[1] = EV_DRAIN;
                    tc::mbar_arrive(ev_bar);
                    tc::mma_commit(acc_full);
                }
                __syncwarp();
                if (!tc::mbar_wait_warp(acc_empty, ndrain & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                ++ndrain;
                started = false;
#pragma unroll
                for (int i = 0; i < 8; ++i) S[i] = B[i];
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) S[i] += B[i];
            }
            tc::tc_fence_after();
            // descriptors are computed by the whole warp (warp-uniform values);
            // one elected lane issues
            const uint32_t a_addr = tiles_addr + (uint32_t)s * STAGE_BYTES;
            const uint64_t ad0 = tc::desc_sw128(a_addr);
            const uint64_t ad1 = tc::desc_sw128(a_addr + A_HALF);
            const uint64_t bd = tc::desc_sw128(a_addr + A_BYTES);
            if (tc::elect_one()) {
#pragma unroll
                for (int j = 0; j < BK / 16; ++j) {  // 32 bytes of K per MMA
                    const uint32_t acc = (started || j > 0) ? 1u : 0u;
                    tc::mma_f16(tmem, ad0 + 2 * j, bd + 2 * j, IDESC, acc);
                    tc::mma_f16(tmem + 256, ad1 + 2 * j, bd + 2 * j, IDESC, acc);
                }
                tc::mma_commit(empty_bar(s));
            }
            started = true;
            __syncwarp();
        }
        if (tc::elect_one()) {
            misc[1] = ok ? EV_FINAL : 0u;
            tc::mbar_arrive(ev_bar);
            tc::mma_commit(acc_full);
            tc::mma_commit(done_bar);
        }
        __syncwarp();
        tc::mbar_wait_drain(done_bar, 0);
        __syncwarp();
    } else {
        // ---------------------------------------------------------- drains + epilogue
        const int q = warp & 3;  // TMEM lane quarter of this warp
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        uint32_t ndrain = 0;
        for (uint32_t ev = 0;; ++ev) {
            if (!tc::mbar_wait_warp(ev_bar, ev & 1u, abort_flag, kIdleSleepNs)) break;
            const uint32_t type = misc[1];
            if (!tc::mbar_wait_warp(acc_full, ev & 1u, abort_flag)) break;
            tc::tc_fence_after();
            if (type != EV_DRAIN && type != EV_FINAL) break;
            const float swz = 0.0f;
            (void)swz;
            for (int h = 0; h < 2; ++h) {
                const int64_t m = m0 + 128 * h + 32 * q + lane;
                const float sxm = (type == EV_FINAL && m < p.M) ? p.sx[m] : 0.0f;
                for (int c = 0; c < bn; c += 16) {
                    __syncwarp();
                    uint32_t a[16];
                    tc::tmem_ld16(tmem + lane_base + 256 * h + c, a);
                    tc::tmem_wait_ld();
                    int tot[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) tot[j] = __float2int_rn(__uint_as_float(a[j]));
                    if (m >= p.M) continue;
                    const int64_t nb = n0 + c;
                    int32_t* dp = dtile + (m - m0) * dld + c;
                    const bool full = (nb + 16 <= p.N) && (p.N % 4 == 0);
                    if (ndrain) {  // add the INT32 sums of earlier drains
                        if (full) {
#pragma unroll
                            for (int j = 0; j < 16; j += 4) {
                                int4 v = *reinterpret_cast<const int4*>(dp + j);
                                tot[j] += v.x;
                                tot[j + 1] += v.y;
                                tot[j + 2] += v.z;
                                tot[j + 3] += v.w;
                            }
                        } else {
                            for (int j = 0; j < 16; ++j)
                                if (nb + j < p.N) tot[j] += dp[j];
                        }
                    }
                    if (type == EV_DRAIN || split) {  // a split tile's final sums go to its slice
                        if (full) {
#pragma unroll
                            for (int j = 0; j < 16; j += 4)
                                *reinterpret_cast<int4*>(dp + j) = make_int4(tot[j], tot[j + 1], tot[j + 2], tot[j + 3]);
                        } else {
                            for (int j = 0; j < 16; ++j)
                                if (nb + j < p.N) dp[j] = tot[j];
                        }
                    } else {
                        store_row<16>(tot, m, nb, p.N, sxm, p.sw, p.y, p.yt, p.acc_out, p.add);
                    }
                }
            }
            if (type == EV_FINAL) break;
            ++ndrain;
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(acc_empty);
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// y / acc_out of the split tail tiles: the tail_split exact INT32 partial sums
// of each output are added and go through the same epilogue as whole tiles.
__global__ void __launch_bounds__(256) k_w8a8_tail(W8TcArgs p, int tail_tiles) {
    using namespace w8tc;
    const int nch = p.bn / 16;  // 16-column chunks of a tile row
    const int per_tile = BM * nch;
    const int total = tail_tiles * per_tile;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        const int t = i / per_tile, rem = i - t * per_tile;
        const int row = rem / nch, ch = rem - row * nch;
        const int64_t tile = p.full_tiles + t;
        const int64_t m = (tile % p.num_m_tiles) * BM + row;
        const int64_t nb = (tile / p.num_m_tiles) * p.bn + ch * 16;
        if (m >= p.M || nb >= p.N) continue;
        int tot[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) tot[j] = 0;
        for (int k = 0; k < p.tail_split; ++k) {
            const int4* src = reinterpret_cast<const int4*>(p.part + ((int64_t)t * p.tail_split + k) * (int64_t)BM * BN +
                                                            row * BN + ch * 16);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int4 v = src[j];
                tot[4 * j] += v.x;
                tot[4 * j + 1] += v.y;
                tot[4 * j + 2] += v.z;
                tot[4 * j + 3] += v.w;
            }
        }
        store_row<16>(tot, m, nb, p.N, p.sx[m], p.sw, p.y, p.yt, p.acc_out, p.add);
    }
}

// ====================================================================== CTA-pair kernel
// A cluster of two CTAs on two SMs owns a 256 x 256 output tile.  One
// M = 256 tcgen05 MMA per 16-k step (cta_group::2) covers the pair: CTA r
// holds activation rows 128 r .. 128 r + 127 of the tile as fp16 in its own
// TMEM (the A operand, written by tcgen05.st, so it never passes through
// shared memory) and weight rows 128 r .. 128 r + 127 as fp16 in its shared
// memory (the B operand; each half is read once for both SMs).
//
// Each converter warp fetches its own int8 rows with cp.async into a private
// ring in shared memory (four k-blocks deep) and reads them back after a
// thread-local wait, so the int8 tiles need no barrier.  The k-blocks
// alternate between two converter groups, so that the fixed cost of a
// warp's hand-off (one wait for a free stage, one arrival) is spent once per
// two k-blocks.  Roles per CTA: group g = 0, 1: warps 8g .. 8g+3 widen
// activation rows (warp w: TMEM lanes 32 (w % 4) .., one row per thread) and
// report each row's sum |q| of the k-block to the even CTA; warps 8g+4 ..
// 8g+7 widen weight rows into the swizzled B tile; warps 16-19 drain and
// finish the accumulators of their TMEM lane quarter; warp 20 owns TMEM and,
// in the even CTA, issues the MMAs; warp 21 of the even CTA tracks the
// running sum |q| of all 256 rows and posts, per stage, whether the
// accumulators must be drained before that k-block.  It decides from the
// sums up to the previous k-block and the bound 64 * 128 on one k-block's
// sum, so the decision is ready as soon as the stage is full and the
// reduction over rows runs while the tensor cores work.
namespace w8p {
constexpr int BM = 256, HM = 128;              // tile rows, rows per CTA
constexpr int BN = 256, HN = 128;              // tile columns, weight rows per CTA
constexpr int BK = 64;
constexpr int S16 = 4;                         // fp16 operand stages (TMEM A + shared B)
constexpr int NGROUP = 2;                      // converter groups (k-blocks alternate)
constexpr int RING = 4;                        // own k-blocks in flight per converter warp
constexpr int SLOT_BYTES = 32 * BK;            // 32 rows x 64 int8 codes
constexpr int WARP_RING_BYTES = RING * SLOT_BYTES;
constexpr int NCONV_WARPS = 8 * NGROUP;
constexpr int B16_BYTES = HN * BK * 2;         // 16 KB swizzled fp16 B half-tile
constexpr int EPI_WARP0 = 16, MMA_WARP = 20, MON_WARP = 21;
constexpr int THREADS = 22 * 32;
constexpr uint32_t ACC_COL = 0;                // accumulator: 128 lanes x 256 fp32 columns
constexpr uint32_t A_COL0 = 256;               // A stage s: 32 columns (64 fp16 k) at A_COL0 + 32 s
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ROWSUM_LIMIT = w8tc::ROWSUM_LIMIT;
constexpr uint32_t KB_SUM_MAX = BK * 128;      // largest sum |q| of one row over one k-block
constexpr uint32_t EV_DRAIN = 1, EV_FINAL = 2;
constexpr int FULL_ARRIVALS = 2 * 8;           // one group's converter warps, both CTAs
constexpr int ACC_EMPTY_ARRIVALS = 2 * 4;      // epilogue warps of both CTAs
constexpr size_t CTRL_BYTES = 8192;
constexpr size_t SMEM_BYTES = 1024 + (size_t)S16 * B16_BYTES + (size_t)NCONV_WARPS * WARP_RING_BYTES + CTRL_BYTES;
constexpr uint32_t kIdleSleepNs = w8tc::kIdleSleepNs;
static_assert(A_COL0 + 32 * S16 <= TMEM_COLS, "TMEM budget");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert((3 * S16 + 4) * 8 + S16 * BM * 4 + S16 * 4 + 16 <= (int)CTRL_BYTES, "control block");
static_assert(S16 % NGROUP == 0, "a stage belongs to one converter group");
}  // namespace w8p

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(w8p::THREADS, 1)
    k_w8a8_pair(const int8_t* __restrict__ qx, const int8_t* __restrict__ qw, W8TcArgs p) {
    using namespace w8p;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* tiles = smem;                                   // S16 x fp16 B half-tile
    uint8_t* rings = smem + S16 * B16_BYTES;                 // per converter warp: RING x 2 KB of int8 rows
    uint64_t* bars = reinterpret_cast<uint64_t*>(rings + NCONV_WARPS * WARP_RING_BYTES);
    // bars: full[S16], empty[S16], acc_full, acc_empty, ev, done, dec[S16]
    uint32_t* rowsum = reinterpret_cast<uint32_t*>(bars + 3 * S16 + 4);  // [S16][BM], even CTA
    volatile uint32_t* drain_dec = reinterpret_cast<volatile uint32_t*>(rowsum + S16 * BM);  // [S16]
    volatile uint32_t* misc = drain_dec + S16;  // tmem, event, abort
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = tc::cluster_rank();
    const bool leader = rank == 0;
    int64_t tile = blockIdx.x >> 1;
    int kpart = 0, nparts = 1;
    if (tile >= p.full_tiles) {
        const int64_t u = tile - p.full_tiles;
        tile = p.full_tiles + u / p.tail_split;
        kpart = (int)(u % p.tail_split);
        nparts = p.tail_split;
    }
    const int64_t m0 = (tile % p.num_m_tiles) * BM;
    const int64_t n0 = (tile / p.num_m_tiles) * BN;
    const int64_t mh = m0 + HM * (int64_t)rank;              // this CTA's first activation row
    const int64_t nh = n0 + HN * (int64_t)rank;              // this CTA's first weight row
    const int nkb_all = (int)ceil_div(p.K, BK);
    const int kb0 = (int)((int64_t)nkb_all * kpart / nparts);
    const int nkb = (int)((int64_t)nkb_all * (kpart + 1) / nparts) - kb0;
    const bool split = nparts > 1;
    int32_t* const dtile = split ? p.part + ((tile - p.full_tiles) * nparts + kpart) * (int64_t)BM * BN
                                 : p.drain + m0 * p.N + n0;
    const int64_t dld = split ? BN : p.N;

    const uint32_t bar0 = tc::smem_addr(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S16 + s); };
    const uint32_t acc_full = bar0 + 8u * (2 * S16);
    const uint32_t acc_empty = acc_full + 8u;
    const uint32_t ev_bar = acc_full + 16u;
    const uint32_t done_bar = acc_full + 24u;
    auto dec_bar = [&](int s) { return bar0 + 8u * (2 * S16 + 4 + s); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S16; ++s) {
            tc::mbar_init(full_bar(s), FULL_ARRIVALS);
            tc::mbar_init(empty_bar(s), 1);
        }
        tc::mbar_init(acc_full, 1);
        tc::mbar_init(acc_empty, ACC_EMPTY_ARRIVALS);
        tc::mbar_init(ev_bar, 1);
        tc::mbar_init(done_bar, 1);
        for (int s = 0; s < S16; ++s) tc::mbar_init(dec_bar(s), 1);
        misc[1] = 0;
        misc[2] = 0;
        tc::mbar_init_fence();
    }
    if (warp == MMA_WARP) {
        tc::tmem_alloc_pair(tc::smem_addr((const void*)&misc[0]), TMEM_COLS);
        tc::tmem_relinquish_pair();
    }
    tc::tc_fence_before();
    tc::cluster_sync();  // both CTAs' barriers initialised and TMEM allocated
    tc::tc_fence_after();
    const uint32_t tmem = misc[0];
    // the even CTA's copies of the barriers and row sums the converters report to
    const uint32_t full_bar_l0 = tc::mapa(full_bar(0), 0);
    const uint32_t rowsum_l0 = tc::mapa(tc::smem_addr(rowsum), 0);
    const uint32_t acc_empty_l0 = tc::mapa(acc_empty, 0);

    if (warp < NCONV_WARPS) {
        // ---------------------------------------------------------- converters
        const int g = warp >> 3;                 // group: k-blocks g, g + 2, ...
        const int q = warp & 3;                  // 32-row quarter of this CTA's half
        const bool is_a = (warp & 4) == 0;
        const uint32_t ring = tc::smem_addr(rings) + (uint32_t)warp * WARP_RING_BYTES;
        const uint8_t* ringp = rings + (size_t)warp * WARP_RING_BYTES;
        const int8_t* src = is_a ? qx : qw;
        const int64_t row0 = (is_a ? mh : nh) + 32 * q;   // first global row of this warp
        const int64_t nrows = is_a ? p.M : p.N;
        // copies: lane l fetches rows 8 j + l / 4 (j = 0..3) of the warp's 32,
        // 16-byte chunk l % 4 of the 64-code k-block; activation rows are
        // stored with a 64-byte swizzle (chunk c of row r at 16 (c ^ (r/2 % 4)))
        // so that reading one row per lane is free of bank conflicts
        const int cc = lane & 3;
        // per-lane copy state, fixed for the whole tile: source row pointers
        // (at this lane's chunk of the first k-block), whether the row exists,
        // and the destination offsets within a slot
        const int8_t* gsrc[4];
        bool row_in[4];
        uint32_t doff[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int rr = 8 * j + (lane >> 2);
            const int64_t row = row0 + rr;
            row_in[j] = row < nrows;
            gsrc[j] = src + (row_in[j] ? row * p.K + (int64_t)kb0 * BK + 16 * cc : 0);
            doff[j] = (uint32_t)rr * 64u + ((is_a ? (uint32_t)(cc ^ ((rr >> 1) & 3)) : (uint32_t)cc) << 4);
        }
        const int64_t k_lane = (int64_t)kb0 * BK + 16 * cc;  // this lane's k in the first k-block
        auto issue = [&](int i) {  // own k-block i of this group
            const int kb = g + NGROUP * i;
            if (kb < nkb) {
                const uint32_t slot = ring + (uint32_t)(i % RING) * SLOT_BYTES;
                const int64_t koff = (int64_t)kb * BK;
                const bool k_in = k_lane + koff < p.K;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const bool in = row_in[j] && k_in;
                    cp_async16_zfill(slot + doff[j], in ? gsrc[j] + koff : src, in);
                }
            }
            cp_async_commit();
        };
        // the failure-detection test hook: no copies and no arrivals, so the
        // monitor's wait for the first stage runs out
        const int nkb_conv = tc::producers_stalled() ? 0 : nkb;
        for (int i = 0; i < RING - 1; ++i) issue(i);
        uint32_t soff[4];  // weight pieces of this lane in the swizzled fp16 tile
#pragma unroll
        for (int j = 0; j < 4; ++j) soff[j] = tc::sw128_off((uint32_t)(32 * q + 8 * j + (lane >> 2)), 2u * (uint32_t)cc);
        for (int i = 0;; ++i) {
            const int kb = g + NGROUP * i;
            if (kb >= nkb_conv) break;
            __syncwarp();  // every lane is done with the slot the next copy overwrites
            issue(i + RING - 1);
            cp_async_wait<RING - 1>();
            __syncwarp();  // all lanes' copies of k-block kb have landed
            const uint8_t* slot = ringp + (size_t)(i % RING) * SLOT_BYTES;
            const int s = kb % S16;
            const uint32_t ph = (uint32_t)(kb / S16) & 1u;
            if (is_a) {
                uint4 cur[4];
                const uint32_t sw = (uint32_t)(lane >> 1) & 3u;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    cur[c] = *reinterpret_cast<const uint4*>(slot + lane * 64 + ((c ^ sw) << 4));
                int rsp[4] = {0, 0, 0, 0};  // four independent dp4a chains
                uint32_t h[32];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    rsp[0] = abs_sum4(cur[c].x, rsp[0]);
                    rsp[1] = abs_sum4(cur[c].y, rsp[1]);
                    rsp[2] = abs_sum4(cur[c].z, rsp[2]);
                    rsp[3] = abs_sum4(cur[c].w, rsp[3]);
                    s8x4_to_f16(cur[c].x, h[8 * c + 0], h[8 * c + 1]);
                    s8x4_to_f16(cur[c].y, h[8 * c + 2], h[8 * c + 3]);
                    s8x4_to_f16(cur[c].z, h[8 * c + 4], h[8 * c + 5]);
                    s8x4_to_f16(cur[c].w, h[8 * c + 6], h[8 * c + 7]);
                }
                const int rs = (rsp[0] + rsp[1]) + (rsp[2] + rsp[3]);
                if (!tc::mbar_wait_warp(empty_bar(s), ph ^ 1u, abort_flag)) break;
                tc::tc_fence_after();
                tc::tmem_st32(tmem + ((uint32_t)(32 * q) << 16) + A_COL0 + 32u * (uint32_t)s, h);
                // row sums: the odd CTA's go to the even CTA by st.async,
                // counted as transaction bytes on the even CTA's barrier
                const int trow = HM * (int)rank + 32 * q + lane;
                if (leader)
                    rowsum[s * BM + trow] = (uint32_t)rs;
                else
                    tc::st_async_b32(rowsum_l0 + 4u * (uint32_t)(s * BM + trow), (uint32_t)rs, full_bar_l0 + 8u * s);
                tc::tmem_wait_st();
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (leader)
                        tc::mbar_arrive(full_bar(s));
                    else
                        tc::mbar_arrive_expect_tx_remote(full_bar_l0 + 8u * s, 32u * 4u);
                }
            } else {
                uint32_t hb[4][8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 v = *reinterpret_cast<const uint4*>(slot + (8 * j + (lane >> 2)) * 64 + 16 * cc);
                    s8x4_to_f16(v.x, hb[j][0], hb[j][1]);
                    s8x4_to_f16(v.y, hb[j][2], hb[j][3]);
                    s8x4_to_f16(v.z, hb[j][4], hb[j][5]);
                    s8x4_to_f16(v.w, hb[j][6], hb[j][7]);
                }
                if (!tc::mbar_wait_warp(empty_bar(s), ph ^ 1u, abort_flag)) break;
                uint8_t* tS = tiles + (size_t)s * B16_BYTES;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    *reinterpret_cast<uint4*>(tS + soff[j]) = make_uint4(hb[j][0], hb[j][1], hb[j][2], hb[j][3]);
                    *reinterpret_cast<uint4*>(tS + (soff[j] ^ 16u)) =
                        make_uint4(hb[j][4], hb[j][5], hb[j][6], hb[j][7]);
                }
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (leader)
                        tc::mbar_arrive(full_bar(s));
                    else
                        tc::mbar_arrive_remote(full_bar_l0 + 8u * s);
                }
            }
        }
        cp_async_wait<0>();
    } else if (warp == MMA_WARP) {
        // ---------------------------------------------------------- MMA issuer (even CTA)
        if (leader) {
            const uint32_t IDESC = p.idesc;
            const uint32_t tiles_addr = tc::smem_addr(tiles);
            const uint32_t peer_misc1 = tc::mapa(tc::smem_addr((const void*)&misc[1]), 1);
            const uint32_t peer_ev = tc::mapa(ev_bar, 1);
            bool started = false;
            uint32_t ndrain = 0;
            bool ok = true;
            // announce an event (drain or final) to the epilogue warps of both CTAs
            auto post_event = [&](uint32_t type) {
                misc[1] = type;
                tc::st_cluster_u32(peer_misc1, type);  // ordered before the release below
                tc::mbar_arrive(ev_bar);
                tc::mbar_arrive_cluster(peer_ev);
                tc::mma_commit_pair(acc_full, 3);
            };
            for (int kb = 0; kb < nkb && ok; ++kb) {
                const int s = kb % S16;
                const uint32_t ph = (uint32_t)(kb / S16) & 1u;
                // the monitor's word for this stage: operands full, drain or not
                if (!tc::mbar_wait_warp(dec_bar(s), ph, abort_flag)) {
                    ok = false;
                    break;
                }
                if (drain_dec[s] != 0) {
                    if (tc::elect_one()) post_event(EV_DRAIN);
                    __syncwarp();
                    if (!tc::mbar_wait_cluster_warp(acc_empty, ndrain & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    ++ndrain;
                    started = false;
                }
                tc::tc_fence_after();
                const uint64_t bd = tc::desc_sw128(tiles_addr + (uint32_t)s * B16_BYTES);
                const uint32_t a_tm = tmem + A_COL0 + 32u * (uint32_t)s;
                if (tc::elect_one()) {
#pragma unroll
                    for (int j = 0; j < BK / 16; ++j)  // 16 k (8 TMEM columns, 32 B of B rows) per MMA
                        tc::mma_f16_pair_tmem_a(tmem + ACC_COL, a_tm + 8u * j, bd + 2 * j, IDESC,
                                                (started || j > 0) ? 1u : 0u);
                    tc::mma_commit_pair(empty_bar(s), 3);
                }
                started = true;
                __syncwarp();
            }
            if (tc::elect_one()) {
                post_event(ok ? EV_FINAL : 0u);
                tc::mma_commit_pair(done_bar, 3);
            }
            __syncwarp();
        }
        tc::mbar_wait_drain(done_bar, 0, leader ? 0u : kIdleSleepNs);
        __syncwarp();
    } else if (warp == MON_WARP) {
        // ---------------------------------------------------------- drain monitor (even CTA)
        if (leader) {
            uint32_t S[8] = {0, 0, 0, 0, 0, 0, 0, 0};  // running sum|qx| of rows 8 lane .. 8 lane + 7
            uint32_t smax = 0;                          // max over the 256 rows of S
            bool started = false;
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = kb % S16;
                const uint32_t ph = (uint32_t)(kb / S16) & 1u;
                if (!tc::mbar_wait_warp(full_bar(s), ph, abort_flag)) break;
                // the stage's row sums, read before the stage is handed on
                const uint4 b0 = *reinterpret_cast<const uint4*>(rowsum + s * BM + lane * 8);
                const uint4 b1 = *reinterpret_cast<const uint4*>(rowsum + s * BM + lane * 8 + 4);
                // drain first if a row could pass the limit with this k-block
                const bool drain = started && smax > ROWSUM_LIMIT - KB_SUM_MAX;
                if (lane == 0) drain_dec[s] = drain ? 1u : 0u;
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(dec_bar(s));
                const uint32_t B[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
                uint32_t mx = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    S[i] = (drain ? 0u : S[i]) + B[i];
                    mx = max(mx, S[i]);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                smax = mx;
                started = true;
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- drains + epilogue (own rows)
        const int q = warp & 3;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const int64_t m = mh + 32 * q + lane;
        const int64_t trow = (int64_t)HM * rank + 32 * q + lane;  // row within the tile
        uint32_t ndrain = 0;
        // this thread's row of the drained sums, staged in the converters' rings
        // (idle once the final event is posted: every k-block has been
        // converted and consumed); 16-byte unit u of the row sits at u ^ (lane & 7)
        uint8_t* const srow = rings + (size_t)(32 * q + lane) * (BN * 4);
        const uint32_t srow_a = tc::smem_addr(srow);
        for (uint32_t ev = 0;; ++ev) {
            if (!tc::mbar_wait_cluster_warp(ev_bar, ev & 1u, abort_flag, kIdleSleepNs)) break;
            const uint32_t type = misc[1];
            // the final event after a drain: fetch the row's drained sums while
            // the last MMAs finish, instead of one global round trip per 16 columns
            const bool staged = type == EV_FINAL && ndrain != 0 && m < p.M && n0 + BN <= p.N && dld % 4 == 0;
            if (staged) {
                const int32_t* src = dtile + trow * dld;
#pragma unroll 8
                for (int u = 0; u < BN / 4; ++u) cp_async16(srow_a + (uint32_t)((u ^ (lane & 7)) << 4), src + 4 * u);
                cp_async_commit();
            }
            if (!tc::mbar_wait_warp(acc_full, ev & 1u, abort_flag)) {
                cp_async_wait<0>();
                break;
            }
            tc::tc_fence_after();
            if (staged) cp_async_wait<0>();
            if (type != EV_DRAIN && type != EV_FINAL) break;
            const float sxm = (type == EV_FINAL && m < p.M) ? p.sx[m] : 0.0f;
            // the next 16 columns' TMEM load is in flight while this chunk is
            // converted and stored
            uint32_t a[16];
            tc::tmem_ld16(tmem + lane_base + ACC_COL, a);
            for (int c = 0; c < BN; c += 16) {
                __syncwarp();
                tc::tmem_wait_ld();
                int tot[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) tot[j] = __float2int_rn(__uint_as_float(a[j]));
                if (c + 16 < BN) tc::tmem_ld16(tmem + lane_base + ACC_COL + c + 16, a);
                if (m >= p.M) continue;
                const int64_t nb = n0 + c;
                if (nb >= p.N) continue;
                int32_t* dp = dtile + trow * dld + c;
                const bool full = (nb + 16 <= p.N) && (p.N % 4 == 0);
                if (staged) {
#pragma unroll
                    for (int j = 0; j < 16; j += 4) {
                        const int u = (c + j) >> 2;
                        const int4 v = *reinterpret_cast<const int4*>(srow + ((u ^ (lane & 7)) << 4));
                        tot[j] += v.x;
                        tot[j + 1] += v.y;
                        tot[j + 2] += v.z;
                        tot[j + 3] += v.w;
                    }
                } else if (ndrain) {
                    if (full) {
#pragma unroll
                        for (int j = 0; j < 16; j += 4) {
                            int4 v = *reinterpret_cast<const int4*>(dp + j);
                            tot[j] += v.x;
                            tot[j + 1] += v.y;
                            tot[j + 2] += v.z;
                            tot[j + 3] += v.w;
                        }
                    } else {
                        for (int j = 0; j < 16; ++j)
                            if (nb + j < p.N) tot[j] += dp[j];
                    }
                }
                if (type == EV_DRAIN || split) {
                    if (full) {
#pragma unroll
                        for (int j = 0; j < 16; j += 4)
                            *reinterpret_cast<int4*>(dp + j) = make_int4(tot[j], tot[j + 1], tot[j + 2], tot[j + 3]);
                    } else {
                        for (int j = 0; j < 16; ++j)
                            if (nb + j < p.N) dp[j] = tot[j];
                    }
                } else {
                    store_row<16>(tot, m, nb, p.N, sxm, p.sw, p.y, p.yt, p.acc_out, p.add);
                }
            }
            if (type == EV_FINAL) break;
            ++ndrain;
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive_cluster(acc_empty_l0);
        }
    }

    tc::tc_fence_before();
    tc::cluster_sync();  // no MMA, remote arrival or remote store of the pair is still in flight
    if (warp == MMA_WARP) {
        tc::tc_fence_after();
        tc::tmem_dealloc_pair(tmem, TMEM_COLS);
    }
}

// Launch plan of k_w8a8_tc: weight rows per CTA and the split of the last,
// partial wave of tiles.
struct W8Plan {
    int bn;
    int64_t tiles, full_tiles, tail_tiles;
    int split;
};

static W8Plan w8_plan(int64_t M, int64_t N, int64_t K) {
    using namespace w8tc;
    W8Plan pl{};
    // Weight rows per CTA: the fewest waves of tiles over bn in {256, 224,
    // ..., 128}, larger bn on ties (measured: a CTA's time per k-block does not
    // shrink with bn, so only the wave count matters).
    const int sms = num_sms();
    const int64_t mt = ceil_div(M, BM);
    pl.bn = BN;
    int64_t best = INT64_MAX;
    for (int cand = BN; cand >= 128; cand -= 32) {
        const int64_t waves = ceil_div(mt * ceil_div(N, cand), sms);
        if (waves < best) {
            best = waves;
            pl.bn = cand;
        }
    }
    pl.tiles = mt * ceil_div(N, pl.bn);
    // The tiles of the last wave would leave SMs idle: cut each into `split`
    // K parts (2..4, at least 4 k-blocks each) when that still fits one wave.
    const int64_t tail = pl.tiles % sms;
    const int64_t nkb = ceil_div(K, BK);
    pl.split = 1;
    if (tail > 0) {
        int64_t sp = sms / tail;
        if (sp > 4) sp = 4;
        while (sp > 1 && nkb < 4 * sp) --sp;
        pl.split = (int)sp;
    }
    pl.tail_tiles = pl.split > 1 ? tail : 0;
    pl.full_tiles = pl.tiles - pl.tail_tiles;
    return pl;
}

// Co-resident clusters of k_w8a8_pair (pairs of SMs that can run at once).
static int w8p_clusters() {
    static int n = 0;
    if (n == 0) {
        int nc = 0;
        if (ensure_smem((const void*)k_w8a8_pair, (int)w8p::SMEM_BYTES) == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)(2 * num_sms()));
            cfg.blockDim = dim3(w8p::THREADS);
            cfg.dynamicSmemBytes = w8p::SMEM_BYTES;
            if (cudaOccupancyMaxActiveClusters(&nc, (const void*)k_w8a8_pair, &cfg) != cudaSuccess) nc = 0;
            (void)cudaGetLastError();
        }
        n = nc > 0 ? nc : num_sms() / 2;
    }
    return n;
}

// Launch plan of k_w8a8_pair: 256 x 256 tiles over the co-resident pairs, the
// last partial wave cut into K parts as for k_w8a8_tc.
static W8Plan w8p_plan(int64_t M, int64_t N, int64_t K) {
    using namespace w8p;
    W8Plan pl{};
    const int units = w8p_clusters();
    pl.bn = BN;
    pl.tiles = ceil_div(M, BM) * ceil_div(N, BN);
    const int64_t tail = pl.tiles % units;
    const int64_t nkb = ceil_div(K, BK);
    pl.split = 1;
    if (tail > 0) {
        int64_t sp = units / tail;
        if (sp > 4) sp = 4;
        while (sp > 1 && nkb < 4 * sp) --sp;
        pl.split = (int)sp;
    }
    pl.tail_tiles = pl.split > 1 ? tail : 0;
    pl.full_tiles = pl.tiles - pl.tail_tiles;
    return pl;
}

// INT32 tile that drains of the exact accumulation add into (touched only
// when a drain occurs), then the partial-sum slices of the split tail tiles.
static size_t w8a8_drain_bytes(int64_t M, int64_t N) { return ((size_t)M * N * sizeof(int32_t) + 15) & ~(size_t)15; }

static size_t w8_part_bytes(const W8Plan& pl) {
    return (size_t)pl.tail_tiles * pl.split * w8tc::BM * w8tc::BN * sizeof(int32_t);
}

// Enough for either tensor-core kernel (the choice can change between calls).
size_t w8a8_ws_bytes(int64_t M, int64_t N, int64_t K) {
    const size_t a = w8_part_bytes(w8_plan(M, N, K)), b = w8_part_bytes(w8p_plan(M, N, K));
    return w8a8_drain_bytes(M, N) + (a > b ? a : b);
}

// QLIN_W8A8_KERNEL: "mma" the legacy mma.sync kernel, "tc1" the single-CTA
// tensor-core kernel; otherwise the CTA-pair kernel.  Read on every call, so
// a process can compare the kernels (all give the same exact INT32 sums).
static int w8a8_kernel_choice() {
    const char* e = getenv("QLIN_W8A8_KERNEL");
    if (e && strcmp(e, "mma") == 0) return 1;
    if (e && strcmp(e, "tc1") == 0) return 0;
    return 2;
}

static cudaError_t run_w8a8_pair(const int8_t* qx, const float* sx, const int8_t* qw, const float* sw, int64_t M,
                                 int64_t N, int64_t K, void* y, int yt, int32_t* acc_out, void* ws, cudaStream_t st,
                                 const float* add) {
    using namespace w8p;
    cudaError_t e = ensure_smem((const void*)k_w8a8_pair, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const W8Plan pl = w8p_plan(M, N, K);
    W8TcArgs a;
    a.sx = sx;
    a.sw = sw;
    a.M = M;
    a.N = N;
    a.K = K;
    a.y = y;
    a.yt = yt;
    a.acc_out = acc_out;
    a.add = add;
    a.drain = reinterpret_cast<int32_t*>(ws);
    a.part = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(ws) + w8a8_drain_bytes(M, N));
    a.full_tiles = pl.full_tiles;
    a.tail_split = pl.split;
    a.num_m_tiles = (int)ceil_div(M, BM);
    a.bn = BN;
    a.idesc = tc::idesc_f16(BM, BN, false);
    const int64_t clusters = pl.full_tiles + pl.tail_tiles * pl.split;
    k_w8a8_pair<<<(unsigned)(2 * clusters), THREADS, SMEM_BYTES, st>>>(qx, qw, a);
    if ((e = cudaGetLastError()) != cudaSuccess || pl.tail_tiles == 0) return e;
    const int64_t work = pl.tail_tiles * BM * (BN / 16);
    k_w8a8_tail<<<(unsigned)ceil_div(work, 256), 256, 0, st>>>(a, (int)pl.tail_tiles);
    return cudaGetLastError();
}

cudaError_t run_gemm_w8a8(const int8_t* qx, const float* sx, const int8_t* qw, const float* sw, int64_t M, int64_t N,
                          int64_t K, void* y, int yt, int32_t* acc_out, void* ws, cudaStream_t st, const float* add) {
    const int choice = w8a8_kernel_choice();
    // With an addend (LLM.int8()'s outlier products) the epilogue reads an
    // fp32 tile per output tile; the single-CTA kernel needs fewer waves for
    // it (measured 381 us against 424 us at 2048 x 11008 x 4096).
    if (choice == 2 && !add) return run_w8a8_pair(qx, sx, qw, sw, M, N, K, y, yt, acc_out, ws, st, add);
    if (choice == 1 && !add) {
        using namespace w8;
        size_t smem = (size_t)2 * STAGES * TILE_BYTES;
        cudaError_t e = ensure_smem((const void*)k_w8a8_mma, (int)smem);
        if (e != cudaSuccess) return e;
        dim3 grid((unsigned)ceil_div(N, BN), (unsigned)ceil_div(M, BM));
        k_w8a8_mma<<<grid, THREADS, smem, st>>>(qx, sx, qw, sw, M, N, K, y, yt, acc_out);
        return cudaGetLastError();
    }
    using namespace w8tc;
    PFN_encodeTiled enc = encode_tiled_fn();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap ta, tb;
    cuuint64_t gda[2] = {(cuuint64_t)K, (cuuint64_t)M};
    cuuint64_t gdb[2] = {(cuuint64_t)K, (cuuint64_t)N};
    cuuint64_t gstride[1] = {(cuuint64_t)K};
    const W8Plan pl = w8_plan(M, N, K);
    const int bn = pl.bn;
    cuuint32_t boxa[2] = {BK, BM}, boxb[2] = {BK, (cuuint32_t)bn};
    cuuint32_t estride[2] = {1, 1};
    if (enc(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(qx), gda, gstride, boxa, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    if (enc(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(qw), gdb, gstride, boxb, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    cudaError_t e = ensure_smem((const void*)k_w8a8_tc, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    W8TcArgs a;
    a.sx = sx;
    a.sw = sw;
    a.M = M;
    a.N = N;
    a.K = K;
    a.y = y;
    a.yt = yt;
    a.acc_out = acc_out;
    a.add = add;
    a.drain = reinterpret_cast<int32_t*>(ws);
    a.part = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(ws) + w8a8_drain_bytes(M, N));  // 16-byte aligned
    a.full_tiles = pl.full_tiles;
    a.tail_split = pl.split;
    a.num_m_tiles = (int)ceil_div(M, BM);
    a.bn = bn;
    a.idesc = tc::idesc_f16(128, bn, false);
    const int64_t ctas = pl.full_tiles + pl.tail_tiles * pl.split;
    k_w8a8_tc<<<(unsigned)ctas, THREADS, SMEM_BYTES, st>>>(ta, tb, a);
    if ((e = cudaGetLastError()) != cudaSuccess || pl.tail_tiles == 0) return e;
    const int64_t work = pl.tail_tiles * BM * (bn / 16);  // < 2^31: tail tiles < SMs
    k_w8a8_tail<<<(unsigned)ceil_div(work, 256), 256, 0, st>>>(a, (int)pl.tail_tiles);
    return cudaGetLastError();
}

}  // namespace qlin
