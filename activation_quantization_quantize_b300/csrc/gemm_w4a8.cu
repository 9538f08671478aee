// gemm_w4a8.cu -- group-wise INT4 weights x per-token INT8 activations.
//
// Method ("第11章 模型量化与压缩" 11.4.5 step 6 -- integer GEMM with INT32
// accumulation, then the scales -- and 11.9.7 / 11.10.2: AWQ-style INT4
// weights combined with SmoothQuant INT8 activations give W4A8).  The weight
// is the packed INT4 blob of qlin_pack_w4 (groups of g consecutive k with a
// binary16 scale and a 4-bit zero point each); the activations are per-token
// INT8 codes qx with binary32 scales sx.  Because every group has its own
// scale, the integer sums are kept per group:
//     acc_g[m,n] = sum_{k in g} qx[m,k] * (q[n,k] - z[n,g])     (exact int32)
//     y[m,n]     = sx[m] * sum_g s[n,g] * acc_g[m,n]            (binary32)
//
// k_w4a8_gemv_dp (M = 1, 2): the same streaming with dp4a dot products on
// the integer pipe.
// k_w4a8_gemv (M <= 16 per CTA row of token tiles): legacy integer MMAs
// (mma.sync m16n8k32, u8 weights x s8 activations).  The packed nibbles are
// used as unsigned codes u (q = u for UINT4, u - 8 for INT4), so
//     sum_k qx (u - z) = sum_k qx u - z * sum_k qx
// and the weight operand needs no arithmetic beyond two masks and a shift per
// word.  The packed layout's k order (lane (g, t), word j holds rows g and g+8
// at k = 16t + 4j + {0, 2, 1, 3} after the masks) is matched by one byte
// permute of each activation word; the dot product does not depend on the
// order of k as long as both operands use the same one.
#include "qlin_common.cuh"
#include "qlin_internal.h"
#include "tc_ptx.cuh"

namespace qlin {

// D (s32, 16x8) += A (u8, 16x32, row) * B (s8, 32x8, col).
__device__ __forceinline__ void mma_u8s8_16832(int c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Sum of the four signed bytes of w.
__device__ __forceinline__ int sum_s8x4(uint32_t w, int acc) { return __dp4a((int)w, 0x01010101, acc); }

struct W4A8Args {
    const int8_t* qx;
    const float* sx;
    const uint8_t* blob;
    qlin_w4_header h;
    int64_t M;
    void* y;
    int yt;
    int32_t* acc_out;  // NULL or [K/g][M][N] exact per-group sums (zeroed by the launcher)
};

constexpr int A8_D = 6;  // cp.async ring depth (chunks of 64 k) per warp

template <int NT>
constexpr int a8_gemv_smem_bytes() {
    return 8 * A8_D * NT * (512 + 256);
}

// CTA: 8 warps; blockIdx.x covers NT 16-row packed tiles, blockIdx.y one
// group of MT*8 tokens.  Warp w takes the contiguous 1/8 of the K chunks.  A
// group cut between two warps gives each warp a partial (exact) integer sum
// that it scales on its own; the 8 warps' binary32 totals are added in a
// fixed order at the end, so results do not depend on timing.
template <int MT, int NT, int G>
__global__ void __launch_bounds__(256, 2) k_w4a8_gemv(W4A8Args a) {
    extern __shared__ __align__(16) uint8_t a8_smem[];
    tc::pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, t = lane & 3;
    const int64_t K = a.h.K, N = a.h.N, nchunk = K / 64, ngr = K / G;
    const int64_t nt0 = (int64_t)blockIdx.x * NT;
    const int64_t m_base = (int64_t)blockIdx.y * (MT * 8);
    const int64_t c_begin = nchunk * warp / 8, c_end = nchunk * (warp + 1) / 8;
    const bool asym = a.h.asym != 0;
    constexpr int CPG = G >= 64 ? G / 64 : 1;  // chunks per group (G = 32: two groups per chunk)

    const uint32_t cring = tc::smem_addr(a8_smem + warp * (A8_D * NT * 512) + lane * 16);
    const uint32_t mring = tc::smem_addr(a8_smem + 8 * A8_D * NT * 512 + warp * (A8_D * NT * 256) + lane * 8);
    const uint8_t* cring_p = a8_smem + warp * (A8_D * NT * 512) + lane * 16;
    const uint8_t* mring_p = a8_smem + 8 * A8_D * NT * 512 + warp * (A8_D * NT * 256) + lane * 8;
    const uint8_t* gcodes = a.blob + a.h.codes_off + lane * 16;
    const uint8_t* gscales = a.blob + a.h.scales_off + gq * 4;
    const uint8_t* gzeros = a.blob + a.h.zeros_off + (gq & 4);
    const int zshift = 8 * (gq & 3);

    // codes and group words of chunk kc for the NT tiles: each lane copies its
    // own 16 code bytes and the group words of its k (group (64 kc + 16 t) / G)
    auto issue = [&](int slot, int64_t kc) {
        if (kc < c_end) {
            const int64_t gi = (kc * 64 + 16 * t) / G;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const int sl = slot * NT + n;
                cp_async16(cring + sl * 512, gcodes + ((nt0 + n) * nchunk + kc) * 512);
                cp_async4(mring + sl * 256, gscales + ((nt0 + n) * ngr + gi) * 32);
                if (asym) cp_async4(mring + sl * 256 + 4, gzeros + ((nt0 + n) * ngr + gi) * 8);
            }
        }
        cp_async_commit();
    };
    // token rows of this lane's activation loads (rows past M read row M-1;
    // their outputs are dropped)
    const int8_t* xr[MT];
#pragma unroll
    for (int u = 0; u < MT; ++u) {
        int64_t m = m_base + u * 8 + gq;
        if (m >= a.M) m = a.M - 1;
        xr[u] = a.qx + m * K + 16 * t;
    }
    auto load_x = [&](uint4 (&xb)[MT], int64_t kc) {
#pragma unroll
        for (int u = 0; u < MT; ++u) xb[u] = __ldg(reinterpret_cast<const uint4*>(xr[u] + kc * 64));
    };

    int acc[NT][MT][4];
    float tot[NT][MT][4];
    int S[MT];  // running sum of this lane's token's codes over the current group (quad-reduced)
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int u = 0; u < MT; ++u)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[n][u][e] = 0;
                tot[n][u][e] = 0.0f;
            }
#pragma unroll
    for (int u = 0; u < MT; ++u) S[u] = 0;

    // Scale the exact sums of one group into tot and restart them.  zw / sw:
    // the zero-point byte (z(g) | z(g+8) << 4, or 0x88 for INT4) and the
    // binary16 scale pair of rows (gq, gq+8) of this group; Sg: the token sums
    // of this lane's quad token gq.  The C fragment of lane (gq, t) holds
    // tokens 2t, 2t+1 of each 8-token tile.
    auto finish_group = [&](int n, int u, uint32_t zw, uint32_t sw2, int Sg, int64_t gi) {
        const int S0 = __shfl_sync(0xffffffffu, Sg, (2 * t) * 4);
        const int S1 = __shfl_sync(0xffffffffu, Sg, (2 * t + 1) * 4);
        const int zg = (int)(zw & 0xFu), zh = (int)((zw >> 4) & 0xFu);
        __half2 h2 = *reinterpret_cast<__half2*>(&sw2);
        const float2 sf = __half22float2(h2);
        const int c0 = acc[n][u][0] - zg * S0, c1 = acc[n][u][1] - zg * S1;
        const int c2 = acc[n][u][2] - zh * S0, c3 = acc[n][u][3] - zh * S1;
        if (a.acc_out) {
            const int64_t ta = m_base + u * 8 + 2 * t, tb = ta + 1;
            const int64_t ra = (nt0 + n) * 16 + gq, rb = ra + 8;
            int32_t* base = a.acc_out + gi * a.M * N;
            if (ta < a.M) {
                atomicAdd(base + ta * N + ra, c0);
                atomicAdd(base + ta * N + rb, c2);
            }
            if (tb < a.M) {
                atomicAdd(base + tb * N + ra, c1);
                atomicAdd(base + tb * N + rb, c3);
            }
        }
        tot[n][u][0] = fmaf(sf.x, (float)c0, tot[n][u][0]);
        tot[n][u][1] = fmaf(sf.x, (float)c1, tot[n][u][1]);
        tot[n][u][2] = fmaf(sf.y, (float)c2, tot[n][u][2]);
        tot[n][u][3] = fmaf(sf.y, (float)c3, tot[n][u][3]);
        acc[n][u][0] = acc[n][u][1] = acc[n][u][2] = acc[n][u][3] = 0;
    };

#pragma unroll 1
    for (int i = 0; i < A8_D - 1; ++i) issue(i, c_begin + i);
    // weights before the wait, activations, scales and outputs after it (as in
    // the W4A16 decode kernels; back to back at 8192 x 28672, M = 8: 50.0 ->
    // 46.7 us)
    tc::pdl_wait();
    uint4 xn[MT];
    if (c_begin < c_end) load_x(xn, c_begin);

    int slot = 0;
    for (int64_t kc = c_begin; kc < c_end; ++kc) {
        issue(slot == 0 ? A8_D - 1 : slot - 1, kc + A8_D - 1);
        uint4 xw[MT];
#pragma unroll
        for (int u = 0; u < MT; ++u) xw[u] = xn[u];
        if (kc + 1 < c_end) load_x(xn, kc + 1);
        // activation words in the weights' k order (bytes 0, 2, 1, 3), and
        // this lane's part of its token's group sums
        uint32_t b[MT][4];
        int p[MT];
#pragma unroll
        for (int u = 0; u < MT; ++u) {
            const uint32_t w4[4] = {xw[u].x, xw[u].y, xw[u].z, xw[u].w};
            int sacc = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                b[u][j] = __byte_perm(w4[j], 0, 0x3120);
                sacc = sum_s8x4(w4[j], sacc);
            }
            p[u] = sacc;
        }
        cp_async_wait<A8_D - 1>();
        if (G >= 64) {
#pragma unroll
            for (int u = 0; u < MT; ++u) {
                int q = p[u] + __shfl_xor_sync(0xffffffffu, p[u], 1);
                q += __shfl_xor_sync(0xffffffffu, q, 2);
                S[u] += q;
            }
        }
        const bool group_end = (G <= 64) || ((kc + 1) % CPG == 0) || (kc + 1 == c_end);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const int sl = slot * NT + n;
            const uint4 cw = *reinterpret_cast<const uint4*>(cring_p + sl * 512);
            const uint2 mw = *reinterpret_cast<const uint2*>(mring_p + sl * 256);
            const uint32_t wd[4] = {cw.x, cw.y, cw.z, cw.w};
            uint32_t lo[4], hi[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                lo[j] = wd[j] & 0x0F0F0F0Fu;          // row gq,   k order (0, 2, 1, 3)
                hi[j] = (wd[j] >> 4) & 0x0F0F0F0Fu;   // row gq+8
            }
            const uint32_t zb = asym ? (mw.y >> zshift) & 0xFFu : 0x88u;
            if (G >= 64) {
#pragma unroll
                for (int u = 0; u < MT; ++u) {
                    mma_u8s8_16832(acc[n][u], lo[0], hi[0], lo[1], hi[1], b[u][0], b[u][1]);
                    mma_u8s8_16832(acc[n][u], lo[2], hi[2], lo[3], hi[3], b[u][2], b[u][3]);
                }
                if (group_end) {
                    const int64_t gi = (kc * 64) / G;
#pragma unroll
                    for (int u = 0; u < MT; ++u) finish_group(n, u, zb, mw.x, S[u], gi);
                }
            } else {
                // G = 32: lanes t < 2 hold group 2 kc, lanes t >= 2 group 2 kc + 1;
                // one MMA pair per group, the other half's lanes supplying zeros
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const bool mine = (t >> 1) == half;
                    uint32_t al[4], ah[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        al[j] = mine ? lo[j] : 0u;
                        ah[j] = mine ? hi[j] : 0u;
                    }
                    const int src = gq * 4 + 2 * half;  // a lane holding this group's words
                    const uint32_t zg = __shfl_sync(0xffffffffu, zb, src);
                    const uint32_t sg = __shfl_sync(0xffffffffu, mw.x, src);
#pragma unroll
                    for (int u = 0; u < MT; ++u) {
                        mma_u8s8_16832(acc[n][u], al[0], ah[0], al[1], ah[1], b[u][0], b[u][1]);
                        mma_u8s8_16832(acc[n][u], al[2], ah[2], al[3], ah[3], b[u][2], b[u][3]);
                        int q = mine ? p[u] : 0;
                        q += __shfl_xor_sync(0xffffffffu, q, 1);
                        q += __shfl_xor_sync(0xffffffffu, q, 2);
                        finish_group(n, u, zg, sg, q, 2 * kc + half);
                    }
                }
            }
        }
        if (G >= 64 && group_end) {
#pragma unroll
            for (int u = 0; u < MT; ++u) S[u] = 0;
        }
        slot = slot + 1 == A8_D ? 0 : slot + 1;
    }
    cp_async_wait<0>();
    __syncthreads();

    // tot[n][u][e]: e = 0, 1 -> (row gq of tile n, tokens u*8 + 2t, +1); e = 2, 3 -> row gq+8
    float(*part)[NT * 16][16] = reinterpret_cast<float(*)[NT * 16][16]>(a8_smem);  // [warp][row][token]
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int u = 0; u < MT; ++u) {
            part[warp][n * 16 + gq][u * 8 + 2 * t] = tot[n][u][0];
            part[warp][n * 16 + gq][u * 8 + 2 * t + 1] = tot[n][u][1];
            part[warp][n * 16 + gq + 8][u * 8 + 2 * t] = tot[n][u][2];
            part[warp][n * 16 + gq + 8][u * 8 + 2 * t + 1] = tot[n][u][3];
        }
    __syncthreads();
    for (int i = threadIdx.x; i < NT * 16 * 16; i += blockDim.x) {
        const int row = i >> 4, tok = i & 15;
        const int64_t m = m_base + tok;
        if (tok < MT * 8 && m < a.M) {
            float s = 0.0f;
#pragma unroll
            for (int w = 0; w < 8; ++w) s += part[w][row][tok];
            const float v = a.sx[m] * s;
            const int64_t o = m * N + nt0 * 16 + row;
            if (a.yt == QLIN_BF16)
                reinterpret_cast<__nv_bfloat16*>(a.y)[o] = __float2bfloat16_rn(v);
            else
                reinterpret_cast<float*>(a.y)[o] = v;
        }
    }
}

// One or two tokens (MX): the m16n8k32 MMA would waste 7/8 of its work on
// absent tokens, so each lane takes dot products of its own 16 codes of rows
// gq and gq+8 with the activation bytes by dp4a (integer pipe, no tensor
// core), and the quad's four partial sums are added exactly at each group's
// end.  Same streaming ring, same group epilogue arithmetic.
template <int MX, int NT, int G>
__global__ void __launch_bounds__(256, 2) k_w4a8_gemv_dp(W4A8Args a) {
    extern __shared__ __align__(16) uint8_t a8_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, t = lane & 3;
    const int64_t K = a.h.K, N = a.h.N, nchunk = K / 64, ngr = K / G;
    const int64_t nt0 = (int64_t)blockIdx.x * NT;
    const int64_t c_begin = nchunk * warp / 8, c_end = nchunk * (warp + 1) / 8;
    const bool asym = a.h.asym != 0;
    constexpr int CPG = G >= 64 ? G / 64 : 1;

    const uint32_t cring = tc::smem_addr(a8_smem + warp * (A8_D * NT * 512) + lane * 16);
    const uint32_t mring = tc::smem_addr(a8_smem + 8 * A8_D * NT * 512 + warp * (A8_D * NT * 256) + lane * 8);
    const uint8_t* cring_p = a8_smem + warp * (A8_D * NT * 512) + lane * 16;
    const uint8_t* mring_p = a8_smem + 8 * A8_D * NT * 512 + warp * (A8_D * NT * 256) + lane * 8;
    const uint8_t* gcodes = a.blob + a.h.codes_off + lane * 16;
    const uint8_t* gscales = a.blob + a.h.scales_off + gq * 4;
    const uint8_t* gzeros = a.blob + a.h.zeros_off + (gq & 4);
    const int zshift = 8 * (gq & 3);

    auto issue = [&](int slot, int64_t kc) {
        if (kc < c_end) {
            const int64_t gi = (kc * 64 + 16 * t) / G;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const int sl = slot * NT + n;
                cp_async16(cring + sl * 512, gcodes + ((nt0 + n) * nchunk + kc) * 512);
                cp_async4(mring + sl * 256, gscales + ((nt0 + n) * ngr + gi) * 32);
                if (asym) cp_async4(mring + sl * 256 + 4, gzeros + ((nt0 + n) * ngr + gi) * 8);
            }
        }
        cp_async_commit();
    };
    const int8_t* xr[MX];
#pragma unroll
    for (int u = 0; u < MX; ++u) xr[u] = a.qx + (u < a.M ? u : a.M - 1) * K + 16 * t;

    int ag[NT][MX], ah[NT][MX];   // this lane's exact partial sums, rows gq and gq+8
    float tot[NT][MX][2];
    int S[MX];                    // this lane's part of the token's code sum over the group
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int u = 0; u < MX; ++u) {
            ag[n][u] = ah[n][u] = 0;
            tot[n][u][0] = tot[n][u][1] = 0.0f;
        }
#pragma unroll
    for (int u = 0; u < MX; ++u) S[u] = 0;

#pragma unroll 1
    for (int i = 0; i < A8_D - 1; ++i) issue(i, c_begin + i);
    uint4 xn[MX];
#pragma unroll
    for (int u = 0; u < MX; ++u)
        if (c_begin < c_end) xn[u] = __ldg(reinterpret_cast<const uint4*>(xr[u] + c_begin * 64));

    int slot = 0;
    for (int64_t kc = c_begin; kc < c_end; ++kc) {
        issue(slot == 0 ? A8_D - 1 : slot - 1, kc + A8_D - 1);
        uint32_t b[MX][4];
#pragma unroll
        for (int u = 0; u < MX; ++u) {
            const uint32_t w4[4] = {xn[u].x, xn[u].y, xn[u].z, xn[u].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                b[u][j] = __byte_perm(w4[j], 0, 0x3120);  // the weights' k order (0, 2, 1, 3)
                S[u] = sum_s8x4(w4[j], S[u]);
            }
        }
        if (kc + 1 < c_end) {
#pragma unroll
            for (int u = 0; u < MX; ++u) xn[u] = __ldg(reinterpret_cast<const uint4*>(xr[u] + (kc + 1) * 64));
        }
        cp_async_wait<A8_D - 1>();
        const bool group_end = (G <= 64) || ((kc + 1) % CPG == 0) || (kc + 1 == c_end);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const int sl = slot * NT + n;
            const uint4 cw = *reinterpret_cast<const uint4*>(cring_p + sl * 512);
            const uint2 mw = *reinterpret_cast<const uint2*>(mring_p + sl * 256);
            const uint32_t wd[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int lo = (int)(wd[j] & 0x0F0F0F0Fu);          // row gq: four codes in [0, 15]
                const int hi = (int)((wd[j] >> 4) & 0x0F0F0F0Fu);   // row gq + 8
#pragma unroll
                for (int u = 0; u < MX; ++u) {
                    ag[n][u] = __dp4a(lo, (int)b[u][j], ag[n][u]);
                    ah[n][u] = __dp4a(hi, (int)b[u][j], ah[n][u]);
                }
            }
            if (G == 32 || group_end) {
                const uint32_t zb = asym ? (mw.y >> zshift) & 0xFFu : 0x88u;
                const int zg = (int)(zb & 0xFu), zh = (int)((zb >> 4) & 0xFu);
                __half2 s2h = *reinterpret_cast<const __half2*>(&mw.x);
                const float2 sf = __half22float2(s2h);
#pragma unroll
                for (int u = 0; u < MX; ++u) {
                    int cg = ag[n][u] - zg * S[u], ch = ah[n][u] - zh * S[u];
                    // G = 32: lanes t < 2 and t >= 2 hold different groups
                    cg += __shfl_xor_sync(0xffffffffu, cg, 1);
                    ch += __shfl_xor_sync(0xffffffffu, ch, 1);
                    if (G != 32) {
                        cg += __shfl_xor_sync(0xffffffffu, cg, 2);
                        ch += __shfl_xor_sync(0xffffffffu, ch, 2);
                    }
                    if (a.acc_out && (t & (G == 32 ? 1 : 3)) == 0 && u < a.M) {
                        const int64_t gi = (kc * 64 + 16 * t) / G;
                        int32_t* base = a.acc_out + gi * a.M * N + (int64_t)u * N;
                        atomicAdd(base + (nt0 + n) * 16 + gq, cg);
                        atomicAdd(base + (nt0 + n) * 16 + gq + 8, ch);
                    }
                    tot[n][u][0] = fmaf(sf.x, (float)cg, tot[n][u][0]);
                    tot[n][u][1] = fmaf(sf.y, (float)ch, tot[n][u][1]);
                    ag[n][u] = ah[n][u] = 0;
                }
            }
        }
        if (G == 32 || group_end) {
#pragma unroll
            for (int u = 0; u < MX; ++u) S[u] = 0;
        }
        slot = slot + 1 == A8_D ? 0 : slot + 1;
    }
    cp_async_wait<0>();
    __syncthreads();
    // G = 32: lanes t and t ^ 2 hold the two groups of a chunk -- add them
    float(*part)[NT * 16][2] = reinterpret_cast<float(*)[NT * 16][2]>(a8_smem);  // [warp][row][token]
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int u = 0; u < MX; ++u) {
            float g0 = tot[n][u][0], g1 = tot[n][u][1];
            if (G == 32) {
                g0 += __shfl_xor_sync(0xffffffffu, g0, 2);
                g1 += __shfl_xor_sync(0xffffffffu, g1, 2);
            }
            if (t == 0) {
                part[warp][n * 16 + gq][u] = g0;
                part[warp][n * 16 + gq + 8][u] = g1;
            }
        }
    __syncthreads();
    for (int i = threadIdx.x; i < NT * 16 * MX; i += blockDim.x) {
        const int row = i / MX, tok = i % MX;
        if (tok < a.M) {
            float s = 0.0f;
#pragma unroll
            for (int w = 0; w < 8; ++w) s += part[w][row][tok];
            const float v = a.sx[tok] * s;
            const int64_t o = (int64_t)tok * N + nt0 * 16 + row;
            if (a.yt == QLIN_BF16)
                reinterpret_cast<__nv_bfloat16*>(a.y)[o] = __float2bfloat16_rn(v);
            else
                reinterpret_cast<float*>(a.y)[o] = v;
        }
    }
}

template <int MX, int NT, int G>
static cudaError_t launch_a8_gemv_dp(const W4A8Args& a, cudaStream_t st) {
    constexpr int smem = a8_gemv_smem_bytes<NT>();
    cudaError_t e = ensure_smem((const void*)k_w4a8_gemv_dp<MX, NT, G>, smem);
    if (e != cudaSuccess) return e;
    // (launched without programmatic dependent launch: back to back, letting
    // the next call start early measured slower for this kernel, 41.8 -> 54.6
    // us at 8192 x 28672, M = 1)
    k_w4a8_gemv_dp<MX, NT, G><<<(unsigned)(a.h.N / (16 * NT)), 256, smem, st>>>(a);
    return cudaGetLastError();
}

template <int MX, int NT>
static cudaError_t launch_a8_gemv_dp_g(const W4A8Args& a, cudaStream_t st) {
    switch (a.h.group) {
    case 32: return launch_a8_gemv_dp<MX, NT, 32>(a, st);
    case 64: return launch_a8_gemv_dp<MX, NT, 64>(a, st);
    default: return launch_a8_gemv_dp<MX, NT, 128>(a, st);
    }
}

template <int MT, int NT, int G>
static cudaError_t launch_a8_gemv(const W4A8Args& a, unsigned mgroups, cudaStream_t st) {
    constexpr int smem = a8_gemv_smem_bytes<NT>();
    static_assert(smem >= 8 * NT * 16 * 16 * 4, "reduction tile must fit in the ring");
    cudaError_t e = ensure_smem((const void*)k_w4a8_gemv<MT, NT, G>, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(k_w4a8_gemv<MT, NT, G>, dim3((unsigned)(a.h.N / (16 * NT)), mgroups), dim3(256), smem, st, a);
}

template <int MT, int NT>
static cudaError_t launch_a8_gemv_g(const W4A8Args& a, unsigned mgroups, cudaStream_t st) {
    switch (a.h.group) {
    case 32: return launch_a8_gemv<MT, NT, 32>(a, mgroups, st);
    case 64: return launch_a8_gemv<MT, NT, 64>(a, mgroups, st);
    default: return launch_a8_gemv<MT, NT, 128>(a, mgroups, st);
    }
}

size_t w4a8_ws_bytes(int64_t M, int64_t N, int64_t K) {
    (void)M;
    (void)N;
    (void)K;
    return 0;
}

cudaError_t run_gemm_w4a8(const int8_t* qx, const float* sx, const void* packed, const qlin_w4_header* h, int64_t M,
                          void* y, int yt, int32_t* acc_out, void* ws, cudaStream_t st) {
    (void)ws;
    W4A8Args a;
    a.qx = qx;
    a.sx = sx;
    a.blob = reinterpret_cast<const uint8_t*>(packed);
    a.h = *h;
    a.M = M;
    a.y = y;
    a.yt = yt;
    a.acc_out = acc_out;
    if (acc_out) {
        cudaError_t e = cudaMemsetAsync(acc_out, 0, (size_t)(h->K / h->group) * M * h->N * sizeof(int32_t), st);
        if (e != cudaSuccess) return e;
    }
    // Two 16-row tiles per CTA (one activation load serves both) when that
    // still leaves at least one CTA per SM.
    const bool two = (h->N % 32 == 0) && (h->N / 32 >= num_sms());
    if (M == 1) return two ? launch_a8_gemv_dp_g<1, 2>(a, st) : launch_a8_gemv_dp_g<1, 1>(a, st);
    if (M == 2) return two ? launch_a8_gemv_dp_g<2, 2>(a, st) : launch_a8_gemv_dp_g<2, 1>(a, st);
    if (M <= 8) return two ? launch_a8_gemv_g<1, 2>(a, 1, st) : launch_a8_gemv_g<1, 1>(a, 1, st);
    const unsigned mg = (unsigned)ceil_div(M, 16);
    return two ? launch_a8_gemv_g<2, 2>(a, mg, st) : launch_a8_gemv_g<2, 1>(a, mg, st);
}

}  // namespace qlin
