// gemm_w4a16.cu -- group-wise INT4 weights x bf16 activations.
//
// Method ("第11章 模型量化与压缩" 11.1.6, INT4 per-group worked case): the weight
// W [N x K] is stored as 4-bit codes in row-wise groups of g with a binary16
// scale (and, for asymmetric codes, a 4-bit zero point) per group; at
// inference each weight is dequantized to the 16-bit compute type,
// w^ = bf16(fl(s * (q - z))), and multiplied with bf16 activations, summing in
// binary32.
//
// Packed layout (version 1), built by k_pack_w4 from the canonical codes:
//   codes  [N/16][K/64][32 lanes][4 words]: the 16 x 64 tile of one warp-wide
//          chunk.  Lane l = 4*gq + t owns rows gq and gq+8 of the tile and the
//          16 consecutive k = 16*t .. 16*t+15 of the chunk.  Word j of the lane
//          holds k = 16*t + 4*j + {0..3} of both rows, nibble layout
//            nib 0/4: row gq,   k+0/k+1     nib 1/5: row gq+8, k+0/k+1
//            nib 2/6: row gq,   k+2/k+3     nib 3/7: row gq+8, k+2/k+3
//          which is an m16n8k16 A fragment (a0..a7) of the k-permutation
//          "logical k (2t+e) <-> real 16t+4j+e, (2t+8+e) <-> real 16t+4j+2+e".
//          Nibble values are unsigned: q for UINT4, q+8 for symmetric INT4.
//   scales [N/16][K/g][16] binary16, rows in the order 0,8,1,9,...,7,15 so a
//          lane reads the (gq, gq+8) pair as one 32-bit word.
//   zeros  [N/16][K/g][8] bytes: byte i = z(row i) | z(row i+8) << 4 (asym only).
//
// The dequantization w^ = bf16_rn(s*d), d = u - z, is formed with packed bf16
// arithmetic: s = s_hi + s_lo with s_hi = bf16_rn(s); s_lo*d is exact in bf16
// (at most 2 + 4 significant bits), so fma.rn.bf16x2(d, s_hi, s_lo*d) rounds
// the exact product s*d once -- bit-identical to rounding fl(s*d).
#include <cuda.h>

#include <mutex>

#include "qlin_common.cuh"
#include "qlin_internal.h"
#include "tc_ptx.cuh"
#include "tma_map.h"

namespace qlin {

// ------------------------------------------------------------------ layout
void w4_layout(int64_t N, int64_t K, int group, int asym, qlin_w4_header* h) {
    auto up = [](uint64_t v) { return (v + 255) & ~(uint64_t)255; };
    h->magic = QLIN_W4_MAGIC;
    h->version = QLIN_W4_VERSION;
    h->N = N;
    h->K = K;
    h->group = group;
    h->asym = asym;
    uint64_t off = up(sizeof(qlin_w4_header));
    h->codes_off = off;
    off = up(off + (uint64_t)N * K / 2);
    h->scales_off = off;
    off = up(off + (uint64_t)N * (K / group) * 2);
    h->zeros_off = asym ? off : 0;
    if (asym) off = up(off + (uint64_t)(N / 16) * (K / group) * 8);
    h->total_bytes = off;
}

// ------------------------------------------------------------------ pack
// One thread per (n_tile, chunk, lane): gathers the 32 nibbles of its word set
// from the canonical row-major nibbles.
__global__ void k_pack_codes(const uint8_t* __restrict__ q, uint32_t* __restrict__ out, int64_t N, int64_t K,
                             int asym) {
    int64_t nchunk = K / 64;
    int64_t total = (N / 16) * nchunk * 32;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        int lane = (int)(i & 31);
        int64_t tile = i >> 5;  // n_tile * nchunk + chunk
        int64_t nt = tile / nchunk, kc = tile % nchunk;
        int gq = lane >> 2, t = lane & 3;
        int64_t r0 = nt * 16 + gq, r1 = r0 + 8;
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int64_t k = kc * 64 + 16 * t + 4 * j;
            uint32_t nib[8];
            // canonical: element c of row r at byte r*K/2 + c/2, low nibble for even c
            auto get = [&](int64_t r, int64_t c) -> uint32_t {
                uint8_t b = q[r * (K / 2) + c / 2];
                uint32_t v = (c & 1) ? (b >> 4) : (b & 0xF);
                return asym ? v : ((v + 8) & 0xF);  // two's complement -> offset binary
            };
            nib[0] = get(r0, k + 0);
            nib[4] = get(r0, k + 1);
            nib[1] = get(r1, k + 0);
            nib[5] = get(r1, k + 1);
            nib[2] = get(r0, k + 2);
            nib[6] = get(r0, k + 3);
            nib[3] = get(r1, k + 2);
            nib[7] = get(r1, k + 3);
            uint32_t v = 0;
#pragma unroll
            for (int p = 0; p < 8; ++p) v |= nib[p] << (4 * p);
            w[j] = v;
        }
        reinterpret_cast<uint4*>(out)[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

__global__ void k_pack_meta(const __half* __restrict__ s, const int32_t* __restrict__ z, __half* __restrict__ s_out,
                            uint8_t* __restrict__ z_out, int64_t N, int64_t ngr) {
    int64_t total = (N / 16) * ngr;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        int64_t nt = i / ngr, gi = i % ngr;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            s_out[i * 16 + 2 * r] = s[(nt * 16 + r) * ngr + gi];
            s_out[i * 16 + 2 * r + 1] = s[(nt * 16 + r + 8) * ngr + gi];
            if (z) {
                uint32_t z0 = (uint32_t)z[(nt * 16 + r) * ngr + gi] & 0xF;
                uint32_t z1 = (uint32_t)z[(nt * 16 + r + 8) * ngr + gi] & 0xF;
                z_out[i * 8 + r] = (uint8_t)(z0 | (z1 << 4));
            }
        }
    }
}

__global__ void k_write_header(qlin_w4_header h, qlin_w4_header* out) { *out = h; }

cudaError_t run_pack_w4(const void* q, const void* s_f16, const int32_t* z, const qlin_w4_header* h, void* packed,
                        cudaStream_t st) {
    uint8_t* base = reinterpret_cast<uint8_t*>(packed);
    int64_t N = h->N, K = h->K, ngr = K / h->group;
    int blocks = num_sms() * 4;
    k_write_header<<<1, 1, 0, st>>>(*h, reinterpret_cast<qlin_w4_header*>(base));
    k_pack_codes<<<blocks, 256, 0, st>>>(reinterpret_cast<const uint8_t*>(q),
                                         reinterpret_cast<uint32_t*>(base + h->codes_off), N, K, h->asym);
    k_pack_meta<<<blocks, 256, 0, st>>>(reinterpret_cast<const __half*>(s_f16), h->asym ? z : nullptr,
                                        reinterpret_cast<__half*>(base + h->scales_off),
                                        h->asym ? base + h->zeros_off : nullptr, N, ngr);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ dequant helpers
__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// Per-row dequantization constants: (s_hi, s_hi), (s_lo, s_lo), (128+z, 128+z).
struct RowDq {
    uint32_t shi2, slo2, c2;
};

__device__ __forceinline__ RowDq row_dq(float s, uint32_t z) {
    RowDq r;
    r.shi2 = f32x2_to_bf16x2(s, s);
    float shi = __uint_as_float(r.shi2 << 16);
    float slo = s - shi;  // exact
    r.slo2 = f32x2_to_bf16x2(slo, slo);
    r.c2 = 0x43004300u | z | (z << 16);  // bf16(128 + z) in both halves
    return r;
}

// Dequantize one word of 8 nibbles into the A fragment (a0a1, a2a3, a4a5, a6a7):
// pairs 0 and 2 use row gq (rg), pairs 1 and 3 row gq+8 (rh).
__device__ __forceinline__ void dq_word(uint32_t w, const RowDq& rg, const RowDq& rh, uint32_t a[4]) {
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        uint32_t v = ((w >> (4 * p)) & 0x000F000Fu) | 0x43004300u;  // bf16x2(128+u)
        const RowDq& R = (p & 1) ? rh : rg;
        uint32_t d = bf16x2_sub(v, R.c2);                            // u - z, exact
        uint32_t lo = bf16x2_mul(d, R.slo2);                         // exact
        a[p] = bf16x2_fma(d, R.shi2, lo);                            // bf16_rn(s*d)
    }
}

// A pure register-to-register operation (no volatile): the compiler may
// interleave independent MMAs with the surrounding dequantization.
__device__ __forceinline__ void mma_bf16_16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Raw dequantization words of lane (gq) for group gi of n-tile nt: the
// (row gq, row gq+8) binary16 scale pair and their packed zero points.
struct DqRaw {
    uint32_t s2;  // two binary16 scales
    uint32_t zb;  // z(row gq) | z(row gq+8) << 4, or 0x88 for symmetric codes
};

__device__ __forceinline__ DqRaw fetch_dq(const uint8_t* __restrict__ blob, const qlin_w4_header& h, int64_t nt,
                                          int64_t ngr, int64_t gi, int gq) {
    DqRaw d;
    d.s2 = __ldg(reinterpret_cast<const uint32_t*>(blob + h.scales_off) + (nt * ngr + gi) * 8 + gq);
    d.zb = h.asym ? (uint32_t)__ldg(blob + h.zeros_off + (nt * ngr + gi) * 8 + gq) : 0x88u;
    return d;
}

__device__ __forceinline__ void build_dq(const DqRaw& d, RowDq& rg, RowDq& rh) {
    uint32_t sw = d.s2;
    __half2 s2 = *reinterpret_cast<__half2*>(&sw);
    float2 sf = __half22float2(s2);
    rg = row_dq(sf.x, d.zb & 0xF);
    rh = row_dq(sf.y, (d.zb >> 4) & 0xF);
}

// Load the dequantization constants of lane (gq) for group gi of n-tile nt.
__device__ __forceinline__ void load_rowdq(const uint8_t* __restrict__ blob, const qlin_w4_header& h, int64_t nt,
                                           int64_t ngr, int64_t gi, int gq, RowDq& rg, RowDq& rh) {
    build_dq(fetch_dq(blob, h, nt, ngr, gi, gq), rg, rh);
}

// ------------------------------------------------------------------ GEMV (M <= 16)
// Two decode kernels share one structure: a CTA covers NT 16-row packed tiles;
// warp w covers a contiguous 1/8 of the k range for all NT tiles, so each
// activation load serves NT tiles.  Codes and group constants stream into a
// per-warp ring in shared memory with cp.async (each lane reads back only what
// it copied, so no barrier is needed).  m16n8k16 with W as A and X^T as B.  The
// 8 partial tiles are summed in a fixed order through shared memory, so the
// result does not depend on timing.  Each accumulation chain covers at most K/8.
//
// k_w4_gemv steps one 64-wide chunk at a time and serves any K % 64 == 0;
// k_w4_gemv2 (below) steps two chunks at a time and serves K % 128 == 0.
constexpr int GV_D = 6;  // ring depth in chunks

template <int NT>
constexpr int gemv_smem_bytes() {
    return 8 * GV_D * NT * (512 + 256);
}

template <int MT, int NT>  // MT: n8 token tiles (1: M <= 8, 2: M <= 16); NT: 16-row tiles per CTA
__global__ void __launch_bounds__(256, 2) k_w4_gemv(const __nv_bfloat16* __restrict__ x, const uint8_t* __restrict__ blob,
                                                    qlin_w4_header h, int64_t M, __nv_bfloat16* __restrict__ y) {
    extern __shared__ __align__(16) uint8_t gv_smem[];
    tc::pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, t = lane & 3;
    const int64_t K = h.K, nchunk = K / 64, ngr = K / h.group;
    const int gshift = __ffs(h.group) - 1;  // group is a power of two
    const int64_t nt0 = (int64_t)blockIdx.x * NT;
    const int64_t c_begin = nchunk * warp / 8, c_end = nchunk * (warp + 1) / 8;
    const bool asym = h.asym != 0;

    // per-lane ring slots: codes [GV_D][NT][32][16 B], group words [GV_D][NT][32][8 B]
    const uint32_t cring = tc::smem_addr(gv_smem + warp * (GV_D * NT * 512) + lane * 16);
    const uint32_t mring = tc::smem_addr(gv_smem + 8 * GV_D * NT * 512 + warp * (GV_D * NT * 256) + lane * 8);
    const uint8_t* gcodes = blob + h.codes_off + lane * 16;
    const uint8_t* gscales = blob + h.scales_off + gq * 4;
    const uint8_t* gzeros = blob + h.zeros_off + (gq & 4);
    const int zshift = 8 * (gq & 3);

    auto issue = [&](int slot, int64_t kc) {
        if (kc < c_end) {
            const int64_t gi = (kc * 64 + 16 * t) >> gshift;
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
    auto load_x = [&](uint4 (&xb)[MT][2], int64_t kc) {
        const int64_t k0 = kc * 64 + 16 * t;
#pragma unroll
        for (int u = 0; u < MT; ++u) {
            const int64_t m = u * 8 + gq;
            if (m < M) {
                const uint4* xp = reinterpret_cast<const uint4*>(x + m * K + k0);
                xb[u][0] = __ldg(xp);
                xb[u][1] = __ldg(xp + 1);
            } else {
                xb[u][0] = make_uint4(0, 0, 0, 0);
                xb[u][1] = make_uint4(0, 0, 0, 0);
            }
        }
    };

    float acc[NT][MT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int u = 0; u < MT; ++u)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[n][u][e] = 0.0f;

#pragma unroll
    for (int i = 0; i < GV_D - 1; ++i) issue(i, c_begin + i);
    // the weights are never written by a kernel that lets its dependents start
    // early, so their first copies are issued before the wait; the activations
    // (and y) are touched only after it
    tc::pdl_wait();
    uint4 xn[MT][2];
    if (c_begin < c_end) load_x(xn, c_begin);

    int slot = 0;
    for (int64_t kc = c_begin; kc < c_end; ++kc) {
        issue(slot == 0 ? GV_D - 1 : slot - 1, kc + GV_D - 1);
        uint4 xb[MT][2];
#pragma unroll
        for (int u = 0; u < MT; ++u) {
            xb[u][0] = xn[u][0];
            xb[u][1] = xn[u][1];
        }
        if (kc + 1 < c_end) load_x(xn, kc + 1);
        cp_async_wait<GV_D - 1>();
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const int sl = slot * NT + n;
            uint4 cw;
            uint32_t s2, zw = 0x88u;
            asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(cw.x), "=r"(cw.y), "=r"(cw.z), "=r"(cw.w)
                         : "r"(cring + sl * 512));
            if (asym) {
                asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(s2), "=r"(zw) : "r"(mring + sl * 256));
                zw = (zw >> zshift) & 0xFFu;
            } else {
                asm volatile("ld.shared.u32 %0, [%1];" : "=r"(s2) : "r"(mring + sl * 256));
            }
            DqRaw d;
            d.s2 = s2;
            d.zb = zw;
            RowDq rg, rh;
            build_dq(d, rg, rh);
            const uint32_t wd[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t a[4];
                dq_word(wd[j], rg, rh, a);
#pragma unroll
                for (int u = 0; u < MT; ++u) {
                    const uint32_t* xw = reinterpret_cast<const uint32_t*>(&xb[u][0]);
                    mma_bf16_16816(acc[n][u], a, xw[2 * j], xw[2 * j + 1]);
                }
            }
        }
        slot = slot + 1 == GV_D ? 0 : slot + 1;
    }
    cp_async_wait<0>();
    __syncthreads();

    // acc[n][u][e]: e=0,1 -> (row gq of tile n, tokens u*8 + 2t, +1); e=2,3 -> row gq+8
    float(*part)[NT * 16][16] = reinterpret_cast<float(*)[NT * 16][16]>(gv_smem);  // [warp][row][token]
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int u = 0; u < MT; ++u) {
            part[warp][n * 16 + gq][u * 8 + 2 * t] = acc[n][u][0];
            part[warp][n * 16 + gq][u * 8 + 2 * t + 1] = acc[n][u][1];
            part[warp][n * 16 + gq + 8][u * 8 + 2 * t] = acc[n][u][2];
            part[warp][n * 16 + gq + 8][u * 8 + 2 * t + 1] = acc[n][u][3];
        }
    __syncthreads();
    for (int i = threadIdx.x; i < NT * 16 * 16; i += blockDim.x) {
        const int row = i >> 4, tok = i & 15;
        if (tok < M && tok < MT * 8) {
            float s = 0.0f;
#pragma unroll
            for (int w = 0; w < 8; ++w) s += part[w][row][tok];
            y[(int64_t)tok * h.N + nt0 * 16 + row] = __float2bfloat16_rn(s);
        }
    }
}

// Pair-chunk variant for K % 128 == 0: one loop step covers the chunks
// (2p, 2p+1) of each of the NT tiles, so groups of >= 128 build their
// dequantization constants once per step (G128).  Codes and group words stream
// through a per-warp ring of GV_P steps; activations are read from L2 at the
// top of the step (rows >= M read row M-1: those token columns are dropped).
constexpr int GV_P = 3;  // ring depth in chunk pairs

template <int NT>
constexpr int gemv2_stage_bytes() {
    return NT * (1024 + 512);
}

template <int MT, int NT, bool G128>
__global__ void __launch_bounds__(256, 2) k_w4_gemv2(const __nv_bfloat16* __restrict__ x,
                                                     const uint8_t* __restrict__ blob, qlin_w4_header h, int64_t M,
                                                     __nv_bfloat16* __restrict__ y) {
    extern __shared__ __align__(16) uint8_t gv_smem[];
    tc::pdl_launch_dependents();
    constexpr int SB = gemv2_stage_bytes<NT>();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, t = lane & 3;
    const int64_t K = h.K, npair = K / 128, ngr = K / h.group;
    const int64_t nt0 = (int64_t)blockIdx.x * NT;
    const int64_t p_begin = npair * warp / 8, p_end = npair * (warp + 1) / 8;
    const bool asym = h.asym != 0;

    const uint32_t ring = tc::smem_addr(gv_smem) + warp * (GV_P * SB) + lane * 16;
    const uint8_t* ringp = gv_smem + warp * (GV_P * SB) + lane * 16;
    // Global streams of this lane, positioned at pair p_begin.  The group of
    // lane t in chunk 2p is (128 p + 16 t) / g; in chunk 2p+1 it is 64 / g
    // groups later (g = 32, 64).  Scale words are 32 B and zero words 8 B per
    // group of a tile.
    const int gpp = 128 / h.group;  // groups per pair: 1, 2 or 4
    const int64_t g0 = (p_begin * 128 + 16 * t) / h.group;
    const int sb_off = 32 * (gpp >> 1), zb_off = 8 * (gpp >> 1);
    const uint8_t* gc[NT];
    const uint8_t* gs[NT];
    const uint8_t* gz[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        gc[n] = blob + h.codes_off + ((nt0 + n) * (K / 64) + 2 * p_begin) * 512 + lane * 16;
        gs[n] = blob + h.scales_off + ((nt0 + n) * ngr + g0) * 32 + gq * 4;
        gz[n] = blob + h.zeros_off + ((nt0 + n) * ngr + g0) * 8 + (gq & 4);
    }
    const int zshift = 8 * (gq & 3);
    const __nv_bfloat16* xr[MT];
#pragma unroll
    for (int u = 0; u < MT; ++u) {
        const int64_t m = (u * 8 + gq) < M ? (u * 8 + gq) : M - 1;
        xr[u] = x + m * K + p_begin * 128 + 16 * t;
    }

    int64_t p_issue = p_begin;
    uint32_t s_issue = 0;
    auto issue = [&]() {
        if (p_issue < p_end) {
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const uint32_t cs = ring + s_issue + n * 1024;
                const uint32_t ms = ring + s_issue + NT * 1024 + n * 512;
                cp_async16(cs, gc[n]);
                cp_async16(cs + 512, gc[n] + 512);
                gc[n] += 1024;
                cp_async4(ms, gs[n]);
                if (asym) cp_async4(ms + 4, gz[n]);
                if (!G128) {
                    cp_async4(ms + 8, gs[n] + sb_off);
                    if (asym) cp_async4(ms + 12, gz[n] + zb_off);
                }
                gs[n] += 32 * gpp;
                gz[n] += 8 * gpp;
            }
        }
        cp_async_commit();
        ++p_issue;
        s_issue = (s_issue + SB == GV_P * SB) ? 0 : s_issue + SB;
    };
    auto load_x = [&](uint4 (&xb)[MT][2][2]) {
#pragma unroll
        for (int u = 0; u < MT; ++u) {
            const uint4* xp = reinterpret_cast<const uint4*>(xr[u]);
            xb[u][0][0] = __ldg(xp);
            xb[u][0][1] = __ldg(xp + 1);
            xb[u][1][0] = __ldg(xp + 8);
            xb[u][1][1] = __ldg(xp + 9);
            xr[u] += 128;
        }
    };

    float acc[NT][MT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int u = 0; u < MT; ++u)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[n][u][e] = 0.0f;

    uint32_t s_use = 0;
    auto step = [&](const uint4 (&xb)[MT][2][2]) {
        issue();
        cp_async_wait<GV_P - 1>();
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const uint8_t* cs = ringp + s_use + n * 1024;
            const uint4 meta = *reinterpret_cast<const uint4*>(ringp + s_use + NT * 1024 + n * 512);
            RowDq rg, rh;
            {
                DqRaw d;
                d.s2 = meta.x;
                d.zb = asym ? (meta.y >> zshift) & 0xFFu : 0x88u;
                build_dq(d, rg, rh);
            }
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (!G128 && c == 1) {
                    DqRaw d;
                    d.s2 = meta.z;
                    d.zb = asym ? (meta.w >> zshift) & 0xFFu : 0x88u;
                    build_dq(d, rg, rh);
                }
                const uint4 cw = *reinterpret_cast<const uint4*>(cs + c * 512);
                const uint32_t wd[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t a[4];
                    dq_word(wd[j], rg, rh, a);
#pragma unroll
                    for (int u = 0; u < MT; ++u) {
                        const uint32_t* xw = reinterpret_cast<const uint32_t*>(&xb[u][c][0]);
                        mma_bf16_16816(acc[n][u], a, xw[2 * j], xw[2 * j + 1]);
                    }
                }
            }
        }
        s_use = (s_use + SB == GV_P * SB) ? 0 : s_use + SB;
    };

#pragma unroll
    for (int i = 0; i < GV_P - 1; ++i) issue();
    // weights before the wait, activations (and y) after it (see k_w4_gemv)
    tc::pdl_wait();

    if (MT == 1) {
        // activations one step ahead, double-buffered by a 2x unrolled loop
        uint4 xa[MT][2][2], xc[MT][2][2];
        if (p_begin < p_end) load_x(xa);
        for (int64_t p = p_begin; p < p_end; p += 2) {
            if (p + 1 < p_end) load_x(xc);
            step(xa);
            if (p + 1 < p_end) {
                if (p + 2 < p_end) load_x(xa);
                step(xc);
            }
        }
    } else {
        for (int64_t p = p_begin; p < p_end; ++p) {
            uint4 xb[MT][2][2];
            load_x(xb);
            step(xb);
        }
    }
    cp_async_wait<0>();
    __syncthreads();

    float(*part)[NT * 16][16] = reinterpret_cast<float(*)[NT * 16][16]>(gv_smem);  // [warp][row][token]
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int u = 0; u < MT; ++u) {
            part[warp][n * 16 + gq][u * 8 + 2 * t] = acc[n][u][0];
            part[warp][n * 16 + gq][u * 8 + 2 * t + 1] = acc[n][u][1];
            part[warp][n * 16 + gq + 8][u * 8 + 2 * t] = acc[n][u][2];
            part[warp][n * 16 + gq + 8][u * 8 + 2 * t + 1] = acc[n][u][3];
        }
    __syncthreads();
    for (int i = threadIdx.x; i < NT * 16 * 16; i += blockDim.x) {
        const int row = i >> 4, tok = i & 15;
        if (tok < M && tok < MT * 8) {
            float s = 0.0f;
#pragma unroll
            for (int w = 0; w < 8; ++w) s += part[w][row][tok];
            y[(int64_t)tok * h.N + nt0 * 16 + row] = __float2bfloat16_rn(s);
        }
    }
}

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel of the stream finishes (it waits with griddepcontrol
// before touching anything that kernel can write).
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int MT, int NT, bool G128>
static cudaError_t launch_gemv2(const __nv_bfloat16* x, const uint8_t* blob, const qlin_w4_header& h, int64_t M,
                                __nv_bfloat16* y, cudaStream_t st) {
    constexpr int smem = 8 * GV_P * gemv2_stage_bytes<NT>();
    static_assert(smem >= 8 * NT * 16 * 16 * 4, "reduction tile must fit in the ring");
    cudaError_t e = ensure_smem((const void*)k_w4_gemv2<MT, NT, G128>, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(k_w4_gemv2<MT, NT, G128>, dim3((unsigned)(h.N / (16 * NT))), dim3(256), smem, st, x, blob, h, M,
                      y);
}

template <int MT, int NT>
static cudaError_t launch_gemv2g(const __nv_bfloat16* x, const uint8_t* blob, const qlin_w4_header& h, int64_t M,
                                 __nv_bfloat16* y, cudaStream_t st) {
    return h.group >= 128 ? launch_gemv2<MT, NT, true>(x, blob, h, M, y, st)
                          : launch_gemv2<MT, NT, false>(x, blob, h, M, y, st);
}

template <int MT, int NT>
static cudaError_t launch_gemv(const __nv_bfloat16* x, const uint8_t* blob, const qlin_w4_header& h, int64_t M,
                               __nv_bfloat16* y, cudaStream_t st) {
    constexpr int smem = gemv_smem_bytes<NT>();
    cudaError_t e = ensure_smem((const void*)k_w4_gemv<MT, NT>, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(k_w4_gemv<MT, NT>, dim3((unsigned)(h.N / (16 * NT))), dim3(256), smem, st, x, blob, h, M, y);
}

// ------------------------------------------------------------------ GEMM (M > 16), mma.sync
// CTA: 8 warps x 16 weight rows = 128 rows of W, BM tokens.  Each warp keeps
// its 16 x 64 weight chunk in registers (dequantized once) and multiplies it
// with all BM/8 token tiles of the chunk's X tile, staged in shared memory.
constexpr int kW4BM = 64;
constexpr int kPromote = 8;  // chunks (of 64 k) per promoted accumulation chain
constexpr int kXStride = 64 + 8;  // bf16 elements per smem row (padding against bank conflicts)

__global__ void __launch_bounds__(256) k_w4_gemm_mma(const __nv_bfloat16* __restrict__ x, const uint8_t* __restrict__ blob,
                                                     qlin_w4_header h, int64_t M, __nv_bfloat16* __restrict__ y) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, t = lane & 3;
    const int64_t K = h.K, nchunk = K / 64, ngr = K / h.group;
    const int64_t nt = (int64_t)blockIdx.x * 8 + warp;  // this warp's n-tile
    const int64_t m0 = (int64_t)blockIdx.y * kW4BM;
    const bool nt_ok = nt < h.N / 16;
    const uint4* __restrict__ codes = reinterpret_cast<const uint4*>(blob + h.codes_off) + nt * nchunk * 32 + lane;

    __shared__ __align__(16) __nv_bfloat16 xs[2][kW4BM * kXStride];

    // The tensor-core accumulator is promoted into `tot` every kPromote chunks
    // so that no single accumulation chain runs over the whole of K.
    float acc[kW4BM / 8][4], tot[kW4BM / 8][4];
#pragma unroll
    for (int u = 0; u < kW4BM / 8; ++u)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[u][e] = tot[u][e] = 0.0f;

    // stage chunk kc of X (BM x 64 bf16 = 512 16-byte pieces; 2 per thread)
    auto stage = [&](int buf, int64_t kc) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            int piece = threadIdx.x + 256 * i;
            int r = piece >> 3, c8 = piece & 7;
            int64_t m = m0 + r;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (m < M) v = __ldg(reinterpret_cast<const uint4*>(x + m * K + kc * 64 + c8 * 8));
            *reinterpret_cast<uint4*>(&xs[buf][r * kXStride + c8 * 8]) = v;
        }
    };

    stage(0, 0);
    __syncthreads();
    int64_t last_g = -1;
    RowDq rg, rh;
    for (int64_t kc = 0; kc < nchunk; ++kc) {
        int buf = (int)(kc & 1);
        uint4 wv = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
        if (nt_ok) wv = __ldg(codes + kc * 32);
        if (kc + 1 < nchunk) stage(buf ^ 1, kc + 1);
        int64_t gi = (kc * 64 + 16 * t) / h.group;
        if (nt_ok && gi != last_g) {
            load_rowdq(blob, h, nt, ngr, gi, gq, rg, rh);
            last_g = gi;
        }
        if (!nt_ok) {
            rg = row_dq(0.0f, 8);
            rh = rg;
        }
        uint32_t wd[4] = {wv.x, wv.y, wv.z, wv.w};
        uint32_t a[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) dq_word(wd[j], rg, rh, a[j]);
#pragma unroll
        for (int u = 0; u < kW4BM / 8; ++u) {
            const __nv_bfloat16* xr = &xs[buf][(u * 8 + gq) * kXStride + 16 * t];
            uint4 b01 = *reinterpret_cast<const uint4*>(xr);
            uint4 b23 = *reinterpret_cast<const uint4*>(xr + 8);
            mma_bf16_16816(acc[u], a[0], b01.x, b01.y);
            mma_bf16_16816(acc[u], a[1], b01.z, b01.w);
            mma_bf16_16816(acc[u], a[2], b23.x, b23.y);
            mma_bf16_16816(acc[u], a[3], b23.z, b23.w);
        }
        if ((kc & (kPromote - 1)) == kPromote - 1 || kc + 1 == nchunk) {
#pragma unroll
            for (int u = 0; u < kW4BM / 8; ++u)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    tot[u][e] += acc[u][e];
                    acc[u][e] = 0.0f;
                }
        }
        __syncthreads();
    }
    if (!nt_ok) return;
#pragma unroll
    for (int u = 0; u < kW4BM / 8; ++u) {
        int64_t mA = m0 + u * 8 + 2 * t, mB = mA + 1;
        int64_t n0 = nt * 16 + gq, n1 = n0 + 8;
        if (mA < M) {
            y[mA * h.N + n0] = __float2bfloat16_rn(tot[u][0]);
            y[mA * h.N + n1] = __float2bfloat16_rn(tot[u][2]);
        }
        if (mB < M) {
            y[mB * h.N + n0] = __float2bfloat16_rn(tot[u][1]);
            y[mB * h.N + n1] = __float2bfloat16_rn(tot[u][3]);
        }
    }
}

// ====================================================================== tcgen05 GEMM (M > 16)
// D[n, m] = sum_k w^[n, k] x[m, k] on the bf16 tensor cores, fp32 in TMEM.
//   A operand: 128 weight rows, dequantized by 8 converter warps from the
//              packed blob into a 128B-swizzled bf16 tile (one 16x64 packed
//              tile per warp per k-block: the lane's 32 nibbles -> rows gq and
//              gq+8, k = 16t..16t+15 of the chunk).
//   B operand: up to 256 tokens of x, loaded by TMA (128B swizzle, rows past M
//              zero-filled).
// K is split across gridDim.y CTAs; each writes fp32 partial sums, which
// k_w4_reduce adds in a fixed order (deterministic) and rounds once to bf16.
// Every `promote` k-blocks the TMEM accumulator is folded into a second fp32
// TMEM region so that no tensor-core accumulation chain spans more than
// promote*64 k.
namespace w4tc {
constexpr int BMW = 128;                  // weight rows per CTA (TMEM lanes)
constexpr int BK = 64;
constexpr int A_STAGES_MAX = 6;           // converted-weight stages (A operand)
constexpr int B_STAGES_MAX = 16;          // activation stages (B operand, TMA)
constexpr int A_BYTES = BMW * BK * 2;     // 16 KB
constexpr int NCONV_WARPS = 16;           // warps 0-15: warp w converts tile w % 8 of k-blocks of parity w / 8
constexpr int EPI_WARP0 = 16;             // warps 16-19
constexpr int MMA_WARP = 20;
constexpr int TMA_WARP = 21;
constexpr int THREADS = 22 * 32;
constexpr uint32_t TMEM_COLS = 512;       // accumulators in [0,256) (two of 128 for ntok <= 128), promoted sums in [256,512)
constexpr int CRING = 6;                  // cp.async ring depth (own k-blocks) of each converter warp
constexpr int CR_WARP_BYTES = CRING * (512 + 256);  // codes [CRING][32][16 B] + group words [CRING][32][8 B]
constexpr int RING_BYTES = NCONV_WARPS * CR_WARP_BYTES;
constexpr int BAR_BYTES = 512;
constexpr size_t SMEM_LIMIT = 232448;     // dynamic shared memory per CTA
// The activation tiles have their own, deeper ring: their TMA latency (L2
// under the weight stream) would otherwise bound the k-block rate.
__host__ __device__ constexpr int b_bytes(int ntok) { return ntok * BK * 2; }  // ntok rows of 128 B
// 256 tokens: 3 A stages, which leaves room for 5 activation stages of 32 KB.
inline int a_stages(int ntok) { return ntok > 128 ? 3 : A_STAGES_MAX; }
inline int b_stages(int ntok) {
    int s = (int)((SMEM_LIMIT - 1024 - RING_BYTES - BAR_BYTES - (size_t)a_stages(ntok) * A_BYTES) / b_bytes(ntok));
    return s < B_STAGES_MAX ? s : B_STAGES_MAX;
}
inline size_t smem_bytes(int ntok) {
    return 1024 + (size_t)a_stages(ntok) * A_BYTES + (size_t)b_stages(ntok) * b_bytes(ntok) + RING_BYTES + BAR_BYTES;
}
}  // namespace w4tc

struct W4TcArgs {
    const uint8_t* blob;
    qlin_w4_header h;
    int64_t M;
    int ntok;         // MMA N: tokens per CTA (multiple of 16, <= 256) = TMA box rows
    int nchunk;       // K / 64
    int nsplit;
    int a_stages;     // converted-weight stages
    int b_stages;     // activation stages
    int promote;      // k-blocks per accumulation chain (0: no promotion)
    uint32_t idesc;
    float* part;            // [nsplit][M][N] fp32 partials, or nullptr when nsplit == 1
    __nv_bfloat16* y;       // [M][N] output when nsplit == 1
};

__global__ void __launch_bounds__(w4tc::THREADS, 1) k_w4_gemm_tc(const __grid_constant__ CUtensorMap tmx, W4TcArgs a) {
    using namespace w4tc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int SA = a.a_stages, SB = a.b_stages;
    const uint32_t B_BYTES = (uint32_t)b_bytes(a.ntok);
    uint8_t* tilesA = smem;                                  // [SA][16 KB], 1024-aligned
    uint8_t* tilesB = smem + (size_t)SA * A_BYTES;           // [SB][ntok * 128 B], 1024-aligned
    uint8_t* cring = tilesB + (size_t)SB * B_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(cring + RING_BYTES);
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(bars + 2 * SA + 2 * SB + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t N = a.h.N;
    const int64_t nblk = blockIdx.x;              // 128-row block of W
    const int split = blockIdx.y;
    const int64_t m0 = (int64_t)blockIdx.z * a.ntok;
    // k-chunk range of this split
    const int c_begin = (int)((int64_t)a.nchunk * split / a.nsplit);
    const int c_end = (int)((int64_t)a.nchunk * (split + 1) / a.nsplit);
    const int nkb = c_end - c_begin;

    const uint32_t bar0 = tc::smem_addr(bars);
    auto fullA = [&](int s) { return bar0 + 8u * s; };
    auto emptyA = [&](int s) { return bar0 + 8u * (SA + s); };
    auto fullB = [&](int s) { return bar0 + 8u * (2 * SA + s); };
    auto emptyB = [&](int s) { return bar0 + 8u * (2 * SA + SB + s); };
    // Accumulation chains: chain c (a.promote k-blocks, the last one shorter)
    // accumulates into TMEM buffer c % nbuf; the epilogue adds every chain but
    // the last into the promoted sums and then frees the buffer.  Each buffer
    // has its own full / empty barrier, so no barrier ever runs two phases
    // ahead of its waiter.
    const uint32_t acc_full0 = bar0 + 8u * (2 * SA + 2 * SB);
    auto acc_full = [&](int b) { return acc_full0 + 8u * b; };
    auto acc_empty = [&](int b) { return acc_full0 + 16u + 8u * b; };
    const uint32_t done_bar = acc_full0 + 32u;
    const bool two_buf = a.ntok <= 128;
    auto buf_of = [&](int c) { return two_buf ? (c & 1) : 0; };        // c % nbuf
    auto use_of = [&](int c) { return (uint32_t)(two_buf ? (c >> 1) : c); };  // c / nbuf
    const int chain_len = a.promote > 0 ? a.promote : (nkb > 0 ? nkb : 1);
    const int nchains = nkb > 0 ? (nkb + chain_len - 1) / chain_len : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < SA; ++s) {
            tc::mbar_init(fullA(s), 8);  // the 8 warps converting this k-block
            tc::mbar_init(emptyA(s), 1);
        }
        for (int s = 0; s < SB; ++s) {
            tc::mbar_init(fullB(s), 1);  // the TMA issuer's expect_tx
            tc::mbar_init(emptyB(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(acc_full(b), 1);
            tc::mbar_init(acc_empty(b), 4);  // one arrival per epilogue warp
        }
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
        // ---------------------------------------------------------- weight dequantization
        // Warp w converts 16-row tile w % 8 for the k-blocks of parity w / 8, so
        // two warps share each tile.  Codes and group words of the warp's next
        // CRING-1 k-blocks stream into its cp.async ring (each lane reads back
        // only what it copied).
        const int ntl = warp & 7;             // 16-row packed tile within the 128-row block
        const int par = warp >> 3;
        const int gq = lane >> 2, t = lane & 3;
        const int64_t nt = nblk * 8 + ntl;
        const int64_t ngr = a.h.K / a.h.group;
        const int gshift = __ffs(a.h.group) - 1;  // group is a power of two
        const bool asym = a.h.asym != 0;
        const int zshift = 8 * (gq & 3);
        const uint8_t* gcodes = a.blob + a.h.codes_off + (nt * a.nchunk + c_begin) * 512 + lane * 16;
        const uint8_t* gsc = a.blob + a.h.scales_off + nt * ngr * 32 + gq * 4;
        const uint8_t* gze = a.blob + a.h.zeros_off + nt * ngr * 8 + (gq & 4);
        uint8_t* rp = cring + warp * CR_WARP_BYTES;
        const uint32_t rc = tc::smem_addr(rp) + lane * 16;               // codes [CRING][32][16 B]
        const uint32_t rm = tc::smem_addr(rp + CRING * 512) + lane * 8;  // words [CRING][32][8 B]
        int kb_issue = par, slot_issue = 0;
        // running source pointers of this lane's next copy: codes advance by
        // two 64-k blocks, the group words by the groups those cover (the
        // lane's k, 64 kb + 16 t, sits in group (64 kb + 16 t) / g)
        const uint8_t* pc = gcodes + (int64_t)par * 512;
        const int64_t gi0 = ((int64_t)(c_begin + par) * 64 + 16 * t) >> gshift;
        const uint8_t* ps = gsc + gi0 * 32;
        const uint8_t* pz = gze + gi0 * 8;
        const int gstep = 128 >> gshift;  // groups per two k-blocks (g <= 128)
        auto issue = [&]() {
            if (kb_issue < nkb) {
                cp_async16(rc + slot_issue * 512, pc);
                cp_async4(rm + slot_issue * 256, ps);
                if (asym) cp_async4(rm + slot_issue * 256 + 4, pz);
            }
            cp_async_commit();
            kb_issue += 2;
            pc += 1024;
            ps += 32 * gstep;
            pz += 8 * gstep;
            slot_issue = slot_issue + 1 == CRING ? 0 : slot_issue + 1;
        };
#pragma unroll 1
        for (int i = 0; i < CRING - 1; ++i) issue();
        const uint32_t r_g = (uint32_t)(ntl * 16 + gq), r_h = r_g + 8;
        int s = par < SA ? par : par - SA, slot = 0;
        uint32_t ph = par < SA ? 0u : 1u;
        for (int kb = par; kb < nkb; kb += 2) {
            issue();
            cp_async_wait<CRING - 1>();
            const uint4 wv = *reinterpret_cast<const uint4*>(rp + slot * 512 + lane * 16);
            const uint2 mw = *reinterpret_cast<const uint2*>(rp + CRING * 512 + slot * 256 + lane * 8);
            slot = slot + 1 == CRING ? 0 : slot + 1;
            DqRaw dq;
            dq.s2 = mw.x;
            dq.zb = asym ? (mw.y >> zshift) & 0xFFu : 0x88u;
            RowDq rg, rh;
            build_dq(dq, rg, rh);
            const uint32_t wd[4] = {wv.x, wv.y, wv.z, wv.w};
            uint32_t og[8], oh[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t f[4];
                dq_word(wd[j], rg, rh, f);
                og[2 * j] = f[0];      // row gq,   k 4j, 4j+1
                og[2 * j + 1] = f[2];  // row gq,   k 4j+2, 4j+3
                oh[2 * j] = f[1];      // row gq+8
                oh[2 * j + 1] = f[3];
            }
            if (!tc::mbar_wait_warp(emptyA(s), ph ^ 1u, abort_flag)) break;
            uint8_t* tA = tilesA + (size_t)s * A_BYTES;
            *reinterpret_cast<uint4*>(tA + tc::sw128_off(r_g, 2 * t)) = make_uint4(og[0], og[1], og[2], og[3]);
            *reinterpret_cast<uint4*>(tA + tc::sw128_off(r_g, 2 * t + 1)) = make_uint4(og[4], og[5], og[6], og[7]);
            *reinterpret_cast<uint4*>(tA + tc::sw128_off(r_h, 2 * t)) = make_uint4(oh[0], oh[1], oh[2], oh[3]);
            *reinterpret_cast<uint4*>(tA + tc::sw128_off(r_h, 2 * t + 1)) = make_uint4(oh[4], oh[5], oh[6], oh[7]);
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(fullA(s));
            s += 2;
            if (s >= SA) {
                s -= SA;
                ph ^= 1u;
            }
        }
        cp_async_wait<0>();
    } else if (warp == TMA_WARP) {
        // ---------------------------------------------------------- activation tiles (TMA)
        if (lane == 0 && !tc::producers_stalled()) {
            const uint32_t tx = (uint32_t)a.ntok * BK * 2;
            int s = 0;
            uint32_t ph = 0;
            for (int kb = 0; kb < nkb; ++kb) {
                if (!tc::mbar_wait(emptyB(s), ph ^ 1u, abort_flag)) break;
                tc::mbar_arrive_expect_tx(fullB(s), tx);
                const uint32_t dstB = tc::smem_addr(tilesB + (size_t)s * B_BYTES);
                tc::tma_load_2d(dstB, &tmx, (c_begin + kb) * BK, (int)m0, fullB(s));
                if (++s == SB) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ---------------------------------------------------------- MMA issuer
        // The warp runs the loop together, so that descriptors and addresses
        // are warp-uniform values; one elected lane issues the MMAs and
        // commits (single-thread operations).
        const uint32_t tA_addr = tc::smem_addr(tilesA), tB_addr = tc::smem_addr(tilesB);
        int c = 0, in_chain = 0;
        int s = 0, sb = 0;
        uint32_t ph = 0, phb = 0;
        for (int kb = 0; kb < nkb; ++kb) {
            if (!tc::mbar_wait_warp(fullB(sb), phb, abort_flag)) break;
            if (!tc::mbar_wait_warp(fullA(s), ph, abort_flag)) break;
            if (in_chain == chain_len) {
                // chain c is complete: hand its buffer to the epilogue and start
                // chain c + 1 once that chain's buffer has been drained
                if (tc::elect_one()) tc::mma_commit(acc_full(buf_of(c)));
                __syncwarp();
                ++c;
                in_chain = 0;
                if (use_of(c) >= 1 && !tc::mbar_wait_warp(acc_empty(buf_of(c)), (use_of(c) - 1) & 1u, abort_flag))
                    break;
            }
            tc::tc_fence_after();
            const uint64_t ad = tc::desc_sw128(tA_addr + (uint32_t)s * A_BYTES);
            const uint64_t bd = tc::desc_sw128(tB_addr + (uint32_t)sb * B_BYTES);
            const uint32_t dacc = tmem + 128u * (uint32_t)buf_of(c);
            if (tc::elect_one()) {
#pragma unroll
                for (int j = 0; j < BK / 16; ++j)
                    tc::mma_f16(dacc, ad + 2 * j, bd + 2 * j, a.idesc, (in_chain > 0 || j > 0) ? 1u : 0u);
                tc::mma_commit(emptyA(s));
                tc::mma_commit(emptyB(sb));
            }
            __syncwarp();
            ++in_chain;
            if (++s == SA) {
                s = 0;
                ph ^= 1u;
            }
            if (++sb == SB) {
                sb = 0;
                phb ^= 1u;
            }
        }
        if (tc::elect_one()) {
            if (nkb > 0) tc::mma_commit(acc_full(buf_of(c)));  // the last chain
            tc::mma_commit(done_bar);
        }
        __syncwarp();
        tc::mbar_wait_drain(done_bar, 0);
        __syncwarp();
    } else {
        // ---------------------------------------------------------- promotions + epilogue
        const int q = warp & 3;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const int64_t n = nblk * BMW + 32 * q + lane;  // output channel of this thread
        const uint32_t t_sum = tmem + lane_base + 256;
        for (int c = 0; c < nchains; ++c) {
            const int b = buf_of(c);
            const uint32_t t_acc = tmem + lane_base + 128u * (uint32_t)b;
            if (!tc::mbar_wait_warp(acc_full(b), use_of(c) & 1u, abort_flag)) break;
            tc::tc_fence_after();
            if (c + 1 < nchains) {
                // promote: sums (+)= chain c
                for (int col = 0; col < a.ntok; col += 16) {
                    uint32_t v[16], r[16];
                    tc::tmem_ld16(t_acc + col, v);
                    if (c > 0) tc::tmem_ld16(t_sum + col, r);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        r[j] = c > 0 ? __float_as_uint(__uint_as_float(r[j]) + __uint_as_float(v[j])) : v[j];
                    tc::tmem_st16(t_sum + col, r);
                }
                tc::tmem_wait_st();
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(acc_empty(b));
                continue;
            }
            for (int col = 0; col < a.ntok; col += 16) {
                __syncwarp();
                uint32_t v[16], r[16];
                tc::tmem_ld16(t_acc + col, v);
                if (c > 0) tc::tmem_ld16(t_sum + col, r);
                tc::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float f = __uint_as_float(v[j]);
                    if (c > 0) f += __uint_as_float(r[j]);
                    const int64_t m = m0 + col + j;
                    if (col + j < a.ntok && m < a.M) {
                        if (a.part)
                            a.part[((int64_t)split * a.M + m) * N + n] = f;
                        else
                            a.y[m * N + n] = __float2bfloat16_rn(f);
                    }
                }
            }
        }
        if (nkb == 0 && !*abort_flag) {
            // an empty split contributes zeros
            for (int64_t j = 0; j < a.ntok; ++j) {
                const int64_t m = m0 + j;
                if (m < a.M) {
                    if (a.part)
                        a.part[((int64_t)split * a.M + m) * N + n] = 0.0f;
                    else
                        a.y[m * N + n] = __float2bfloat16_rn(0.0f);
                }
            }
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ W4A16 GEMM, A operand in TMEM (M <= 128 per CTA)
// The same roles as k_w4_gemm_tc, but the converters write the dequantized
// weight tile into tensor memory with tcgen05.st and the MMA reads A from there
// (tcgen05.mma with an [a-tmem] operand).  That takes the 16 KB store of each
// 64-k block and the tensor core's 16 KB read of it off the shared-memory
// ports, which bound the shared-memory version at these sizes.  Stages cover
// 128 k, so the single MMA-issuing warp pays its waits and commits once per
// two 64-k blocks.  TMEM holds everything for up to 128 tokens: two
// accumulators, the promoted sums and 2 (or 4, for <= 64 tokens) A stages of
// 64 columns.
namespace w4tm {
constexpr int BMW = 128;
constexpr int BK = 64;
constexpr int NCONV_WARPS = 16;  // warp w: TMEM quarter w % 4, tile half (w >> 2) & 1, 64-k half w >> 3 of each stage
constexpr int EPI_WARP0 = 16;
constexpr int MMA_WARP = 20;
constexpr int TMA_WARP = 21;
constexpr int THREADS = 22 * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr int B_STAGES_MAX = 16;
constexpr int BAR_BYTES = 512;
constexpr size_t SMEM_LIMIT = 232448;
// A pipeline stage covers 128 k: two 64-k blocks, one per converter half, and
// two 64-k activation boxes.  One stage costs the MMA warp one wait per
// operand, 8 MMAs and 2 commits.
__host__ __device__ constexpr int b_bytes(int ntok) { return ntok * BK * 2; }  // one 64-k box of X
__host__ __device__ constexpr int b_stage_bytes(int ntok) { return 2 * b_bytes(ntok); }
// TMEM columns: accumulator b at b * acc_stride, promoted sums at
// 2 * acc_stride, A stage s (128 lanes x 64 columns = 128 rows x 128 bf16, k
// pairs packed low-first; columns 0-31 hold k 0-63) at a_col0 + 64 s.
__host__ __device__ inline int acc_stride(int ntok) { return ntok <= 64 ? 64 : 128; }
__host__ __device__ inline int a_col0(int ntok) { return ntok <= 64 ? 256 : 384; }
__host__ __device__ inline int a_stages(int ntok) { return ntok <= 64 ? 4 : 2; }
constexpr int CRING = 6;  // cp.async ring depth (own k-blocks) of each converter warp
constexpr int CR_WARP_BYTES = CRING * (512 + 256);  // codes [CRING][32 chunks][16 B] + group words [CRING][32][8 B]
constexpr int RING_BYTES = NCONV_WARPS * CR_WARP_BYTES;
inline int b_stages(int ntok) {
    int s = (int)((SMEM_LIMIT - 1024 - RING_BYTES - BAR_BYTES) / b_stage_bytes(ntok));
    return s < B_STAGES_MAX ? s : B_STAGES_MAX;
}
inline size_t smem_bytes(int ntok) {
    return 1024 + (size_t)b_stages(ntok) * b_stage_bytes(ntok) + RING_BYTES + BAR_BYTES;
}
}  // namespace w4tm

// 16 TMEM lanes x 4 x 256 bits: in repetition r, thread (g = lane / 4, t = lane % 4)
// writes r[4r], r[4r+1] to lane g, columns 8r + 2t, 8r + 2t + 1, and r[4r+2],
// r[4r+3] to lane g + 8, same columns (base lane and column from taddr).
__device__ __forceinline__ void tmem_st_16x256b_x4(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f16; A is 128 lanes (rows) x 8
// columns (16 k) from a_tmem.
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__global__ void __launch_bounds__(w4tm::THREADS, 1) k_w4_gemm_tm(const __grid_constant__ CUtensorMap tmx, W4TcArgs a) {
    using namespace w4tm;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int SA = a_stages(a.ntok), SB = a.b_stages;
    const uint32_t B_HALF = (uint32_t)b_bytes(a.ntok), B_BYTES = 2u * B_HALF;
    uint8_t* tilesB = smem;                                  // [SB][2][ntok * 128 B], 1024-aligned
    uint8_t* cring = tilesB + (size_t)SB * B_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(cring + RING_BYTES);
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(bars + 2 * SA + 2 * SB + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t N = a.h.N;
    const int64_t nblk = blockIdx.x;
    const int split = blockIdx.y;
    const int64_t m0 = (int64_t)blockIdx.z * a.ntok;
    const int c_begin = (int)((int64_t)a.nchunk * split / a.nsplit);
    const int c_end = (int)((int64_t)a.nchunk * (split + 1) / a.nsplit);
    const int nkb = c_end - c_begin;
    const int nst = (nkb + 1) >> 1;  // stages; with an odd count the last holds one 64-k block
    const uint32_t ACC_STRIDE = (uint32_t)acc_stride(a.ntok), A_COL0 = (uint32_t)a_col0(a.ntok);

    const uint32_t bar0 = tc::smem_addr(bars);
    auto fullA = [&](int s) { return bar0 + 8u * s; };
    auto emptyA = [&](int s) { return bar0 + 8u * (SA + s); };
    auto fullB = [&](int s) { return bar0 + 8u * (2 * SA + s); };
    auto emptyB = [&](int s) { return bar0 + 8u * (2 * SA + SB + s); };
    const uint32_t acc_full0 = bar0 + 8u * (2 * SA + 2 * SB);
    auto acc_full = [&](int b) { return acc_full0 + 8u * b; };
    auto acc_empty = [&](int b) { return acc_full0 + 16u + 8u * b; };
    const uint32_t done_bar = acc_full0 + 32u;
    // chains of a.promote 64-k blocks, rounded up to whole stages
    const int chain_st = a.promote > 0 ? (a.promote + 1) >> 1 : (nst > 0 ? nst : 1);
    const int nchains = nst > 0 ? (nst + chain_st - 1) / chain_st : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < SA; ++s) {
            tc::mbar_init(fullA(s), 16);  // every converter warp, each stage
            tc::mbar_init(emptyA(s), 1);
        }
        for (int s = 0; s < SB; ++s) {
            tc::mbar_init(fullB(s), 1);
            tc::mbar_init(emptyB(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(acc_full(b), 1);
            tc::mbar_init(acc_empty(b), 4);
        }
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
        // Warp w converts the 16-row tile 2 (w % 4) + ((w >> 2) & 1), 64-k half
        // w >> 3 of every stage, and stores it into its own TMEM quarter.
        // Lane (g, t) copies its packed 16 bytes (k 16t .. 16t+15 of rows g and
        // g+8) to ring chunk 8t + g; after the warp's copies land it reads word t
        // of chunks 8r + g, r = 0..3, i.e. k 16r + 4t .. 16r + 4t + 3, which is
        // what the 16x256b TMEM store wants from this lane.
        const int q = warp & 3, hsel = (warp >> 2) & 1, par = warp >> 3;
        const int ntl = 2 * q + hsel;
        const int gq = lane >> 2, t = lane & 3;
        const int64_t nt = nblk * 8 + ntl;
        const int64_t ngr = a.h.K / a.h.group;
        const int gshift = __ffs(a.h.group) - 1;
        const bool asym = a.h.asym != 0;
        const bool g32 = a.h.group == 32;
        const int zshift = 8 * (gq & 3);
        const uint8_t* gcodes = a.blob + a.h.codes_off + (nt * a.nchunk + c_begin) * 512 + lane * 16;
        const uint8_t* gsc = a.blob + a.h.scales_off + nt * ngr * 32 + gq * 4;
        const uint8_t* gze = a.blob + a.h.zeros_off + nt * ngr * 8 + (gq & 4);
        uint8_t* rp = cring + warp * CR_WARP_BYTES;
        const uint32_t rc = tc::smem_addr(rp) + (uint32_t)(8 * t + gq) * 16;  // codes [CRING][32 chunks][16 B]
        const uint32_t rm = tc::smem_addr(rp + CRING * 512) + lane * 8;          // words [CRING][32][8 B]
        const uint32_t t_lane = (uint32_t)(32 * q + 16 * hsel) << 16;
        int kb_issue = par, slot_issue = 0;
        // running source pointers of this lane's next copy: codes advance by
        // two 64-k blocks, the group words by the groups those cover (the
        // lane's k, 64 kb + 16 t, sits in group (64 kb + 16 t) / g)
        const uint8_t* pc = gcodes + (int64_t)par * 512;
        const int64_t gi0 = ((int64_t)(c_begin + par) * 64 + 16 * t) >> gshift;
        const uint8_t* ps = gsc + gi0 * 32;
        const uint8_t* pz = gze + gi0 * 8;
        const int gstep = 128 >> gshift;  // groups per two k-blocks (g <= 128)
        auto issue = [&]() {
            if (kb_issue < nkb) {
                cp_async16(rc + slot_issue * 512, pc);
                cp_async4(rm + slot_issue * 256, ps);
                if (asym) cp_async4(rm + slot_issue * 256 + 4, pz);
            }
            cp_async_commit();
            kb_issue += 2;
            pc += 1024;
            ps += 32 * gstep;
            pz += 8 * gstep;
            slot_issue = slot_issue + 1 == CRING ? 0 : slot_issue + 1;
        };
#pragma unroll 1
        for (int i = 0; i < CRING - 1; ++i) issue();
        int s = 0, slot = 0, pend = -1;
        uint32_t ph = 0u;
        for (int st_i = 0; st_i < nst; ++st_i) {
            // With an odd k-block count the second half of the last stage is
            // empty: those warps still take the stage (wait, arrive) so that
            // its barrier phase completes, but store nothing.
            const bool has = 2 * st_i + par < nkb;
            issue();
            cp_async_wait<CRING - 1>();
            __syncwarp();  // the other lanes' copies of this slot have landed
            const uint8_t* cs = rp + slot * 512 + gq * 16 + t * 4;
            uint32_t u[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) u[r] = *reinterpret_cast<const uint32_t*>(cs + r * 128);
            // group words of lanes (g, 0) and (g, 2): k 0..31 and 32..63 of the block
            const uint8_t* ms = rp + CRING * 512 + slot * 256 + gq * 32;
            const uint2 mw0 = *reinterpret_cast<const uint2*>(ms);
            const uint2 mw1 = g32 ? *reinterpret_cast<const uint2*>(ms + 16) : mw0;
            __syncwarp();  // every lane has read the slot before it is refilled
            slot = slot + 1 == CRING ? 0 : slot + 1;
            DqRaw d0, d1;
            d0.s2 = mw0.x;
            d0.zb = asym ? (mw0.y >> zshift) & 0xFFu : 0x88u;
            d1.s2 = mw1.x;
            d1.zb = asym ? (mw1.y >> zshift) & 0xFFu : 0x88u;
            RowDq rg0, rh0, rg1, rh1;
            build_dq(d0, rg0, rh0);
            if (g32)
                build_dq(d1, rg1, rh1);
            else {
                rg1 = rg0;
                rh1 = rh0;
            }
            uint32_t st[16];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                uint32_t f[4];
                if (r < 2)
                    dq_word(u[r], rg0, rh0, f);
                else
                    dq_word(u[r], rg1, rh1, f);
                st[4 * r + 0] = f[0];  // row g,   k 16r+4t, +1
                st[4 * r + 1] = f[2];  // row g,   k 16r+4t+2, +3
                st[4 * r + 2] = f[1];  // row g+8
                st[4 * r + 3] = f[3];
            }
            // A stage's TMEM store is waited for (and the stage handed to the
            // MMA warp) only after the next stage is converted, so the store's
            // latency overlaps that conversion instead of stalling the warp.
            if (pend >= 0) {
                tc::tmem_wait_st();
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(fullA(pend));
                pend = -1;
            }
            if (!tc::mbar_wait_warp(emptyA(s), ph ^ 1u, abort_flag)) break;
            tc::tc_fence_after();
            if (has) tmem_st_16x256b_x4(tmem + t_lane + A_COL0 + 64u * (uint32_t)s + 32u * (uint32_t)par, st);
            pend = s;
            if (++s == SA) {
                s = 0;
                ph ^= 1u;
            }
        }
        tc::tmem_wait_st();
        if (pend >= 0) {
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(fullA(pend));
        }
        cp_async_wait<0>();
    } else if (warp == TMA_WARP) {
        if (lane == 0 && !tc::producers_stalled()) {
            int s = 0;
            uint32_t ph = 0;
            for (int st_i = 0; st_i < nst; ++st_i) {
                const int nh = 2 * st_i + 1 < nkb ? 2 : 1;  // 64-k boxes in this stage
                if (!tc::mbar_wait(emptyB(s), ph ^ 1u, abort_flag)) break;
                tc::mbar_arrive_expect_tx(fullB(s), (uint32_t)nh * B_HALF);
                const uint32_t dstB = tc::smem_addr(tilesB + (size_t)s * B_BYTES);
                for (int hh = 0; hh < nh; ++hh)
                    tc::tma_load_2d(dstB + (uint32_t)hh * B_HALF, &tmx, (c_begin + 2 * st_i + hh) * BK, (int)m0,
                                    fullB(s));
                if (++s == SB) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        const uint32_t tB_addr = tc::smem_addr(tilesB);
        int c = 0, in_chain = 0;
        int s = 0, sb = 0;
        uint32_t ph = 0, phb = 0;
        for (int st_i = 0; st_i < nst; ++st_i) {
            if (!tc::mbar_wait_warp(fullB(sb), phb, abort_flag)) break;
            if (!tc::mbar_wait_warp(fullA(s), ph, abort_flag)) break;
            if (in_chain == chain_st) {
                if (tc::elect_one()) tc::mma_commit(acc_full(c & 1));
                __syncwarp();
                ++c;
                in_chain = 0;
                if (c >= 2 && !tc::mbar_wait_warp(acc_empty(c & 1), ((c >> 1) - 1) & 1u, abort_flag)) break;
            }
            tc::tc_fence_after();
            const int nh = 2 * st_i + 1 < nkb ? 2 : 1;
            const uint32_t at = tmem + A_COL0 + 64u * (uint32_t)s;
            const uint32_t dacc = tmem + ACC_STRIDE * (uint32_t)(c & 1);
            if (tc::elect_one()) {
                for (int hh = 0; hh < nh; ++hh) {
                    const uint64_t bd = tc::desc_sw128(tB_addr + (uint32_t)sb * B_BYTES + (uint32_t)hh * B_HALF);
#pragma unroll
                    for (int j = 0; j < BK / 16; ++j)
                        mma_f16_tmem_a(dacc, at + 32u * hh + 8u * j, bd + 2 * j, a.idesc,
                                       (in_chain > 0 || hh > 0 || j > 0) ? 1u : 0u);
                }
                tc::mma_commit(emptyA(s));
                tc::mma_commit(emptyB(sb));
            }
            __syncwarp();
            ++in_chain;
            if (++s == SA) {
                s = 0;
                ph ^= 1u;
            }
            if (++sb == SB) {
                sb = 0;
                phb ^= 1u;
            }
        }
        if (tc::elect_one()) {
            if (nst > 0) tc::mma_commit(acc_full(c & 1));  // the last chain
            tc::mma_commit(done_bar);
        }
        __syncwarp();
        tc::mbar_wait_drain(done_bar, 0);
        __syncwarp();
    } else {
        const int q = warp & 3;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const int64_t n = nblk * BMW + 32 * q + lane;
        const uint32_t t_sum = tmem + lane_base + 2u * ACC_STRIDE;
        for (int c = 0; c < nchains; ++c) {
            const int b = c & 1;
            const uint32_t t_acc = tmem + lane_base + ACC_STRIDE * (uint32_t)b;
            if (!tc::mbar_wait_warp(acc_full(b), (uint32_t)(c >> 1) & 1u, abort_flag)) break;
            tc::tc_fence_after();
            if (c + 1 < nchains) {
                for (int col = 0; col < a.ntok; col += 16) {
                    uint32_t v[16], r[16];
                    tc::tmem_ld16(t_acc + col, v);
                    if (c > 0) tc::tmem_ld16(t_sum + col, r);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        r[j] = c > 0 ? __float_as_uint(__uint_as_float(r[j]) + __uint_as_float(v[j])) : v[j];
                    tc::tmem_st16(t_sum + col, r);
                }
                tc::tmem_wait_st();
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(acc_empty(b));
                continue;
            }
            for (int col = 0; col < a.ntok; col += 16) {
                __syncwarp();
                uint32_t v[16], r[16];
                tc::tmem_ld16(t_acc + col, v);
                if (c > 0) tc::tmem_ld16(t_sum + col, r);
                tc::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float f = __uint_as_float(v[j]);
                    if (c > 0) f += __uint_as_float(r[j]);
                    const int64_t m = m0 + col + j;
                    if (col + j < a.ntok && m < a.M) {
                        if (a.part)
                            a.part[((int64_t)split * a.M + m) * N + n] = f;
                        else
                            a.y[m * N + n] = __float2bfloat16_rn(f);
                    }
                }
            }
        }
        if (nkb == 0 && !*abort_flag) {
            for (int64_t j = 0; j < a.ntok; ++j) {
                const int64_t m = m0 + j;
                if (m < a.M) {
                    if (a.part)
                        a.part[((int64_t)split * a.M + m) * N + n] = 0.0f;
                    else
                        a.y[m * N + n] = __float2bfloat16_rn(0.0f);
                }
            }
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// y[m, n] = bf16( sum_s part[s, m, n] ), summed in split order.
__global__ void k_w4_reduce(const float* __restrict__ part, int nsplit, int64_t MN, __nv_bfloat16* __restrict__ y) {
    for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4; i < MN; i += (int64_t)gridDim.x * blockDim.x * 4) {
        float4 acc = *reinterpret_cast<const float4*>(part + i);
        for (int s = 1; s < nsplit; ++s) {
            float4 v = *reinterpret_cast<const float4*>(part + (int64_t)s * MN + i);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        __nv_bfloat162 p0 = __floats2bfloat162_rn(acc.x, acc.y);
        __nv_bfloat162 p1 = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&p0);
        u.y = *reinterpret_cast<uint32_t*>(&p1);
        *reinterpret_cast<uint2*>(y + i) = u;
    }
}

// ------------------------------------------------------------------ planning
struct W4Plan {
    bool tc;          // tensor-core path
    int ntok;         // tokens per CTA (TMA box rows, MMA N)
    int64_t mtiles;
    int nsplit;
};

static W4Plan w4_plan(int64_t M, int64_t N, int64_t K) {
    W4Plan p{};
    p.tc = (M > 16) && (N % w4tc::BMW == 0) && (K % 64 == 0);
    if (!p.tc) return p;
    p.ntok = (int)((M >= 256) ? 256 : ((M + 15) / 16) * 16);
    p.mtiles = ceil_div(M, p.ntok);
    const int64_t tiles = (N / w4tc::BMW) * p.mtiles;
    const int64_t nchunk = K / 64;
    const int sms = num_sms();
    // pick the split that minimizes (wave-quantized compute) + (partial-sum traffic)
    double best = 1e30;
    int best_s = 1;
    for (int s = 1; s <= 16; ++s) {
        if (nchunk / s < 8 && s > 1) break;  // at least 512 k per split
        int64_t ctas = tiles * s;
        double waves = (double)ceil_div(ctas, sms);
        double compute = waves / s;                  // in units of one full-K tile per SM
        double traffic = (s > 1) ? (double)s * M * N * 8.0 : 0.0;  // partial write + read bytes
        // convert traffic to the compute unit: one full-K 128 x ntok tile on one SM
        double tile_flops = 2.0 * w4tc::BMW * p.ntok * (double)K;
        double per_sm_flops = 8.0e12;                // ~ one SM's bf16 rate
        double traffic_units = traffic / 6.0e12 / (tile_flops / per_sm_flops);
        double cost = compute + traffic_units;
        if (cost < best - 1e-9) {
            best = cost;
            best_s = s;
        }
    }
    p.nsplit = best_s;
    return p;
}

size_t w4a16_ws_bytes(int64_t M, int64_t N, int64_t K) {
    W4Plan p = w4_plan(M, N, K);
    if (!p.tc || p.nsplit <= 1) return 0;
    return (size_t)p.nsplit * M * N * sizeof(float);
}

// QLIN_W4A16_KERNEL=mma forces the mma.sync GEMM for M > 16, =smem the
// tcgen05 GEMM with the A operand in shared memory (comparisons); read on
// every call.
static bool w4_force_mma() {
    const char* e = getenv("QLIN_W4A16_KERNEL");
    return e && strcmp(e, "mma") == 0;
}
static bool w4_force_smem_a() {
    const char* e = getenv("QLIN_W4A16_KERNEL");
    return e && strcmp(e, "smem") == 0;
}

// k-blocks per accumulation chain.  The tensor cores' fp32 accumulation loses
// accuracy over long chains; promoting every 8 k-blocks (512 k) keeps the
// error near 2e-5 of the output scale, every 32 near 2e-4 (8192 x 28672 UINT4).
// With ntok <= 128 two TMEM accumulators alternate and promotion does not
// stall the MMAs; above that one accumulator must be drained in place, so the
// chains are longer.  Both lengths are even, so the TMEM-operand kernel
// (128-k stages) and the shared-memory-operand kernel (64-k blocks) promote
// after the same k-blocks and give the same bits.
static int w4_promote(int ntok) { return ntok <= 128 ? 8 : 32; }

cudaError_t run_gemm_w4a16(const void* x, const void* packed, const qlin_w4_header* h, int64_t M, void* y, void* ws,
                           cudaStream_t st) {
    const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(x);
    const uint8_t* blob = reinterpret_cast<const uint8_t*>(packed);
    __nv_bfloat16* yb = reinterpret_cast<__nv_bfloat16*>(y);
    if (M <= 16) {
        // Two 16-row tiles per CTA (one activation load serves both) when that
        // still leaves at least one CTA per SM.
        const bool two = (h->N % 32 == 0) && (h->N / 32 >= num_sms());
        if (h->K % 128 == 0) {
            if (M <= 8)
                return two ? launch_gemv2g<1, 2>(xb, blob, *h, M, yb, st) : launch_gemv2g<1, 1>(xb, blob, *h, M, yb, st);
            return two ? launch_gemv2g<2, 2>(xb, blob, *h, M, yb, st) : launch_gemv2g<2, 1>(xb, blob, *h, M, yb, st);
        }
        if (M <= 8) return two ? launch_gemv<1, 2>(xb, blob, *h, M, yb, st) : launch_gemv<1, 1>(xb, blob, *h, M, yb, st);
        return two ? launch_gemv<2, 2>(xb, blob, *h, M, yb, st) : launch_gemv<2, 1>(xb, blob, *h, M, yb, st);
    }
    unsigned ntiles = (unsigned)(h->N / 16);
    W4Plan plan = w4_plan(M, h->N, h->K);
    PFN_encodeTiled enc = plan.tc ? encode_tiled_fn() : nullptr;
    if (!plan.tc || !enc || w4_force_mma()) {
        dim3 grid((unsigned)ceil_div(ntiles, 8), (unsigned)ceil_div(M, kW4BM));
        k_w4_gemm_mma<<<grid, 256, 0, st>>>(xb, blob, *h, M, yb);
        return cudaGetLastError();
    }
    CUtensorMap tmap;
    cuuint64_t gdim[2] = {(cuuint64_t)h->K, (cuuint64_t)M};
    cuuint64_t gstride[1] = {(cuuint64_t)h->K * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)plan.ntok};
    cuuint32_t estride[2] = {1, 1};
    if (enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), gdim, gstride, box, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    W4TcArgs a;
    a.blob = blob;
    a.h = *h;
    a.M = M;
    a.ntok = plan.ntok;
    a.nchunk = (int)(h->K / 64);
    a.nsplit = plan.nsplit;
    const bool tmem_a = plan.ntok <= 128 && !w4_force_smem_a();  // A operand in TMEM (k_w4_gemm_tm)
    a.a_stages = tmem_a ? w4tm::a_stages(plan.ntok) : w4tc::a_stages(plan.ntok);
    a.b_stages = tmem_a ? w4tm::b_stages(plan.ntok) : w4tc::b_stages(plan.ntok);
    a.promote = w4_promote(plan.ntok);
    a.idesc = tc::idesc_f16(w4tc::BMW, plan.ntok, true);
    a.part = (plan.nsplit > 1) ? reinterpret_cast<float*>(ws) : nullptr;
    a.y = yb;
    const void* kern = tmem_a ? (const void*)k_w4_gemm_tm : (const void*)k_w4_gemm_tc;
    const size_t smem = tmem_a ? w4tm::smem_bytes(plan.ntok) : w4tc::smem_bytes(plan.ntok);
    cudaError_t e = ensure_smem(kern, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(h->N / w4tc::BMW), (unsigned)plan.nsplit, (unsigned)plan.mtiles);
    if (tmem_a)
        k_w4_gemm_tm<<<grid, w4tm::THREADS, smem, st>>>(tmap, a);
    else
        k_w4_gemm_tc<<<grid, w4tc::THREADS, smem, st>>>(tmap, a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (plan.nsplit > 1) {
        int64_t MN = M * h->N;
        k_w4_reduce<<<num_sms() * 4, 256, 0, st>>>(a.part, plan.nsplit, MN, yb);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace qlin
