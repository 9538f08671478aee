// kvcache.cu -- KV-cache quantization in token groups outside a recent window.
//
// Method ("第11章 模型量化与压缩" 11.6.3 granularity, 11.6.4 K/V sensitivity,
// 11.6.5 low-bit schemes and KIVI's grouped on-demand quantization): K is
// quantized per channel (one scale / zero point per channel over a group of
// G tokens, since K's outliers sit in channels), V per token (one per token
// and head, over head_dim channels); the most recent tokens stay in 16-bit
// and a group of G tokens is quantized once it has left the window of R
// recent tokens.  Codes are asymmetric, [0, 2^bits - 1], with the quantizer
// of qlin_quantize (range widened to contain 0, round-half-even of the
// correctly rounded quotient, zero point added after rounding).
//
// State: the quantized store (codes, scales, zero points of tokens
// [0, quantized)) and a bf16 ring of R + G slots holding tokens
// [quantized, length) at slot t mod (R + G).
#include "qlin_common.cuh"
#include "qlin_internal.h"

namespace qlin {

struct KvArgs {
    const __nv_bfloat16* k_new;  // [n x C] tokens [T, T + n)
    const __nv_bfloat16* v_new;
    int64_t T;                   // length before this append
    int64_t q0;                  // first token to quantize (multiple of G)
    int64_t ngroups;             // groups [q0 / G, q0 / G + ngroups)
    int C, D, G, slots, bits;
    uint8_t* k_codes;
    uint8_t* v_codes;
    float* k_scale;
    int32_t* k_zero;
    float* v_scale;
    int32_t* v_zero;
    __nv_bfloat16* k_ring;
    __nv_bfloat16* v_ring;
};

__device__ __forceinline__ const __nv_bfloat16* kv_src(const __nv_bfloat16* ring, const __nv_bfloat16* fresh,
                                                     int64_t t, int64_t T, int slots, int C) {
    return t < T ? ring + (t % slots) * (int64_t)C : fresh + (t - T) * (int64_t)C;
}

__device__ __forceinline__ uint32_t kv_code(float v, const ScopeParams& sp, int qmax) {
    return code_bits(v, sp, make_range(0, qmax));
}

// K: a CTA of 32 channel pairs x 8 token slices per (group, 64 channels).
// Each thread reduces its slice of the group's G tokens for its two
// channels; thread row 0 combines the 8 slices into the scales and zero
// points; then every thread writes the codes of its slice (adjacent channels
// share a byte for 4-bit codes).
constexpr int KV_KX = 32, KV_KY = 8;

__global__ void __launch_bounds__(KV_KX * KV_KY) k_kv_quant_k(KvArgs a) {
    __shared__ float red[4][KV_KY][KV_KX];
    __shared__ float sc_s[2][KV_KX];
    __shared__ int sc_z[2][KV_KX];
    const int qmax = (1 << a.bits) - 1;
    const int tx = threadIdx.x % KV_KX, ty = threadIdx.x / KV_KX;
    const int c = (blockIdx.x * KV_KX + tx) * 2;
    const bool live = c < a.C;
    const int64_t g = blockIdx.y;
    const int64_t t0 = a.q0 + g * a.G;
    float lo0 = 0.0f, hi0 = 0.0f, lo1 = 0.0f, hi1 = 0.0f;
    if (live) {
        for (int j = ty; j < a.G; j += KV_KY) {
            const float2 f = __bfloat1622float2(
                *reinterpret_cast<const __nv_bfloat162*>(kv_src(a.k_ring, a.k_new, t0 + j, a.T, a.slots, a.C) + c));
            hi0 = fmaxf(hi0, f.x);
            lo0 = fminf(lo0, f.x);
            hi1 = fmaxf(hi1, f.y);
            lo1 = fminf(lo1, f.y);
        }
    }
    red[0][ty][tx] = hi0;
    red[1][ty][tx] = lo0;
    red[2][ty][tx] = hi1;
    red[3][ty][tx] = lo1;
    __syncthreads();
    const int64_t gi = t0 / a.G;
    if (ty == 0) {
#pragma unroll
        for (int y = 1; y < KV_KY; ++y) {
            hi0 = fmaxf(hi0, red[0][y][tx]);
            lo0 = fminf(lo0, red[1][y][tx]);
            hi1 = fmaxf(hi1, red[2][y][tx]);
            lo1 = fminf(lo1, red[3][y][tx]);
        }
        float s0, s1;
        int z0, z1;
        scale_zero(lo0, hi0, 0, qmax, false, false, s0, z0);
        scale_zero(lo1, hi1, 0, qmax, false, false, s1, z1);
        sc_s[0][tx] = s0;
        sc_s[1][tx] = s1;
        sc_z[0][tx] = z0;
        sc_z[1][tx] = z1;
        if (live) {
            a.k_scale[gi * a.C + c] = s0;
            a.k_scale[gi * a.C + c + 1] = s1;
            a.k_zero[gi * a.C + c] = z0;
            a.k_zero[gi * a.C + c + 1] = z1;
        }
    }
    __syncthreads();
    if (!live) return;
    const ScopeParams sp0 = make_scope(sc_s[0][tx], sc_z[0][tx]), sp1 = make_scope(sc_s[1][tx], sc_z[1][tx]);
    for (int j = ty; j < a.G; j += KV_KY) {
        const int64_t t = t0 + j;
        const float2 f = __bfloat1622float2(
            *reinterpret_cast<const __nv_bfloat162*>(kv_src(a.k_ring, a.k_new, t, a.T, a.slots, a.C) + c));
        const uint32_t q0 = kv_code(f.x, sp0, qmax) & 0xFFu, q1 = kv_code(f.y, sp1, qmax) & 0xFFu;
        if (a.bits == 4) {
            a.k_codes[t * (a.C / 2) + c / 2] = (uint8_t)((q0 & 0xFu) | ((q1 & 0xFu) << 4));
        } else {
            a.k_codes[t * a.C + c] = (uint8_t)q0;
            a.k_codes[t * a.C + c + 1] = (uint8_t)q1;
        }
    }
}

// V: one warp per (token, head) -- min/max over head_dim channels, the scale
// and zero point, then the codes (lane l takes channel pairs 2l, 2l + 64, ...).
__global__ void k_kv_quant_v(KvArgs a) {
    const int qmax = (1 << a.bits) - 1;
    const int lane = threadIdx.x & 31;
    const int heads = a.C / a.D;
    const int64_t units = (int64_t)a.ngroups * a.G * heads;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t u = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < units; u += nwarps) {
        const int64_t t = a.q0 + u / heads;
        const int h = (int)(u % heads);
        const __nv_bfloat16* row = kv_src(a.v_ring, a.v_new, t, a.T, a.slots, a.C) + (int64_t)h * a.D;
        float lo = 0.0f, hi = 0.0f;
        for (int c = 2 * lane; c < a.D; c += 64) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(row + c));
            hi = fmaxf(hi, fmaxf(f.x, f.y));
            lo = fminf(lo, fminf(f.x, f.y));
        }
        hi = warp_max(hi);
        lo = warp_min(lo);
        float s;
        int z;
        scale_zero(lo, hi, 0, qmax, false, false, s, z);
        if (lane == 0) {
            a.v_scale[t * heads + h] = s;
            a.v_zero[t * heads + h] = z;
        }
        const ScopeParams sp = make_scope(s, z);
        for (int c = 2 * lane; c < a.D; c += 64) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(row + c));
            const uint32_t q0 = kv_code(f.x, sp, qmax) & 0xFFu, q1 = kv_code(f.y, sp, qmax) & 0xFFu;
            const int64_t e = t * a.C + (int64_t)h * a.D + c;
            if (a.bits == 4) {
                a.v_codes[e / 2] = (uint8_t)((q0 & 0xFu) | ((q1 & 0xFu) << 4));
            } else {
                a.v_codes[e] = (uint8_t)q0;
                a.v_codes[e + 1] = (uint8_t)q1;
            }
        }
    }
}

// New tokens [first, T + n) that stay in 16-bit go to their ring slots.
__global__ void k_kv_to_ring(KvArgs a, int64_t first, int64_t n) {
    const int64_t last = a.T + n;
    const int64_t per = a.C / 8;  // 16-byte pieces per token
    const int64_t total = (last - first) * per;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = first + i / per, p = i % per;
        const int64_t src = (t - a.T) * per + p, dst = (t % a.slots) * per + p;
        reinterpret_cast<uint4*>(a.k_ring)[dst] = __ldg(reinterpret_cast<const uint4*>(a.k_new) + src);
        reinterpret_cast<uint4*>(a.v_ring)[dst] = __ldg(reinterpret_cast<const uint4*>(a.v_new) + src);
    }
}

// The cache as attention reads it: tokens [0, quantized) dequantized,
// fl(s * (q - z)) rounded to bf16, tokens [quantized, length) from the ring.
// One thread per 8 consecutive channels of one token.
struct KvReadArgs {
    const uint8_t *k_codes, *v_codes;
    const float *k_scale, *v_scale;
    const int32_t *k_zero, *v_zero;
    const __nv_bfloat16 *k_ring, *v_ring;
    int64_t length, quantized;
    int C, D, G, slots, bits;
    __nv_bfloat16 *k_out, *v_out;
};

__device__ __forceinline__ void kv_codes8(const uint8_t* codes, int64_t e, int bits, int q[8]) {
    if (bits == 4) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(codes + e / 2);
#pragma unroll
        for (int j = 0; j < 8; ++j) q[j] = (w >> (4 * j)) & 0xF;
    } else {
        const uint2 w = *reinterpret_cast<const uint2*>(codes + e);
#pragma unroll
        for (int j = 0; j < 8; ++j) q[j] = ((j < 4 ? w.x : w.y) >> (8 * (j & 3))) & 0xFF;
    }
}

constexpr int KV_READ_TOK = 8;  // tokens per thread in k_kv_read

// Thread unit: 8 consecutive channels of 8 consecutive tokens; K's scales
// and zero points (per group and channel) are loaded once per group.
__global__ void __launch_bounds__(256) k_kv_read(KvReadArgs a) {
    const int64_t per = a.C / 8;
    const int64_t tblocks = ceil_div(a.length, (int64_t)KV_READ_TOK);
    const int64_t total = tblocks * per;
    const int heads = a.C / a.D;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tb = i / per;
        const int c0 = (int)(i - tb * per) * 8;
        int64_t g_loaded = -1;
        float ks[8];
        int kz[8];
        for (int u = 0; u < KV_READ_TOK; ++u) {
            const int64_t t = tb * KV_READ_TOK + u;
            if (t >= a.length) break;
            const int64_t o = t * per + c0 / 8;
            uint4 ko, vo;
            if (t < a.quantized) {
                const int64_t g = t / a.G;
                if (g != g_loaded) {
                    const float4* sp = reinterpret_cast<const float4*>(a.k_scale + g * a.C + c0);
                    const int4* zp = reinterpret_cast<const int4*>(a.k_zero + g * a.C + c0);
                    const float4 s0 = __ldg(sp), s1 = __ldg(sp + 1);
                    const int4 z0 = __ldg(zp), z1 = __ldg(zp + 1);
                    ks[0] = s0.x; ks[1] = s0.y; ks[2] = s0.z; ks[3] = s0.w;
                    ks[4] = s1.x; ks[5] = s1.y; ks[6] = s1.z; ks[7] = s1.w;
                    kz[0] = z0.x; kz[1] = z0.y; kz[2] = z0.z; kz[3] = z0.w;
                    kz[4] = z1.x; kz[5] = z1.y; kz[6] = z1.z; kz[7] = z1.w;
                    g_loaded = g;
                }
                const int64_t e = t * a.C + c0;
                int qk[8], qv[8];
                kv_codes8(a.k_codes, e, a.bits, qk);
                kv_codes8(a.v_codes, e, a.bits, qv);
                const int64_t sv = t * heads + c0 / a.D;  // 8 channels never straddle a head (D % 8 == 0)
                const float vs = __ldg(a.v_scale + sv);
                const int vz = __ldg(a.v_zero + sv);
                uint32_t kw[4], vw[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float k0 = __fmul_rn(ks[2 * j], (float)(qk[2 * j] - kz[2 * j]));
                    const float k1 = __fmul_rn(ks[2 * j + 1], (float)(qk[2 * j + 1] - kz[2 * j + 1]));
                    const float v0 = __fmul_rn(vs, (float)(qv[2 * j] - vz));
                    const float v1 = __fmul_rn(vs, (float)(qv[2 * j + 1] - vz));
                    __nv_bfloat162 kb = __floats2bfloat162_rn(k0, k1), vb = __floats2bfloat162_rn(v0, v1);
                    kw[j] = *reinterpret_cast<uint32_t*>(&kb);
                    vw[j] = *reinterpret_cast<uint32_t*>(&vb);
                }
                ko = make_uint4(kw[0], kw[1], kw[2], kw[3]);
                vo = make_uint4(vw[0], vw[1], vw[2], vw[3]);
            } else {
                const int64_t r = (t % a.slots) * per + c0 / 8;
                ko = __ldg(reinterpret_cast<const uint4*>(a.k_ring) + r);
                vo = __ldg(reinterpret_cast<const uint4*>(a.v_ring) + r);
            }
            reinterpret_cast<uint4*>(a.k_out)[o] = ko;
            reinterpret_cast<uint4*>(a.v_out)[o] = vo;
        }
    }
}

// ------------------------------------------------------------------ layout and launchers
void kv_layout(int64_t capacity, int C, int D, int G, int R, int bits, size_t off[8], size_t* total) {
    auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
    const size_t code_bytes = (size_t)capacity * C * bits / 8;
    const size_t groups = (size_t)(capacity / G);
    const size_t heads = (size_t)(C / D);
    const size_t slots = (size_t)(R + G);
    size_t o = 0;
    off[0] = o; o = up(o + code_bytes);                 // k codes
    off[1] = o; o = up(o + code_bytes);                 // v codes
    off[2] = o; o = up(o + groups * C * 4);             // k scales
    off[3] = o; o = up(o + groups * C * 4);             // k zero points
    off[4] = o; o = up(o + (size_t)capacity * heads * 4);  // v scales
    off[5] = o; o = up(o + (size_t)capacity * heads * 4);  // v zero points
    off[6] = o; o = up(o + slots * C * 2);              // k ring
    off[7] = o; o = up(o + slots * C * 2);              // v ring
    *total = o;
}

cudaError_t run_kv_append(const qlin_kv_cache* c, const void* k_new, const void* v_new, int64_t n, int64_t q_new,
                          cudaStream_t st) {
    KvArgs a;
    a.k_new = reinterpret_cast<const __nv_bfloat16*>(k_new);
    a.v_new = reinterpret_cast<const __nv_bfloat16*>(v_new);
    a.T = c->length;
    a.q0 = c->quantized;
    a.ngroups = (q_new - c->quantized) / c->group;
    a.C = c->channels;
    a.D = c->head_dim;
    a.G = c->group;
    a.slots = c->residual + c->group;
    a.bits = c->bits;
    a.k_codes = reinterpret_cast<uint8_t*>(c->k_codes);
    a.v_codes = reinterpret_cast<uint8_t*>(c->v_codes);
    a.k_scale = c->k_scale;
    a.k_zero = c->k_zero;
    a.v_scale = c->v_scale;
    a.v_zero = c->v_zero;
    a.k_ring = reinterpret_cast<__nv_bfloat16*>(c->k_recent);
    a.v_ring = reinterpret_cast<__nv_bfloat16*>(c->v_recent);
    cudaError_t e;
    if (a.ngroups > 0) {
        for (int64_t g0 = 0; g0 < a.ngroups; g0 += 65535) {  // grid.y holds at most 65535 groups
            KvArgs b = a;
            b.q0 = a.q0 + g0 * a.G;
            b.ngroups = a.ngroups - g0 < 65535 ? a.ngroups - g0 : 65535;
            dim3 gk((unsigned)ceil_div(a.C / 2, KV_KX), (unsigned)b.ngroups);
            k_kv_quant_k<<<gk, KV_KX * KV_KY, 0, st>>>(b);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
        const int64_t warps = a.ngroups * a.G * (a.C / a.D);
        int64_t grid = ceil_div(warps, 8);
        if (grid > (int64_t)num_sms() * 8) grid = (int64_t)num_sms() * 8;
        k_kv_quant_v<<<(unsigned)grid, 256, 0, st>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    const int64_t first = q_new > a.T ? q_new : a.T;  // new tokens that stay in 16-bit
    if (a.T + n > first) {
        const int64_t pieces = (a.T + n - first) * (a.C / 8);
        int64_t grid = ceil_div(pieces, 256);
        if (grid > (int64_t)num_sms() * 8) grid = (int64_t)num_sms() * 8;
        k_kv_to_ring<<<(unsigned)grid, 256, 0, st>>>(a, first, n);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t run_kv_read(const qlin_kv_cache* c, void* k_out, void* v_out, cudaStream_t st) {
    KvReadArgs a;
    a.k_codes = reinterpret_cast<const uint8_t*>(c->k_codes);
    a.v_codes = reinterpret_cast<const uint8_t*>(c->v_codes);
    a.k_scale = c->k_scale;
    a.v_scale = c->v_scale;
    a.k_zero = c->k_zero;
    a.v_zero = c->v_zero;
    a.k_ring = reinterpret_cast<const __nv_bfloat16*>(c->k_recent);
    a.v_ring = reinterpret_cast<const __nv_bfloat16*>(c->v_recent);
    a.length = c->length;
    a.quantized = c->quantized;
    a.C = c->channels;
    a.D = c->head_dim;
    a.G = c->group;
    a.slots = c->residual + c->group;
    a.bits = c->bits;
    a.k_out = reinterpret_cast<__nv_bfloat16*>(k_out);
    a.v_out = reinterpret_cast<__nv_bfloat16*>(v_out);
    const int64_t total = ceil_div(a.length, (int64_t)KV_READ_TOK) * (a.C / 8);
    int64_t grid = ceil_div(total, 256);
    if (grid > (int64_t)num_sms() * 8) grid = (int64_t)num_sms() * 8;
    if (grid < 1) return cudaSuccess;
    k_kv_read<<<(unsigned)grid, 256, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace qlin
