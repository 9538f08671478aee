// qlin_common.cuh -- device helpers shared by the qlin kernels (sm_103a).
//
// The arithmetic here is the affine quantizer of the pages "量化、蒸馏与模型压缩"
// (core formula) and "第11章 模型量化与压缩" 11.1.1-11.1.2: codes are
// clip(rne(fl(x/s)) + z, qmin, qmax) with fl() the correctly rounded binary32
// quotient.  The fast path below reaches exactly that result without a
// division per element.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/qlin.h"

namespace qlin {

// ---------------------------------------------------------------- device error word
// Set by kernels whose bounded waits give up; read and cleared by
// qlin_device_error().
__device__ int g_device_error = 0;

__device__ __forceinline__ void raise_device_error(int code) { atomicExch(&g_device_error, code); }

// Cycle limit of every bounded device-side wait (about 2 s at 2 GHz), in
// constant memory: the waits read it from the constant cache.  Changed only
// between kernels (qlin_debug_stall_producers synchronizes the device).
constexpr long long kDefaultWaitLimitCycles = 4000000000LL;
__constant__ long long g_wait_limit_cycles = kDefaultWaitLimitCycles;
// Failure-detection test hook (qlin_debug_stall_producers): while non-zero,
// the producer roles of the pipelined kernels issue no copies, so the
// consumers' bounded waits run out and the kernels take their abort path.
__constant__ int g_stall_producers = 0;

// ---------------------------------------------------------------- loads / stores
template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <>
__device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }

// Widen 8 consecutive elements starting at p (16-byte aligned for the 16-bit
// types, 32-byte aligned for binary32) into v[0..7].
template <typename T>
__device__ __forceinline__ void load8(const T* p, float v[8]);

template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float v[8]) {
    uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

template <>
__device__ __forceinline__ void load8<__half>(const __half* p, float v[8]) {
    uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h = *reinterpret_cast<__half2*>(&w[i]);
        float2 f = __half22float2(h);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}

template <>
__device__ __forceinline__ void load8<float>(const float* p, float v[8]) {
    float4 a = __ldg(reinterpret_cast<const float4*>(p));
    float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <typename T>
__device__ __forceinline__ float load1(const T* p) { return to_f32<T>(p[0]); }

// Widen 8 packed 16-bit values (one 16-byte chunk) to binary32.
template <typename T>
__device__ __forceinline__ void unpack8(const uint4 u, float v[8]);
template <>
__device__ __forceinline__ void unpack8<__nv_bfloat16>(const uint4 u, float v[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}
template <>
__device__ __forceinline__ void unpack8<__half>(const uint4 u, float v[8]) {
    uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __half22float2(*reinterpret_cast<__half2*>(&w[i]));
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}
template <>
__device__ __forceinline__ void unpack8<float>(const uint4, float v[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 0.0f;  // not used: binary32 rows take another kernel
}

// ---------------------------------------------------------------- scale / zero point
struct ScopeParams {
    float s;      // stored scale (binary32 value of the stored scale)
    float r;      // approximate 1/s, only used to guess the code
    float hs;     // s * (0.5 - 2^-11): half-step minus a safety margin
    float cz;     // 1.5*2^23 + z
};

// Clamp bounds of code_bits() in the 1.5*2^23 + code domain.
// lo2 / hi2: qmin / qmax in both 16-bit lanes, for clamp_pair16.
struct CodeRange {
    float lo, hi;
    uint32_t lo2, hi2;
};
__device__ __forceinline__ CodeRange make_range(int qmin, int qmax) {
    CodeRange c;
    c.lo = 12582912.0f + (float)qmin;
    c.hi = 12582912.0f + (float)qmax;
    c.lo2 = (uint32_t)(uint16_t)qmin * 0x10001u;
    c.hi2 = (uint32_t)(uint16_t)qmax * 0x10001u;
    return c;
}

// Round a scale to binary16 (nearest-even) saturating at 65504, as a binary32 value.
__device__ __forceinline__ float round_f16_sat(float s) {
    float r = __half2float(__float2half_rn(s));
    if (isinf(r)) r = copysignf(65504.0f, s);
    return r;
}

// Dynamic scale and zero point from the scope statistics
// ([CH11] 11.1.1-11.1.2; [CSDN] symmetric / asymmetric sections).
//   symmetric : hi = max|x|          -> s = fl(hi / qmax), z = 0
//   asymmetric: lo = min(min x, 0), hi = max(max x, 0)
//               -> s = fl(fl(hi - lo) / (qmax - qmin)), z = clip(qmin + rne(fl(-lo/s)))
__device__ __forceinline__ void scale_zero(float lo, float hi, int qmin, int qmax, bool sym,
                                           bool f16, float& s, int& z) {
    if (sym) {
        s = __fdiv_rn(hi, (float)qmax);
    } else {
        s = __fdiv_rn(__fsub_rn(hi, lo), (float)(qmax - qmin));
    }
    if (f16) s = round_f16_sat(s);
    if (s == 0.0f) s = 1.0f;
    if (sym) {
        z = 0;
    } else {
        float t = rintf(__fdiv_rn(-lo, s));
        float zz = fminf(fmaxf(t + (float)qmin, (float)qmin), (float)qmax);
        z = (int)zz;
    }
}

__device__ __forceinline__ ScopeParams make_scope(float s, int z);

// scale_zero then make_scope, out of line: per-group loops call it once per
// group and unrolled copies of the correctly rounded divisions would fill the
// instruction cache.
struct ScopeOf {
    float s;
    int z;
};
__device__ __noinline__ ScopeOf scope_of_range(float lo, float hi, int qmin, int qmax, bool sym, bool f16) {
    ScopeOf r;
    scale_zero(lo, hi, qmin, qmax, sym, f16, r.s, r.z);
    return r;
}

__device__ __forceinline__ ScopeParams make_scope(float s, int z) {
    ScopeParams p;
    p.s = s;
    p.r = __frcp_rn(s);
    p.hs = s * 0.49951171875f;
    p.cz = 12582912.0f + (float)z;
    return p;
}

// Code of one (already smoothed) value, returned as the bit pattern of the
// binary32 number 1.5*2^23 + code, so that its low byte is the two's-complement
// code byte and its low nibble the 4-bit code.
//
// Exactness: t = v*r is within a few ulp of v/s.  When |t| < 4096 the
// candidate n = rne(t) (1.5*2^23 trick, exact round-half-even) gives an exact
// remainder d = v - n*s (fma; n*s and v share the quantum of s).  If |d| stays
// below (0.5 - 2^-11)*s the true quotient is more than 2^-11 away from a
// half-integer, so fl(v/s) (within 2^-13 of v/s here) rounds to the same n and
// rne(t) + z = rne(t + z).  Every other case -- a near-tie, a value far
// outside the code range, an overflowing reciprocal -- takes the correctly
// rounded division.
__device__ __forceinline__ uint32_t code_bits(float v, const ScopeParams& p, const CodeRange& cr) {
    float t = v * p.r;
    float m;
    if (fabsf(t) < 4096.0f) {
        m = t + p.cz;                          // rne(t) + 1.5*2^23 + z
        float n = m - p.cz;                    // rne(t), exact
        float d = fmaf(-n, p.s, v);            // exact remainder
        if (!(fabsf(d) < p.hs)) {
            float q = rintf(__fdiv_rn(v, p.s));
            m = fminf(fmaxf(q, -8388608.0f), 8388608.0f) + p.cz;
        }
    } else {
        float q = rintf(__fdiv_rn(v, p.s));
        m = fminf(fmaxf(q, -8388608.0f), 8388608.0f) + p.cz;
    }
    m = fminf(fmaxf(m, cr.lo), cr.hi);
    return __float_as_uint(m);
}

// code_bits() for values known to satisfy |v/s| <= qmax + 1 (dynamic scales
// computed from the same scope): the far-range branch is dropped; near-ties
// still take the correctly rounded division.
__device__ __forceinline__ uint32_t code_bits_inrange(float v, const ScopeParams& p, const CodeRange& cr) {
    const float t = v * p.r;
    float m = t + p.cz;
    const float n = m - p.cz;
    const float d = fmaf(-n, p.s, v);
    if (!(fabsf(d) < p.hs)) {
        const float q = rintf(__fdiv_rn(v, p.s));
        m = fminf(fmaxf(q, -8388608.0f), 8388608.0f) + p.cz;
    }
    m = fminf(fmaxf(m, cr.lo), cr.hi);
    return __float_as_uint(m);
}

// Packed binary32 pairs (sm_100 family): each lane of the pair is an IEEE
// operation rounded to nearest, exactly as its scalar counterpart.
__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 f2_add(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// The exact per-element path of a chunk that failed the fast test (a
// near-tie, or a value far outside the code range), out of line: kernels
// that unroll many chunks with little register pressure take it (inlined
// at every unrolled chunk it fills the instruction cache), kernels with many
// live registers keep it inline (a call would save them around it).
__device__ __noinline__ void code_bits8_exact(float v0, float v1, float v2, float v3, float v4, float v5, float v6,
                                              float v7, ScopeParams p, CodeRange cr, uint32_t* cb) {
    const float v[8] = {v0, v1, v2, v3, v4, v5, v6, v7};
#pragma unroll 1
    for (int j = 0; j < 8; ++j) cb[j] = code_bits(v[j], p, cr);
}

// code_bits() of eight values with one branch.  The fast candidates of all
// eight are formed in one basic block on packed pairs, and the near-tie test
// |d| < hs becomes the sign of d*d - hs*hs (one fused multiply-add per pair;
// its rounding can only move the outcome for |d| within an ulp of hs, where
// either path gives the right code, since hs keeps a 2^-11 * s margin from
// the tie; a NaN has a clear sign bit and fails the test).  Likewise
// |t| < 4096 is tested as t*t - 2^24 < 0 unless kInRange.  A chunk that fails
// re-derives every element through the scalar function.  kClamp = false drops
// the clamp to [qmin, qmax]; callers use it only for symmetric scopes whose
// scale came from the scope's own absmax, where |rne(v/s)| <= qmax always
// holds.  Same results as code_bits() / code_bits_inrange() per element.
// Two code candidates m0, m1 (bit patterns of 1.5*2^23 + z + n, |z + n| <
// 2^15) as one word of two 16-bit lanes, each z + n in two's complement (the
// low 16 bits of the pattern), clamped to [qmin, qmax] lane by lane: the same
// integers as clamping the binary32 candidates, for one permute and two
// instructions per pair.
__device__ __forceinline__ uint32_t clamp_pair16(uint32_t m0, uint32_t m1, const CodeRange& cr) {
    const uint32_t p = __byte_perm(m0, m1, 0x5410);
    uint32_t d;
    asm("max.s16x2 %0, %1, %2;" : "=r"(d) : "r"(p), "r"(cr.lo2));
    asm("min.s16x2 %0, %1, %2;" : "=r"(d) : "r"(d), "r"(cr.hi2));
    return d;
}
// Eight codes from four clamp_pair16 words: bytes (code j in byte j), or
// nibbles (element 2i in the low nibble of byte i).
__device__ __forceinline__ uint2 pack_pairs_bytes(const uint32_t p[4]) {
    return make_uint2(__byte_perm(p[0], p[1], 0x6420), __byte_perm(p[2], p[3], 0x6420));
}
__device__ __forceinline__ uint32_t pack_pairs_nibbles(const uint32_t p[4]) {
    uint32_t b0 = __byte_perm(p[0], p[1], 0x6420) & 0x0F0F0F0Fu;
    uint32_t b1 = __byte_perm(p[2], p[3], 0x6420) & 0x0F0F0F0Fu;
    b0 = b0 | (b0 >> 4);
    b1 = b1 | (b1 >> 4);
    return __byte_perm(b0, b1, 0x6420);
}

// kPairs (with kClamp): cb[0..3] receive the codes as clamp_pair16 words
// (for pack_pairs_bytes / pack_pairs_nibbles) instead of eight clamped
// candidates.
template <bool kInRange, bool kClamp = true, bool kOutline = false, bool kPairs = false>
__device__ __forceinline__ void code_bits8(const float v[8], const ScopeParams& p, const CodeRange& cr,
                                           uint32_t cb[8]) {
    static_assert(!kPairs || kClamp, "pair words carry clamped codes");
    float m[8];
    uint32_t neg = 0xFFFFFFFFu;  // AND of the sign bits of the tests
    const float2 r2 = make_float2(p.r, p.r), cz2 = make_float2(p.cz, p.cz), ncz2 = make_float2(-p.cz, -p.cz);
    const float2 ns2 = make_float2(-p.s, -p.s);
    const float hs_sq = p.hs * p.hs;
    const float2 nhs2 = make_float2(-hs_sq, -hs_sq);
    const float2 nlim2 = make_float2(-16777216.0f, -16777216.0f);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 v2 = make_float2(v[2 * j], v[2 * j + 1]);
        const float2 t2 = f2_mul(v2, r2);
        const float2 m2 = f2_add(t2, cz2);      // rne(t) + 1.5*2^23 + z
        const float2 n2 = f2_add(m2, ncz2);     // rne(t), exact
        const float2 d2 = f2_fma(n2, ns2, v2);  // v - n*s, exact
        const float2 e2 = f2_fma(d2, d2, nhs2);
        neg &= __float_as_uint(e2.x) & __float_as_uint(e2.y);
        if (!kInRange) {
            const float2 g2 = f2_fma(t2, t2, nlim2);
            neg &= __float_as_uint(g2.x) & __float_as_uint(g2.y);
        }
        m[2 * j] = m2.x;
        m[2 * j + 1] = m2.y;
    }
    if (neg & 0x80000000u) {
        if constexpr (kPairs) {
#pragma unroll
            for (int k = 0; k < 4; ++k) cb[k] = clamp_pair16(__float_as_uint(m[2 * k]), __float_as_uint(m[2 * k + 1]), cr);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) cb[j] = __float_as_uint(kClamp ? fminf(fmaxf(m[j], cr.lo), cr.hi) : m[j]);
        }
    } else {
        uint32_t t8[8];
        if (kOutline) {
            // (code_bits equals code_bits_inrange wherever the latter applies)
            code_bits8_exact(v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7], p, cr, t8);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) t8[j] = kInRange ? code_bits_inrange(v[j], p, cr) : code_bits(v[j], p, cr);
        }
        if constexpr (kPairs) {
            // clamped candidates: their low 16 bits are the codes
#pragma unroll
            for (int k = 0; k < 4; ++k) cb[k] = __byte_perm(t8[2 * k], t8[2 * k + 1], 0x5410);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) cb[j] = t8[j];
        }
    }
}

// Constants of two adjacent per-column scopes as packed pairs: 1/s
// (approximate), 1.5*2^23 + z, -s and -(hs*hs).
struct ColPair {
    float2 r, cz, ns, nhs2;
};
__device__ __forceinline__ ColPair make_colpair(const ScopeParams& p0, const ScopeParams& p1) {
    ColPair c;
    c.r = make_float2(p0.r, p1.r);
    c.cz = make_float2(p0.cz, p1.cz);
    c.ns = make_float2(-p0.s, -p1.s);
    c.nhs2 = make_float2(-(p0.hs * p0.hs), -(p1.hs * p1.hs));
    return c;
}
// The ScopeParams of one lane of a pair, rebuilt exactly as make_scope
// builds them (s = -(-s); hs = s * (0.5 - 2^-11)).
__device__ __forceinline__ ScopeParams colpair_scope(const ColPair& c, int lane) {
    ScopeParams p;
    p.s = -(lane ? c.ns.y : c.ns.x);
    p.r = lane ? c.r.y : c.r.x;
    p.hs = p.s * 0.49951171875f;
    p.cz = lane ? c.cz.y : c.cz.x;
    return p;
}
__device__ __forceinline__ float2 f2_sub(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __noinline__ uint32_t code_bits_outline(float v, ScopeParams p, CodeRange cr) { return code_bits(v, p, cr); }

// code_bits8 with one scope per element (per-column scopes): the same packed
// fast path with per-lane constants (m - cz is the same operation as
// m + (-cz)); a chunk that fails takes the exact per-element path out of line.
template <bool kInRange, bool kClamp, bool kPairs = false>
__device__ __forceinline__ void code_bits8_cols(const float v[8], const ColPair cp[4], const CodeRange& cr,
                                                uint32_t cb[8]) {
    static_assert(!kPairs || kClamp, "pair words carry clamped codes");
    float m[8];
    uint32_t neg = 0xFFFFFFFFu;
    const float2 nlim2 = make_float2(-16777216.0f, -16777216.0f);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 v2 = make_float2(v[2 * j], v[2 * j + 1]);
        const float2 t2 = f2_mul(v2, cp[j].r);
        const float2 m2 = f2_add(t2, cp[j].cz);
        const float2 n2 = f2_sub(m2, cp[j].cz);
        const float2 d2 = f2_fma(n2, cp[j].ns, v2);
        const float2 e2 = f2_fma(d2, d2, cp[j].nhs2);
        neg &= __float_as_uint(e2.x) & __float_as_uint(e2.y);
        if (!kInRange) {
            const float2 g2 = f2_fma(t2, t2, nlim2);
            neg &= __float_as_uint(g2.x) & __float_as_uint(g2.y);
        }
        m[2 * j] = m2.x;
        m[2 * j + 1] = m2.y;
    }
    if (neg & 0x80000000u) {
        if constexpr (kPairs) {
#pragma unroll
            for (int k = 0; k < 4; ++k) cb[k] = clamp_pair16(__float_as_uint(m[2 * k]), __float_as_uint(m[2 * k + 1]), cr);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) cb[j] = __float_as_uint(kClamp ? fminf(fmaxf(m[j], cr.lo), cr.hi) : m[j]);
        }
    } else {
        uint32_t t8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) t8[j] = code_bits_outline(v[j], colpair_scope(cp[j / 2], j & 1), cr);
        if constexpr (kPairs) {
#pragma unroll
            for (int k = 0; k < 4; ++k) cb[k] = __byte_perm(t8[2 * k], t8[2 * k + 1], 0x5410);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) cb[j] = t8[j];
        }
    }
}

// Pack the low bytes of four code_bits() words: byte i <- a[i].
__device__ __forceinline__ uint32_t pack_bytes4(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3) {
    uint32_t lo = __byte_perm(a0, a1, 0x0040);
    uint32_t hi = __byte_perm(a2, a3, 0x0040);
    return __byte_perm(lo, hi, 0x5410);
}

// Pack eight codes into four bytes of nibbles: element 2i in the low nibble.
__device__ __forceinline__ uint32_t pack_nibbles8(const uint32_t c[8]) {
    uint32_t b0 = pack_bytes4(c[0], c[1], c[2], c[3]) & 0x0F0F0F0Fu;
    uint32_t b1 = pack_bytes4(c[4], c[5], c[6], c[7]) & 0x0F0F0F0Fu;
    b0 = b0 | (b0 >> 4);   // bytes 0 and 2 now hold (c0|c1<<4), (c2|c3<<4)
    b1 = b1 | (b1 >> 4);
    return __byte_perm(b0, b1, 0x6420);
}

// ---------------------------------------------------------------- reductions
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ---------------------------------------------------------------- misc
__host__ __device__ __forceinline__ int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }


// ------------------------------------------------------------------ cp.async
// 16-byte global -> shared copy that writes zeros when !pred.
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, bool pred) {
    int n = pred ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's committed groups are still pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace qlin
