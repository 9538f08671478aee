// quantize.cu -- quantize / dequantize / absmax / smoothing-factor kernels.
//
// Method: the affine quantizer q = clip(round(x/s) + z, qmin, qmax),
// x^ = s(q - z) of "量化、蒸馏与模型压缩" (core formula) and
// "第11章 模型量化与压缩" 11.1.1-11.1.5, at the granularities of
// "十九：模型压缩：量化、ZeroQuant、LLM.int8() 与 SmoothQuant" section 4.
//
// Kernels (all HBM-bound; the design target is one read of x and one write of
// the codes per element where the scope is row-local):
//   k_quant_rows    per-row / per-group scopes: the row is held in registers,
//                   reduced with warp shuffles, quantized and packed in one pass.
//   k_stats_strip   per-tensor / per-column range statistics (atomic max of
//                   non-negative binary32 bit patterns: order-independent, so
//                   deterministic).
//   k_finalize      statistics -> (s, z) per scope.
//   k_quant_strip   per-tensor / per-column codes from stored (s, z).
//   k_*_generic     scalar fallbacks for unaligned or odd shapes.
//   k_hist*/k_select percentile clipping (exact radix select on |x| bits).
//   k_dequant       x^ = fl(s (q - z)) rounded to the output type.
#include <map>
#include <mutex>
#include <tuple>
#include <type_traits>

#include "qlin_common.cuh"
#include "qlin_internal.h"
#include "tc_ptx.cuh"

namespace qlin {

// ------------------------------------------------------------------ parameters
struct QuantArgs {
    const void* x;
    int64_t rows, cols, ld;
    const float* smooth;
    int smooth_mode;
    int qmin, qmax;
    int sym;
    int gran;
    int group;
    int scale_f16;
    int static_scale;
    int code4;        // 1: two codes per byte
    void* q;
    void* s;
    int32_t* z;
    float* absmax_out;  // stats-only mode (qlin_absmax), else nullptr
    // per-tensor / per-column range statistics (see k_stats_strip): when set,
    // the codes kernels derive each scope's (s, z) from them and the scope's
    // first reader writes s / z out; else s / z are read from s / z
    const uint32_t* stat_in = nullptr;
};

__device__ __forceinline__ float load_scale(const void* s, int64_t i, int f16) {
    return f16 ? __half2float(reinterpret_cast<const __half*>(s)[i]) : reinterpret_cast<const float*>(s)[i];
}
__device__ __forceinline__ void store_scale(void* s, int64_t i, int f16, float v) {
    if (f16)
        reinterpret_cast<__half*>(s)[i] = __float2half_rn(v);  // v is already a binary16 value
    else
        reinterpret_cast<float*>(s)[i] = v;
}

// (s, z) of scope i from the range statistics words, exactly as k_finalize
// stores them.
__device__ __forceinline__ ScopeOf scope_from_stat(const QuantArgs& a, const uint32_t* stat, int64_t i) {
    return scope_of_range(-__uint_as_float(stat[2 * i + 1]), __uint_as_float(stat[2 * i]), a.qmin, a.qmax, a.sym,
                          a.scale_f16);
}
// (s, z) of scope i: derived from a.stat_in (the writer stores them), else
// read from s / z.
__device__ __forceinline__ ScopeOf scope_in(const QuantArgs& a, int64_t i, bool writer) {
    ScopeOf o;
    if (a.stat_in) {
        o = scope_from_stat(a, a.stat_in, i);
        if (writer) {
            store_scale(a.s, i, a.scale_f16, o.s);
            if (a.z) a.z[i] = o.z;
        }
    } else {
        o.s = load_scale(a.s, i, a.scale_f16);
        o.z = a.z ? a.z[i] : 0;
    }
    return o;
}

// Optional smoothing of 8 elements of columns c0..c0+7: x / s_c (correctly
// rounded binary32 division) or x * s_c.
__device__ __forceinline__ void smooth8(float v[8], int mode, const float* __restrict__ sm, int64_t c0) {
    if (mode == QLIN_SMOOTH_NONE) return;
    float4 a = __ldg(reinterpret_cast<const float4*>(sm + c0));
    float4 b = __ldg(reinterpret_cast<const float4*>(sm + c0) + 1);
    float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = (mode == QLIN_SMOOTH_DIVIDE) ? __fdiv_rn(v[j], f[j]) : v[j] * f[j];
}

// Store 8 codes of chunk `chunk` of row r (codes as code_bits words).
__device__ __forceinline__ void store_codes8(void* q, int64_t r, int64_t cols, int64_t chunk, int code4,
                                             const uint32_t c[8]) {
    if (code4) {
        uint32_t w = pack_nibbles8(c);
        reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(q) + r * (cols / 2))[chunk] = w;
    } else {
        uint2 w;
        w.x = pack_bytes4(c[0], c[1], c[2], c[3]);
        w.y = pack_bytes4(c[4], c[5], c[6], c[7]);
        reinterpret_cast<uint2*>(reinterpret_cast<int8_t*>(q) + r * cols)[chunk] = w;
    }
}

// ------------------------------------------------------------------ row-local scopes
// One CTA walks rows r = blockIdx.x, blockIdx.x + gridDim.x, ...; thread t holds
// chunks c = i*blockDim.x + t (8 elements each) of the row in registers.
// PER_ROW reduces over the CTA; PER_GROUP over the g/8 adjacent lanes holding
// one group.  CPT = max chunks per thread.
template <typename T, int CPT>
__global__ void __launch_bounds__(512) k_quant_rows(QuantArgs a) {
    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    const int64_t nchunks = a.cols / 8;
    const bool per_row = (a.gran == QLIN_PER_ROW);
    const int gl = per_row ? 0 : a.group / 8;  // lanes per group
    const T* __restrict__ x = reinterpret_cast<const T*>(a.x);
    const CodeRange cr = make_range(a.qmin, a.qmax);
    __shared__ float red_hi[32], red_lo[32];
    __shared__ float bc[2];

    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        float v[CPT][8];
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            int64_t c = (int64_t)i * nt + tid;
            if (c < nchunks) {
                load8<T>(x + r * a.ld + c * 8, v[i]);
                smooth8(v[i], a.smooth_mode, a.smooth, c * 8);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) v[i][j] = 0.0f;
            }
        }

        if (per_row) {
            float s;
            int z;
            if (a.static_scale) {
                s = load_scale(a.s, r, a.scale_f16);
                z = a.z ? a.z[r] : 0;
            } else {
                float hi = 0.0f, lo = 0.0f;
#pragma unroll
                for (int i = 0; i < CPT; ++i)
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (a.sym) {
                            hi = fmaxf(hi, fabsf(v[i][j]));
                        } else {
                            hi = fmaxf(hi, v[i][j]);
                            lo = fminf(lo, v[i][j]);
                        }
                    }
                hi = warp_max(hi);
                lo = warp_min(lo);
                if ((tid & 31) == 0) {
                    red_hi[tid >> 5] = hi;
                    red_lo[tid >> 5] = lo;
                }
                __syncthreads();
                if (tid < 32) {
                    int nw = nt >> 5;
                    float h = (tid < nw) ? red_hi[tid] : 0.0f;
                    float l = (tid < nw) ? red_lo[tid] : 0.0f;
                    h = warp_max(h);
                    l = warp_min(l);
                    if (tid == 0) {
                        bc[0] = h;
                        bc[1] = l;
                    }
                }
                __syncthreads();
                hi = bc[0];
                lo = bc[1];
                __syncthreads();  // bc / red_* are reused by the next row
                if (a.absmax_out) {
                    if (tid == 0) a.absmax_out[r] = hi;
                    continue;
                }
                scale_zero(lo, hi, a.qmin, a.qmax, a.sym, a.scale_f16, s, z);
                if (tid == 0) {
                    store_scale(a.s, r, a.scale_f16, s);
                    if (a.z) a.z[r] = z;
                }
            }
            const ScopeParams p = make_scope(s, z);
#pragma unroll
            for (int i = 0; i < CPT; ++i) {
                int64_t c = (int64_t)i * nt + tid;
                if (c < nchunks) {
                    uint32_t cb[8];
                    code_bits8<false>(v[i], p, cr, cb);
                    store_codes8(a.q, r, a.cols, c, a.code4, cb);
                }
            }
        } else {
            const int64_t ngr = a.cols / a.group;
#pragma unroll
            for (int i = 0; i < CPT; ++i) {
                int64_t c = (int64_t)i * nt + tid;
                int64_t grp = (c * 8) / a.group;  // group index within the row
                float s;
                int z;
                if (a.static_scale) {
                    s = (c < nchunks) ? load_scale(a.s, r * ngr + grp, a.scale_f16) : 1.0f;
                    z = (c < nchunks && a.z) ? a.z[r * ngr + grp] : 0;
                } else {
                    float hi = 0.0f, lo = 0.0f;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (a.sym) {
                            hi = fmaxf(hi, fabsf(v[i][j]));
                        } else {
                            hi = fmaxf(hi, v[i][j]);
                            lo = fminf(lo, v[i][j]);
                        }
                    }
                    for (int o = 1; o < gl; o <<= 1) {
                        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
                        lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
                    }
                    const bool leader = (c < nchunks) && ((c % gl) == 0);
                    if (a.absmax_out) {
                        if (leader) a.absmax_out[r * ngr + grp] = hi;
                        continue;
                    }
                    scale_zero(lo, hi, a.qmin, a.qmax, a.sym, a.scale_f16, s, z);
                    if (leader) {
                        store_scale(a.s, r * ngr + grp, a.scale_f16, s);
                        if (a.z) a.z[r * ngr + grp] = z;
                    }
                }
                if (c < nchunks) {
                    const ScopeParams p = make_scope(s, z);
                    uint32_t cb[8];
                    code_bits8<false>(v[i], p, cr, cb);
                    store_codes8(a.q, r, a.cols, c, a.code4, cb);
                }
            }
        }
    }
}

// ------------------------------------------------------------------ long rows, per-row scopes
// For rows longer than 4096 elements: one CTA of 512 threads per row at a
// time, the smoothed binary32 row staged in shared memory (so registers stay
// few and two CTAs fit on an SM): pass 1 loads (four chunks in flight per
// thread), smooths, stores and reduces; pass 2 reads the staged values back
// and writes the codes.
template <typename T>
__global__ void __launch_bounds__(512, 2) k_quant_longrows(QuantArgs a) {
    extern __shared__ float xs[];  // [cols]
    __shared__ float red_hi[32], red_lo[32];
    const int tid = threadIdx.x, nt = blockDim.x;
    const int64_t nchunks = a.cols / 8;
    const T* __restrict__ x = reinterpret_cast<const T*>(a.x);
    const CodeRange cr = make_range(a.qmin, a.qmax);
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        float hi = 0.0f, lo = 0.0f;
        for (int64_t c0 = tid; c0 < nchunks; c0 += 4 * (int64_t)nt) {
            float v[4][8];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                int64_t c = c0 + (int64_t)u * nt;
                if (c < nchunks) load8<T>(x + r * a.ld + c * 8, v[u]);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                int64_t c = c0 + (int64_t)u * nt;
                if (c >= nchunks) break;
                smooth8(v[u], a.smooth_mode, a.smooth, c * 8);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (a.sym) {
                        hi = fmaxf(hi, fabsf(v[u][j]));
                    } else {
                        hi = fmaxf(hi, v[u][j]);
                        lo = fminf(lo, v[u][j]);
                    }
                }
                float4* d = reinterpret_cast<float4*>(xs + c * 8);
                d[0] = make_float4(v[u][0], v[u][1], v[u][2], v[u][3]);
                d[1] = make_float4(v[u][4], v[u][5], v[u][6], v[u][7]);
            }
        }
        hi = warp_max(hi);
        lo = warp_min(lo);
        if ((tid & 31) == 0) {
            red_hi[tid >> 5] = hi;
            red_lo[tid >> 5] = lo;
        }
        __syncthreads();
        hi = 0.0f;
        lo = 0.0f;
        for (int w = 0; w < (nt >> 5); ++w) {
            hi = fmaxf(hi, red_hi[w]);
            lo = fminf(lo, red_lo[w]);
        }
        float s;
        int z;
        if (a.static_scale) {
            s = load_scale(a.s, r, a.scale_f16);
            z = a.z ? a.z[r] : 0;
        } else {
            scale_zero(lo, hi, a.qmin, a.qmax, a.sym, a.scale_f16, s, z);
            if (tid == 0) {
                store_scale(a.s, r, a.scale_f16, s);
                if (a.z) a.z[r] = z;
            }
        }
        const ScopeParams p = make_scope(s, z);
        for (int64_t c = tid; c < nchunks; c += nt) {
            const float4* d = reinterpret_cast<const float4*>(xs + c * 8);
            float4 u0 = d[0], u1 = d[1];
            float v[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
            uint32_t cb[8];
            code_bits8<false>(v, p, cr, cb);
            store_codes8(a.q, r, a.cols, c, a.code4, cb);
        }
        __syncthreads();  // xs and red_* are reused by the next row
    }
}

// ------------------------------------------------------------------ row-local kernels for 16-bit rows
// The kernels below take per-row and per-group scopes of bf16 / fp16 rows
// without smoothing (the activation path: SmoothQuant's 1/s is folded into
// the previous layer).  Their modes are compile-time parameters, so the chunk
// loops carry no run-time branches; indices inside a row are 32-bit.
//   SYM / STATIC : dynamic symmetric scopes (no clamp, since |rne(x/s)| <=
//                  qmax when s comes from the scope's own max|x|), dynamic
//                  asymmetric scopes (clamp), or static scales (clamp and
//                  far-range test).
//   CODE4        : two codes per byte.
// Per-tensor scopes (GL = 0, gran = QLIN_PER_TENSOR) use one (s, z) for every
// row: static, or derived from the statistics words of the pass before (the
// first CTA's thread 0 writes it out); dynamic per-tensor scopes take the
// dynamic arithmetic, since the tensor's own range bounds every |x / s|.

// Running range of packed 16-bit pairs: |x| max (symmetric) or max and min.
template <typename T>
struct PairRange;
template <>
struct PairRange<__nv_bfloat16> {
    __nv_bfloat162 hi = __floats2bfloat162_rn(0.0f, 0.0f), lo = __floats2bfloat162_rn(0.0f, 0.0f);
    __device__ __forceinline__ void add(const uint4 u, bool sym) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
            if (sym) {
                hi = __hmax2(hi, __habs2(v));
            } else {
                hi = __hmax2(hi, v);
                lo = __hmin2(lo, v);
            }
        }
    }
    __device__ __forceinline__ void result(bool sym, float& h, float& l) const {
        h = fmaxf(__low2float(hi), __high2float(hi));
        l = sym ? 0.0f : fminf(__low2float(lo), __high2float(lo));
    }
};
template <>
struct PairRange<__half> {
    __half2 hi = __floats2half2_rn(0.0f, 0.0f), lo = __floats2half2_rn(0.0f, 0.0f);
    __device__ __forceinline__ void add(const uint4 u, bool sym) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 v = *reinterpret_cast<const __half2*>(&w[i]);
            if (sym) {
                hi = __hmax2(hi, __habs2(v));
            } else {
                hi = __hmax2(hi, v);
                lo = __hmin2(lo, v);
            }
        }
    }
    __device__ __forceinline__ void result(bool sym, float& h, float& l) const {
        h = fmaxf(__low2float(hi), __high2float(hi));
        l = sym ? 0.0f : fminf(__low2float(lo), __high2float(lo));
    }
};

template <bool CODE4>
__device__ __forceinline__ void put_codes8(uint8_t* __restrict__ qrow, uint32_t c, const uint32_t cb[8]) {
    if (CODE4)
        reinterpret_cast<uint32_t*>(qrow)[c] = pack_nibbles8(cb);
    else
        reinterpret_cast<uint2*>(qrow)[c] =
            make_uint2(pack_bytes4(cb[0], cb[1], cb[2], cb[3]), pack_bytes4(cb[4], cb[5], cb[6], cb[7]));
}

template <typename T, bool SYM, bool STATIC, bool OUTLINE = false>
__device__ __forceinline__ void codes_of_chunk(const uint4 raw, const ScopeParams& sp, const CodeRange& cr,
                                               uint32_t cb[8]) {
    float v[8];
    unpack8<T>(raw, v);
    if (STATIC)
        code_bits8<false, true, OUTLINE>(v, sp, cr, cb);
    else if (SYM)
        code_bits8<true, false, OUTLINE>(v, sp, cr, cb);
    else
        code_bits8<true, true, OUTLINE>(v, sp, cr, cb);
}

// Codes of one chunk stored at chunk index c of the code row.  Scopes with a
// clamp clamp and pack the codes as 16-bit pairs (clamp_pair16); dynamic
// symmetric scopes need no clamp and pack the candidates directly.
template <typename T, bool SYM, bool STATIC, bool OUTLINE, bool CODE4>
__device__ __forceinline__ void quant_chunk(const uint4 raw, const ScopeParams& sp, const CodeRange& cr,
                                            uint8_t* __restrict__ qrow, uint32_t c) {
    uint32_t cb[8];
    if constexpr (STATIC || !SYM) {
        float v[8];
        unpack8<T>(raw, v);
        code_bits8<!STATIC, true, OUTLINE, true>(v, sp, cr, cb);
        if (CODE4)
            reinterpret_cast<uint32_t*>(qrow)[c] = pack_pairs_nibbles(cb);
        else
            reinterpret_cast<uint2*>(qrow)[c] = pack_pairs_bytes(cb);
    } else {
        codes_of_chunk<T, SYM, STATIC, OUTLINE>(raw, sp, cr, cb);
        put_codes8<CODE4>(qrow, c, cb);
    }
}

// Row-local scopes of 16-bit rows streamed through shared memory by bulk
// copies.  Each persistent CTA keeps `nbuf` row buffers: while it reduces and
// quantizes one row, the copies of its next rows land in the others.  NT
// threads per CTA: 512 for long rows (two such CTAs with two buffers fit an SM
// for rows of up to 28,672 values, so one CTA's barriers overlap the other's
// work), 128 for rows of up to 8192 values (a dozen CTAs share an SM, so many
// rows are in flight and each row's reduction spans only four warps).
// GL = 0: per-row scopes (a range pass, a CTA-wide maximum, a code pass);
// GL > 0: groups of 8 GL values, one pass, a group's chunks spread over up
// to GL / 4 lanes that reduce with shuffles (no CTA-wide step besides the
// buffer release).
template <typename T, bool SYM, bool STATIC, bool CODE4, int NT, int GL>
__global__ void __launch_bounds__(NT) k_qrow_bulk(QuantArgs a, uint32_t buf_stride, int nbuf) {
    extern __shared__ __align__(128) uint8_t qb_smem[];
    __shared__ float red_hi[NT / 32], red_lo[NT / 32];
    __shared__ __align__(8) uint64_t bar[3];
    __shared__ int abort_flag;
    const int tid = threadIdx.x;
    const uint32_t nchunks = (uint32_t)(a.cols / 8);
    const uint32_t row_bytes = (uint32_t)(a.cols * 2);
    const CodeRange cr = make_range(a.qmin, a.qmax);
    const uint32_t bar0 = tc::smem_addr(&bar[0]);
    const uint32_t buf0 = tc::smem_addr(qb_smem);
    const uint8_t* xg = reinterpret_cast<const uint8_t*>(a.x);
    if (tid == 0) {
        for (int b = 0; b < nbuf; ++b) tc::mbar_init(bar0 + 8u * b, 1);
        abort_flag = 0;
        tc::mbar_init_fence();
    }
    __syncthreads();
    // thread 0: start the copy of row r into buffer b (whose earlier readers
    // have all passed a __syncthreads)
    auto issue = [&](int64_t r, int b) {
        tc::fence_proxy_async_smem();
        tc::mbar_arrive_expect_tx(bar0 + 8u * b, row_bytes);
        tc::bulk_load(buf0 + (uint32_t)b * buf_stride, xg + r * a.ld * 2, row_bytes, bar0 + 8u * b);
    };
    const bool stalled = tc::producers_stalled();
    if (tid == 0 && !stalled) {
        for (int b = 0; b < nbuf; ++b)
            if (blockIdx.x + (int64_t)b * gridDim.x < a.rows) issue(blockIdx.x + (int64_t)b * gridDim.x, b);
    }
    const int64_t qld = CODE4 ? a.cols / 2 : a.cols;
    // per-tensor scopes (GL = 0), static or from the statistics pass: one
    // (s, z) for every row (dynamic ones only below 512 threads: longer rows
    // of dynamic per-tensor scopes take the strip kernel, and the 512-thread
    // per-row kernels keep no run-time test of it)
    float s_t = 0.0f;
    int z_t = 0;
    const bool one_scope = GL == 0 && a.gran == QLIN_PER_TENSOR && (STATIC || NT < 512);
    if (one_scope) {
        const ScopeOf o = scope_in(a, 0, blockIdx.x == 0 && tid == 0);
        s_t = o.s;
        z_t = o.z;
    }
    int b = 0;
    uint32_t ph = 0;
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        const bool ok = tc::mbar_wait(bar0 + 8u * b, ph, &abort_flag);
        if (!__syncthreads_and(ok)) break;
        const uint4* xs16 = reinterpret_cast<const uint4*>(qb_smem + (size_t)b * buf_stride);
        if constexpr (GL > 0) {
            // per-group scopes, one pass: a group's GL chunks go to LPG lanes
            // of CPL chunks each (chunk p + LPG j of the group for lane p), so
            // the group's scale is computed once per CPL chunks and the LPG
            // lanes reduce with shuffles; the lanes of a group read adjacent
            // chunks (at most two-way bank conflicts)
            constexpr int CPL = GL < 4 ? GL : 4;
            constexpr int LPG = GL / CPL;
            const uint32_t ngr = (uint32_t)(a.cols / a.group);
            uint8_t* qrow = reinterpret_cast<uint8_t*>(a.q) + r * qld;
            for (uint32_t g0 = 0; g0 < ngr; g0 += NT / LPG) {
                const uint32_t gidx = g0 + (uint32_t)tid / LPG;
                const bool live = gidx < ngr;  // a group's lanes are all live or all idle
                const uint32_t c0 = gidx * GL + (uint32_t)tid % LPG;
                uint4 raw[CPL];
#pragma unroll
                for (int j = 0; j < CPL; ++j) raw[j] = live ? xs16[c0 + LPG * j] : make_uint4(0, 0, 0, 0);
                const int64_t sc = r * ngr + gidx;
                float s;
                int z;
                if (STATIC) {
                    s = live ? load_scale(a.s, sc, a.scale_f16) : 1.0f;
                    z = (a.z && live) ? a.z[sc] : 0;
                } else {
                    PairRange<T> pr;
#pragma unroll
                    for (int j = 0; j < CPL; ++j) pr.add(raw[j], SYM);
                    float hi, lo;
                    pr.result(SYM, hi, lo);
#pragma unroll
                    for (int o = 1; o < LPG; o <<= 1) {
                        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
                        if (!SYM) lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
                    }
                    scale_zero(lo, hi, a.qmin, a.qmax, SYM, a.scale_f16, s, z);
                    if (live && tid % LPG == 0) {
                        store_scale(a.s, sc, a.scale_f16, s);
                        if (!SYM) a.z[sc] = z;
                    }
                }
                if (live) {
                    const ScopeParams sp = make_scope(s, z);
#pragma unroll
                    for (int j = 0; j < CPL; ++j) {
                        quant_chunk<T, SYM, STATIC, false, CODE4>(raw[j], sp, cr, qrow, c0 + LPG * j);
                    }
                }
            }
            __syncthreads();  // buffer b is free
            if (tid == 0 && !stalled && r + (int64_t)nbuf * gridDim.x < a.rows) issue(r + (int64_t)nbuf * gridDim.x, b);
            if (++b == nbuf) {
                b = 0;
                ph ^= 1u;
            }
            continue;
        }
        float s;
        int z;
        if (one_scope) {
            s = s_t;
            z = z_t;
        } else if (STATIC) {
            s = load_scale(a.s, r, a.scale_f16);
            z = a.z ? a.z[r] : 0;
        } else {
            PairRange<T> pr;
#pragma unroll 4
            for (uint32_t c = tid; c < nchunks; c += NT) pr.add(xs16[c], SYM);
            float hi, lo;
            pr.result(SYM, hi, lo);
            hi = warp_max(hi);
            if (!SYM) lo = warp_min(lo);
            if ((tid & 31) == 0) {
                red_hi[tid >> 5] = hi;
                red_lo[tid >> 5] = lo;
            }
            __syncthreads();
            hi = red_hi[0];
            lo = red_lo[0];
#pragma unroll
            for (int w = 1; w < NT / 32; ++w) {
                hi = fmaxf(hi, red_hi[w]);
                if (!SYM) lo = fminf(lo, red_lo[w]);
            }
            scale_zero(lo, hi, a.qmin, a.qmax, SYM, a.scale_f16, s, z);
            if (tid == 0) {
                store_scale(a.s, r, a.scale_f16, s);
                if (!SYM) a.z[r] = z;
            }
        }
        const ScopeParams sp = make_scope(s, z);
        uint8_t* qrow = reinterpret_cast<uint8_t*>(a.q) + r * qld;
#pragma unroll 4
        for (uint32_t c = tid; c < nchunks; c += NT) {
            quant_chunk<T, SYM, STATIC, false, CODE4>(xs16[c], sp, cr, qrow, c);
        }
        __syncthreads();  // buffer b and red_* are free
        if (tid == 0 && !stalled && r + (int64_t)nbuf * gridDim.x < a.rows) issue(r + (int64_t)nbuf * gridDim.x, b);
        if (++b == nbuf) {
            b = 0;
            ph ^= 1u;
        }
    }
}

// Maximum / minimum of NW per-warp slots in shared memory (16-byte aligned),
// read four at a time when NW is a multiple of 4.
template <int NW>
__device__ __forceinline__ float slots_max(const float* p) {
    if constexpr (NW % 4 == 0) {
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < NW / 4; ++i) {
            const float4 q = reinterpret_cast<const float4*>(p)[i];
            m = fmaxf(m, fmaxf(fmaxf(q.x, q.y), fmaxf(q.z, q.w)));
        }
        return m;
    } else {
        float m = p[0];
#pragma unroll
        for (int i = 1; i < NW; ++i) m = fmaxf(m, p[i]);
        return m;
    }
}
template <int NW>
__device__ __forceinline__ float slots_min(const float* p) {
    if constexpr (NW % 4 == 0) {
        float m = INFINITY;
#pragma unroll
        for (int i = 0; i < NW / 4; ++i) {
            const float4 q = reinterpret_cast<const float4*>(p)[i];
            m = fminf(m, fminf(fminf(q.x, q.y), fminf(q.z, q.w)));
        }
        return m;
    } else {
        float m = p[0];
#pragma unroll
        for (int i = 1; i < NW; ++i) m = fminf(m, p[i]);
        return m;
    }
}

// k_qrow_bulk with the row held in registers: each thread copies its chunks
// of the row (at most NC of them) out of the row buffer, so the buffer is free
// -- and thread 0 starts the copy of a later row into it -- as soon as the
// CTA has passed one barrier, which is also the barrier of the per-row
// maximum.  One barrier per row; the reduction slots alternate between two
// sets by row parity, so a fast thread writing the next row's slot never
// overwrites one that a slow thread still reads.  Chunk c of a per-row scope
// sits in slot (c - tid) / NT; per-group scopes (GL > 0) take the chunk
// assignment of k_qrow_bulk, iteration `it` of its group loop in slots
// it * CPT ... it * CPT + CPT - 1.  Rows of more than NC * NT chunks take
// k_qrow_bulk.
template <typename T, bool SYM, bool STATIC, bool CODE4, int NT, int GL, int NC>
__global__ void __launch_bounds__(NT, NT >= 512 ? 2 : 1) k_qrow_reg(QuantArgs a, uint32_t buf_stride, int nbuf) {
    constexpr int CPT = GL == 0 ? 1 : (GL < 4 ? GL : 4);
    constexpr int LPG = GL == 0 ? 1 : GL / CPT;
    constexpr int NI = NC / CPT;  // group-loop iterations held (GL > 0)
    static_assert(NC % CPT == 0, "slots hold whole group iterations");
    extern __shared__ __align__(128) uint8_t qb_smem[];
    __shared__ __align__(16) float red_hi[2][NT / 32];
    __shared__ __align__(16) float red_lo[2][NT / 32];
    __shared__ __align__(8) uint64_t bar[3];
    __shared__ int abort_flag;
    const int tid = threadIdx.x;
    const uint32_t nchunks = (uint32_t)(a.cols / 8);
    const uint32_t row_bytes = (uint32_t)(a.cols * 2);
    const CodeRange cr = make_range(a.qmin, a.qmax);
    const uint32_t bar0 = tc::smem_addr(&bar[0]);
    const uint32_t buf0 = tc::smem_addr(qb_smem);
    const uint8_t* xg = reinterpret_cast<const uint8_t*>(a.x);
    if (tid == 0) {
        for (int b = 0; b < nbuf; ++b) tc::mbar_init(bar0 + 8u * b, 1);
        abort_flag = 0;
        tc::mbar_init_fence();
    }
    __syncthreads();
    auto issue = [&](int64_t r, int b) {
        tc::fence_proxy_async_smem();
        tc::mbar_arrive_expect_tx(bar0 + 8u * b, row_bytes);
        tc::bulk_load(buf0 + (uint32_t)b * buf_stride, xg + r * a.ld * 2, row_bytes, bar0 + 8u * b);
    };
    const bool stalled = tc::producers_stalled();
    if (tid == 0 && !stalled) {
        for (int b = 0; b < nbuf; ++b)
            if (blockIdx.x + (int64_t)b * gridDim.x < a.rows) issue(blockIdx.x + (int64_t)b * gridDim.x, b);
    }
    const int64_t qld = CODE4 ? a.cols / 2 : a.cols;
    float s_t = 0.0f;
    int z_t = 0;
    const bool one_scope = GL == 0 && a.gran == QLIN_PER_TENSOR && (STATIC || NT < 512);  // as in k_qrow_bulk
    if (one_scope) {
        const ScopeOf o = scope_in(a, 0, blockIdx.x == 0 && tid == 0);
        s_t = o.s;
        z_t = o.z;
    }
    // chunk index of slot i (>= nchunks: no chunk)
    auto chunk_of = [&](int i) -> uint32_t {
        if constexpr (GL == 0) {
            return (uint32_t)tid + (uint32_t)NT * (uint32_t)i;
        } else {
            const uint32_t gidx = (uint32_t)(i / CPT) * (uint32_t)(NT / LPG) + (uint32_t)tid / LPG;
            return gidx * GL + (uint32_t)tid % LPG + (uint32_t)LPG * (uint32_t)(i % CPT);
        }
    };
    int b = 0, par = 0;
    uint32_t ph = 0;
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        const bool ok = tc::mbar_wait(bar0 + 8u * b, ph, &abort_flag);
        const uint4* xs16 = reinterpret_cast<const uint4*>(qb_smem + (size_t)b * buf_stride);
        uint4 raw[NC];
#pragma unroll
        for (int i = 0; i < NC; ++i) {
            const uint32_t c = chunk_of(i);
            raw[i] = (ok && c < nchunks) ? xs16[c] : make_uint4(0, 0, 0, 0);
        }
        if (GL == 0 && !STATIC && !one_scope) {
            // zero padding: the range of a scope always includes 0
            PairRange<T> pr;
#pragma unroll
            for (int i = 0; i < NC; ++i) pr.add(raw[i], SYM);
            float hi, lo;
            pr.result(SYM, hi, lo);
            hi = warp_max(hi);
            if (!SYM) lo = warp_min(lo);
            if ((tid & 31) == 0) {
                red_hi[par][tid >> 5] = hi;
                red_lo[par][tid >> 5] = lo;
            }
        }
        if (!__syncthreads_and(ok)) break;
        // every thread holds its chunks: buffer b is free
        if (tid == 0 && !stalled && r + (int64_t)nbuf * gridDim.x < a.rows) issue(r + (int64_t)nbuf * gridDim.x, b);
        uint8_t* qrow = reinterpret_cast<uint8_t*>(a.q) + r * qld;
        if constexpr (GL == 0) {
            float s;
            int z;
            if (one_scope) {
                s = s_t;
                z = z_t;
            } else if (STATIC) {
                s = load_scale(a.s, r, a.scale_f16);
                z = a.z ? a.z[r] : 0;
            } else {
                const float hi = slots_max<NT / 32>(red_hi[par]);
                const float lo = SYM ? 0.0f : slots_min<NT / 32>(red_lo[par]);
                scale_zero(lo, hi, a.qmin, a.qmax, SYM, a.scale_f16, s, z);
                if (tid == 0) {
                    store_scale(a.s, r, a.scale_f16, s);
                    if (!SYM) a.z[r] = z;
                }
            }
            const ScopeParams sp = make_scope(s, z);
#pragma unroll
            for (int i = 0; i < NC; ++i) {
                const uint32_t c = chunk_of(i);
                if (c < nchunks) {
                    quant_chunk<T, SYM, STATIC, false, CODE4>(raw[i], sp, cr, qrow, c);
                }
            }
        } else {
            const uint32_t ngr = (uint32_t)(a.cols / a.group);
#pragma unroll
            for (int it = 0; it < NI; ++it) {
                const uint32_t gidx = (uint32_t)it * (uint32_t)(NT / LPG) + (uint32_t)tid / LPG;
                const bool live = gidx < ngr;  // a group's lanes are all live or all idle
                if (it > 0 && (uint32_t)it * (uint32_t)(NT / LPG) >= ngr) break;  // CTA-uniform
                const int64_t sc = r * ngr + gidx;
                float s;
                int z;
                if (STATIC) {
                    s = live ? load_scale(a.s, sc, a.scale_f16) : 1.0f;
                    z = (a.z && live) ? a.z[sc] : 0;
                } else {
                    PairRange<T> pr;
#pragma unroll
                    for (int j = 0; j < CPT; ++j) pr.add(raw[it * CPT + j], SYM);
                    float hi, lo;
                    pr.result(SYM, hi, lo);
#pragma unroll
                    for (int o = 1; o < LPG; o <<= 1) {
                        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
                        if (!SYM) lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
                    }
                    scale_zero(lo, hi, a.qmin, a.qmax, SYM, a.scale_f16, s, z);
                    if (live && tid % LPG == 0) {
                        store_scale(a.s, sc, a.scale_f16, s);
                        if (!SYM) a.z[sc] = z;
                    }
                }
                if (live) {
                    const ScopeParams sp = make_scope(s, z);
#pragma unroll
                    for (int j = 0; j < CPT; ++j) {
                        quant_chunk<T, SYM, STATIC, false, CODE4>(raw[it * CPT + j], sp, cr, qrow,
                                                                   chunk_of(it * CPT + j));
                    }
                }
            }
        }
        par ^= 1;
        if (++b == nbuf) {
            b = 0;
            ph ^= 1u;
        }
    }
}

// Per-row scopes of 16-bit rows of at most 32 * NC eight-value chunks: one
// warp per row, the row held in registers (lane l holds chunks l, l + 32,
// ...), every reduction a register shuffle, many warps per SM in flight.
template <typename T, bool SYM, bool STATIC, bool CODE4, int NC>
__global__ void __launch_bounds__(256) k_qrow_warp(QuantArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const uint32_t nchunks = (uint32_t)(a.cols / 8);
    const CodeRange cr = make_range(a.qmin, a.qmax);
    const int64_t qld = CODE4 ? a.cols / 2 : a.cols;
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < a.rows; r += nwarps) {
        const uint4* __restrict__ xr = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(a.x) + r * a.ld * 2);
        uint8_t* qrow = reinterpret_cast<uint8_t*>(a.q) + r * qld;
        uint4 raw[NC];
#pragma unroll
        for (int i = 0; i < NC; ++i) {
            const uint32_t c = lane + 32u * i;
            raw[i] = c < nchunks ? __ldg(xr + c) : make_uint4(0, 0, 0, 0);
        }
        {
            float s;
            int z;
            if (STATIC) {
                s = load_scale(a.s, r, a.scale_f16);
                z = a.z ? a.z[r] : 0;
            } else {
                PairRange<T> pr;
#pragma unroll
                for (int i = 0; i < NC; ++i) pr.add(raw[i], SYM);  // zero padding: the range includes 0
                float hi, lo;
                pr.result(SYM, hi, lo);
                hi = warp_max(hi);
                if (!SYM) lo = warp_min(lo);
                scale_zero(lo, hi, a.qmin, a.qmax, SYM, a.scale_f16, s, z);
                if (lane == 0) {
                    store_scale(a.s, r, a.scale_f16, s);
                    if (!SYM) a.z[r] = z;
                }
            }
            const ScopeParams sp = make_scope(s, z);
#pragma unroll
            for (int i = 0; i < NC; ++i) {
                const uint32_t c = lane + 32u * i;
                if (c < nchunks) {
                    uint32_t cb[8];
                    codes_of_chunk<T, SYM, STATIC, true>(raw[i], sp, cr, cb);
                    put_codes8<CODE4>(qrow, c, cb);
                }
            }
        }
    }
}

// Per-group scopes of 16-bit rows (g = 8 * GL values, GL a power of two <=
// 32): a warp takes slabs of 32 chunks (256 values) in a grid-stride loop
// over every (row, slab), one chunk per lane; the GL lanes of a group reduce
// with shuffles and compute its scale in registers.  Little register
// pressure, so many warps per SM keep many slabs in flight.
template <typename T, bool SYM, bool STATIC, bool CODE4, int GL>
__global__ void __launch_bounds__(256) k_qgrp_slab(QuantArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const uint32_t nchunks = (uint32_t)(a.cols / 8);
    const uint32_t slabs = (nchunks + 31) / 32;
    const uint32_t ngr = (uint32_t)(a.cols / a.group);
    const int64_t units = a.rows * (int64_t)slabs;
    const CodeRange cr = make_range(a.qmin, a.qmax);
    const int64_t qld = CODE4 ? a.cols / 2 : a.cols;
#pragma unroll 2
    for (int64_t u = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < units; u += nwarps) {
        const int64_t r = u / slabs;
        const uint32_t c = (uint32_t)(u - r * slabs) * 32u + lane;
        const bool live = c < nchunks;  // whole groups: a group's lanes are all live or all idle
        const uint4 raw = live ? __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(a.x) +
                                                                      r * a.ld * 2) + c)
                               : make_uint4(0, 0, 0, 0);
        const int64_t sc = r * ngr + c / GL;
        float s;
        int z;
        if (STATIC) {
            s = live ? load_scale(a.s, sc, a.scale_f16) : 1.0f;
            z = (a.z && live) ? a.z[sc] : 0;
        } else {
            PairRange<T> pr;
            pr.add(raw, SYM);
            float hi, lo;
            pr.result(SYM, hi, lo);
#pragma unroll
            for (int o = 1; o < GL; o <<= 1) {
                hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
                if (!SYM) lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
            }
            scale_zero(lo, hi, a.qmin, a.qmax, SYM, a.scale_f16, s, z);
            if (live && (lane & (GL - 1)) == 0) {
                store_scale(a.s, sc, a.scale_f16, s);
                if (!SYM) a.z[sc] = z;
            }
        }
        if (live) {
            uint32_t cb[8];
            codes_of_chunk<T, SYM, STATIC, true>(raw, make_scope(s, z), cr, cb);
            put_codes8<CODE4>(reinterpret_cast<uint8_t*>(a.q) + r * qld, c, cb);
        }
    }
}

// ------------------------------------------------------------------ column-strip kernels
// Tiling shared by the per-tensor / per-column kernels.  A block of NT
// threads covers cpb = min(nchunks, 32) chunk columns (8 values each) x
// rpi = NT / cpb adjacent rows per step, so a warp reads 32 adjacent chunks
// of one row.  The grid holds gx blocks across the chunk columns and gy
// blocks down the rows, sized by the host to the blocks that fit on the GPU
// at once; block y takes row groups y, y + gy, y + 2 gy, ... of rpi rows, so
// all blocks sweep the matrix together.
constexpr int kStripThreads = 256;

struct Strip {
    int64_t chunk;  // chunk column of this thread (-1 when idle)
    int64_t r0;     // first row of this thread
    int64_t step;   // rows between this thread's consecutive rows (gy * rpi)
    int64_t nr;     // rows of this thread: r0 + i * step, i < nr
};

template <int NT = kStripThreads>
__device__ __forceinline__ Strip strip_of(int64_t nchunks, int64_t rows) {
    Strip s;
    const int t = threadIdx.x;
    const int cpb = nchunks < 32 ? (int)nchunks : 32;
    const int rpi = NT / cpb;
    const int rl = t / cpb;
    const int64_t c = (int64_t)blockIdx.x * cpb + t % cpb;
    s.chunk = (rl < rpi && c < nchunks) ? c : -1;
    s.r0 = (int64_t)blockIdx.y * rpi + rl;
    s.step = (int64_t)gridDim.y * rpi;
    s.nr = s.r0 < rows ? (rows - 1 - s.r0) / s.step + 1 : 0;
    return s;
}

// One chunk of eight input values as loaded (16 bytes of a 16-bit type, 32
// of binary32), zero when the row is outside the slab.
template <typename T>
struct Raw8 {
    uint4 w[sizeof(T) == 4 ? 2 : 1];
};
template <typename T>
__device__ __forceinline__ Raw8<T> raw8_load(const T* p, bool live) {
    Raw8<T> c;
#pragma unroll
    for (int i = 0; i < (int)(sizeof(c.w) / sizeof(uint4)); ++i)
        c.w[i] = live ? __ldg(reinterpret_cast<const uint4*>(p) + i) : make_uint4(0u, 0u, 0u, 0u);
    return c;
}

template <typename T>
__device__ __forceinline__ void raw8_widen(const Raw8<T>& c, float v[8]) {
    if constexpr (sizeof(T) == 4) {
        const uint32_t w[8] = {c.w[0].x, c.w[0].y, c.w[0].z, c.w[0].w, c.w[1].x, c.w[1].y, c.w[1].z, c.w[1].w};
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(w[j]);
    } else {
        unpack8<T>(c.w[0], v);
    }
}

// Packed pair type of a 16-bit input type.
template <typename T>
struct Pair16;
template <>
struct Pair16<__nv_bfloat16> {
    using P = __nv_bfloat162;
};
template <>
struct Pair16<__half> {
    using P = __half2;
};

// Range statistics into ws words (binary32 bit patterns of non-negative values,
// atomicMax): stat[2*scope] = max(max x, 0) (or max|x| when SYM),
// stat[2*scope+1] = -min(min x, 0).  The words start at 0 (memset by the
// host).  PACKED (unsmoothed 16-bit input) keeps the running maxima as packed
// pairs in the input's own format: max and min are exact in any format, and
// both ignore NaN like fmaxf / fminf.  A zero chunk leaves every statistic
// unchanged, so rows past the slab load as zeros.  Per-column statistics are
// reduced over the block's row lanes in shared memory before one atomic per
// column and statistic.
template <typename T, bool SYM, bool PER_COL, bool PACKED>
__global__ void __launch_bounds__(kStripThreads) k_stats_strip(QuantArgs a, uint32_t* stat) {
    constexpr int U = 8;  // loads in flight per thread
    const int64_t nchunks = a.cols / 8;
    const Strip st = strip_of(nchunks, a.rows);
    float hi[8], lo[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        hi[j] = 0.0f;
        lo[j] = 0.0f;
    }
    if (st.chunk >= 0 && st.nr > 0) {
        const int64_t rstep = st.step * a.ld;  // elements between this thread's rows
        const T* p = reinterpret_cast<const T*>(a.x) + st.r0 * a.ld + st.chunk * 8;
        int64_t left = st.nr;
        if constexpr (PACKED) {
            using P = typename Pair16<T>::P;
            const uint32_t zbits = 0u;
            const P zero = *reinterpret_cast<const P*>(&zbits);
            P h[4], l[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                h[i] = zero;
                l[i] = zero;
            }
            for (; left > 0; left -= U, p += U * rstep) {
                Raw8<T> c[U];
#pragma unroll
                for (int k = 0; k < U; ++k) c[k] = raw8_load<T>(p + k * rstep, k < left);
#pragma unroll
                for (int k = 0; k < U; ++k) {
                    const uint32_t w[4] = {c[k].w[0].x, c[k].w[0].y, c[k].w[0].z, c[k].w[0].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const P v = *reinterpret_cast<const P*>(&w[i]);
                        if (SYM) {
                            h[i] = __hmax2(h[i], __habs2(v));
                        } else {
                            h[i] = __hmax2(h[i], v);
                            l[i] = __hmin2(l[i], v);
                        }
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                hi[2 * i] = __low2float(h[i]);
                hi[2 * i + 1] = __high2float(h[i]);
                lo[2 * i] = __low2float(l[i]);
                lo[2 * i + 1] = __high2float(l[i]);
            }
        } else {
            constexpr int UF = sizeof(T) == 4 ? 2 : 4;
            for (; left > 0; left -= UF, p += UF * rstep) {
                Raw8<T> c[UF];
#pragma unroll
                for (int k = 0; k < UF; ++k) c[k] = raw8_load<T>(p + k * rstep, k < left);
#pragma unroll
                for (int k = 0; k < UF; ++k) {
                    float v[8];
                    raw8_widen<T>(c[k], v);
                    smooth8(v, a.smooth_mode, a.smooth, st.chunk * 8);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (SYM) {
                            hi[j] = fmaxf(hi[j], fabsf(v[j]));
                        } else {
                            hi[j] = fmaxf(hi[j], v[j]);
                            lo[j] = fminf(lo[j], v[j]);
                        }
                    }
                }
            }
        }
    }
    if constexpr (PER_COL) {
        __shared__ __align__(16) float sh_hi[kStripThreads * 8];
        __shared__ __align__(16) float sh_lo[SYM ? 4 : kStripThreads * 8];
        const int cpb = nchunks < 32 ? (int)nchunks : 32;
        const int rpi = kStripThreads / cpb;
        const int ncol = cpb * 8;
        if (st.chunk >= 0) {
            const int base = ((int)threadIdx.x / cpb) * ncol + (threadIdx.x % cpb) * 8;
            reinterpret_cast<float4*>(sh_hi + base)[0] = make_float4(hi[0], hi[1], hi[2], hi[3]);
            reinterpret_cast<float4*>(sh_hi + base)[1] = make_float4(hi[4], hi[5], hi[6], hi[7]);
            if (!SYM) {
                reinterpret_cast<float4*>(sh_lo + base)[0] = make_float4(lo[0], lo[1], lo[2], lo[3]);
                reinterpret_cast<float4*>(sh_lo + base)[1] = make_float4(lo[4], lo[5], lo[6], lo[7]);
            }
        }
        __syncthreads();
        const int t = threadIdx.x;
        const int64_t c = (int64_t)blockIdx.x * ncol + t;
        if (t < ncol && c < a.cols) {
            float h = 0.0f, l = 0.0f;
            for (int k = 0; k < rpi; ++k) {
                h = fmaxf(h, sh_hi[k * ncol + t]);
                if (!SYM) l = fminf(l, sh_lo[k * ncol + t]);
            }
            if (h > 0.0f) atomicMax(&stat[2 * c], __float_as_uint(h));
            if (l < 0.0f) atomicMax(&stat[2 * c + 1], __float_as_uint(-l));
        }
    } else {
        float h = 0.0f, l = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            h = fmaxf(h, hi[j]);
            l = fminf(l, lo[j]);
        }
        h = warp_max(h);
        if (!SYM) l = warp_min(l);
        if ((threadIdx.x & 31) == 0) {
            if (h > 0.0f) atomicMax(&stat[0], __float_as_uint(h));
            if (l < 0.0f) atomicMax(&stat[1], __float_as_uint(-l));
        }
    }
}

// Statistics -> stored scale and zero point of every scope.
__global__ void k_finalize(QuantArgs a, const uint32_t* stat, int64_t nscopes) {
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= nscopes) return;
    float hi = __uint_as_float(stat[2 * i]);
    float lo = -__uint_as_float(stat[2 * i + 1]);
    if (a.absmax_out) {
        a.absmax_out[i] = hi;
        return;
    }
    float s;
    int z;
    scale_zero(lo, hi, a.qmin, a.qmax, a.sym, a.scale_f16, s, z);
    store_scale(a.s, i, a.scale_f16, s);
    if (a.z) a.z[i] = z;
}

// Codes for per-tensor / per-column scopes.  MODE 0: dynamic symmetric (no
// clamp; |rne(x/s)| <= qmax since s came from the same data), 1: dynamic
// asymmetric (clamp), 2: static scales (clamp and far-range test).  The
// eight codes of a chunk are decided together on packed pairs; per-column
// scopes give each element its own constants.  Each thread stages its
// chunks through a ring of S slots of its own in shared memory by
// asynchronous copies (S - 1 rows in flight per thread, no registers held
// for them, no barrier: a thread reads only what it copied); the row loop is
// unrolled by S so that every slot offset is a constant.  SMOOTHED instances
// apply the smoothing factors (their divisions take registers).
template <typename T, int MODE, bool PER_COL, bool SMOOTHED>
__global__ void __launch_bounds__(kStripThreads, SMOOTHED ? 2 : (PER_COL ? 3 : 4))
    k_quant_strip(QuantArgs a) {
    constexpr int W = sizeof(T) == 4 ? 2 : 1;  // 16-byte words per chunk
    constexpr int S = sizeof(T) == 4 ? 4 : 8;  // ring slots per thread
    constexpr uint32_t kSlotBytes = W * kStripThreads * 16;
    __shared__ __align__(16) uint4 ring[S * W * kStripThreads];
    const int64_t nchunks = a.cols / 8;
    const Strip st = strip_of(nchunks, a.rows);
    if (st.chunk < 0 || st.nr == 0) return;
    const int nr = (int)st.nr;
    const int64_t rstep = st.step * a.ld;
    // codes: 8 bytes (or 4 of nibbles) per chunk, rows of cols (cols/2) bytes
    const int64_t qrow = a.code4 ? a.cols / 2 : a.cols;
    const int64_t qstep = st.step * qrow;
    uint8_t* qp = reinterpret_cast<uint8_t*>(a.q) + st.r0 * qrow + st.chunk * (a.code4 ? 4 : 8);
    const T* src = reinterpret_cast<const T*>(a.x) + st.r0 * a.ld + st.chunk * 8;  // next row to copy
    const uint32_t slot0 = (uint32_t)__cvta_generic_to_shared(&ring[threadIdx.x]);
    auto copy_row = [&](int slot, bool live) {
        if (live) {
#pragma unroll
            for (int w = 0; w < W; ++w)
                cp_async16(slot0 + (uint32_t)slot * kSlotBytes + (uint32_t)w * kStripThreads * 16,
                           reinterpret_cast<const uint4*>(src) + w);
        }
        src += rstep;
        cp_async_commit();
    };
#pragma unroll
    for (int u = 0; u < S - 1; ++u) copy_row(u, u < nr);
    // (the first copies are in flight while the scopes are set up)
    const CodeRange cr = make_range(a.qmin, a.qmax);
    // the first row group's threads write the scopes they derive
    const bool writer = st.r0 == 0;
    ScopeParams sp;
    ColPair cp[4];
    if constexpr (PER_COL) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t c0 = st.chunk * 8 + 2 * j;
            const ScopeOf o0 = scope_in(a, c0, writer), o1 = scope_in(a, c0 + 1, writer);
            cp[j] = make_colpair(make_scope(o0.s, o0.z), make_scope(o1.s, o1.z));
        }
    } else {
        const ScopeOf o = scope_in(a, 0, writer && st.chunk == 0);
        sp = make_scope(o.s, o.z);
    }
    for (int j0 = 0; j0 < nr; j0 += S) {
#pragma unroll
        for (int u = 0; u < S; ++u) {
            if (j0 + u >= nr) break;
            copy_row((u + S - 1) % S, j0 + u + S - 1 < nr);
            cp_async_wait<S - 1>();
            Raw8<T> c;
#pragma unroll
            for (int w = 0; w < W; ++w) c.w[w] = ring[(u * W + w) * kStripThreads + threadIdx.x];
            float v[8];
            raw8_widen<T>(c, v);
            if constexpr (SMOOTHED) smooth8(v, a.smooth_mode, a.smooth, st.chunk * 8);
            // clamped codes as 16-bit pairs (clamp_pair16), except static
            // per-column scopes, whose far-range test already fills the
            // registers (the pairs spill there)
            constexpr bool kP = MODE == 1 || (MODE == 2 && !PER_COL);
            uint32_t cb[8];
            if constexpr (PER_COL)
                code_bits8_cols<MODE != 2, MODE != 0, kP>(v, cp, cr, cb);
            else
                code_bits8<MODE != 2, MODE != 0, true, kP>(v, sp, cr, cb);
            if (a.code4) {
                *reinterpret_cast<uint32_t*>(qp) = kP ? pack_pairs_nibbles(cb) : pack_nibbles8(cb);
            } else {
                uint2 w;
                if constexpr (kP) {
                    w = pack_pairs_bytes(cb);
                } else {
                    w.x = pack_bytes4(cb[0], cb[1], cb[2], cb[3]);
                    w.y = pack_bytes4(cb[4], cb[5], cb[6], cb[7]);
                }
                *reinterpret_cast<uint2*>(qp) = w;
            }
            qp += qstep;
        }
    }
    cp_async_wait<0>();
}

// ------------------------------------------------------------------ generic (scalar) path
__device__ __forceinline__ int64_t scope_index(int gran, int64_t r, int64_t c, int64_t cols, int group) {
    switch (gran) {
    case QLIN_PER_TENSOR: return 0;
    case QLIN_PER_ROW: return r;
    case QLIN_PER_COL: return c;
    default: return r * (cols / group) + c / group;
    }
}

template <typename T>
__device__ __forceinline__ float load_smoothed(const QuantArgs& a, int64_t r, int64_t c) {
    float v = load1<T>(reinterpret_cast<const T*>(a.x) + r * a.ld + c);
    if (a.smooth_mode == QLIN_SMOOTH_DIVIDE) return __fdiv_rn(v, a.smooth[c]);
    if (a.smooth_mode == QLIN_SMOOTH_MULTIPLY) return v * a.smooth[c];
    return v;
}

// Row-local scopes (per-row, per-group) of rows the vector kernels cannot
// take (unaligned, odd lengths, very long rows): one CTA per scope reduces its
// range and writes the stored scale and zero point straight into the caller's
// s / z (or the statistic into absmax_out), so no workspace is needed; the
// codes then come from k_quant_generic.
template <typename T>
__global__ void __launch_bounds__(256) k_scope_stats(QuantArgs a) {
    const bool grp = a.gran == QLIN_PER_GROUP;
    const int64_t ngr = grp ? a.cols / a.group : 1;
    const int64_t len = grp ? a.group : a.cols;
    const int64_t nsc = a.rows * ngr;
    __shared__ float red_hi[8], red_lo[8];
    const int tid = threadIdx.x;
    for (int64_t sc = blockIdx.x; sc < nsc; sc += gridDim.x) {
        const int64_t r = sc / ngr, c0 = (sc - r * ngr) * len;
        float hi = 0.0f, lo = 0.0f;
        for (int64_t i = tid; i < len; i += blockDim.x) {
            const float v = load_smoothed<T>(a, r, c0 + i);
            if (a.sym) {
                hi = fmaxf(hi, fabsf(v));
            } else {
                hi = fmaxf(hi, v);
                lo = fminf(lo, v);
            }
        }
        hi = warp_max(hi);
        lo = warp_min(lo);
        if ((tid & 31) == 0) {
            red_hi[tid >> 5] = hi;
            red_lo[tid >> 5] = lo;
        }
        __syncthreads();
        if (tid == 0) {
            for (int w = 1; w < (int)(blockDim.x >> 5); ++w) {
                hi = fmaxf(hi, red_hi[w]);
                lo = fminf(lo, red_lo[w]);
            }
            if (a.absmax_out) {
                a.absmax_out[sc] = hi;
            } else {
                float s;
                int z;
                scale_zero(lo, hi, a.qmin, a.qmax, a.sym, a.scale_f16, s, z);
                store_scale(a.s, sc, a.scale_f16, s);
                if (a.z) a.z[sc] = z;
            }
        }
        __syncthreads();  // red_* are reused by the next scope
    }
}

template <typename T>
__global__ void k_stats_generic(QuantArgs a, uint32_t* stat) {
    int64_t n = a.rows * a.cols;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        int64_t r = i / a.cols, c = i % a.cols;
        float v = load_smoothed<T>(a, r, c);
        int64_t sc = scope_index(a.gran, r, c, a.cols, a.group);
        if (a.sym) {
            float h = fabsf(v);
            if (h > 0.0f) atomicMax(&stat[2 * sc], __float_as_uint(h));
        } else {
            if (v > 0.0f) atomicMax(&stat[2 * sc], __float_as_uint(v));
            if (v < 0.0f) atomicMax(&stat[2 * sc + 1], __float_as_uint(-v));
        }
    }
}

// One thread per code byte (one or two elements).
template <typename T>
__global__ void k_quant_generic(QuantArgs a) {
    int64_t per_row = a.code4 ? a.cols / 2 : a.cols;
    int64_t n = a.rows * per_row;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        int64_t r = i / per_row, b = i % per_row;
        int ne = a.code4 ? 2 : 1;
        uint32_t byte = 0;
        for (int e = 0; e < ne; ++e) {
            int64_t c = b * ne + e;
            int64_t sc = scope_index(a.gran, r, c, a.cols, a.group);
            float s = load_scale(a.s, sc, a.scale_f16);
            int z = a.z ? a.z[sc] : 0;
            ScopeParams p = make_scope(s, z);
            uint32_t cbits = code_bits(load_smoothed<T>(a, r, c), p, make_range(a.qmin, a.qmax));
            byte |= a.code4 ? ((cbits & 0xFu) << (4 * e)) : (cbits & 0xFFu);
        }
        reinterpret_cast<uint8_t*>(a.q)[r * per_row + b] = (uint8_t)byte;
    }
}

// ------------------------------------------------------------------ percentile clipping
// Exact nearest-rank selection of |x| by its binary32 bit pattern (for
// non-negative floats the pattern order is the value order): a 32768-bin
// histogram of the top 16 bits, a selection, then (when the low 16 bits can be
// non-zero) a 65536-bin histogram of the low bits inside the selected bin.
// ws words: hist1[32768] | hist2[65536] | sel[4].
constexpr int kHist1 = 32768, kHist2 = 65536;

constexpr int kHistThreads = 1024;

// Level-1 histogram in shared memory, merged into hist1.  Aligned rows of
// whole chunks (strip != 0) take the column-strip tiling with several
// loads in flight per thread; the bin of unsmoothed bf16 input is its own bit
// pattern without the sign (the top half of the binary32 pattern of |x|).
// Other rows (strip = 0) take a scalar grid-stride walk.
template <typename T>
__global__ void __launch_bounds__(kHistThreads) k_hist1(QuantArgs a, uint32_t* hist1, int strip) {
    extern __shared__ uint32_t sh[];
    for (int i = threadIdx.x; i < kHist1; i += blockDim.x) sh[i] = 0;
    __syncthreads();
    if (strip) {
        constexpr int U = 4;  // loads in flight per thread
        const int64_t nchunks = a.cols / 8;
        const Strip sp = strip_of<kHistThreads>(nchunks, a.rows);
        const bool bits = std::is_same<T, __nv_bfloat16>::value && a.smooth_mode == QLIN_SMOOTH_NONE;
        if (sp.chunk >= 0) {
            const int64_t rstep = sp.step * a.ld;
            const T* p = reinterpret_cast<const T*>(a.x) + sp.r0 * a.ld + sp.chunk * 8;
            for (int64_t left = sp.nr; left > 0; left -= U, p += U * rstep) {
                Raw8<T> c[U];
#pragma unroll
                for (int k = 0; k < U; ++k) c[k] = raw8_load<T>(p + k * rstep, k < left);
#pragma unroll
                for (int k = 0; k < U; ++k) {
                    if (k >= left) break;
                    if (bits) {
                        const uint32_t w[4] = {c[k].w[0].x, c[k].w[0].y, c[k].w[0].z, c[k].w[0].w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            atomicAdd(&sh[w[i] & 0x7FFFu], 1u);
                            atomicAdd(&sh[(w[i] >> 16) & 0x7FFFu], 1u);
                        }
                    } else {
                        float v[8];
                        raw8_widen<T>(c[k], v);
                        smooth8(v, a.smooth_mode, a.smooth, sp.chunk * 8);
#pragma unroll
                        for (int j = 0; j < 8; ++j) atomicAdd(&sh[__float_as_uint(fabsf(v[j])) >> 16], 1u);
                    }
                }
            }
        }
    } else {
        for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x)
            for (int64_t c = threadIdx.x; c < a.cols; c += blockDim.x) {
                float v = fabsf(load_smoothed<T>(a, r, c));
                atomicAdd(&sh[__float_as_uint(v) >> 16], 1u);
            }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kHist1; i += blockDim.x)
        if (sh[i]) atomicAdd(&hist1[i], sh[i]);
}

template <typename T>
__global__ void k_hist2(QuantArgs a, const uint32_t* sel, uint32_t* hist2) {
    uint32_t bin = sel[0];
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x)
        for (int64_t c = threadIdx.x; c < a.cols; c += blockDim.x) {
            uint32_t u = __float_as_uint(fabsf(load_smoothed<T>(a, r, c)));
            if ((u >> 16) == bin) atomicAdd(&hist2[u & 0xFFFFu], 1u);
        }
}

// Single CTA of 1024 threads: the bin holding rank k (1-based) of `hist`
// (1024 * PER bins, PER a multiple of 32; total count below 2^32) -- the
// first bin whose inclusive prefix count reaches k -- and the rank inside
// it, written to {*out_bin, *out_rank}.  Warp w owns the PER rows of 32 bins
// from bin w * 32 * PER on and reads them coalesced, keeping each row's sum
// (lane l holds rows l, l + 32, ...).  A scan of the warp totals picks the
// warp holding rank k; a scan of its row sums picks the row; a scan of the
// row picks the bin.  (Were k above the total, the last bin would be
// returned.)
template <int PER>
__device__ void select_rank(const uint32_t* hist, uint64_t k, uint32_t* out_bin, uint64_t* out_rank) {
    __shared__ unsigned long long wtot[32];
    constexpr int NP = PER / 32;
    const unsigned full = 0xFFFFFFFFu;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const uint32_t* seg = hist + (size_t)wid * 32 * PER;
    uint32_t rsum[NP];
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const uint32_t r = __reduce_add_sync(full, seg[j * 32 + lane]);
        if ((j & 31) == lane) rsum[j >> 5] = r;
    }
    unsigned long long sum = 0;
#pragma unroll
    for (int i = 0; i < NP; ++i) sum += rsum[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(full, sum, o);
    if (lane == 0) wtot[wid] = sum;
    __syncthreads();
    if (wid == 0) {
        unsigned long long v = wtot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long u = __shfl_up_sync(full, v, o);
            if (lane >= o) v += u;
        }
        wtot[lane] = v;  // inclusive totals of warps 0..lane
    }
    __syncthreads();
    const unsigned long long incl = wtot[wid];
    const unsigned long long excl = wid > 0 ? wtot[wid - 1] : 0ull;
    if ((incl >= k && (wid == 0 || excl < k)) || (wid == 31 && incl < k)) {
        // exclusive scan: the lowest lane whose inclusive prefix reaches k
        auto first_reaching = [&](unsigned long long v, unsigned long long base, int& at,
                                  unsigned long long& before) -> bool {
            unsigned long long x = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = __shfl_up_sync(full, x, o);
                if (lane >= o) x += y;
            }
            const unsigned hit = __ballot_sync(full, base + x >= k);
            if (hit) {
                at = __ffs(hit) - 1;
                before = __shfl_sync(full, x - v, at);
                return true;
            }
            before = __shfl_sync(full, x, 31);
            return false;
        };
        unsigned long long acc = excl, before = 0;
        int row = -1, at = 0;
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            if (row < 0) {
                if (first_reaching(rsum[i], acc, at, before)) row = i * 32 + at;
                acc += before;
            }
        }
        uint32_t bin = (uint32_t)(wid * 32 * PER + 32 * PER - 1);
        if (row >= 0) {
            const uint32_t h = seg[row * 32 + lane];
            first_reaching(h, acc, at, before);
            bin = (uint32_t)(wid * 32 * PER + row * 32 + at);
            acc += before;
        }
        if (lane == 0) {
            *out_bin = bin;
            *out_rank = k - acc;
        }
    }
    __syncthreads();
}

// Level 1: select the top-16-bit bin; when `final_` the low bits are known to
// be zero and the scale is written directly.
__global__ void __launch_bounds__(1024) k_select1(QuantArgs a, const uint32_t* hist1, uint32_t* sel, uint64_t k, int final_) {
    __shared__ uint32_t bin;
    __shared__ uint64_t rk;
    select_rank<kHist1 / 1024>(hist1, k, &bin, &rk);
    if (threadIdx.x == 0) {
        sel[0] = bin;
        sel[1] = (uint32_t)rk;
        if (final_) {
            float T_ = __uint_as_float(bin << 16);
            float s;
            int z;
            scale_zero(0.0f, T_, a.qmin, a.qmax, true, a.scale_f16, s, z);
            store_scale(a.s, 0, a.scale_f16, s);
            if (a.z) a.z[0] = 0;
        }
    }
}

__global__ void __launch_bounds__(1024) k_select2(QuantArgs a, const uint32_t* hist2, const uint32_t* sel) {
    __shared__ uint32_t bin;
    __shared__ uint64_t rk;
    select_rank<kHist2 / 1024>(hist2, sel[1], &bin, &rk);
    if (threadIdx.x == 0) {
        float T_ = __uint_as_float((sel[0] << 16) | bin);
        float s;
        int z;
        scale_zero(0.0f, T_, a.qmin, a.qmax, true, a.scale_f16, s, z);
        store_scale(a.s, 0, a.scale_f16, s);
        if (a.z) a.z[0] = 0;
    }
}

// ------------------------------------------------------------------ dequantize
struct DequantArgs {
    const void* q;
    const void* s;
    const int32_t* z;
    int64_t rows, cols;
    int gran, group, scale_f16, code4, code_signed;
    void* y;
    int yt;
};

__device__ __forceinline__ int code_at(const DequantArgs& d, int64_t r, int64_t c) {
    if (d.code4) {
        uint8_t b = reinterpret_cast<const uint8_t*>(d.q)[r * (d.cols / 2) + c / 2];
        int v = (c & 1) ? (b >> 4) : (b & 0xF);
        if (d.code_signed && v >= 8) v -= 16;
        return v;
    }
    if (d.code_signed) return reinterpret_cast<const int8_t*>(d.q)[r * d.cols + c];
    return reinterpret_cast<const uint8_t*>(d.q)[r * d.cols + c];
}

__device__ __forceinline__ void store_y(const DequantArgs& d, int64_t i, float v) {
    if (d.yt == QLIN_BF16)
        reinterpret_cast<__nv_bfloat16*>(d.y)[i] = __float2bfloat16_rn(v);
    else if (d.yt == QLIN_F16)
        reinterpret_cast<__half*>(d.y)[i] = __float2half_rn(v);
    else
        reinterpret_cast<float*>(d.y)[i] = v;
}

// Vector path: 8 elements per thread (cols % 8 == 0, group % 8 == 0).
__global__ void k_dequant_vec(DequantArgs d) {
    int64_t nchunks = d.rows * (d.cols / 8);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nchunks; i += (int64_t)gridDim.x * blockDim.x) {
        int64_t r = i / (d.cols / 8), c0 = (i % (d.cols / 8)) * 8;
        int code[8];
        if (d.code4) {
            uint32_t w = reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint8_t*>(d.q) + r * (d.cols / 2))[c0 / 8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                int v = (w >> (4 * j)) & 0xF;
                code[j] = (d.code_signed && v >= 8) ? v - 16 : v;
            }
        } else {
            uint2 w = reinterpret_cast<const uint2*>(reinterpret_cast<const uint8_t*>(d.q) + r * d.cols)[c0 / 8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint32_t b = ((j < 4 ? w.x : w.y) >> (8 * (j & 3))) & 0xFFu;
                code[j] = d.code_signed ? (int)(int8_t)b : (int)b;
            }
        }
        float out[8];
        if (d.gran == QLIN_PER_COL) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float s = load_scale(d.s, c0 + j, d.scale_f16);
                int z = d.z ? d.z[c0 + j] : 0;
                out[j] = s * (float)(code[j] - z);
            }
        } else {
            // one scope for the whole chunk (groups are whole chunks)
            int64_t sc = (d.gran == QLIN_PER_TENSOR) ? 0
                       : (d.gran == QLIN_PER_ROW) ? r
                       : r * (d.cols / d.group) + c0 / d.group;
            float s = load_scale(d.s, sc, d.scale_f16);
            int z = d.z ? d.z[sc] : 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) out[j] = s * (float)(code[j] - z);
        }
        int64_t base = r * d.cols + c0;
        if (d.yt == QLIN_BF16) {
            uint4 u;
            __nv_bfloat162 p0 = __floats2bfloat162_rn(out[0], out[1]);
            __nv_bfloat162 p1 = __floats2bfloat162_rn(out[2], out[3]);
            __nv_bfloat162 p2 = __floats2bfloat162_rn(out[4], out[5]);
            __nv_bfloat162 p3 = __floats2bfloat162_rn(out[6], out[7]);
            u.x = *reinterpret_cast<uint32_t*>(&p0);
            u.y = *reinterpret_cast<uint32_t*>(&p1);
            u.z = *reinterpret_cast<uint32_t*>(&p2);
            u.w = *reinterpret_cast<uint32_t*>(&p3);
            reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(d.y) + base)[0] = u;
        } else if (d.yt == QLIN_F32) {
            float4* yp = reinterpret_cast<float4*>(reinterpret_cast<float*>(d.y) + base);
            yp[0] = make_float4(out[0], out[1], out[2], out[3]);
            yp[1] = make_float4(out[4], out[5], out[6], out[7]);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) store_y(d, base + j, out[j]);
        }
    }
}

// Row-segment path (per-tensor / per-row / per-group with g % 16 == 0,
// cols % 16 == 0): a CTA takes one segment of kDqUnroll * 256 chunks of 16
// codes of one row and issues all of its loads before converting, so each
// thread keeps kDqUnroll loads in flight; the row and segment come from one
// division per CTA iteration.  Same arithmetic as k_dequant_vec.
constexpr int kDqUnroll = 4;

__device__ __forceinline__ void store16_y(const DequantArgs& d, int64_t base, const float (&o)[16]) {
    if (d.yt == QLIN_F32) {
        float4* yp = reinterpret_cast<float4*>(reinterpret_cast<float*>(d.y) + base);
#pragma unroll
        for (int j = 0; j < 4; ++j) yp[j] = make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
        return;
    }
    uint32_t w[8];
    if (d.yt == QLIN_BF16) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            __nv_bfloat162 p2 = __floats2bfloat162_rn(o[2 * j], o[2 * j + 1]);
            w[j] = *reinterpret_cast<uint32_t*>(&p2);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            __half2 p2 = __floats2half2_rn(o[2 * j], o[2 * j + 1]);
            w[j] = *reinterpret_cast<uint32_t*>(&p2);
        }
    }
    uint4* yp = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(d.y) + base);
    yp[0] = make_uint4(w[0], w[1], w[2], w[3]);
    yp[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// s * (code - z) of the 16 codes of a chunk (INT8: raw.x..w; INT4: raw.x,
// raw.y, code j in nibble j), as binary32 values.  INT4 codes take no
// integer-to-float conversions: each nibble, made non-negative (signed codes
// get their sign bit flipped, i.e. code + 8), is placed below the exponent of
// 2^23 by a byte permute, and one subtraction of 2^23 + offset + z leaves the
// integer code - z exactly (every quantity is an integer below 2^24, and the
// two operands are within a factor of two); the product with s is the same
// binary32 multiplication as s * (float)(code - z).  Measured on 16384 x 4096
// per-group-128 INT4 / UINT4: 53.8 -> 48.0 us and 55.8 -> 49.9 us.  The same
// for INT8 codes was slower on the 28672-value rows (65.5 -> 71.9 us), so
// those keep the integer conversion.
__device__ __forceinline__ void dq16(const uint4 raw, bool code4, bool code_signed, int z, float s, float o[16]) {
    if (code4) {
        const float c = 8388608.0f + (float)((code_signed ? 8 : 0) + z);
        uint32_t m[16];
        const uint32_t flip = code_signed ? 0x88888888u : 0u;
        const uint32_t w[2] = {raw.x ^ flip, raw.y ^ flip};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t lo = w[h] & 0x0F0F0F0Fu, hi = (w[h] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                m[8 * h + 2 * k] = __byte_perm(lo, 0x4B000000u, 0x7540u | k);
                m[8 * h + 2 * k + 1] = __byte_perm(hi, 0x4B000000u, 0x7540u | k);
            }
        }
        const float2 nc2 = make_float2(-c, -c), s2 = make_float2(s, s);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float2 d2 = f2_add(make_float2(__uint_as_float(m[2 * j]), __uint_as_float(m[2 * j + 1])), nc2);
            const float2 p2 = f2_mul(d2, s2);
            o[2 * j] = p2.x;
            o[2 * j + 1] = p2.y;
        }
    } else {
        const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const uint32_t b = (wv[j >> 2] >> (8 * (j & 3))) & 0xFFu;
            const int code = code_signed ? (int)(int8_t)b : (int)b;
            o[j] = s * (float)(code - z);
        }
    }
}

__global__ void __launch_bounds__(256) k_dequant_rows(DequantArgs d) {
    const int tid = threadIdx.x, nt = blockDim.x;
    const int64_t nch = d.cols / 16;
    const int64_t seg_len = (int64_t)kDqUnroll * nt;
    const int64_t nseg = (nch + seg_len - 1) / seg_len;
    const int64_t units = d.rows * nseg;
    for (int64_t unit = blockIdx.x; unit < units; unit += gridDim.x) {
        const int64_t r = unit / nseg, c0 = (unit - r * nseg) * seg_len + tid;
        uint4 raw[kDqUnroll];
#pragma unroll
        for (int u = 0; u < kDqUnroll; ++u) {
            const int64_t c = c0 + (int64_t)u * nt;
            if (c < nch) {
                if (d.code4) {
                    const uint2 w = reinterpret_cast<const uint2*>(reinterpret_cast<const uint8_t*>(d.q) + r * (d.cols / 2))[c];
                    raw[u] = make_uint4(w.x, w.y, 0, 0);
                } else {
                    raw[u] = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(d.q) + r * d.cols)[c];
                }
            }
        }
        const bool row_scope = d.gran != QLIN_PER_GROUP;
        float s_row = 0.0f;
        int z_row = 0;
        if (row_scope) {
            const int64_t sc = (d.gran == QLIN_PER_TENSOR) ? 0 : r;
            s_row = load_scale(d.s, sc, d.scale_f16);
            z_row = d.z ? d.z[sc] : 0;
        }
#pragma unroll
        for (int u = 0; u < kDqUnroll; ++u) {
            const int64_t c = c0 + (int64_t)u * nt;
            if (c >= nch) break;
            float s = s_row;
            int z = z_row;
            if (!row_scope) {
                const int64_t sc = r * (d.cols / d.group) + (c * 16) / d.group;
                s = load_scale(d.s, sc, d.scale_f16);
                z = d.z ? d.z[sc] : 0;
            }
            float o[16];
            dq16(raw[u], d.code4, d.code_signed, z, s, o);
            store16_y(d, r * d.cols + c * 16, o);
        }
    }
}

// Short rows (row-segment conditions, and a row's chunk count divides
// kDqUnroll * 256): a CTA takes a unit of several whole rows, so each thread
// keeps kDqUnroll code and scale loads in flight where k_dequant_rows would
// have one.  Same arithmetic as k_dequant_vec.
__global__ void __launch_bounds__(256) k_dequant_short(DequantArgs d) {
    const int tid = threadIdx.x, nt = blockDim.x;
    const int64_t nch = d.cols / 16;
    const int64_t rows_per_unit = (int64_t)kDqUnroll * nt / nch;
    const int64_t units = (d.rows + rows_per_unit - 1) / rows_per_unit;
    // chunk u of this thread: row offset roff[u], chunk column coff[u] of every unit
    int roff[kDqUnroll];
    int coff[kDqUnroll];
#pragma unroll
    for (int u = 0; u < kDqUnroll; ++u) {
        const int f = tid + u * nt;
        roff[u] = (int)(f / nch);
        coff[u] = (int)(f % nch);
    }
    const bool row_scope = d.gran != QLIN_PER_GROUP;
    for (int64_t unit = blockIdx.x; unit < units; unit += gridDim.x) {
        const int64_t r0 = unit * rows_per_unit;
        uint4 raw[kDqUnroll];
        float sv[kDqUnroll];
        int zv[kDqUnroll];
#pragma unroll
        for (int u = 0; u < kDqUnroll; ++u) {
            const int64_t r = r0 + roff[u];
            const int64_t c = coff[u];
            if (r < d.rows) {
                if (d.code4) {
                    const uint2 w = reinterpret_cast<const uint2*>(reinterpret_cast<const uint8_t*>(d.q) + r * (d.cols / 2))[c];
                    raw[u] = make_uint4(w.x, w.y, 0, 0);
                } else {
                    raw[u] = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(d.q) + r * d.cols)[c];
                }
                const int64_t sc = row_scope ? ((d.gran == QLIN_PER_TENSOR) ? 0 : r)
                                             : r * (d.cols / d.group) + (c * 16) / d.group;
                sv[u] = load_scale(d.s, sc, d.scale_f16);
                zv[u] = d.z ? d.z[sc] : 0;
            }
        }
#pragma unroll
        for (int u = 0; u < kDqUnroll; ++u) {
            const int64_t r = r0 + roff[u];
            const int64_t c = coff[u];
            if (r >= d.rows) continue;
            const float s = sv[u];
            const int z = zv[u];
            float o[16];
            dq16(raw[u], d.code4, d.code_signed, z, s, o);
            store16_y(d, r * d.cols + c * 16, o);
        }
    }
}

__global__ void k_dequant_generic(DequantArgs d) {
    int64_t n = d.rows * d.cols;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        int64_t r = i / d.cols, c = i % d.cols;
        int64_t sc = scope_index(d.gran, r, c, d.cols, d.group);
        float s = load_scale(d.s, sc, d.scale_f16);
        int z = d.z ? d.z[sc] : 0;
        store_y(d, i, s * (float)(code_at(d, r, c) - z));
    }
}

// ------------------------------------------------------------------ smoothing factors
// s_j = max|X_j|^alpha / max|W_j|^(1-alpha) ("量化、蒸馏与模型压缩" 2.3 eq. 1).
__global__ void k_smooth_factors(const float* xmax, const float* wmax, int64_t K, float alpha, float* s) {
    int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= K) return;
    float mx = xmax[j], mw = wmax[j];
    float v;
    if (mx == 0.0f || mw == 0.0f)
        v = 1.0f;
    else if (alpha == 0.5f)
        v = __fdiv_rn(__fsqrt_rn(mx), __fsqrt_rn(mw));
    else
        v = __fdiv_rn(powf(mx, alpha), powf(mw, 1.0f - alpha));
    s[j] = v;
}

// ------------------------------------------------------------------ host launchers
static int g_num_sms = 0;
cudaError_t ensure_smem(const void* kernel, int bytes) {
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, int> raised;  // (kernel, device) -> bytes
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    int& have = raised[std::make_pair(kernel, dev)];
    if (have >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) have = bytes;
    return e;
}

int num_sms() {
    if (g_num_sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (g_num_sms <= 0) g_num_sms = 148;
    }
    return g_num_sms;
}

static inline int elem_size(int xt) { return xt == QLIN_F32 ? 4 : 2; }

// Whether the row kernel applies: 8-element chunks, 16-byte aligned rows,
// groups that are whole chunks and fit a warp.
static bool rows_kernel_ok(const QuantArgs& a, int xt) {
    int es = elem_size(xt);
    if (a.cols % 8 != 0) return false;
    if (((uintptr_t)a.x) % 16 != 0 || (a.ld * es) % 16 != 0) return false;
    if (a.code4 && ((uintptr_t)a.q) % 4 != 0) return false;
    if (!a.code4 && ((uintptr_t)a.q) % 8 != 0) return false;
    if (a.gran == QLIN_PER_GROUP) {
        if (a.group % 8 != 0 || a.group > 256) return false;
        int gl = a.group / 8;
        if (gl & (gl - 1)) return false;  // power of two lanes
    }
    if (a.cols / 8 > 8 * 512) return false;
    if (a.smooth_mode != QLIN_SMOOTH_NONE && ((uintptr_t)a.smooth) % 16 != 0) return false;
    return true;
}

template <typename T, bool SYM, bool STATIC, bool CODE4, int GL>
static cudaError_t launch_qgrp_warp(const QuantArgs& a, int64_t nchunks, int64_t grid, cudaStream_t st) {
    (void)grid;
    const int64_t units = a.rows * ceil_div(nchunks, 32);
    int64_t g = ceil_div(units, 8);  // 8 warps per CTA
    const int64_t cap = (int64_t)num_sms() * 16;
    if (g > cap) g = cap;
    k_qgrp_slab<T, SYM, STATIC, CODE4, GL><<<(unsigned)g, 256, 0, st>>>(a);
    return cudaGetLastError();
}

template <typename T, bool SYM, bool STATIC, bool CODE4>
static cudaError_t launch_qrow_warp_m(const QuantArgs& a, cudaStream_t st) {
    const int64_t nchunks = a.cols / 8;
    int64_t grid = ceil_div(a.rows, 8);  // 8 warps (rows) per CTA
    const int64_t cap = (int64_t)num_sms() * 8;
    if (grid > cap) grid = cap;
    const bool row = a.gran == QLIN_PER_ROW;
    if (row) {
        if (nchunks <= 128)
            k_qrow_warp<T, SYM, STATIC, CODE4, 4><<<(unsigned)grid, 256, 0, st>>>(a);
        else
            k_qrow_warp<T, SYM, STATIC, CODE4, 16><<<(unsigned)grid, 256, 0, st>>>(a);
        return cudaGetLastError();
    }
    // per-group: lanes per group as a compile-time constant (g = 8 * GL)
    switch (a.group / 8) {
    case 1: return launch_qgrp_warp<T, SYM, STATIC, CODE4, 1>(a, nchunks, grid, st);
    case 2: return launch_qgrp_warp<T, SYM, STATIC, CODE4, 2>(a, nchunks, grid, st);
    case 4: return launch_qgrp_warp<T, SYM, STATIC, CODE4, 4>(a, nchunks, grid, st);
    case 8: return launch_qgrp_warp<T, SYM, STATIC, CODE4, 8>(a, nchunks, grid, st);
    case 16: return launch_qgrp_warp<T, SYM, STATIC, CODE4, 16>(a, nchunks, grid, st);
    default: return launch_qgrp_warp<T, SYM, STATIC, CODE4, 32>(a, nchunks, grid, st);
    }
}

template <typename T>
static cudaError_t launch_qrow_warp(const QuantArgs& a, cudaStream_t st) {
    if (a.static_scale)
        return a.code4 ? launch_qrow_warp_m<T, true, true, true>(a, st) : launch_qrow_warp_m<T, true, true, false>(a, st);
    if (a.sym)
        return a.code4 ? launch_qrow_warp_m<T, true, false, true>(a, st) : launch_qrow_warp_m<T, true, false, false>(a, st);
    return a.code4 ? launch_qrow_warp_m<T, false, false, true>(a, st) : launch_qrow_warp_m<T, false, false, false>(a, st);
}

// Shared memory of one SM: two CTAs of two row buffers each fit it for rows of
// up to 28,672 16-bit values; longer rows take one CTA with three buffers.
constexpr size_t kSmemPerSM = 233472;

static int qrow_choice();

template <typename T, bool SYM, bool STATIC, bool CODE4, int NT, int GL>
static cudaError_t launch_qrow_bulk_k(const QuantArgs& a, uint32_t buf_stride, cudaStream_t st) {
    // rows of up to NC * NT chunks are held in registers (k_qrow_reg) at 128
    // threads and for per-row scopes at 512 threads; per-group scopes at 512
    // threads take the row-buffer kernel: there the 64-register cap of two
    // CTAs per SM spills, and the register-held kernel measured slower
    // (4096 x 28672 bf16 at g = 128: 92 us against 78 us).  Eight chunks a
    // thread at 64 threads measured slower too (16384 x 4096 per-token INT8
    // 47.7 us against 41.5 us): its unrolled copies of the exact fallback
    // fill the instruction cache, and out of line the call spills.
    constexpr int NC = NT >= 512 ? 8 : 4;
    constexpr bool kReg = NT == 128 || (NT == 512 && GL == 0);
    const bool reg = kReg && a.cols / 8 <= (int64_t)NC * NT && qrow_choice() != 2;
    const void* kern = (const void*)k_qrow_bulk<T, SYM, STATIC, CODE4, NT, GL>;
    if constexpr (kReg)
        if (reg) kern = (const void*)k_qrow_reg<T, SYM, STATIC, CODE4, NT, GL, NC>;
    int nbuf, smem;
    int64_t grid;
    if (NT == 512) {
        const bool two = 2 * (2 * (size_t)buf_stride + 1024 + 512) <= kSmemPerSM;
        nbuf = two ? 2 : (3 * (size_t)buf_stride <= 200 * 1024 ? 3 : 2);
        smem = nbuf * (int)buf_stride;
        grid = (int64_t)num_sms() * (two ? 2 : 1);
    } else {
        nbuf = 2;
        smem = nbuf * (int)buf_stride;
    }
    cudaError_t e = ensure_smem(kern, smem);
    if (e != cudaSuccess) return e;
    if (NT != 512) {
        int per_sm = 0;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT, smem)) != cudaSuccess) return e;
        grid = (int64_t)num_sms() * (per_sm > 0 ? per_sm : 1);
    }
    if (grid > a.rows) grid = a.rows;
    if constexpr (kReg) {
        if (reg) {
            k_qrow_reg<T, SYM, STATIC, CODE4, NT, GL, NC><<<(unsigned)grid, NT, smem, st>>>(a, buf_stride, nbuf);
            return cudaGetLastError();
        }
    }
    k_qrow_bulk<T, SYM, STATIC, CODE4, NT, GL><<<(unsigned)grid, NT, smem, st>>>(a, buf_stride, nbuf);
    return cudaGetLastError();
}

// NT = 512 threads for rows of more than 8192 values, 128 for shorter ones;
// dynamic symmetric per-token INT8 codes of rows of up to 4096 values take
// the row-buffer kernel at 64 threads, whose smaller CTAs keep more rows in
// flight per SM (16384 x 4096 bf16: 39.8 us against 41.3 us; the other code
// widths and scopes measured slower there).  Measured on 16384 x 4096 and
// 4096 x 28672 bf16.
template <typename T, bool SYM, bool STATIC, bool CODE4, int GL>
static cudaError_t launch_qrow_bulk_g(const QuantArgs& a, uint32_t buf_stride, cudaStream_t st) {
    if constexpr (GL == 0 && SYM && !STATIC && !CODE4) {
        if (a.cols <= 4096) return launch_qrow_bulk_k<T, SYM, STATIC, CODE4, 64, GL>(a, buf_stride, st);
    }
    if (a.cols <= 8192) return launch_qrow_bulk_k<T, SYM, STATIC, CODE4, 128, GL>(a, buf_stride, st);
    return launch_qrow_bulk_k<T, SYM, STATIC, CODE4, 512, GL>(a, buf_stride, st);
}

template <typename T, bool SYM, bool STATIC, bool CODE4>
static cudaError_t launch_qrow_bulk_m(const QuantArgs& a, uint32_t buf_stride, cudaStream_t st) {
    if (a.gran == QLIN_PER_ROW) return launch_qrow_bulk_g<T, SYM, STATIC, CODE4, 0>(a, buf_stride, st);
    switch (a.group / 8) {
    case 1: return launch_qrow_bulk_g<T, SYM, STATIC, CODE4, 1>(a, buf_stride, st);
    case 2: return launch_qrow_bulk_g<T, SYM, STATIC, CODE4, 2>(a, buf_stride, st);
    case 4: return launch_qrow_bulk_g<T, SYM, STATIC, CODE4, 4>(a, buf_stride, st);
    case 8: return launch_qrow_bulk_g<T, SYM, STATIC, CODE4, 8>(a, buf_stride, st);
    case 16: return launch_qrow_bulk_g<T, SYM, STATIC, CODE4, 16>(a, buf_stride, st);
    default: return launch_qrow_bulk_g<T, SYM, STATIC, CODE4, 32>(a, buf_stride, st);
    }
}

template <typename T>
static cudaError_t launch_qrow_bulk(const QuantArgs& a, uint32_t buf_stride, cudaStream_t st) {
    if (a.static_scale)
        return a.code4 ? launch_qrow_bulk_m<T, true, true, true>(a, buf_stride, st)
                       : launch_qrow_bulk_m<T, true, true, false>(a, buf_stride, st);
    if (a.sym)
        return a.code4 ? launch_qrow_bulk_m<T, true, false, true>(a, buf_stride, st)
                       : launch_qrow_bulk_m<T, true, false, false>(a, buf_stride, st);
    return a.code4 ? launch_qrow_bulk_m<T, false, false, true>(a, buf_stride, st)
                   : launch_qrow_bulk_m<T, false, false, false>(a, buf_stride, st);
}

template <typename T>
static cudaError_t launch_rows(const QuantArgs& a, cudaStream_t st) {
    int64_t nchunks = a.cols / 8;
    int cpt = (nchunks <= 512) ? 1 : (nchunks <= 1024) ? 2 : (nchunks <= 2048) ? 4 : 8;
    int64_t nt = ceil_div(nchunks, cpt);
    nt = ceil_div(nt, 32) * 32;
    if (a.gran == QLIN_PER_GROUP) {
        int gl = a.group / 8;
        if (nt % gl) nt = ceil_div(nt, gl) * gl;
    }
    if (nt < 32) nt = 32;
    int per_sm = (int)(2048 / nt);
    if (per_sm < 1) per_sm = 1;
    int64_t grid = (int64_t)num_sms() * per_sm;
    if (grid > a.rows) grid = a.rows;
    if (grid < 1) grid = 1;
    switch (cpt) {
    case 1: k_quant_rows<T, 1><<<(unsigned)grid, (unsigned)nt, 0, st>>>(a); break;
    case 2: k_quant_rows<T, 2><<<(unsigned)grid, (unsigned)nt, 0, st>>>(a); break;
    case 4: k_quant_rows<T, 4><<<(unsigned)grid, (unsigned)nt, 0, st>>>(a); break;
    default: k_quant_rows<T, 8><<<(unsigned)grid, (unsigned)nt, 0, st>>>(a); break;
    }
    return cudaGetLastError();
}

// Grid of the column-strip kernels (nt threads a block): gx blocks across
// the chunk columns and as many down the rows as fill the GPU once at
// `per_sm` resident blocks per SM (no more than there are row groups).
static dim3 strip_grid(int64_t nchunks, int64_t rows, int nt, int per_sm) {
    const int64_t cpb = nchunks < 32 ? nchunks : 32;
    const int64_t rpi = nt / cpb;
    const int64_t gx = ceil_div(nchunks, cpb);
    const int64_t target = (int64_t)num_sms() * (per_sm > 0 ? per_sm : 1);
    int64_t gy = target / gx;
    if (gy > ceil_div(rows, rpi)) gy = ceil_div(rows, rpi);
    if (gy > 65535) gy = 65535;
    if (gy < 1) gy = 1;
    return dim3((unsigned)gx, (unsigned)gy);
}

template <typename T>
using QuantStripFn = void (*)(QuantArgs);
template <typename T, bool SM>
static QuantStripFn<T> quant_strip_fn_s(int mode, bool pc) {
    switch (mode * 2 + (pc ? 1 : 0)) {
    case 0: return k_quant_strip<T, 0, false, SM>;
    case 1: return k_quant_strip<T, 0, true, SM>;
    case 2: return k_quant_strip<T, 1, false, SM>;
    case 3: return k_quant_strip<T, 1, true, SM>;
    case 4: return k_quant_strip<T, 2, false, SM>;
    default: return k_quant_strip<T, 2, true, SM>;
    }
}
template <typename T>
static QuantStripFn<T> quant_strip_fn(int mode, bool pc, bool smoothed) {
    return smoothed ? quant_strip_fn_s<T, true>(mode, pc) : quant_strip_fn_s<T, false>(mode, pc);
}
template <typename T, bool PACKED>
static void (*stats_strip_fn_p(bool sym, bool pc))(QuantArgs, uint32_t*) {
    if (sym) return pc ? k_stats_strip<T, true, true, PACKED> : k_stats_strip<T, true, false, PACKED>;
    return pc ? k_stats_strip<T, false, true, PACKED> : k_stats_strip<T, false, false, PACKED>;
}
// PACKED statistics for unsmoothed 16-bit input.
template <typename T>
static void (*stats_strip_fn(bool sym, bool pc, bool smoothed))(QuantArgs, uint32_t*) {
    if constexpr (sizeof(T) == 2) {
        if (!smoothed) return stats_strip_fn_p<T, true>(sym, pc);
    }
    return stats_strip_fn_p<T, false>(sym, pc);
}

// Resident blocks per SM of a kernel launch shape (queried once per kernel,
// shape and device).
static int blocks_per_sm(const void* kern, int nt, size_t smem) {
    static std::mutex mu;
    static std::map<std::tuple<const void*, int, size_t, int>, int> known;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_tuple(kern, nt, smem, dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = known.find(key);
        if (it != known.end()) return it->second;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, nt, smem) != cudaSuccess || n < 1) n = 1;
    std::lock_guard<std::mutex> lock(mu);
    known[key] = n;
    return n;
}

// QLIN_QROW: "warp" keeps the register-resident row kernels (per-row rows of
// up to 4096 values, per-group slabs), "smem" the row-streaming kernel that
// reads its chunks from the row buffer (k_qrow_bulk), and "strip" the strip
// kernel for the codes of dynamic symmetric per-tensor scopes, for
// comparisons; read on every call, same codes.
static int qrow_choice() {
    const char* e = getenv("QLIN_QROW");
    if (e && strcmp(e, "warp") == 0) return 1;
    if (e && strcmp(e, "smem") == 0) return 2;
    if (e && strcmp(e, "strip") == 0) return 3;
    return 0;
}

static bool strip_ok(const QuantArgs& a, int xt) {
    int es = elem_size(xt);
    if (a.cols % 8 != 0 || a.rows == 0) return false;
    if (a.smooth_mode != QLIN_SMOOTH_NONE && ((uintptr_t)a.smooth) % 16 != 0) return false;
    if (((uintptr_t)a.x) % 16 != 0 || (a.ld * es) % 16 != 0) return false;
    if (a.code4 && ((uintptr_t)a.q) % 4 != 0) return false;
    if (!a.code4 && ((uintptr_t)a.q) % 8 != 0) return false;
    return true;
}

static int64_t nscopes_of(const QuantArgs& a) {
    switch (a.gran) {
    case QLIN_PER_TENSOR: return 1;
    case QLIN_PER_ROW: return a.rows;
    case QLIN_PER_COL: return a.cols;
    default: return a.rows * (a.cols / a.group);
    }
}

size_t quantize_ws_bytes(int64_t rows, int64_t cols, const qlin_qparams* p) {
    if (p->static_scale) return 0;
    if (p->clip_percentile > 0.0) return (size_t)(kHist1 + kHist2 + 4) * 4;
    if (p->gran == QLIN_PER_TENSOR) return 2 * 4;
    if (p->gran == QLIN_PER_COL) return (size_t)cols * 2 * 4;
    // per-row / per-group: every kernel that serves these scopes (the fused
    // row kernels and k_scope_stats) keeps its statistics on chip
    return 0;
}

template <typename T>
static cudaError_t run_quantize_t(QuantArgs a, int xt, const qlin_qparams* p, void* ws, cudaStream_t st) {
    cudaError_t e = cudaSuccess;
    const int64_t n = a.rows * a.cols;
    const int gblocks = num_sms() * 4;
    const bool row_local = (a.gran == QLIN_PER_ROW || a.gran == QLIN_PER_GROUP);
    if (row_local && rows_kernel_ok(a, xt) && p->clip_percentile <= 0.0) {
        const int64_t nchunks = a.cols / 8;
        const size_t row_bytes = (size_t)a.cols * sizeof(float);
        const size_t raw_bytes = (size_t)a.cols * 2;
        const uint32_t buf_stride = (uint32_t)((raw_bytes + 127) & ~(size_t)127);
        if constexpr (!std::is_same<T, float>::value) {
            // binary16 scales can saturate at 65504, and then |x/s| is not
            // bounded by qmax: those calls take kernels that clamp and test
            // the range of every code
            const bool fast16 = !a.absmax_out && a.smooth_mode == QLIN_SMOOTH_NONE && !a.scale_f16;
            if (fast16 && qrow_choice() == 1 && nchunks <= 512) return launch_qrow_warp<T>(a, st);
            if (fast16 && 2 * (size_t)buf_stride <= 200 * 1024) return launch_qrow_bulk<T>(a, buf_stride, st);
        }
        if (a.gran == QLIN_PER_ROW && !a.absmax_out && nchunks > 1024 && row_bytes <= 113 * 1024) {
            cudaError_t e = ensure_smem((const void*)k_quant_longrows<T>, (int)row_bytes);
            if (e != cudaSuccess) return e;
            int64_t grid = (int64_t)num_sms() * 2;
            if (grid > a.rows) grid = a.rows;
            k_quant_longrows<T><<<(unsigned)grid, 512, row_bytes, st>>>(a);
            return cudaGetLastError();
        }
        return launch_rows<T>(a, st);
    }

    if (row_local) {
        // rows the vector kernels cannot take: per-scope statistics straight
        // into s / z, then scalar codes
        if (!a.static_scale) {
            int64_t nsc = nscopes_of(a);
            int64_t grid = nsc < (int64_t)gblocks * 2 ? nsc : (int64_t)gblocks * 2;
            k_scope_stats<T><<<(unsigned)grid, 256, 0, st>>>(a);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
        if (a.absmax_out) return cudaSuccess;
        k_quant_generic<T><<<gblocks, 256, 0, st>>>(a);
        return cudaGetLastError();
    }

    // Per-tensor / per-column: statistics (dynamic) -> codes.  The codes
    // kernels derive the scopes' (s, z) from the statistics themselves (and
    // write them out); the scalar fallback and qlin_absmax take k_finalize.
    const bool strip = strip_ok(a, xt);
    const bool pc = a.gran == QLIN_PER_COL;
    const bool smoothed = a.smooth_mode != QLIN_SMOOTH_NONE;
    // percentile scales clip values beyond the percentile, and binary16
    // scales can saturate: both take the fully checked codes
    const int mode = (a.static_scale || p->clip_percentile > 0.0 || a.scale_f16) ? 2 : (a.sym ? 0 : 1);
    // per-tensor codes of unsmoothed 16-bit rows: the row-streaming kernels
    // with one scope for all rows.  Dynamic scopes (modes 0 and 1, rows of up
    // to 8192 values) take the per-row kernels' arithmetic -- no far-range
    // test, and no clamp for symmetric codes, since the tensor's own max|x|
    // (or range) bounds every |x / s| -- and the other scales the fully
    // checked one.
    uint32_t buf_stride = 0;
    bool rowcodes = false;
    if constexpr (!std::is_same<T, float>::value) {
        buf_stride = (uint32_t)(((size_t)a.cols * 2 + 127) & ~(size_t)127);
        rowcodes = !pc && !smoothed && strip && a.cols / 8 <= 8 * 512 && 2 * (size_t)buf_stride <= 200 * 1024 &&
                   (mode == 2 || a.cols <= 8192) && !(mode == 0 && qrow_choice() == 3);
    }
    if (!a.static_scale) {
        uint32_t* stat = reinterpret_cast<uint32_t*>(ws);
        if (p->clip_percentile > 0.0) {
            uint32_t* hist1 = stat;
            uint32_t* hist2 = stat + kHist1;
            uint32_t* sel = hist2 + kHist2;
            uint64_t k = (uint64_t)percentile_rank(n, p->clip_percentile);
            if ((e = cudaMemsetAsync(ws, 0, (size_t)(kHist1 + kHist2 + 4) * 4, st)) != cudaSuccess) return e;
            if ((e = ensure_smem((const void*)k_hist1<T>, kHist1 * 4)) != cudaSuccess) return e;
            if (strip) {
                const dim3 hgrid = strip_grid(a.cols / 8, a.rows, kHistThreads,
                                              blocks_per_sm((const void*)k_hist1<T>, kHistThreads, kHist1 * 4));
                k_hist1<T><<<hgrid, kHistThreads, kHist1 * 4, st>>>(a, hist1, 1);
            } else {
                k_hist1<T><<<num_sms(), kHistThreads, kHist1 * 4, st>>>(a, hist1, 0);
            }
            // Low 16 bits of |x| are zero for unsmoothed bf16 input.
            bool need2 = !(xt == QLIN_BF16 && a.smooth_mode == QLIN_SMOOTH_NONE);
            k_select1<<<1, 1024, 0, st>>>(a, hist1, sel, k, need2 ? 0 : 1);
            if (need2) {
                k_hist2<T><<<gblocks, 256, 0, st>>>(a, sel, hist2);
                k_select2<<<1, 1024, 0, st>>>(a, hist2, sel);
            }
        } else {
            int64_t ns = nscopes_of(a);
            if ((e = cudaMemsetAsync(ws, 0, (size_t)ns * 8, st)) != cudaSuccess) return e;
            if (strip) {
                auto ks = stats_strip_fn<T>(a.sym, pc, smoothed);
                ks<<<strip_grid(a.cols / 8, a.rows, kStripThreads, blocks_per_sm((const void*)ks, kStripThreads, 0)),
                     kStripThreads, 0, st>>>(a, stat);
            } else {
                k_stats_generic<T><<<gblocks, 256, 0, st>>>(a, stat);
            }
            if (a.absmax_out || !strip)
                k_finalize<<<(unsigned)ceil_div(ns, 256), 256, 0, st>>>(a, stat, ns);
            else
                a.stat_in = stat;
        }
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (a.absmax_out) return cudaGetLastError();
    if (rowcodes) {
        if constexpr (!std::is_same<T, float>::value) {
            if (mode == 0)
                return a.code4 ? launch_qrow_bulk_g<T, true, false, true, 0>(a, buf_stride, st)
                               : launch_qrow_bulk_g<T, true, false, false, 0>(a, buf_stride, st);
            if (mode == 1)
                return a.code4 ? launch_qrow_bulk_g<T, false, false, true, 0>(a, buf_stride, st)
                               : launch_qrow_bulk_g<T, false, false, false, 0>(a, buf_stride, st);
            return a.code4 ? launch_qrow_bulk_g<T, true, true, true, 0>(a, buf_stride, st)
                           : launch_qrow_bulk_g<T, true, true, false, 0>(a, buf_stride, st);
        }
    }
    if (strip) {
        const QuantStripFn<T> kq = quant_strip_fn<T>(mode, pc, smoothed);
        kq<<<strip_grid(a.cols / 8, a.rows, kStripThreads, blocks_per_sm((const void*)kq, kStripThreads, 0)),
             kStripThreads, 0, st>>>(a);
    } else {
        k_quant_generic<T><<<gblocks, 256, 0, st>>>(a);
    }
    return cudaGetLastError();
}

cudaError_t run_quantize(const void* x, int xt, int64_t rows, int64_t cols, int64_t ld, const float* smooth,
                         const qlin_qparams* p, void* q, void* s, int32_t* z, void* ws, cudaStream_t st) {
    QuantArgs a;
    a.x = x;
    a.rows = rows;
    a.cols = cols;
    a.ld = ld;
    a.smooth = smooth;
    a.smooth_mode = p->smooth_mode;
    a.qmin = p->qmin;
    a.qmax = p->qmax;
    a.sym = p->symmetric;
    a.gran = p->gran;
    a.group = p->group;
    a.scale_f16 = (p->scale_dtype == QLIN_F16);
    a.static_scale = p->static_scale;
    a.code4 = (p->code == QLIN_S4 || p->code == QLIN_U4);
    a.q = q;
    a.s = s;
    a.z = z;
    a.absmax_out = nullptr;
    switch (xt) {
    case QLIN_BF16: return run_quantize_t<__nv_bfloat16>(a, xt, p, ws, st);
    case QLIN_F16: return run_quantize_t<__half>(a, xt, p, ws, st);
    default: return run_quantize_t<float>(a, xt, p, ws, st);
    }
}

cudaError_t run_absmax(const void* x, int xt, int64_t rows, int64_t cols, int64_t ld, int gran, int group,
                       float* out, void* ws, cudaStream_t st) {
    qlin_qparams p{};
    p.code = QLIN_S8;
    p.qmin = -127;
    p.qmax = 127;
    p.symmetric = 1;
    p.gran = (qlin_gran)gran;
    p.group = group;
    p.scale_dtype = QLIN_F32;
    QuantArgs a{};
    a.x = x;
    a.rows = rows;
    a.cols = cols;
    a.ld = ld;
    a.smooth_mode = QLIN_SMOOTH_NONE;
    a.qmin = -127;
    a.qmax = 127;
    a.sym = 1;
    a.gran = gran;
    a.group = group;
    a.absmax_out = out;
    a.q = nullptr;
    switch (xt) {
    case QLIN_BF16: return run_quantize_t<__nv_bfloat16>(a, xt, &p, ws, st);
    case QLIN_F16: return run_quantize_t<__half>(a, xt, &p, ws, st);
    default: return run_quantize_t<float>(a, xt, &p, ws, st);
    }
}

cudaError_t run_dequantize(const void* q, const void* s, const int32_t* z, const qlin_qparams* p, int64_t rows,
                           int64_t cols, void* y, int yt, cudaStream_t st) {
    DequantArgs d;
    d.q = q;
    d.s = s;
    d.z = z;
    d.rows = rows;
    d.cols = cols;
    d.gran = p->gran;
    d.group = p->group;
    d.scale_f16 = (p->scale_dtype == QLIN_F16);
    d.code4 = (p->code == QLIN_S4 || p->code == QLIN_U4);
    d.code_signed = (p->code == QLIN_S8 || p->code == QLIN_S4);
    d.y = y;
    d.yt = yt;
    int blocks = num_sms() * 8;
    int ys = (yt == QLIN_F32) ? 4 : 2;
    bool vec = (cols % 8 == 0) && (p->gran != QLIN_PER_GROUP || p->group % 8 == 0) &&
               ((uintptr_t)q % (d.code4 ? 4 : 8) == 0) && ((uintptr_t)y % (8 * ys) == 0);
    const bool seg16 = (cols % 16 == 0) && (p->gran != QLIN_PER_COL) &&
                        (p->gran != QLIN_PER_GROUP || p->group % 16 == 0) &&
                        ((uintptr_t)q % (d.code4 ? 8 : 16) == 0) && ((uintptr_t)y % 16 == 0);
    const int64_t nch16 = cols / 16, seg = (int64_t)kDqUnroll * 256;
    if (seg16 && nch16 > 0 && nch16 <= seg && seg % nch16 == 0)
        k_dequant_short<<<blocks, 256, 0, st>>>(d);
    else if (seg16)
        k_dequant_rows<<<blocks, 256, 0, st>>>(d);
    else if (vec)
        k_dequant_vec<<<blocks, 256, 0, st>>>(d);
    else
        k_dequant_generic<<<blocks, 256, 0, st>>>(d);
    return cudaGetLastError();
}

cudaError_t run_smooth_factors(const float* xmax, const float* wmax, int64_t K, float alpha, float* s,
                               cudaStream_t st) {
    k_smooth_factors<<<(unsigned)ceil_div(K, 256), 256, 0, st>>>(xmax, wmax, K, alpha, s);
    return cudaGetLastError();
}

int64_t percentile_rank(int64_t n, double p) {
    double k = ceil((double)n * p / 100.0);
    if (k < 1.0) k = 1.0;
    if (k > (double)n) k = (double)n;
    return (int64_t)k;
}

}  // namespace qlin
