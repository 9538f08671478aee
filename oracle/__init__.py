"""CPU oracle for the quantized linear layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps ``liborc.so`` (plain C, see
``qlin_oracle.c``) with numpy marshalling and shares nothing with the CUDA
library.
"""
import ctypes as C

import numpy as np

from . import build as _build

PER_TENSOR, PER_ROW, PER_COL, PER_GROUP = 0, 1, 2, 3
SMOOTH_NONE, SMOOTH_DIVIDE, SMOOTH_MULTIPLY = 0, 1, 2

_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(_build.build())
        _declare(_lib)
    return _lib


_f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(np.int64, flags="C_CONTIGUOUS")
_i8p = np.ctypeslib.ndpointer(np.int8, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")
_i64 = C.c_int64


def _declare(L):
    L.orc_bf16_to_f32.argtypes = [C.c_uint16]
    L.orc_bf16_to_f32.restype = C.c_float
    L.orc_f32_to_bf16.argtypes = [C.c_float]
    L.orc_f32_to_bf16.restype = C.c_uint16
    L.orc_round_bf16.argtypes = [C.c_float]
    L.orc_round_bf16.restype = C.c_float
    L.orc_round_f16.argtypes = [C.c_float]
    L.orc_round_f16.restype = C.c_float
    L.orc_round_bf16_n.argtypes = [_f32p, _i64, _f32p]
    L.orc_round_bf16_n.restype = None
    L.orc_round_f16_n.argtypes = [_f32p, _i64, _f32p]
    L.orc_round_f16_n.restype = None
    L.orc_num_scopes.argtypes = [C.c_int, _i64, _i64, _i64]
    L.orc_num_scopes.restype = _i64
    L.orc_percentile_rank.argtypes = [_i64, C.c_double]
    L.orc_percentile_rank.restype = _i64
    L.orc_quantize.argtypes = [_f32p, _i64, _i64, C.c_void_p, C.c_int,
                               C.c_int, C.c_int, C.c_int, C.c_int, _i64,
                               C.c_double, C.c_int, C.c_int, _i32p, _f32p, _i32p]
    L.orc_quantize.restype = C.c_int
    L.orc_dequantize.argtypes = [_i32p, _f32p, C.c_void_p, _i64, _i64, C.c_int, _i64, _f32p]
    L.orc_dequantize.restype = C.c_int
    L.orc_absmax.argtypes = [_f32p, _i64, _i64, C.c_int, _i64, _f32p]
    L.orc_absmax.restype = C.c_int
    L.orc_smooth_factors.argtypes = [_f32p, _f32p, _i64, C.c_float, _f32p]
    L.orc_smooth_factors.restype = None
    L.orc_pack_nibbles.argtypes = [_i32p, _i64, _u8p]
    L.orc_pack_nibbles.restype = None
    L.orc_unpack_nibbles.argtypes = [_u8p, _i64, C.c_int, _i32p]
    L.orc_unpack_nibbles.restype = None
    L.orc_w8a8_acc.argtypes = [_i8p, _i8p, _i64, _i64, _i64, _i64p]
    L.orc_w8a8_acc.restype = None
    L.orc_w8a8_out.argtypes = [_i64p, _f32p, _f32p, _i64, _i64, _f64p]
    L.orc_w8a8_out.restype = None
    L.orc_w4_dequant.argtypes = [_i32p, _f32p, C.c_void_p, _i64, _i64, _i64, _f32p]
    L.orc_w4_dequant.restype = None
    L.orc_matmul_f64.argtypes = [_f32p, _f32p, _i64, _i64, _i64, _f64p]
    L.orc_matmul_f64.restype = None
    L.orc_w4a8_acc.argtypes = [_i8p, _i32p, C.c_void_p, _i64, _i64, _i64, _i64, _i64p]
    L.orc_w4a8_acc.restype = None
    L.orc_w4a8_out.argtypes = [_i64p, _f32p, _f32p, _i64, _i64, _i64, _f64p]
    L.orc_w4a8_out.restype = None
    L.orc_channel_absmax_update.argtypes = [_f32p, _i64, _i64, _f32p]
    L.orc_channel_absmax_update.restype = None
    L.orc_fold_layernorm.argtypes = [_f32p, C.c_void_p, _f32p, _i64, _f32p, C.c_void_p]
    L.orc_fold_layernorm.restype = None
    L.orc_quant_error.argtypes = [_f32p, _i64, _i64, C.c_void_p, C.c_int, _i32p, _f32p, C.c_void_p, C.c_int,
                                  _i64, _f64p]
    L.orc_quant_error.restype = None
    L.orc_llmint8_outlier_cols.argtypes = [_f32p, _i64, _i64, C.c_float, _i32p]
    L.orc_llmint8_outlier_cols.restype = _i64
    L.orc_llmint8_out.argtypes = [_f32p, _i8p, _f32p, _f32p, _i64p, _i32p, _i64, _i64, _i64, _i64, _f64p]
    L.orc_llmint8_out.restype = None
    L.orc_set_threads.argtypes = [C.c_int]
    L.orc_set_threads.restype = C.c_int


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


# ---------------------------------------------------------------- formats
def bf16_bits_to_f32(bits):
    """Widen bf16 bit patterns (uint16 array) to binary32 values."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def round_bf16(x):
    """Round binary32 values to bf16 (nearest-even) using the oracle's routine."""
    x = _f32(x)
    out = np.zeros_like(x)
    lib().orc_round_bf16_n(x, x.size, out)
    return out


def f32_to_bf16_bits(x):
    L = lib()
    x = _f32(x)
    return np.array([L.orc_f32_to_bf16(float(v)) for v in x.ravel()],
                    dtype=np.uint16).reshape(x.shape)


def round_f16(x):
    x = _f32(x)
    out = np.zeros_like(x)
    lib().orc_round_f16_n(x, x.size, out)
    return out


def num_scopes(gran, rows, cols, group=0):
    return int(lib().orc_num_scopes(gran, rows, cols, group))


def percentile_rank(n, p):
    return int(lib().orc_percentile_rank(n, p))


def set_threads(n):
    return int(lib().orc_set_threads(n))


# ---------------------------------------------------------------- quantizer
def quantize(x, qmin, qmax, symmetric, gran, group=0, smooth=None,
             smooth_mode=SMOOTH_NONE, percentile=0.0, scale_f16=False,
             static_s=None, static_z=None):
    """Quantize a 2-D binary32 array; returns (q int32, s float32, z int32)."""
    x = _f32(x)
    if x.ndim == 1:
        x = x.reshape(1, -1)
    rows, cols = x.shape
    nsc = num_scopes(gran, rows, cols, group)
    if nsc < 0:
        raise ValueError("bad granularity/group")
    q = np.zeros((rows, cols), dtype=np.int32)
    if static_s is not None:
        s = _f32(static_s).copy()
        z = np.ascontiguousarray(static_z if static_z is not None else np.zeros(nsc), dtype=np.int32).copy()
    else:
        s = np.zeros(nsc, dtype=np.float32)
        z = np.zeros(nsc, dtype=np.int32)
    sm = None if smooth is None else _f32(smooth)
    rc = lib().orc_quantize(x, rows, cols, _ptr(sm), smooth_mode, int(qmin), int(qmax),
                            int(bool(symmetric)), gran, int(group), float(percentile),
                            int(bool(scale_f16)), int(static_s is not None), q, s, z)
    if rc != 0:
        raise ValueError("orc_quantize rejected the arguments (rc=%d)" % rc)
    return q, s, z


def dequantize(q, s, z, gran, group=0):
    q = np.ascontiguousarray(q, dtype=np.int32)
    if q.ndim == 1:
        q = q.reshape(1, -1)
    rows, cols = q.shape
    y = np.zeros((rows, cols), dtype=np.float32)
    zz = None if z is None else np.ascontiguousarray(z, dtype=np.int32)
    rc = lib().orc_dequantize(q, _f32(s), _ptr(zz), rows, cols, gran, int(group), y)
    if rc != 0:
        raise ValueError("orc_dequantize rejected the arguments")
    return y


def absmax(x, gran, group=0):
    x = _f32(x)
    rows, cols = x.shape
    out = np.zeros(num_scopes(gran, rows, cols, group), dtype=np.float32)
    if lib().orc_absmax(x, rows, cols, gran, int(group), out) != 0:
        raise ValueError("orc_absmax rejected the arguments")
    return out


def smooth_factors(xmax, wmax, alpha):
    xmax, wmax = _f32(xmax), _f32(wmax)
    s = np.zeros_like(xmax)
    lib().orc_smooth_factors(xmax, wmax, xmax.size, float(alpha), s)
    return s


def pack_nibbles(q):
    q = np.ascontiguousarray(q, dtype=np.int32).ravel()
    out = np.zeros((q.size + 1) // 2, dtype=np.uint8)
    lib().orc_pack_nibbles(q, q.size, out)
    return out


def unpack_nibbles(b, n, signed):
    b = np.ascontiguousarray(b, dtype=np.uint8).ravel()
    q = np.zeros(n, dtype=np.int32)
    lib().orc_unpack_nibbles(b, n, int(bool(signed)), q)
    return q


# ---------------------------------------------------------------- GEMMs
def w8a8_acc(qx, qw):
    qx = np.ascontiguousarray(qx, dtype=np.int8)
    qw = np.ascontiguousarray(qw, dtype=np.int8)
    M, K = qx.shape
    N = qw.shape[0]
    acc = np.zeros((M, N), dtype=np.int64)
    lib().orc_w8a8_acc(qx, qw, M, N, K, acc)
    return acc


def w8a8_out(acc, sx, sw):
    acc = np.ascontiguousarray(acc, dtype=np.int64)
    M, N = acc.shape
    y = np.zeros((M, N), dtype=np.float64)
    lib().orc_w8a8_out(acc, _f32(sx), _f32(sw), M, N, y)
    return y


def w4_dequant(q, s, z, g):
    q = np.ascontiguousarray(q, dtype=np.int32)
    N, K = q.shape
    w = np.zeros((N, K), dtype=np.float32)
    zz = None if z is None else np.ascontiguousarray(z, dtype=np.int32)
    lib().orc_w4_dequant(q, _f32(s), _ptr(zz), N, K, int(g), w)
    return w


def matmul_f64(x, w):
    x, w = _f32(x), _f32(w)
    M, K = x.shape
    N = w.shape[0]
    y = np.zeros((M, N), dtype=np.float64)
    lib().orc_matmul_f64(x, w, M, N, K, y)
    return y


def w4a8_acc(qx, q, z, g):
    """Exact per-group integer sums acc[g][m][n] = sum_{k in g} qx[m,k] (q[n,k] - z[n,g])."""
    qx = np.ascontiguousarray(qx, dtype=np.int8)
    q = np.ascontiguousarray(q, dtype=np.int32)
    M, K = qx.shape
    N = q.shape[0]
    acc = np.zeros((K // g, M, N), dtype=np.int64)
    zz = None if z is None else np.ascontiguousarray(z, dtype=np.int32)
    lib().orc_w4a8_acc(qx, q, _ptr(zz), M, N, K, int(g), acc)
    return acc


def w4a8_out(acc, sx, s):
    """y[m,n] = sx[m] * sum_g s[n,g] * acc[g][m][n] in binary64."""
    acc = np.ascontiguousarray(acc, dtype=np.int64)
    ng, M, N = acc.shape
    y = np.zeros((M, N), dtype=np.float64)
    lib().orc_w4a8_out(acc, _f32(sx), _f32(s), M, N, ng, y)
    return y


# ---------------------------------------------------------------- SmoothQuant calibration
def channel_absmax_update(x, running):
    """running[j] = max(running[j], max_i |x[i, j]|), in place; returns running."""
    x = _f32(x)
    assert running.dtype == np.float32 and running.flags["C_CONTIGUOUS"]
    lib().orc_channel_absmax_update(x, x.shape[0], x.shape[1], running)
    return running


def fold_layernorm(gamma, beta, s):
    """(gamma / s, beta / s) in binary32 (beta may be None)."""
    gamma, s = _f32(gamma), _f32(s)
    g_out = np.zeros_like(gamma)
    b = None if beta is None else _f32(beta)
    b_out = None if beta is None else np.zeros_like(gamma)
    lib().orc_fold_layernorm(gamma, _ptr(b), s, gamma.size, g_out, _ptr(b_out))
    return g_out, b_out


def quant_error(x, q, s, z, gran, group=0, smooth=None, smooth_mode=SMOOTH_NONE):
    """(sum (x' - x^)^2, sum x'^2, max |x' - x^|) in binary64."""
    x = _f32(x)
    rows, cols = x.shape
    q = np.ascontiguousarray(q, dtype=np.int32)
    out = np.zeros(3, dtype=np.float64)
    sm = None if smooth is None else _f32(smooth)
    zz = None if z is None else np.ascontiguousarray(z, dtype=np.int32)
    lib().orc_quant_error(x, rows, cols, _ptr(sm), smooth_mode, q, _f32(s), _ptr(zz), gran, int(group), out)
    return out


# ---------------------------------------------------------------- LLM.int8()
def llmint8_outlier_cols(x, threshold):
    x = _f32(x)
    cols = np.zeros(x.shape[1], dtype=np.int32)
    n = lib().orc_llmint8_outlier_cols(x, x.shape[0], x.shape[1], float(threshold), cols)
    return cols[:n].copy()


def llmint8_out(x, qw, sw, sx, acc, cols):
    x = _f32(x)
    M, K = x.shape
    qw = np.ascontiguousarray(qw, dtype=np.int8)
    N = qw.shape[0]
    y = np.zeros((M, N), dtype=np.float64)
    cols = np.ascontiguousarray(cols, dtype=np.int32)
    lib().orc_llmint8_out(x, qw, _f32(sw), _f32(sx), np.ascontiguousarray(acc, dtype=np.int64), cols, cols.size,
                          M, N, K, y)
    return y


def llmint8(x, qw, sw, threshold):
    """The whole decomposition: outlier channels, per-token INT8 codes of the
    normal channels (outlier channels zeroed, so they neither widen the scale
    nor add to the INT8 sums), the INT8 sums, and y in binary64."""
    x = _f32(x)
    cols = llmint8_outlier_cols(x, threshold)
    xn = x.copy()
    xn[:, cols] = 0.0
    qx, sx, _ = quantize(xn, -127, 127, True, PER_ROW)
    acc = w8a8_acc(qx.astype(np.int8), qw)
    return cols, qx, sx, acc, llmint8_out(x, qw, sw, sx, acc, cols)


# ---------------------------------------------------------------- KV-cache quantization
def kv_cache_reference(k, v, group, residual, head_dim, bits):
    """KV-cache quantization in token groups outside a recent window ([CH11]
    11.6.3-11.6.5: K per channel, V per token, the most recent tokens kept in
    16-bit; KIVI's grouped, on-demand quantization).

    k, v: binary32 [T x C] (the 16-bit values the cache received).  The first
    Tq = group * floor(max(T - residual, 0) / group) tokens are quantized in
    groups of `group` tokens with asymmetric codes [0, 2^bits - 1]: K with one
    scale / zero point per (group, channel) (min-max over the group's tokens),
    V with one per (token, head) (min-max over head_dim channels).  Returns a
    dict with the codes, scales and zero points of the quantized part, Tq,
    and the cache as read back (binary32): dequantized s * (q - z) for
    t < Tq, the original values for t >= Tq."""
    k, v = _f32(k), _f32(v)
    T, C = k.shape
    qmax = (1 << bits) - 1
    tq = group * (max(T - residual, 0) // group)
    ng = tq // group
    kq = np.zeros((tq, C), np.int32)
    ks = np.zeros((ng, C), np.float32)
    kz = np.zeros((ng, C), np.int32)
    for gi in range(ng):
        blk = k[gi * group:(gi + 1) * group]
        q, s, z = quantize(blk, 0, qmax, False, PER_COL)
        kq[gi * group:(gi + 1) * group], ks[gi], kz[gi] = q, s, z
    vq, vs, vz = (quantize(v[:tq], 0, qmax, False, PER_GROUP, head_dim) if tq
                  else (np.zeros((0, C), np.int32), np.zeros(0, np.float32), np.zeros(0, np.int32)))
    khat, vhat = k.copy(), v.copy()
    if tq:
        for gi in range(ng):
            khat[gi * group:(gi + 1) * group] = dequantize(kq[gi * group:(gi + 1) * group], ks[gi], kz[gi], PER_COL)
        vhat[:tq] = dequantize(vq, vs, vz, PER_GROUP, head_dim)
    return dict(tq=tq, k_codes=kq, k_scale=ks, k_zero=kz, v_codes=vq, v_scale=vs.reshape(tq, C // head_dim),
                v_zero=vz.reshape(tq, C // head_dim), k_hat=khat, v_hat=vhat)
