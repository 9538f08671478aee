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
