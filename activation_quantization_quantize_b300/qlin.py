"""Thin ctypes binding of libqlin.so (include/qlin.h).

Every entry point keeps its C name; arguments are torch tensors (device
memory) or plain numbers, converted to pointers and sizes here.  All
arithmetic runs in the CUDA library: there is no CPU fallback, and a missing
library raises ``QlinError`` on first use.
"""
import ctypes as C
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libqlin.so")

# qlin_status
QLIN_OK, QLIN_ERR_ARG, QLIN_ERR_UNSUPPORTED, QLIN_ERR_CUDA = 0, -1, -2, -3
QLIN_ERR_TIMEOUT, QLIN_ERR_WORKSPACE, QLIN_ERR_LAYOUT = -4, -5, -6
# qlin_gran
QLIN_PER_TENSOR, QLIN_PER_ROW, QLIN_PER_COL, QLIN_PER_GROUP = 0, 1, 2, 3
# qlin_dtype
QLIN_F32, QLIN_BF16, QLIN_F16, QLIN_S8, QLIN_U8, QLIN_S4, QLIN_U4, QLIN_S32 = range(8)
# qlin_smooth
QLIN_SMOOTH_NONE, QLIN_SMOOTH_DIVIDE, QLIN_SMOOTH_MULTIPLY = 0, 1, 2
# operations
QLIN_OP_QUANTIZE, QLIN_OP_ABSMAX, QLIN_OP_GEMM_W8A8, QLIN_OP_GEMM_W4A16, QLIN_OP_GEMM_W4A8 = 0, 1, 2, 3, 4
QLIN_OP_QUANT_ERROR = 5
QLIN_W4_MAGIC, QLIN_W4_VERSION = 0x34574C51, 1


class QlinError(RuntimeError):
    def __init__(self, fn, status, text):
        super().__init__("%s failed: %s (%d)" % (fn, text, status))
        self.status = status


class qlin_qparams(C.Structure):
    _fields_ = [("code", C.c_int), ("qmin", C.c_int), ("qmax", C.c_int), ("symmetric", C.c_int),
                ("gran", C.c_int), ("group", C.c_int), ("clip_percentile", C.c_double),
                ("scale_dtype", C.c_int), ("static_scale", C.c_int), ("smooth_mode", C.c_int)]


class qlin_w4_header(C.Structure):
    _fields_ = [("magic", C.c_uint32), ("version", C.c_uint32), ("N", C.c_int64), ("K", C.c_int64),
                ("group", C.c_int32), ("asym", C.c_int32), ("codes_off", C.c_uint64),
                ("scales_off", C.c_uint64), ("zeros_off", C.c_uint64), ("total_bytes", C.c_uint64)]


class qlin_kv_cache(C.Structure):
    _fields_ = [("capacity", C.c_int64), ("channels", C.c_int32), ("head_dim", C.c_int32), ("group", C.c_int32),
                ("residual", C.c_int32), ("bits", C.c_int32), ("reserved", C.c_int32), ("length", C.c_int64),
                ("quantized", C.c_int64), ("k_codes", C.c_void_p), ("v_codes", C.c_void_p),
                ("k_scale", C.c_void_p), ("k_zero", C.c_void_p), ("v_scale", C.c_void_p), ("v_zero", C.c_void_p),
                ("k_recent", C.c_void_p), ("v_recent", C.c_void_p)]


_lib = None
_P = C.c_void_p
_I64 = C.c_int64


def load():
    """Load libqlin.so (built in-tree by build.py); raise if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise QlinError("load", QLIN_ERR_CUDA, "libqlin.so is not built (run build.py)")
        L = C.CDLL(LIB_PATH)
        L.qlin_version.restype = C.c_int
        L.qlin_status_string.argtypes = [C.c_int]
        L.qlin_status_string.restype = C.c_char_p
        L.qlin_workspace_size.argtypes = [C.c_int, _I64, _I64, _I64, C.POINTER(qlin_qparams)]
        L.qlin_workspace_size.restype = C.c_size_t
        L.qlin_quantize.argtypes = [_P, C.c_int, _I64, _I64, _I64, _P, C.POINTER(qlin_qparams),
                                    _P, _P, _P, _P, C.c_size_t, _P]
        L.qlin_dequantize.argtypes = [_P, _P, _P, C.POINTER(qlin_qparams), _I64, _I64, _P, C.c_int, _P]
        L.qlin_absmax.argtypes = [_P, C.c_int, _I64, _I64, _I64, C.c_int, C.c_int, _P, _P, C.c_size_t, _P]
        L.qlin_smooth_factors.argtypes = [_P, _P, _I64, C.c_float, _P, _P]
        L.qlin_pack_w4_size.argtypes = [_I64, _I64, C.c_int, C.c_int]
        L.qlin_pack_w4_size.restype = C.c_size_t
        L.qlin_pack_w4.argtypes = [_P, _P, _P, _I64, _I64, C.c_int, _P, C.c_size_t,
                                   C.POINTER(qlin_w4_header), _P]
        L.qlin_gemm_w8a8.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _P, C.c_int, _P, _P, C.c_size_t, _P]
        L.qlin_gemm_w4a16.argtypes = [_P, _P, C.POINTER(qlin_w4_header), _I64, _P, _P, C.c_size_t, _P]
        L.qlin_gemm_w4a8.argtypes = [_P, _P, _P, C.POINTER(qlin_w4_header), _I64, _P, C.c_int, _P, _P, C.c_size_t, _P]
        L.qlin_gemm_w4a8.restype = C.c_int
        L.qlin_absmax_update.argtypes = [_P, C.c_int, _I64, _I64, _I64, _P, _P]
        L.qlin_fold_layernorm.argtypes = [_P, _P, _P, _I64, _P, _P, _P]
        L.qlin_quant_error.argtypes = [_P, C.c_int, _I64, _I64, _I64, _P, C.POINTER(qlin_qparams), _P, _P, _P, _P,
                                       _P, C.c_size_t, _P]
        for name in ("qlin_absmax_update", "qlin_fold_layernorm", "qlin_quant_error"):
            getattr(L, name).restype = C.c_int
        L.qlin_llmint8_workspace_size.argtypes = [_I64, _I64, _I64, _I64]
        L.qlin_llmint8_workspace_size.restype = C.c_size_t
        L.qlin_gemm_llmint8.argtypes = [_P, C.c_int, _I64, _I64, _I64, _P, _P, _I64, C.c_float, _I64, _P, C.c_int,
                                        _P, _P, C.c_size_t, _P]
        L.qlin_gemm_llmint8.restype = C.c_int
        L.qlin_kv_cache_bytes.argtypes = [_I64, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int]
        L.qlin_kv_cache_bytes.restype = C.c_size_t
        L.qlin_kv_cache_init.argtypes = [C.POINTER(qlin_kv_cache), _P, C.c_size_t, _I64, C.c_int, C.c_int, C.c_int,
                                         C.c_int, C.c_int]
        L.qlin_kv_append.argtypes = [C.POINTER(qlin_kv_cache), _P, _P, _I64, _P]
        L.qlin_kv_read.argtypes = [C.POINTER(qlin_kv_cache), _P, _P, _P]
        for name in ("qlin_kv_cache_init", "qlin_kv_append", "qlin_kv_read"):
            getattr(L, name).restype = C.c_int
        L.qlin_device_error.argtypes = [_P]
        L.qlin_debug_stall_producers.argtypes = [C.c_int, C.c_longlong]
        L.qlin_debug_stall_producers.restype = C.c_int
        L.qlin_quantize_noalloc.argtypes = [_P, C.c_int, _I64, _I64, _I64, _P, C.POINTER(qlin_qparams),
                                            _P, _P, _P, _P]
        L.qlin_quantize_noalloc.restype = C.c_int
        for name in ("qlin_quantize", "qlin_dequantize", "qlin_absmax", "qlin_smooth_factors",
                     "qlin_pack_w4", "qlin_gemm_w8a8", "qlin_gemm_w4a16", "qlin_device_error"):
            getattr(L, name).restype = C.c_int
        _lib = L
    return _lib


def _check(fn, rc):
    if rc != QLIN_OK:
        raise QlinError(fn, rc, load().qlin_status_string(rc).decode())
    return rc


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


_TORCH_DT = {torch.float32: QLIN_F32, torch.bfloat16: QLIN_BF16, torch.float16: QLIN_F16}


def dtype_code(t):
    return _TORCH_DT[t.dtype]


# ----------------------------------------------------------------------------- C names
def qlin_version():
    return load().qlin_version()


def qlin_status_string(status):
    return load().qlin_status_string(status).decode()


def qlin_workspace_size(op, M, N, K, p=None):
    return load().qlin_workspace_size(op, M, N, K, C.byref(p) if p is not None else None)


def qlin_quantize(x, xt, rows, cols, ld, smooth, p, q, s, z, ws, ws_bytes, stream=None):
    return _check("qlin_quantize", load().qlin_quantize(
        _ptr(x), xt, rows, cols, ld, _ptr(smooth), C.byref(p), _ptr(q), _ptr(s), _ptr(z), _ptr(ws),
        ws_bytes, _stream(stream)))


def qlin_dequantize(q, s, z, p, rows, cols, y, yt, stream=None):
    return _check("qlin_dequantize", load().qlin_dequantize(
        _ptr(q), _ptr(s), _ptr(z), C.byref(p), rows, cols, _ptr(y), yt, _stream(stream)))


def qlin_absmax(x, xt, rows, cols, ld, gran, group, out, ws, ws_bytes, stream=None):
    return _check("qlin_absmax", load().qlin_absmax(
        _ptr(x), xt, rows, cols, ld, gran, group, _ptr(out), _ptr(ws), ws_bytes, _stream(stream)))


def qlin_smooth_factors(xmax, wmax, K, alpha, s, stream=None):
    return _check("qlin_smooth_factors", load().qlin_smooth_factors(
        _ptr(xmax), _ptr(wmax), K, alpha, _ptr(s), _stream(stream)))


def qlin_pack_w4_size(N, K, group, asym):
    return load().qlin_pack_w4_size(N, K, group, 1 if asym else 0)


def qlin_pack_w4(q, s_f16, z, N, K, group, packed, packed_cap, hdr, stream=None):
    return _check("qlin_pack_w4", load().qlin_pack_w4(
        _ptr(q), _ptr(s_f16), _ptr(z), N, K, group, _ptr(packed), packed_cap,
        C.byref(hdr) if hdr is not None else None, _stream(stream)))


def qlin_gemm_w8a8(qx, sx, qw, sw, M, N, K, y, yt, acc_out, ws, ws_bytes, stream=None):
    return _check("qlin_gemm_w8a8", load().qlin_gemm_w8a8(
        _ptr(qx), _ptr(sx), _ptr(qw), _ptr(sw), M, N, K, _ptr(y), yt, _ptr(acc_out), _ptr(ws), ws_bytes,
        _stream(stream)))


def qlin_gemm_w4a16(x, packed, hdr, M, y, ws, ws_bytes, stream=None):
    return _check("qlin_gemm_w4a16", load().qlin_gemm_w4a16(
        _ptr(x), _ptr(packed), C.byref(hdr), M, _ptr(y), _ptr(ws), ws_bytes, _stream(stream)))


def qlin_gemm_w4a8(qx, sx, packed, hdr, M, y, yt, acc_out, ws, ws_bytes, stream=None):
    return _check("qlin_gemm_w4a8", load().qlin_gemm_w4a8(
        _ptr(qx), _ptr(sx), _ptr(packed), C.byref(hdr), M, _ptr(y), yt, _ptr(acc_out), _ptr(ws), ws_bytes,
        _stream(stream)))


def qlin_quantize_noalloc(x, xt, rows, cols, ld, smooth, p, q, s, z, stream=None):
    return _check("qlin_quantize_noalloc", load().qlin_quantize_noalloc(
        _ptr(x), xt, rows, cols, ld, _ptr(smooth), C.byref(p), _ptr(q), _ptr(s), _ptr(z), _stream(stream)))


def qlin_device_error(stream=None):
    return load().qlin_device_error(_stream(stream))


def qlin_debug_stall_producers(enable, wait_limit_cycles=0):
    return _check("qlin_debug_stall_producers", load().qlin_debug_stall_producers(1 if enable else 0,
                                                                                 int(wait_limit_cycles)))


# ----------------------------------------------------------------------------- conveniences
CODE_RANGES = {"s8": (QLIN_S8, -127, 127), "u8": (QLIN_U8, 0, 255),
               "s4": (QLIN_S4, -7, 7), "u4": (QLIN_U4, 0, 15)}
GRANS = {"tensor": QLIN_PER_TENSOR, "row": QLIN_PER_ROW, "col": QLIN_PER_COL, "group": QLIN_PER_GROUP}


def make_params(code="s8", gran="row", group=0, symmetric=None, qmin=None, qmax=None, percentile=0.0,
                scale_f16=False, static_scale=False, smooth_mode=QLIN_SMOOTH_NONE):
    ct, lo, hi = CODE_RANGES[code]
    if symmetric is None:
        symmetric = code in ("s8", "s4")
    p = qlin_qparams()
    p.code = ct
    p.qmin = lo if qmin is None else qmin
    p.qmax = hi if qmax is None else qmax
    p.symmetric = 1 if symmetric else 0
    p.gran = GRANS[gran] if isinstance(gran, str) else gran
    p.group = group
    p.clip_percentile = float(percentile)
    p.scale_dtype = QLIN_F16 if scale_f16 else QLIN_F32
    p.static_scale = 1 if static_scale else 0
    p.smooth_mode = smooth_mode
    return p


def num_scopes(p, rows, cols):
    return {QLIN_PER_TENSOR: 1, QLIN_PER_ROW: rows, QLIN_PER_COL: cols,
            QLIN_PER_GROUP: rows * (cols // max(p.group, 1))}[p.gran]


def workspace(op, M, N, K, p=None, device="cuda"):
    n = qlin_workspace_size(op, M, N, K, p)
    return (torch.empty(n, dtype=torch.uint8, device=device) if n else None), n


def quantize(x, p, smooth=None, s=None, z=None, ws=None, stream=None):
    """Quantize a 2-D device tensor; returns (codes, scales, zero points)."""
    rows, cols = x.shape
    ld = x.stride(0)
    assert x.stride(1) == 1
    code4 = p.code in (QLIN_S4, QLIN_U4)
    cdt = torch.int8 if p.code in (QLIN_S8, QLIN_S4) else torch.uint8
    q = torch.empty((rows, cols // 2 if code4 else cols), dtype=cdt, device=x.device)
    ns = num_scopes(p, rows, cols)
    if s is None:
        s = torch.empty(ns, dtype=torch.float16 if p.scale_dtype == QLIN_F16 else torch.float32, device=x.device)
    if z is None and not p.symmetric:
        z = torch.empty(ns, dtype=torch.int32, device=x.device)
    nbytes = qlin_workspace_size(QLIN_OP_QUANTIZE, rows, cols, 0, p)
    if ws is None and nbytes:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=x.device)
    qlin_quantize(x, dtype_code(x), rows, cols, ld, smooth, p, q, s, z, ws, nbytes, stream)
    return q, s, z


def dequantize(q, s, z, p, rows, cols, out_dtype=torch.bfloat16, stream=None):
    y = torch.empty((rows, cols), dtype=out_dtype, device=q.device)
    qlin_dequantize(q, s, z, p, rows, cols, y, _TORCH_DT[out_dtype], stream)
    return y


def absmax(x, gran, group=0, stream=None):
    rows, cols = x.shape
    p = make_params("s8", gran, group)
    ns = num_scopes(p, rows, cols)
    out = torch.empty(ns, dtype=torch.float32, device=x.device)
    nbytes = qlin_workspace_size(QLIN_OP_ABSMAX, rows, cols, 0, p)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=x.device) if nbytes else None
    qlin_absmax(x, dtype_code(x), rows, cols, x.stride(0), p.gran, group, out, ws, nbytes, stream)
    return out


def smooth_factors(xmax, wmax, alpha, stream=None):
    s = torch.empty_like(xmax)
    qlin_smooth_factors(xmax, wmax, xmax.numel(), alpha, s, stream)
    return s


def pack_w4(q, s_f16, z, N, K, group, stream=None):
    """Pack canonical INT4 codes; returns (packed uint8 tensor, header)."""
    n = qlin_pack_w4_size(N, K, group, z is not None)
    if n == 0:
        raise QlinError("qlin_pack_w4_size", QLIN_ERR_ARG, "invalid sizes")
    packed = torch.empty(n, dtype=torch.uint8, device=q.device)
    hdr = qlin_w4_header()
    qlin_pack_w4(q, s_f16, z, N, K, group, packed, n, hdr, stream)
    return packed, hdr


def gemm_w8a8(qx, sx, qw, sw, out_dtype=torch.bfloat16, acc_out=None, stream=None):
    M, K = qx.shape
    N = qw.shape[0]
    y = torch.empty((M, N), dtype=out_dtype, device=qx.device)
    nbytes = qlin_workspace_size(QLIN_OP_GEMM_W8A8, M, N, K)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=qx.device) if nbytes else None
    qlin_gemm_w8a8(qx, sx, qw, sw, M, N, K, y, _TORCH_DT[out_dtype], acc_out, ws, nbytes, stream)
    return y


def gemm_w4a16(x, packed, hdr, stream=None, y=None):
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, hdr.N), dtype=torch.bfloat16, device=x.device)
    nbytes = qlin_workspace_size(QLIN_OP_GEMM_W4A16, M, hdr.N, hdr.K)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=x.device) if nbytes else None
    qlin_gemm_w4a16(x, packed, hdr, M, y, ws, nbytes, stream)
    return y


def gemm_w4a8(qx, sx, packed, hdr, out_dtype=torch.bfloat16, acc_out=None, stream=None, y=None):
    """W4A8: per-token INT8 codes qx [M x K] with scales sx, packed INT4 weight."""
    M = qx.shape[0]
    if y is None:
        y = torch.empty((M, hdr.N), dtype=out_dtype, device=qx.device)
    nbytes = qlin_workspace_size(QLIN_OP_GEMM_W4A8, M, hdr.N, hdr.K)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=qx.device) if nbytes else None
    qlin_gemm_w4a8(qx, sx, packed, hdr, M, y, _TORCH_DT[y.dtype], acc_out, ws, nbytes, stream)
    return y


def qlin_absmax_update(x, xt, rows, cols, ld, running, stream=None):
    return _check("qlin_absmax_update", load().qlin_absmax_update(_ptr(x), xt, rows, cols, ld, _ptr(running),
                                                                  _stream(stream)))


def qlin_fold_layernorm(gamma, beta, s, K, gamma_out, beta_out, stream=None):
    return _check("qlin_fold_layernorm", load().qlin_fold_layernorm(_ptr(gamma), _ptr(beta), _ptr(s), K,
                                                                    _ptr(gamma_out), _ptr(beta_out), _stream(stream)))


def qlin_quant_error(x, xt, rows, cols, ld, smooth, p, q, s, z, out, ws, ws_bytes, stream=None):
    return _check("qlin_quant_error", load().qlin_quant_error(
        _ptr(x), xt, rows, cols, ld, _ptr(smooth), C.byref(p), _ptr(q), _ptr(s), _ptr(z), _ptr(out), _ptr(ws),
        ws_bytes, _stream(stream)))


def absmax_update(x, running, stream=None):
    rows, cols = x.shape
    qlin_absmax_update(x, dtype_code(x), rows, cols, x.stride(0), running, stream)
    return running


def fold_layernorm(gamma, beta, s, stream=None):
    g2 = torch.empty_like(gamma)
    b2 = None if beta is None else torch.empty_like(beta)
    qlin_fold_layernorm(gamma, beta, s, gamma.numel(), g2, b2, stream)
    return g2, b2


def quant_error(x, p, q, s, z, smooth=None, stream=None):
    """(sum (x' - x^)^2, sum x'^2, max |x' - x^|) as a device binary64 tensor."""
    rows, cols = x.shape
    out = torch.empty(3, dtype=torch.float64, device=x.device)
    n = qlin_workspace_size(QLIN_OP_QUANT_ERROR, 0, 0, 0)
    ws = torch.empty(n, dtype=torch.uint8, device=x.device)
    qlin_quant_error(x, dtype_code(x), rows, cols, x.stride(0), smooth, p, q, s, z, out, ws, n, stream)
    return out


def qlin_llmint8_workspace_size(M, N, K, max_outliers):
    return load().qlin_llmint8_workspace_size(M, N, K, max_outliers)


def qlin_gemm_llmint8(x, xt, M, K, ld, qw, sw, N, threshold, max_outliers, y, yt, outliers, ws, ws_bytes,
                      stream=None):
    return _check("qlin_gemm_llmint8", load().qlin_gemm_llmint8(
        _ptr(x), xt, M, K, ld, _ptr(qw), _ptr(sw), N, threshold, max_outliers, _ptr(y), yt, _ptr(outliers),
        _ptr(ws), ws_bytes, _stream(stream)))


def gemm_llmint8(x, qw, sw, threshold=6.0, max_outliers=None, out_dtype=torch.bfloat16, outliers=None,
                 stream=None):
    """LLM.int8(): bf16/fp16 activations x [M x K], INT8 weight qw [N x K] with
    per-channel scales sw; returns y [M x N]."""
    M, K = x.shape
    N = qw.shape[0]
    if max_outliers is None:
        max_outliers = K
    n = qlin_llmint8_workspace_size(M, N, K, max_outliers)
    ws = torch.empty(n, dtype=torch.uint8, device=x.device)
    y = torch.empty((M, N), dtype=out_dtype, device=x.device)
    qlin_gemm_llmint8(x, dtype_code(x), M, K, x.stride(0), qw, sw, N, threshold, max_outliers, y,
                      _TORCH_DT[out_dtype], outliers, ws, n, stream)
    return y


def qlin_kv_cache_bytes(capacity, channels, head_dim, group, residual, bits):
    return load().qlin_kv_cache_bytes(capacity, channels, head_dim, group, residual, bits)


def qlin_kv_cache_init(c, mem, mem_bytes, capacity, channels, head_dim, group, residual, bits):
    return _check("qlin_kv_cache_init", load().qlin_kv_cache_init(C.byref(c), _ptr(mem), mem_bytes, capacity,
                                                                  channels, head_dim, group, residual, bits))


def qlin_kv_append(c, k_new, v_new, n, stream=None):
    return _check("qlin_kv_append", load().qlin_kv_append(C.byref(c), _ptr(k_new), _ptr(v_new), n, _stream(stream)))


def qlin_kv_read(c, k_out, v_out, stream=None):
    return _check("qlin_kv_read", load().qlin_kv_read(C.byref(c), _ptr(k_out), _ptr(v_out), _stream(stream)))


class KVCache:
    """A quantized KV cache in one device buffer (see qlin_kv_cache)."""

    def __init__(self, capacity, channels, head_dim, group, residual, bits, device="cuda"):
        n = qlin_kv_cache_bytes(capacity, channels, head_dim, group, residual, bits)
        if n == 0:
            raise QlinError("qlin_kv_cache_bytes", QLIN_ERR_ARG, "invalid cache parameters")
        self.mem = torch.empty(n, dtype=torch.uint8, device=device)
        self.c = qlin_kv_cache()
        qlin_kv_cache_init(self.c, self.mem, n, capacity, channels, head_dim, group, residual, bits)

    def append(self, k, v, stream=None):
        qlin_kv_append(self.c, k, v, k.shape[0], stream)

    def read(self, stream=None):
        T, C_ = self.c.length, self.c.channels
        k = torch.empty((T, C_), dtype=torch.bfloat16, device=self.mem.device)
        v = torch.empty((T, C_), dtype=torch.bfloat16, device=self.mem.device)
        qlin_kv_read(self.c, k, v, stream)
        return k, v

    def _view(self, ptr, count, dtype):
        off = ptr - self.mem.data_ptr()
        item = torch.empty((), dtype=dtype).element_size()
        return self.mem[off:off + count * item].view(dtype)

    def state(self):
        """Device views of the quantized store: (k_codes, k_scale, k_zero,
        v_codes, v_scale, v_zero) of the tokens below c.quantized."""
        c = self.c
        tq, C_, heads = c.quantized, c.channels, c.channels // c.head_dim
        nb = tq * C_ * c.bits // 8
        return (self._view(c.k_codes, nb, torch.uint8), self._view(c.k_scale, tq // c.group * C_, torch.float32),
                self._view(c.k_zero, tq // c.group * C_, torch.int32), self._view(c.v_codes, nb, torch.uint8),
                self._view(c.v_scale, tq * heads, torch.float32), self._view(c.v_zero, tq * heads, torch.int32))
