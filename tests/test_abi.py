"""C-ABI checks that need no GPU: the library loads, exports every entry
point include/qlin.h declares, and rejects bad arguments on the host before
any CUDA call."""
import ctypes as C
import os
import re

import pytest

from activation_quantization_quantize_b300 import build, qlin

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return qlin.load()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(qlin_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 12
    for n in ["qlin_quantize", "qlin_pack_w4", "qlin_gemm_w8a8", "qlin_gemm_w4a16"]:
        assert n in names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    assert qlin.qlin_version() >= 10000
    for st in range(-6, 1):
        assert qlin.qlin_status_string(st) != "unknown status"
    assert qlin.qlin_status_string(7) == "unknown status"


def test_qparams_layout_matches_header():
    # int code, qmin, qmax, symmetric, gran, group (6 x 4) + pad to 8 + double + 3 ints + pad
    assert C.sizeof(qlin.qlin_qparams) == 48
    assert qlin.qlin_qparams.clip_percentile.offset == 24
    assert C.sizeof(qlin.qlin_w4_header) == 64


def test_workspace_sizes(lib):
    p = qlin.make_params("s8", "row")
    assert qlin.qlin_workspace_size(qlin.QLIN_OP_QUANTIZE, 16, 4096, 0, p) >= 0
    p = qlin.make_params("s8", "tensor")
    assert qlin.qlin_workspace_size(qlin.QLIN_OP_QUANTIZE, 16384, 4096, 0, p) == 8
    p = qlin.make_params("u8", "col")
    assert qlin.qlin_workspace_size(qlin.QLIN_OP_QUANTIZE, 16384, 4096, 0, p) == 4096 * 8
    p = qlin.make_params("s8", "tensor", percentile=99.9)
    assert qlin.qlin_workspace_size(qlin.QLIN_OP_QUANTIZE, 16384, 4096, 0, p) == (32768 + 65536 + 4) * 4
    p = qlin.make_params("s8", "tensor", static_scale=True)
    assert qlin.qlin_workspace_size(qlin.QLIN_OP_QUANTIZE, 16384, 4096, 0, p) == 0


def test_pack_w4_size_closed_form(lib):
    # codes N*K/2 + fp16 scales N*K/g*2 (+ 4-bit zeros N*K/g/2), each 256-aligned, after a header
    N, K, g = 4096, 4096, 128
    n = qlin.qlin_pack_w4_size(N, K, g, False)
    assert n == 256 + N * K // 2 + N * (K // g) * 2
    N, K = 8192, 28672
    n = qlin.qlin_pack_w4_size(N, K, g, True)
    assert n == 256 + N * K // 2 + N * (K // g) * 2 + N * (K // g) // 2
    assert qlin.qlin_pack_w4_size(N, K, 100, False) == 0


def _bad(fn, *args):
    rc = getattr(qlin.load(), fn)(*args)
    return rc


def test_host_validation_without_gpu(lib):
    L = lib
    fake = C.c_void_p(0x10000)          # never dereferenced: validation fails first
    p = qlin.make_params("s8", "row")
    p.qmin, p.qmax = -128, 127          # symmetric needs qmin == -qmax
    assert L.qlin_quantize(fake, qlin.QLIN_BF16, 4, 64, 64, None, C.byref(p), fake, fake, None, None, 0,
                           None) == qlin.QLIN_ERR_ARG
    p = qlin.make_params("s4", "group", group=48)   # 64 % 48 != 0
    assert L.qlin_quantize(fake, qlin.QLIN_BF16, 4, 64, 64, None, C.byref(p), fake, fake, None, None, 0,
                           None) == qlin.QLIN_ERR_ARG
    p = qlin.make_params("u8", "row", percentile=99.9)  # percentile: symmetric per-tensor only
    assert L.qlin_quantize(fake, qlin.QLIN_BF16, 4, 64, 64, None, C.byref(p), fake, fake, fake, None, 0,
                           None) == qlin.QLIN_ERR_UNSUPPORTED
    p = qlin.make_params("s8", "tensor")               # needs a workspace
    assert L.qlin_quantize(fake, qlin.QLIN_BF16, 4, 64, 64, None, C.byref(p), fake, fake, None, None, 0,
                           None) == qlin.QLIN_ERR_WORKSPACE
    p = qlin.make_params("u8", "row")                  # asymmetric needs z
    assert L.qlin_quantize(fake, qlin.QLIN_BF16, 4, 64, 64, None, C.byref(p), fake, fake, None, None, 0,
                           None) == qlin.QLIN_ERR_ARG
    p = qlin.make_params("s8", "row", smooth_mode=qlin.QLIN_SMOOTH_DIVIDE)  # smoothing needs factors
    assert L.qlin_quantize(fake, qlin.QLIN_BF16, 4, 64, 64, None, C.byref(p), fake, fake, None, None, 0,
                           None) == qlin.QLIN_ERR_ARG
    p = qlin.make_params("s8", "row")
    assert L.qlin_quantize(fake, qlin.QLIN_BF16, 4, 64, 32, None, C.byref(p), fake, fake, None, None, 0,
                           None) == qlin.QLIN_ERR_ARG   # ld < cols
    # empty input is a no-op
    assert L.qlin_quantize(None, qlin.QLIN_BF16, 0, 64, 64, None, C.byref(p), None, None, None, None, 0,
                           None) == qlin.QLIN_OK
    # W8A8: K must be a multiple of 16, operands 16-byte aligned
    assert L.qlin_gemm_w8a8(fake, fake, fake, fake, 8, 8, 24, fake, qlin.QLIN_F32, None, None, 0,
                            None) == qlin.QLIN_ERR_UNSUPPORTED
    assert L.qlin_gemm_w8a8(C.c_void_p(0x10001), fake, fake, fake, 8, 8, 32, fake, qlin.QLIN_F32, None,
                            None, 0, None) == qlin.QLIN_ERR_ARG
    assert L.qlin_gemm_w8a8(fake, fake, fake, fake, 8, 8, 32, fake, qlin.QLIN_S8, None, None, 0,
                            None) == qlin.QLIN_ERR_ARG
    # W4: header checks
    h = qlin.qlin_w4_header()
    assert L.qlin_gemm_w4a16(fake, fake, C.byref(h), 1, fake, None, 0, None) == qlin.QLIN_ERR_LAYOUT
    h.magic, h.version, h.N, h.K, h.group, h.asym = qlin.QLIN_W4_MAGIC, 1, 64, 256, 128, 0
    assert L.qlin_gemm_w4a16(fake, fake, C.byref(h), 1, fake, None, 0, None) == qlin.QLIN_ERR_LAYOUT
    assert L.qlin_pack_w4(fake, fake, None, 64, 256, 96, fake, 1 << 20, None, None) == qlin.QLIN_ERR_UNSUPPORTED
    assert L.qlin_pack_w4(fake, fake, None, 64, 256, 128, C.c_void_p(0x10010), 1 << 20, None,
                          None) == qlin.QLIN_ERR_ARG   # packed must be 256-byte aligned
    assert L.qlin_smooth_factors(fake, fake, 16, C.c_float(1.5), fake, None) == qlin.QLIN_ERR_ARG


def test_noalloc_reports_argument_errors_first(lib):
    """qlin_quantize_noalloc checks its arguments exactly as qlin_quantize does
    before it looks at the scratch limit: a bad group is QLIN_ERR_ARG, not
    QLIN_ERR_WORKSPACE, even for a size whose statistics would not fit."""
    L = lib
    fake = C.c_void_p(0x10000)
    p = qlin.make_params("s8", "col")
    p.group = -5
    p.gran = 7                                          # no such granularity
    assert L.qlin_quantize_noalloc(fake, qlin.QLIN_BF16, 4, 1 << 20, 1 << 20, None, C.byref(p), fake, fake,
                                   None, None) == qlin.QLIN_ERR_ARG
    p = qlin.make_params("s8", "group", group=-128)
    assert L.qlin_quantize_noalloc(fake, qlin.QLIN_BF16, 4, 4096, 4096, None, C.byref(p), fake, fake,
                                   None, None) == qlin.QLIN_ERR_ARG
    p = qlin.make_params("u8", "col", percentile=99.9)  # percentile: symmetric per-tensor only
    assert L.qlin_quantize_noalloc(fake, qlin.QLIN_BF16, 4, 1 << 20, 1 << 20, None, C.byref(p), fake, fake,
                                   fake, None) == qlin.QLIN_ERR_UNSUPPORTED
    p = qlin.make_params("s8", "col")                   # valid, but 8 MB of statistics > the scratch
    assert L.qlin_quantize_noalloc(fake, qlin.QLIN_BF16, 4, 1 << 20, 1 << 20, None, C.byref(p), fake, fake,
                                   None, None) == qlin.QLIN_ERR_WORKSPACE


def test_row_local_scopes_need_no_workspace(lib):
    for code, gran, g in [("s8", "row", 0), ("u4", "group", 128), ("u8", "group", 7), ("s4", "row", 0)]:
        p = qlin.make_params(code, gran, group=g)
        for rows, cols in [(1, 14), (4096, 4096), (8192, 28672), (3, 100003 * 7 if g == 7 else 100002)]:
            assert qlin.qlin_workspace_size(qlin.QLIN_OP_QUANTIZE, rows, cols, 0, p) == 0


def test_stall_hook_validates_without_gpu(lib):
    assert lib.qlin_debug_stall_producers(1, 0) == qlin.QLIN_ERR_ARG


def test_kv_cache_struct_and_validation(lib):
    assert C.sizeof(qlin.qlin_kv_cache) == 112
    assert qlin.qlin_kv_cache.length.offset == 32
    assert qlin.qlin_kv_cache_bytes(1024, 512, 128, 32, 48, 4) > 0
    assert qlin.qlin_kv_cache_bytes(1000, 512, 128, 32, 48, 4) == 0   # capacity % group
    assert qlin.qlin_kv_cache_bytes(1024, 500, 128, 32, 48, 4) == 0   # channels % 16
    assert qlin.qlin_kv_cache_bytes(1024, 512, 128, 32, 48, 3) == 0   # bits
    # closed form: codes + K scales/zeros per (group, channel) + V per (token, head) + two bf16 rings
    cap, Cc, D, G, R = 1024, 512, 128, 32, 48
    up = lambda b: (b + 255) // 256 * 256  # noqa: E731
    want = 2 * up(cap * Cc // 2) + 2 * up(cap // G * Cc * 4) + 2 * up(cap * (Cc // D) * 4) + 2 * up((R + G) * Cc * 2)
    assert qlin.qlin_kv_cache_bytes(cap, Cc, D, G, R, 4) == want
    c = qlin.qlin_kv_cache()
    assert lib.qlin_kv_cache_init(C.byref(c), C.c_void_p(0x10000), want - 1, cap, Cc, D, G, R, 4) == \
        qlin.QLIN_ERR_WORKSPACE
    assert lib.qlin_kv_cache_init(C.byref(c), C.c_void_p(0x10000), want, cap, Cc, D, G, R, 4) == qlin.QLIN_OK
    assert c.length == 0 and c.quantized == 0 and c.k_codes == 0x10000
    fake = C.c_void_p(0x20000)
    assert lib.qlin_kv_append(C.byref(c), fake, fake, cap + 1, None) == qlin.QLIN_ERR_ARG   # past capacity
    assert lib.qlin_kv_append(C.byref(c), C.c_void_p(0x20008), fake, 4, None) == qlin.QLIN_ERR_ARG  # alignment
    assert lib.qlin_kv_append(C.byref(c), fake, fake, 0, None) == qlin.QLIN_OK
