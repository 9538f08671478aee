"""GPU parity of qlin_quantize / qlin_dequantize / qlin_absmax /
qlin_smooth_factors against the CPU oracle: codes, scales (binary32 bits or
binary16 values), zero points and dequantized values must be bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from activation_quantization_quantize_b300 import inputs, qlin
from helpers import codes_to_int, host_f32, oracle_quantize, scales_f32

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


def make_x(rows, cols, seed, dtype, special=True):
    x = inputs.normal((rows, cols), 1.0, seed)
    if special and rows * cols > 0:
        rng = np.random.default_rng(seed + 100)
        x[:, rng.integers(0, cols)] *= 40.0                       # an outlier channel
        x.reshape(-1)[rng.integers(0, rows * cols, max(1, rows * cols // 500))] = 100.0
        x[rows // 2] = 0.0                                        # an all-zero row
        if rows > 2:
            x[1] = -np.abs(x[1])                                  # a negative-only row
    t = torch.from_numpy(x).to(DT[dtype])
    return t.cuda(), host_f32(t)


def run_case(xd, xh, p, smooth=None):
    rows, cols = xh.shape
    sm_d = None if smooth is None else torch.from_numpy(smooth).cuda()
    q, s, z = qlin.quantize(xd, p, smooth=sm_d)
    torch.cuda.synchronize()
    qo, so, zo = oracle_quantize(xh, p, smooth=smooth)
    np.testing.assert_array_equal(codes_to_int(q, p, rows, cols), qo)
    sg = scales_f32(s)
    if p.scale_dtype == qlin.QLIN_F32:
        np.testing.assert_array_equal(sg.view(np.uint32), so.view(np.uint32))
    else:
        np.testing.assert_array_equal(sg, so)
    if not p.symmetric:
        np.testing.assert_array_equal(z.cpu().numpy(), zo)
    return q, s, z, qo, so, zo


CODES = ["s8", "s4", "u8", "u4"]
SHAPES = [(1, 8), (3, 40), (17, 264), (64, 4096), (5, 1024), (33, 384)]


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("code", CODES)
@pytest.mark.parametrize("gran", ["tensor", "row", "col"])
@pytest.mark.parametrize("shape", SHAPES)
def test_quantize_dynamic(dtype, code, gran, shape):
    rows, cols = shape
    xd, xh = make_x(rows, cols, seed=rows * 7 + cols, dtype=dtype)
    run_case(xd, xh, qlin.make_params(code, gran))


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("code", CODES)
@pytest.mark.parametrize("group", [8, 32, 64, 128])
@pytest.mark.parametrize("shape", [(3, 128), (17, 384), (64, 4096), (5, 6144), (2, 28672), (3, 40960)])
def test_quantize_groups(dtype, code, group, shape):
    rows, cols = shape
    if cols % group:
        pytest.skip("group does not divide cols")
    xd, xh = make_x(rows, cols, seed=cols + group, dtype=dtype)
    run_case(xd, xh, qlin.make_params(code, "group", group=group))


@pytest.mark.parametrize("code", CODES)
@pytest.mark.parametrize("gran,group", [("row", 0), ("group", 128), ("group", 32), ("tensor", 0)])
def test_quantize_f16_scales(code, gran, group):
    xd, xh = make_x(24, 512, seed=3, dtype="bf16")
    xd = (xd.float() * 0.02).to(torch.bfloat16)
    xh = host_f32(xd)
    run_case(xd, xh, qlin.make_params(code, gran, group=group, scale_f16=True))


@pytest.mark.parametrize("code", ["s8", "u8", "s4"])
@pytest.mark.parametrize("gran,group,cols", [("row", 0, 512), ("row", 0, 8192), ("group", 64, 512),
                                             ("tensor", 0, 512), ("col", 0, 512)])
def test_quantize_f16_scale_saturation(code, gran, group, cols):
    """Values whose scale overflows binary16 (max|x| / qmax > 65504): the
    stored scale saturates at 65504 and the codes must clip, as the oracle's
    do (every kernel that serves binary16 scales clamps and range-tests)."""
    rows = 16
    xf = inputs.normal((rows, cols), 1.0, 77)
    xf[:, 3] = 3.0e7                                          # far beyond 65504 * 127
    xf[5, :] *= 2.0e6
    xd = torch.from_numpy(xf).to(torch.bfloat16).cuda()
    run_case(xd, host_f32(xd), qlin.make_params(code, gran, group=group, scale_f16=True))


@pytest.mark.parametrize("mode", [qlin.QLIN_SMOOTH_DIVIDE, qlin.QLIN_SMOOTH_MULTIPLY])
@pytest.mark.parametrize("gran", ["row", "tensor", "col", "group"])
def test_quantize_smoothing(mode, gran):
    rows, cols = 32, 1024
    xd, xh = make_x(rows, cols, seed=11, dtype="bf16")
    rng = np.random.default_rng(12)
    sm = rng.uniform(0.05, 30.0, cols).astype(np.float32)
    run_case(xd, xh, qlin.make_params("s8", gran, group=64 if gran == "group" else 0, smooth_mode=mode),
             smooth=sm)


@pytest.mark.parametrize("code", CODES)
@pytest.mark.parametrize("gran", ["tensor", "row", "col", "group"])
def test_quantize_static_scales(code, gran):
    rows, cols = 16, 256
    xd, xh = make_x(rows, cols, seed=21, dtype="bf16")
    group = 64 if gran == "group" else 0
    p = qlin.make_params(code, gran, group=group)
    _, so, zo = oracle_quantize(xh * 0.7, p)               # scales from other data -> clipping
    ps = qlin.make_params(code, gran, group=group, static_scale=True)
    s = torch.from_numpy(so).cuda()
    z = torch.from_numpy(zo).cuda()
    q, _, _ = qlin.quantize(xd, ps, s=s, z=z)
    qo, _, _ = oracle_quantize(xh, ps, static_s=so, static_z=zo)
    np.testing.assert_array_equal(codes_to_int(q, ps, rows, cols), qo)


def test_quantize_unaligned_rows_generic_path():
    base = torch.from_numpy(inputs.normal((9, 100), 1.0, 5)).to(torch.bfloat16).cuda()
    xd = base[:, 3:3 + 90]                                   # ld = 100, odd offset
    xh = host_f32(xd)
    for code, gran, group in [("s8", "row", 0), ("u8", "tensor", 0), ("s4", "group", 10), ("u4", "col", 0)]:
        p = qlin.make_params(code, gran, group=group)
        q, s, z = qlin.quantize(xd, p)
        qo, so, zo = oracle_quantize(np.ascontiguousarray(xh), p)
        np.testing.assert_array_equal(codes_to_int(q, p, 9, 90), qo)
        np.testing.assert_array_equal(scales_f32(s).view(np.uint32), so.view(np.uint32))


@pytest.mark.parametrize("shape", [(37, 1024), (300, 4096)])
def test_quantize_aligned_strided_rows(shape):
    """A 16-byte-aligned view with ld > cols takes the vector kernels (strip,
    row-streaming, percentile): every scope against the oracle on the
    contiguous copy."""
    rows, cols = shape
    base = torch.from_numpy(inputs.normal((rows, cols + 64), 1.0, rows + 3)).to(torch.bfloat16).cuda()
    xd = base[:, 32:32 + cols]                               # ld = cols + 64, 64-byte offset
    xh = np.ascontiguousarray(host_f32(xd))
    cases = [("s8", "tensor", 0, 0.0), ("u8", "tensor", 0, 0.0), ("s4", "tensor", 0, 0.0), ("s8", "col", 0, 0.0),
             ("u8", "col", 0, 0.0), ("s8", "row", 0, 0.0), ("u4", "group", 64, 0.0), ("s8", "tensor", 0, 99.9)]
    for code, gran, group, pct in cases:
        p = qlin.make_params(code, gran, group=group, percentile=pct)
        q, s, z = qlin.quantize(xd, p)
        qo, so, zo = oracle_quantize(xh, p)
        np.testing.assert_array_equal(codes_to_int(q, p, rows, cols), qo)
        np.testing.assert_array_equal(scales_f32(s).view(np.uint32), so.view(np.uint32))
        if not p.symmetric:
            np.testing.assert_array_equal(z.cpu().numpy(), zo)


def test_exhaustive_bf16_static_scales():
    """Every finite bf16 value against the oracle at a set of scales and zero
    points (the code decision near half-integers)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = oracle.bf16_bits_to_f32(bits)
    v = v[np.isfinite(v)]
    v = v[: (v.size // 8) * 8]
    cols = 8
    rows = v.size // cols
    xt = torch.from_numpy(v.reshape(rows, cols)).to(torch.bfloat16).cuda()
    rng = np.random.default_rng(31)
    scales = [0.016535433, 1.0, 2.0 ** -10, 3.7e-3, 0.787401, 1e-30, 3e5] + list(rng.uniform(1e-3, 2, 20))
    for sc in scales:
        for code, z in [("s8", 0), ("u8", 93), ("s4", 0), ("u4", 8), ("u8", 0)]:
            p = qlin.make_params(code, "tensor", static_scale=True)
            s = torch.tensor([sc], dtype=torch.float32).cuda()
            zt = torch.tensor([z], dtype=torch.int32).cuda()
            q, _, _ = qlin.quantize(xt, p, s=s, z=zt)
            qo, _, _ = oracle_quantize(v.reshape(rows, cols), p, static_s=np.array([sc], np.float32),
                                       static_z=np.array([z], np.int32))
            np.testing.assert_array_equal(codes_to_int(q, p, rows, cols), qo)


def test_near_ties_binary32():
    """Values whose binary32 quotient lands on (or next to) a half-integer."""
    rng = np.random.default_rng(41)
    s = np.float32(0.0123)
    n = rng.integers(-120, 120, 4096)
    base = ((n + 0.5) * np.float64(s)).astype(np.float32)
    neigh = np.stack([np.nextafter(base, np.float32(-np.inf)), base, np.nextafter(base, np.float32(np.inf))], 1)
    x = neigh.reshape(-1, 8)
    xt = torch.from_numpy(x).cuda()
    for code, z in [("s8", 0), ("u8", 3), ("u8", 128)]:
        p = qlin.make_params(code, "tensor", static_scale=True)
        q, _, _ = qlin.quantize(xt, p, s=torch.tensor([s]).cuda(), z=torch.tensor([z], dtype=torch.int32).cuda())
        qo, _, _ = oracle_quantize(x, p, static_s=np.array([s]), static_z=np.array([z], np.int32))
        np.testing.assert_array_equal(codes_to_int(q, p, *x.shape), qo)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_percentile_per_tensor(dtype):
    xd, xh = make_x(200, 1024, seed=51, dtype=dtype)
    run_case(xd, xh, qlin.make_params("s8", "tensor", percentile=99.9))
    run_case(xd, xh, qlin.make_params("s4", "tensor", percentile=99.0))
    sm = np.random.default_rng(52).uniform(0.5, 4, 1024).astype(np.float32)
    run_case(xd, xh, qlin.make_params("s8", "tensor", percentile=99.9, smooth_mode=qlin.QLIN_SMOOTH_DIVIDE),
             smooth=sm)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("code", CODES)
@pytest.mark.parametrize("shape", [(1, 4104), (300, 28672), (517, 8200), (3, 40960)])
def test_quantize_per_token_long_rows(dtype, code, shape):
    """Per-token scopes of rows longer than 4096 16-bit values: the rows are
    streamed through shared memory (several rows per CTA when rows > SMs),
    held in registers up to 32,768 values and read from the row buffer
    beyond."""
    rows, cols = shape
    xd, xh = make_x(rows, cols, seed=rows + cols, dtype=dtype)
    run_case(xd, xh, qlin.make_params(code, "row"))


@pytest.mark.parametrize("code", ["s8", "u4"])
def test_quantize_per_token_long_rows_static(code):
    """Static per-token scales taken from other data (so codes clip) on rows
    streamed through shared memory."""
    rows, cols = 200, 12288
    xd, xh = make_x(rows, cols, seed=91, dtype="bf16")
    p = qlin.make_params(code, "row")
    _, so, zo = oracle_quantize(xh * 0.7, p)
    ps = qlin.make_params(code, "row", static_scale=True)
    q, _, _ = qlin.quantize(xd, ps, s=torch.from_numpy(so).cuda(),
                            z=None if zo is None else torch.from_numpy(zo).cuda())
    qo, _, _ = oracle_quantize(xh, ps, static_s=so, static_z=zo)
    np.testing.assert_array_equal(codes_to_int(q, ps, rows, cols), qo)


@pytest.mark.parametrize("code", CODES)
@pytest.mark.parametrize("gran,group", [("tensor", 0), ("row", 0), ("col", 0), ("group", 32), ("group", 128)])
@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32, torch.float16])
def test_dequantize(code, gran, group, out):
    rows, cols = 19, 256
    xd, xh = make_x(rows, cols, seed=61, dtype="bf16")
    p = qlin.make_params(code, gran, group=group, scale_f16=(gran == "group"))
    q, s, z = qlin.quantize(xd, p)
    y = qlin.dequantize(q, s, z, p, rows, cols, out_dtype=out)
    qo, so, zo = oracle_quantize(xh, p)
    yo = oracle.dequantize(qo, so, zo if not p.symmetric else None, {0: 0, 1: 1, 2: 2, 3: 3}[p.gran], group)
    if out == torch.bfloat16:
        yo = oracle.round_bf16(yo)
    elif out == torch.float16:
        yo = yo.astype(np.float16).astype(np.float32)
    np.testing.assert_array_equal(host_f32(y), yo)


@pytest.mark.parametrize("gran,group", [("tensor", 0), ("row", 0), ("col", 0), ("group", 64)])
def test_absmax(gran, group):
    xd, xh = make_x(37, 512, seed=71, dtype="bf16")
    a = qlin.absmax(xd, qlin.GRANS[gran], group)
    ao = oracle.absmax(xh, {"tensor": 0, "row": 1, "col": 2, "group": 3}[gran], group)
    np.testing.assert_array_equal(a.cpu().numpy(), ao)


@pytest.mark.parametrize("alpha", [0.5, 0.0, 1.0, 0.7])
def test_smooth_factors(alpha):
    rng = np.random.default_rng(81)
    mx = rng.uniform(0.1, 60, 4099).astype(np.float32)
    mw = rng.uniform(1e-3, 0.1, 4099).astype(np.float32)
    mx[5] = 0.0
    s = qlin.smooth_factors(torch.from_numpy(mx).cuda(), torch.from_numpy(mw).cuda(), alpha).cpu().numpy()
    so = oracle.smooth_factors(mx, mw, alpha)
    if alpha in (0.5, 1.0):
        np.testing.assert_array_equal(s, so)
    else:
        np.testing.assert_allclose(s, so, rtol=4 * 2 ** -23)


def test_empty_input_is_noop():
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    q, s, z = qlin.quantize(x, qlin.make_params("s8", "row"))
    assert q.numel() == 0


# ------------------------------------------------------------- full-size sweep (16384 x 4096)
@pytest.fixture(scope="module")
def sweep():
    t = inputs.sweep_tensor()
    return t.cuda(), host_f32(t)


@pytest.mark.parametrize("code", ["s8", "s4", "u8"])
@pytest.mark.parametrize("gran,group", [("row", 0), ("group", 32), ("group", 64), ("group", 128)])
def test_sweep_rowlocal_sampled(sweep, code, gran, group):
    xd, xh = sweep
    p = qlin.make_params(code, gran, group=group)
    q, s, z = qlin.quantize(xd, p)
    rows = np.random.default_rng(91).choice(xh.shape[0], 64, replace=False)
    rows.sort()
    qo, so, zo = oracle_quantize(xh[rows], p)
    qg = codes_to_int(q, p, *xh.shape)[rows]
    np.testing.assert_array_equal(qg, qo)
    ngr = 1 if gran == "row" else xh.shape[1] // group
    sg = scales_f32(s).reshape(xh.shape[0], ngr)[rows].reshape(-1)
    np.testing.assert_array_equal(sg.view(np.uint32), so.view(np.uint32))


@pytest.mark.parametrize("code,gran", [("s8", "tensor"), ("u8", "tensor"), ("s8", "col"), ("u8", "col"),
                                       ("s4", "col")])
def test_sweep_global_scopes(sweep, code, gran):
    xd, xh = sweep
    run_case(xd, xh, qlin.make_params(code, gran))


def test_sweep_percentile(sweep):
    xd, xh = sweep
    run_case(xd, xh, qlin.make_params("s8", "tensor", percentile=99.9))


# ------------------------------------------------------------- dequantize at full size
def _dequant_check(q, s, z, p, rows, cols, out=torch.bfloat16, row_sets=None):
    """GPU dequantize of the whole tensor against the oracle's dequantize of
    the same codes / scales / zero points, element by element, bit-exact
    (one binary32 product s*(q-z), then one rounding to the output type).
    The oracle side runs on row_sets (all rows in blocks when None)."""
    y = qlin.dequantize(q, s, z, p, rows, cols, out_dtype=out)
    torch.cuda.synchronize()
    gran = {0: 0, 1: 1, 2: 2, 3: 3}[p.gran]
    ngr = {0: 1, 1: 1, 2: 1, 3: cols // max(p.group, 1)}[p.gran]
    sh = scales_f32(s)
    zh = None if p.symmetric else z.cpu().numpy()
    if row_sets is None:
        row_sets = [np.arange(r0, min(rows, r0 + 1024)) for r0 in range(0, rows, 1024)]
    for rs in row_sets:
        idx = torch.from_numpy(rs).cuda()
        qi = codes_to_int(q[idx], p, len(rs), cols)
        if p.gran == qlin.QLIN_PER_ROW:
            ss, zz = sh[rs], (None if zh is None else zh[rs])
        elif p.gran == qlin.QLIN_PER_GROUP:
            ss = sh.reshape(rows, ngr)[rs].reshape(-1)
            zz = None if zh is None else zh.reshape(rows, ngr)[rs].reshape(-1)
        else:
            ss, zz = sh, zh
        yo = oracle.dequantize(qi, ss, zz, gran, p.group)
        if out == torch.bfloat16:
            yo = oracle.round_bf16(yo)
        elif out == torch.float16:
            yo = yo.astype(np.float16).astype(np.float32)
        np.testing.assert_array_equal(host_f32(y[idx]), yo)


@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32, torch.float16])
def test_dequantize_downproj_rows_full_size(out):
    """4096 x 28672 per-token INT8 (the step's call): every row takes two
    segments of 1024 16-code chunks, and the 8192 (row, segment) units exceed
    the grid, so the kernel grid-strides.  Whole tensor, bit-exact."""
    rows, cols = 4096, 28672
    x = inputs.downproj_activation(rows, outliers=True).cuda()
    p = qlin.make_params("s8", "row")
    q, s, z = qlin.quantize(x, p)
    del x
    _dequant_check(q, s, z, p, rows, cols, out)


@pytest.mark.parametrize("code,gran,group", [("s8", "row", 0), ("s4", "group", 128), ("u8", "tensor", 0),
                                             ("u8", "group", 64)])
def test_dequantize_sweep_full_size(sweep, code, gran, group):
    """The 16384 x 4096 sweep tensor (16384 units, far more than the grid)
    dequantized at full size; the oracle checks every row."""
    xd, xh = sweep
    rows, cols = xh.shape
    p = qlin.make_params(code, gran, group=group, scale_f16=(gran == "group"))
    q, s, z = qlin.quantize(xd, p)
    _dequant_check(q, s, z, p, rows, cols)


def test_dequantize_asym_groups_long_rows():
    """Asymmetric UINT8 per-group (g = 128) on rows of 17,408 values (more
    than one 16,384-value segment per row) and a ragged row count."""
    rows, cols = 33, 17408
    xd, xh = make_x(rows, cols, seed=1717, dtype="bf16")
    p = qlin.make_params("u8", "group", group=128)
    q, s, z = qlin.quantize(xd, p)
    qo, so, zo = oracle_quantize(xh, p)
    np.testing.assert_array_equal(codes_to_int(q, p, rows, cols), qo)
    for out in (torch.bfloat16, torch.float32):
        _dequant_check(q, s, z, p, rows, cols, out)


@pytest.mark.parametrize("code", ["s8", "u8", "s4", "u4"])
@pytest.mark.parametrize("cols", [256, 4096, 28672])
def test_dequantize_every_code(code, cols):
    """Every bit pattern of the code type (all 256 bytes, all 16 nibbles, the
    ones outside [qmin, qmax] included) with zero points at both ends of the
    code range, negative ones for signed codes, and scales from tiny to
    binary16's largest, through the short-row and long-row dequantize
    kernels: bit-exact against the oracle's s * (q - z)."""
    bits = 4 if code in ("s4", "u4") else 8
    signed = code.startswith("s")
    allv = np.arange(-(1 << (bits - 1)), 1 << (bits - 1)) if signed else np.arange(0, 1 << bits)
    zs = [0, int(allv[0]), int(allv[-1]), 3] + ([-5] if signed else [])
    ss = np.array([0.37, 1e-3, 3.0, 65504.0, 2.0 ** -20], dtype=np.float32)
    rows = 2 * len(zs) * len(ss)
    rng = np.random.default_rng(cols + bits)
    qi = np.empty((rows, cols), dtype=np.int32)
    for r in range(rows):
        qi[r] = np.resize(np.roll(allv, r), cols)
        qi[r, rng.integers(0, cols, 16)] = allv[rng.integers(0, len(allv), 16)]
    zi = np.array([zs[(r // len(ss)) % len(zs)] for r in range(rows)], dtype=np.int32)
    sf = np.array([ss[r % len(ss)] for r in range(rows)], dtype=np.float32)
    if bits == 4:
        u = (qi & 0xF).astype(np.uint8)
        packed = (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)
        qd = torch.from_numpy(packed).cuda()
    else:
        qd = torch.from_numpy(qi.astype(np.int8 if signed else np.uint8)).cuda()
    p = qlin.make_params(code, "row", symmetric=False)
    y = qlin.dequantize(qd, torch.from_numpy(sf).cuda(), torch.from_numpy(zi).cuda(), p, rows, cols,
                        out_dtype=torch.float32)
    torch.cuda.synchronize()
    yo = oracle.dequantize(qi, sf, zi, oracle.PER_ROW)
    np.testing.assert_array_equal(host_f32(y).view(np.uint32), yo.view(np.uint32))


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("code", CODES)
@pytest.mark.parametrize("shape", [(9, 6144), (4, 8192), (17, 8200), (5, 12288)])
def test_quantize_per_tensor_long_rows(dtype, code, shape):
    """Dynamic per-tensor scopes on both sides of the routing boundary: rows
    of up to 8192 values take the row-streaming kernels' one-scope mode,
    longer rows the strip kernel."""
    rows, cols = shape
    xd, xh = make_x(rows, cols, seed=rows * 3 + cols, dtype=dtype)
    run_case(xd, xh, qlin.make_params(code, "tensor"))
