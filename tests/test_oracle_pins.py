"""Pins of the CPU oracle to values and properties fixed by the pages and by
mathematics (no GPU).  Each test names the passage it checks; a plausible
slip in the oracle (wrong rounding, dropped zero point, transposed operand,
wrong scale index, double instead of float division) fails at least one."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = (t.strip() for t in line.split("=", 1))
            out[k] = [float(t) for t in v.split()]
    return out


def f32_bits(v):
    return int(np.array([v], dtype=np.float32).view(np.uint32)[0])


def rne_fraction(fr):
    """Round a rational to the nearest integer, ties to even (exact)."""
    fl = math.floor(fr)
    d = fr - fl
    if d > Fraction(1, 2):
        return fl + 1
    if d < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


# ------------------------------------------------------------- worked examples
def test_page5_symmetric_example(orc):
    g = read_golden("page5_symmetric.txt")
    x = np.array(g["input"], dtype=np.float32)
    q, s, z = orc.quantize(x, -127, 127, True, orc.PER_TENSOR)
    q = q.ravel()
    # scale = max|x|/127 in binary32; page prints ~0.0165.
    assert f32_bits(s[0]) == 0x3C877551
    assert abs(float(s[0]) - g["printed_scale"][0]) < 5e-5
    assert z[0] == 0
    # every code equals round-half-even of the exact quotient x/s (no value is
    # within a rounding of a half-integer here, so fl() does not matter).
    for xi, qi in zip(x, q):
        assert qi == rne_fraction(Fraction(float(xi)) / Fraction(float(s[0])))
    printed = [int(v) for v in g["printed_codes"]]
    bad = [int(v) for v in g["disagree_codes"]]
    for i, (a, b) in enumerate(zip(q, printed)):
        if i in bad:
            assert a != b and abs(a - b) == 1, "logged disagreement moved"
        else:
            assert a == b
    assert list(q) == [30, -73, 127, -48, 103]
    xh = orc.dequantize(q, s, z, orc.PER_TENSOR).ravel()
    pd = g["printed_dequant"]
    bad_d = [int(v) for v in g["disagree_dequant"]]
    for i, (a, b) in enumerate(zip(xh, pd)):
        if i not in bad_d:
            assert abs(a - b) < 6e-4
    np.testing.assert_array_equal(
        xh, np.array([0.496063, -1.2070866, 2.1, -0.7937008, 1.7031496], dtype=np.float32))


def test_page5_asymmetric_example(orc):
    g = read_golden("page5_asymmetric.txt")
    x = np.array(g["input"], dtype=np.float32)
    qmin, qmax = int(g["qmin"][0]), int(g["qmax"][0])
    q, s, z = orc.quantize(x, qmin, qmax, False, orc.PER_TENSOR)
    q = q.ravel()
    # scale = (max - min)/255 in binary32, zero point = round(-min/scale).
    assert f32_bits(s[0]) == 0x3C54073A
    assert z[0] == 93
    assert list(q) == [132, 0, 255, 31, 224]
    # the page's own formula round(x/s + z) gives the same codes here.
    for xi, qi in zip(x, q):
        assert qi == rne_fraction(Fraction(float(xi)) / Fraction(float(s[0])) + int(z[0]))
    # errors stay within s/2 (the printed asymmetric error list is unpinned).
    xh = orc.dequantize(q, s, z, orc.PER_TENSOR).ravel()
    assert np.all(np.abs(x.astype(np.float64) - xh) <= float(s[0]) / 2 * (1 + 1e-6))
    # exact zero: 0 -> z -> 0
    q0, _, _ = orc.quantize(np.array([0.0], np.float32), qmin, qmax, False, orc.PER_TENSOR,
                            static_s=s, static_z=z)
    assert q0[0, 0] == z[0]
    assert orc.dequantize(q0, s, z, orc.PER_TENSOR)[0, 0] == 0.0


def test_page5_outlier_example(orc):
    g = read_golden("page5_outlier.txt")
    rng = np.random.default_rng(5)
    x = rng.uniform(g["normal_lo"][0], g["normal_hi"][0], 999).astype(np.float32)
    x = np.concatenate([x, np.array([g["outlier"][0], 2.0, -2.0], np.float32)])
    q, s, _ = orc.quantize(x, -127, 127, True, orc.PER_TENSOR)
    assert abs(float(s[0]) - g["printed_scale"][0]) < 5e-3
    lo, hi = (int(v) for v in g["printed_code_range"])
    assert q[0, -2] == hi and q[0, -3 + 2] == lo and q[0, -3] == 127
    assert q[0, :999].min() >= lo and q[0, :999].max() <= hi


def test_round_half_to_even_ties(orc):
    # absmax 127 -> s = 1 exactly, so x/s = x and every .5 is an exact tie.
    x = np.array([127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.5, 126.5], np.float32)
    q, s, _ = orc.quantize(x, -127, 127, True, orc.PER_TENSOR)
    assert s[0] == 1.0
    assert list(q.ravel()) == [127, 0, 2, 2, 0, -2, -2, 4, 126]
    assert list(q.ravel()[1:]) == [round(float(v)) for v in x[1:]]  # Python rounds half to even


def test_round_then_add_zero_point(orc):
    # With an odd zero point, round(x/s)+z and round(x/s+z) differ at ties; the
    # core formula (round first, then add z) is the one implemented.
    s = np.array([1.0], np.float32)
    z = np.array([3], np.int32)
    q, _, _ = orc.quantize(np.array([0.5, 1.5, -0.5], np.float32), 0, 255, False,
                           orc.PER_TENSOR, static_s=s, static_z=z)
    assert list(q.ravel()) == [3, 5, 3]


# ------------------------------------------------------------- exhaustive / brute force
def _all_finite_bf16():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = (bits.astype(np.uint32) << 16).view(np.float32)
    return v[np.isfinite(v)]


@pytest.mark.parametrize("scale", [0.016535433, 1.0, 2.0 ** -10, 3.7e-3, 0.787401, 1e-30, 3e5])
@pytest.mark.parametrize("qmin,qmax,z", [(-127, 127, 0), (-7, 7, 0), (0, 255, 93), (0, 15, 8)])
def test_exhaustive_bf16_codes(orc, scale, qmin, qmax, z):
    """All finite bf16 values against an independent binary32 evaluation
    (numpy's IEEE float32 divide and round-half-even rint)."""
    x = _all_finite_bf16()
    s = np.array([scale], np.float32)
    zz = np.array([z], np.int32)
    q, _, _ = orc.quantize(x, qmin, qmax, qmin == -qmax, orc.PER_TENSOR, static_s=s, static_z=zz)
    with np.errstate(over="ignore"):
        t = x / s[0]
    expect = np.clip(np.rint(t).astype(np.float64) + z, qmin, qmax).astype(np.int32)
    np.testing.assert_array_equal(q.ravel(), expect)


def test_division_is_binary32_not_binary64(orc):
    """Pairs (x, s) whose exact quotient is NOT a half-integer but whose
    binary32 quotient rounds onto one: the code is the even neighbour of that
    binary32 tie, which a binary64 division would not give."""
    found = 0
    rng = np.random.default_rng(1)
    for _ in range(20000):
        n = int(rng.integers(1, 100))
        s = np.float32(rng.uniform(0.01, 1.0))
        x = np.float32((n + 0.5) * float(s))
        t32 = x / s
        if float(t32) == n + 0.5 and Fraction(float(x)) / Fraction(float(s)) != Fraction(2 * n + 1, 2):
            q, _, _ = orc.quantize(np.array([x]), -127, 127, True, orc.PER_TENSOR,
                                   static_s=np.array([s]), static_z=np.zeros(1, np.int32))
            assert q[0, 0] == (n if n % 2 == 0 else n + 1)
            found += 1
    assert found > 10


def test_bound_half_step_unclipped(orc):
    """|x - s(q-z)| <= s/2 for values that are not clipped ([QDC] core formula
    bound), for every granularity and both code families."""
    rng = np.random.default_rng(2)
    x = rng.standard_normal((64, 256)).astype(np.float32)
    x[:, 5] *= 30
    for gran, group in [(orc.PER_TENSOR, 0), (orc.PER_ROW, 0), (orc.PER_COL, 0),
                        (orc.PER_GROUP, 32), (orc.PER_GROUP, 128)]:
        for qmin, qmax, sym in [(-127, 127, True), (-7, 7, True), (0, 255, False), (0, 15, False)]:
            q, s, z = orc.quantize(x, qmin, qmax, sym, gran, group)
            rows, cols = x.shape
            r = np.arange(rows)[:, None]
            c = np.arange(cols)[None, :]
            sc = {orc.PER_TENSOR: 0 * r + 0 * c, orc.PER_ROW: r + 0 * c, orc.PER_COL: 0 * r + c,
                  orc.PER_GROUP: r * (cols // max(group, 1)) + c // max(group, 1)}[gran]
            ss = s[sc].astype(np.float64)
            err = np.abs(x.astype(np.float64) - ss * (q - z[sc]))
            unclipped = (q > qmin) & (q < qmax)
            assert np.all(err[unclipped] <= ss[unclipped] / 2 * (1 + 2.0 ** -20))
            # min-max scales never clip more than rounding at the extreme
            assert np.all(err <= ss / 2 * (1 + 2.0 ** -20) + 0)


def test_asymmetric_zero_exact_and_relu(orc):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((16, 64)).astype(np.float32) + 0.7
    x[:, 0] = 0.0
    q, s, z = orc.quantize(x, 0, 255, False, orc.PER_ROW)
    xh = orc.dequantize(q, s, z, orc.PER_ROW)
    assert np.all(q[:, 0] == z) and np.all(xh[:, 0] == 0.0)
    # non-negative (ReLU-like) data: the zero point is 0 ([CH11] 11.1.2)
    xr = np.abs(x)
    q2, s2, z2 = orc.quantize(xr, 0, 255, False, orc.PER_ROW)
    assert np.all(z2 == 0)
    assert np.all(s2 == (xr.max(axis=1) / np.float32(255)).astype(np.float32))


def test_degenerate_scope_scale_one(orc):
    x = np.zeros((3, 8), np.float32)
    x[1] = 1.0
    q, s, z = orc.quantize(x, -127, 127, True, orc.PER_ROW)
    assert s[0] == 1.0 and s[2] == 1.0 and np.all(q[0] == 0)
    q, s, z = orc.quantize(x, 0, 15, False, orc.PER_ROW)
    assert s[0] == 1.0 and z[0] == 0
    # an fp16 scale that underflows to zero is stored as 1
    q, s, z = orc.quantize(np.full((1, 4), 1e-9, np.float32), -7, 7, True, orc.PER_ROW,
                           scale_f16=True)
    assert s[0] == 1.0 and np.all(q == 0)


def test_scale_f16_is_the_stored_scale(orc):
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((8, 256)) * 0.02).astype(np.float32)
    q, s, z = orc.quantize(x, -7, 7, True, orc.PER_GROUP, 128, scale_f16=True)
    # group maxima by numpy (8 rows x 2 groups of 128), binary32 division by 7,
    # then numpy's nearest-even binary16 rounding
    gmax = np.abs(x).reshape(8, 2, 128).max(axis=2).reshape(-1)
    s32 = (gmax / np.float32(7)).astype(np.float32)
    np.testing.assert_array_equal(s, s32.astype(np.float16).astype(np.float32))
    sc = np.arange(8)[:, None] * 2 + np.arange(256)[None, :] // 128
    expect = np.clip(np.rint(x / s[sc]), -7, 7)
    np.testing.assert_array_equal(q, expect)


@pytest.mark.parametrize("shape", [(1, 1), (5, 24), (37, 512)])
def test_absmax_every_granularity_against_numpy(orc, shape):
    """orc_absmax against numpy's max of |x| along the scope's axes: per tensor,
    per row (axis 1), per column (axis 0) and per group of g consecutive
    elements of a row ([L19] section 4; [CH11] table 11-1; [CH11] 11.4.5
    step 1 for the channel maxima)."""
    rows, cols = shape
    rng = np.random.default_rng(rows * 31 + cols)
    x = rng.standard_normal((rows, cols)).astype(np.float32)
    x[rows // 2, cols // 2] = -1000.0                      # a negative extreme: |x| must be taken
    a = np.abs(x)
    np.testing.assert_array_equal(orc.absmax(x, orc.PER_TENSOR), np.array([a.max()], np.float32))
    np.testing.assert_array_equal(orc.absmax(x, orc.PER_ROW), a.max(axis=1))
    np.testing.assert_array_equal(orc.absmax(x, orc.PER_COL), a.max(axis=0))
    for g in (1, 8, cols):
        if cols % g == 0:
            np.testing.assert_array_equal(orc.absmax(x, orc.PER_GROUP, g),
                                          a.reshape(rows, cols // g, g).max(axis=2).reshape(-1))
    assert orc.absmax(np.zeros((3, 8), np.float32), orc.PER_ROW).tolist() == [0.0, 0.0, 0.0]


def test_granularity_scopes(orc):
    """Per-row / per-col / per-group scales equal the per-tensor scale of the
    corresponding slice ([L19] section 4; [CH11] table 11-1)."""
    rng = np.random.default_rng(6)
    x = rng.standard_normal((6, 64)).astype(np.float32)
    _, s_row, _ = orc.quantize(x, -127, 127, True, orc.PER_ROW)
    _, s_col, _ = orc.quantize(x, -127, 127, True, orc.PER_COL)
    _, s_grp, _ = orc.quantize(x, 0, 255, False, orc.PER_GROUP, 16)
    for r in range(6):
        assert s_row[r] == orc.quantize(x[r:r + 1], -127, 127, True, orc.PER_TENSOR)[1][0]
        for j in range(4):
            sl = x[r:r + 1, 16 * j:16 * (j + 1)]
            assert s_grp[r * 4 + j] == orc.quantize(sl, 0, 255, False, orc.PER_TENSOR)[1][0]
    for c in range(64):
        assert s_col[c] == orc.quantize(x[:, c:c + 1].T.copy(), -127, 127, True, orc.PER_TENSOR)[1][0]


def test_percentile_nearest_rank(orc):
    rng = np.random.default_rng(7)
    v = rng.permutation(np.arange(1, 1001)).astype(np.float32)
    v[::2] *= -1
    q, s, _ = orc.quantize(v, -127, 127, True, orc.PER_TENSOR, percentile=99.9)
    assert s[0] == np.float32(999) / np.float32(127)
    assert q.max() == 127 and q.min() == -127
    _, s100, _ = orc.quantize(v, -127, 127, True, orc.PER_TENSOR, percentile=100.0)
    assert s100[0] == np.float32(1000) / np.float32(127)
    for n in [1, 7, 1000, 4097]:
        x = rng.standard_normal(n).astype(np.float32)
        _, s, _ = orc.quantize(x, -127, 127, True, orc.PER_TENSOR, percentile=99.9)
        srt = np.sort(np.abs(x))
        k = max(1, min(n, math.ceil(n * 99.9 / 100.0)))   # binary64 percentile
        assert s[0] == srt[k - 1] / np.float32(127)
        assert orc.percentile_rank(n, 99.9) == k


def test_noise_variance_delta_sq_over_12(orc):
    """Uniform quantization noise has variance ~ Delta^2/12 ([CH11] 11.1.5)."""
    rng = np.random.default_rng(8)
    x = rng.uniform(-1, 1, 1 << 20).astype(np.float32)
    q, s, z = orc.quantize(x, -127, 127, True, orc.PER_TENSOR)
    err = x.astype(np.float64) - float(s[0]) * q.ravel()
    var = err.var()
    assert abs(var / (float(s[0]) ** 2 / 12) - 1) < 0.02


# ------------------------------------------------------------- formats
def test_bf16_rounding_matches_torch(orc):
    rng = np.random.default_rng(9)
    v = np.concatenate([
        rng.standard_normal(200000).astype(np.float32),
        (rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32)).view(np.float32),
        np.array([0x3F808000, 0x3F818000, 0x7F7FFFFF, 0x00008000, 0x80018000],
                 np.uint32).view(np.float32)])
    v = v[np.isfinite(v)]
    ours = orc.round_bf16(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(ours.view(np.uint32), ref.view(np.uint32))


def test_f16_rounding_matches_numpy_and_saturates(orc):
    rng = np.random.default_rng(10)
    v = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10.0 ** rng.integers(-9, 5, 100000),
                        np.array([65504.0, 65519.0, 65520.0, 1e6, -1e6, 2.0 ** -24, 2.0 ** -25, 3e-8],
                                 np.float32)]).astype(np.float32)
    ours = orc.round_f16(v)
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).astype(np.float32)
    ref = np.where(np.isinf(ref), np.sign(ref) * 65504.0, ref).astype(np.float32)
    np.testing.assert_array_equal(ours, ref)


def test_nibble_packing(orc):
    packed = orc.pack_nibbles(np.array([1, -1, 7, -7], np.int32))
    assert list(packed) == [0xF1, 0x97]
    rng = np.random.default_rng(11)
    q = rng.integers(-7, 8, 1001).astype(np.int32)
    np.testing.assert_array_equal(orc.unpack_nibbles(orc.pack_nibbles(q), q.size, True), q)
    u = rng.integers(0, 16, 1000).astype(np.int32)
    np.testing.assert_array_equal(orc.unpack_nibbles(orc.pack_nibbles(u), u.size, False), u)


# ------------------------------------------------------------- group metadata
def test_metadata_counts(orc):
    g = read_golden("metadata_overhead.txt")
    dout, din, grp, ngroups = (int(v) for v in g["llama7b_attn"])
    assert orc.num_scopes(orc.PER_GROUP, dout, din, grp) == ngroups == dout * din // grp
    assert orc.num_scopes(orc.PER_GROUP, 8192, 28672, 128) == 1835008
    # fp16 scale per group over 4-bit codes
    frac128 = 16 / (128 * 4)
    frac32 = 16 / (32 * 4)
    frac128_z = (16 + 4) / (128 * 4)
    assert g["overhead_g128_lo"][0] <= frac128 <= g["overhead_g128_hi"][0]
    assert g["overhead_g128_lo"][0] <= frac128_z <= g["overhead_g128_hi"][0]
    assert g["overhead_g32_lo"][0] <= frac32 <= g["overhead_g32_hi"][0]
    # the oracle writes exactly that many scales on a smaller grouped weight
    x = np.ones((64, 512), np.float32)
    _, s, _ = orc.quantize(x, -7, 7, True, orc.PER_GROUP, 128)
    assert s.size == 64 * 512 // 128


# ------------------------------------------------------------- W8A8 / W4A16
def test_w8a8_integer_sums_brute_force(orc):
    rng = np.random.default_rng(12)
    for M, N, K in [(1, 1, 1), (3, 5, 7), (4, 3, 33)]:
        qx = rng.integers(-127, 128, (M, K)).astype(np.int8)
        qw = rng.integers(-127, 128, (N, K)).astype(np.int8)
        acc = orc.w8a8_acc(qx, qw)
        for m in range(M):
            for n in range(N):
                assert acc[m, n] == sum(int(qx[m, k]) * int(qw[n, k]) for k in range(K))
    # extreme: all +-127 over K=1040 reaches 16129*1040
    K = 1040
    acc = orc.w8a8_acc(np.full((1, K), 127, np.int8), np.full((2, K), -127, np.int8))
    assert acc[0, 0] == -16129 * K


def test_w8a8_error_identity(orc):
    """y^ - y = dW x + W dx + dW dx ([QDC] section 1, eq. 2) with the oracle's
    quantized path for y^ (per-token X, per-output-channel W)."""
    rng = np.random.default_rng(13)
    M, N, K = 5, 7, 64
    x = rng.standard_normal((M, K)).astype(np.float32)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    qx, sx, _ = orc.quantize(x, -127, 127, True, orc.PER_ROW)
    qw, sw, _ = orc.quantize(w, -127, 127, True, orc.PER_ROW)
    yhat = orc.w8a8_out(orc.w8a8_acc(qx, qw), sx, sw)
    X = x.astype(np.float64)
    W = w.astype(np.float64)
    dX = sx.astype(np.float64)[:, None] * qx - X
    dW = sw.astype(np.float64)[:, None] * qw - W
    y = X @ W.T
    rhs = dX @ W.T + X @ dW.T + dX @ dW.T
    np.testing.assert_allclose(yhat - y, rhs, rtol=1e-9, atol=1e-12)


def test_w4_dequant_bits(orc):
    rng = np.random.default_rng(14)
    N, K, g = 16, 256, 128
    w = (rng.standard_normal((N, K)) * 0.015).astype(np.float32)
    q, s, z = orc.quantize(w, 0, 15, False, orc.PER_GROUP, g, scale_f16=True)
    what = orc.w4_dequant(q, s, z, g)
    sc = np.arange(N)[:, None] * (K // g) + np.arange(K)[None, :] // g
    prod = (s[sc] * (q - z[sc]).astype(np.float32)).astype(np.float32)
    # the product of an fp16 scale and a 5-bit integer is exact in binary32
    np.testing.assert_array_equal(prod.astype(np.float64), s[sc].astype(np.float64) * (q - z[sc]))
    ref = torch.from_numpy(prod).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(what, ref)
    x = rng.standard_normal((3, K)).astype(np.float32)
    np.testing.assert_allclose(orc.matmul_f64(x, what), x.astype(np.float64) @ what.T.astype(np.float64),
                               rtol=1e-12, atol=1e-12)


def test_matmul_f64_orientation(orc):
    x = np.array([[1, 2, 3]], np.float32)
    w = np.array([[1, 0, 0], [0, 0, 1]], np.float32)
    np.testing.assert_array_equal(orc.matmul_f64(x, w), [[1.0, 3.0]])


# ------------------------------------------------------------- SmoothQuant
def test_smooth_factor_closed_forms(orc):
    rng = np.random.default_rng(15)
    mx = rng.uniform(0.1, 60, 257).astype(np.float32)
    mw = rng.uniform(0.001, 0.1, 257).astype(np.float32)
    np.testing.assert_array_equal(orc.smooth_factors(mx, mw, 1.0), mx)
    np.testing.assert_array_equal(orc.smooth_factors(mx, mw, 0.0),
                                  (1.0 / mw.astype(np.float64)).astype(np.float32))
    np.testing.assert_array_equal(orc.smooth_factors(mx, mw, 0.5), np.sqrt(mx) / np.sqrt(mw))
    a7 = orc.smooth_factors(mx, mw, 0.7)
    ref = (mx.astype(np.float64) ** np.float64(np.float32(0.7))
           / mw.astype(np.float64) ** (1 - np.float64(np.float32(0.7))))
    np.testing.assert_allclose(a7, ref, rtol=2 ** -23)
    z = orc.smooth_factors(np.array([0.0, 1.0], np.float32), np.array([1.0, 0.0], np.float32), 0.5)
    assert list(z) == [1.0, 1.0]


def test_smoothing_equivalence_and_orientation(orc):
    """XW = (X diag(s)^-1)(diag(s)W) ([QDC] 2.3; [CH11] 11.4.2); after
    smoothing with alpha=0.5 the channel maxima of X and W match."""
    rng = np.random.default_rng(16)
    M, N, K = 32, 24, 96
    x = rng.standard_normal((M, K)).astype(np.float32)
    x[:, [4, 50]] *= 40
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    s = orc.smooth_factors(orc.absmax(x, orc.PER_COL), orc.absmax(w, orc.PER_COL), 0.5)
    xs = x / s[None, :]
    ws = w * s[None, :]
    np.testing.assert_allclose(xs.astype(np.float64) @ ws.T.astype(np.float64),
                               x.astype(np.float64) @ w.T.astype(np.float64), rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(np.abs(xs).max(0), np.abs(ws).max(0), rtol=1e-5)
    # quantizing with divide-mode smoothing == quantizing the pre-divided X
    a = orc.quantize(x, -127, 127, True, orc.PER_ROW, smooth=s, smooth_mode=orc.SMOOTH_DIVIDE)
    b = orc.quantize(xs, -127, 127, True, orc.PER_ROW)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)
    c = orc.quantize(x, -127, 127, True, orc.PER_ROW, smooth=s, smooth_mode=orc.SMOOTH_MULTIPLY)
    d = orc.quantize(x * s[None, :], -127, 127, True, orc.PER_ROW)
    for u, v in zip(c, d):
        np.testing.assert_array_equal(u, v)
    # per-token quantization error of X shrinks after smoothing
    def qerr(v):
        q, sc, _ = orc.quantize(v, -127, 127, True, orc.PER_ROW)
        return np.abs(sc[:, None] * q - v).mean() / np.abs(v).mean()
    assert qerr(xs) < qerr(x)


def test_oracle_rejects_undefined_arguments(orc):
    x = np.ones((2, 10), np.float32)
    with pytest.raises(ValueError):
        orc.quantize(x, -127, 127, True, orc.PER_GROUP, 3)      # 10 % 3 != 0
    with pytest.raises(ValueError):
        orc.quantize(x, 0, 255, False, orc.PER_TENSOR, percentile=99.9)  # percentile is symmetric
    with pytest.raises(ValueError):
        orc.quantize(x, -128, 127, True, orc.PER_TENSOR)          # symmetric needs qmin = -qmax


# ------------------------------------------------------------- W4A8 (group-wise INT4 x per-token INT8)
def test_w4a8_group_sums_brute_force(orc):
    """Exact per-group integer sums by plain Python loops ([CH11] 11.4.5
    step 6: integer products summed exactly; groups of g consecutive k)."""
    rng = np.random.default_rng(21)
    M, N, K, g = 3, 5, 64, 16
    qx = rng.integers(-127, 128, (M, K)).astype(np.int8)
    q = rng.integers(0, 16, (N, K)).astype(np.int32)
    z = rng.integers(0, 16, (N, K // g)).astype(np.int32)
    acc = orc.w4a8_acc(qx, q, z.reshape(-1), g)
    assert acc.shape == (K // g, M, N)
    for gi in range(K // g):
        for m in range(M):
            for n in range(N):
                want = sum(int(qx[m, k]) * (int(q[n, k]) - int(z[n, gi])) for k in range(gi * g, (gi + 1) * g))
                assert acc[gi, m, n] == want
    # extremes: 127 * 15 * 128 per group
    qx = np.full((1, 128), 127, np.int8)
    q = np.full((1, 128), 15, np.int32)
    assert orc.w4a8_acc(qx, q, np.zeros(1, np.int32), 128)[0, 0, 0] == 127 * 15 * 128
    # symmetric codes: z = NULL means z = 0
    qx = rng.integers(-127, 128, (2, 32)).astype(np.int8)
    q = rng.integers(-7, 8, (4, 32)).astype(np.int32)
    np.testing.assert_array_equal(orc.w4a8_acc(qx, q, None, 32)[0], qx.astype(np.int64) @ q.T.astype(np.int64))


def test_w4a8_one_group_is_w8a8(orc):
    """With a single group per row and z = 0 the W4A8 layer is the W8A8 layer
    with per-output-channel scales ([L19] section 6): same sums, same y."""
    rng = np.random.default_rng(22)
    M, N, K = 4, 6, 96
    qx = rng.integers(-127, 128, (M, K)).astype(np.int8)
    q = rng.integers(-7, 8, (N, K)).astype(np.int32)
    sx = rng.uniform(1e-3, 1e-1, M).astype(np.float32)
    s = rng.uniform(1e-3, 1e-1, N).astype(np.float32)
    acc = orc.w4a8_acc(qx, q, None, K)
    acc8 = orc.w8a8_acc(qx, q.astype(np.int8))
    np.testing.assert_array_equal(acc[0], acc8)
    np.testing.assert_array_equal(orc.w4a8_out(acc, sx, s), orc.w8a8_out(acc8, sx, s))


def test_w4a8_error_identity(orc):
    """y^ - y = dW x + W dx + dW dx ([QDC] section 1, the error of y = W x when
    both operands are quantized): the oracle's W4A8 output is the product of
    the dequantized operands x^ = sx qx (per token) and w^ = s (q - z) (per
    group), with the orientation y[m,n] = sum_k x[m,k] w[n,k]."""
    rng = np.random.default_rng(23)
    M, N, K, g = 6, 10, 256, 64
    x = rng.standard_normal((M, K)).astype(np.float32)
    x[:, 7] *= 30.0
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    qx, sx, _ = orc.quantize(x, -127, 127, True, orc.PER_ROW)
    q, s, z = orc.quantize(w, 0, 15, False, orc.PER_GROUP, g, scale_f16=True)
    yq = orc.w4a8_out(orc.w4a8_acc(qx.astype(np.int8), q, z, g), sx, s)
    xh = sx.astype(np.float64)[:, None] * qx
    sc = np.repeat(s.reshape(N, K // g).astype(np.float64), g, axis=1)
    zc = np.repeat(z.reshape(N, K // g), g, axis=1)
    wh = sc * (q - zc)
    x64, w64 = x.astype(np.float64), w.astype(np.float64)
    dx, dw = xh - x64, wh - w64
    y = x64 @ w64.T
    lhs = yq - y
    rhs = x64 @ dw.T + dx @ w64.T + dx @ dw.T
    np.testing.assert_allclose(lhs, rhs, rtol=0, atol=1e-12 * np.abs(y).max())
    np.testing.assert_allclose(yq, xh @ wh.T, rtol=1e-13, atol=1e-15)
    # a weight row whose codes all equal their zero point contributes exactly 0
    q2 = q.copy()
    q2[3] = np.repeat(z.reshape(N, K // g)[3], g)
    assert np.all(orc.w4a8_out(orc.w4a8_acc(qx.astype(np.int8), q2, z, g), sx, s)[:, 3] == 0.0)


# ------------------------------------------------------------- SmoothQuant calibration
def test_channel_absmax_update_is_the_max_over_all_batches(orc):
    """Calibration keeps max|X_j| over every batch seen ([CH11] 11.4.5 steps
    1-2): the running maxima equal numpy's max over the concatenated batches."""
    rng = np.random.default_rng(31)
    batches = [rng.standard_normal((n, 48)).astype(np.float32) * rng.uniform(0.5, 3) for n in (3, 7, 1, 12)]
    batches[2][0, 5] = -900.0
    run = np.zeros(48, np.float32)
    for b in batches:
        orc.channel_absmax_update(b, run)
    np.testing.assert_array_equal(run, np.abs(np.concatenate(batches)).max(axis=0))


def test_fold_layernorm_equivalence(orc):
    """LN(x) diag(s)^-1 is the LayerNorm with gamma / s and beta / s ([CH11]
    11.4.4: the smoothing is absorbed by the previous LayerNorm's gamma): the
    folded parameters are binary32 quotients, and the folded LayerNorm equals
    the unfolded one divided by s up to those roundings."""
    rng = np.random.default_rng(32)
    K = 256
    gamma = rng.uniform(0.5, 1.5, K).astype(np.float32)
    beta = rng.uniform(-0.2, 0.2, K).astype(np.float32)
    s = rng.uniform(0.1, 20.0, K).astype(np.float32)
    g2, b2 = orc.fold_layernorm(gamma, beta, s)
    np.testing.assert_array_equal(g2, gamma / s)           # IEEE binary32 division
    np.testing.assert_array_equal(b2, beta / s)
    x = rng.standard_normal((5, K)) * 3 + 1
    mu = x.mean(axis=1, keepdims=True)
    sd = np.sqrt(x.var(axis=1, keepdims=True) + 1e-5)
    ln = (x - mu) / sd * gamma + beta
    ln2 = (x - mu) / sd * g2.astype(np.float64) + b2.astype(np.float64)
    np.testing.assert_allclose(ln2, ln / s, rtol=2e-7, atol=1e-7 * np.abs(ln / s).max())
    g3, b3 = orc.fold_layernorm(gamma, None, s)
    assert b3 is None and np.array_equal(g3, g2)


def test_quant_error_statistics(orc):
    """Sum of squared errors, sum of squares and max error of x' - s(q - z) in
    binary64, against numpy on the same dequantized values; a value on the
    grid has no error."""
    rng = np.random.default_rng(33)
    x = rng.standard_normal((6, 40)).astype(np.float32)
    sm = rng.uniform(0.5, 2.0, 40).astype(np.float32)
    for mode, xs in ((orc.SMOOTH_NONE, x), (orc.SMOOTH_DIVIDE, x / sm), (orc.SMOOTH_MULTIPLY, x * sm)):
        q, s, z = orc.quantize(x, 0, 255, False, orc.PER_GROUP, 8, smooth=sm if mode else None, smooth_mode=mode)
        e = orc.quant_error(x, q, s, z, orc.PER_GROUP, 8, smooth=sm if mode else None, smooth_mode=mode)
        sc = np.repeat(s.reshape(6, 5), 8, axis=1)
        zc = np.repeat(z.reshape(6, 5), 8, axis=1)
        xh = (sc * (q - zc).astype(np.float32)).astype(np.float32)
        d = xs.astype(np.float64) - xh.astype(np.float64)
        np.testing.assert_allclose(e[0], (d * d).sum(), rtol=1e-12)
        np.testing.assert_allclose(e[1], (xs.astype(np.float64) ** 2).sum(), rtol=1e-12)
        assert e[2] == np.abs(d).max()
    g = np.array([[0.5, -1.0, 2.0, 0.25]], np.float32)      # multiples of s = 0.25: exact codes
    q, s, z = orc.quantize(g, -8, 8, True, orc.PER_TENSOR)
    assert list(orc.quant_error(g, q, s, z, orc.PER_TENSOR)) == [0.0, float((g.astype(np.float64) ** 2).sum()), 0.0]


def _outlier_layer(seed, M=64, N=96, K=256, n_out=4):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32)
    cols = np.sort(rng.choice(K, n_out, replace=False))
    x[:, cols] *= rng.uniform(20, 60, n_out).astype(np.float32)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    return x, w, cols


def test_smoothquant_alpha_table(orc):
    """[CH11] table 11-4: raising alpha moves quantization difficulty from the
    activations to the weights -- the INT8 error of the smoothed activations
    (per token) falls and that of the smoothed weights (per output channel)
    rises, alpha = 0.3 < 0.5 < 0.7.  Relative Frobenius errors on inputs with
    outlier channels."""
    x, w, _ = _outlier_layer(34, M=128, N=128, K=512, n_out=6)
    xmax, wmax = orc.absmax(x, orc.PER_COL), orc.absmax(w, orc.PER_COL)
    act, wgt = [], []
    for alpha in (0.3, 0.5, 0.7):
        s = orc.smooth_factors(xmax, wmax, alpha)
        qx, sx, zx = orc.quantize(x, -127, 127, True, orc.PER_ROW, smooth=s, smooth_mode=orc.SMOOTH_DIVIDE)
        qw, sw, zw = orc.quantize(w, -127, 127, True, orc.PER_ROW, smooth=s, smooth_mode=orc.SMOOTH_MULTIPLY)
        ea = orc.quant_error(x, qx, sx, None, orc.PER_ROW, smooth=s, smooth_mode=orc.SMOOTH_DIVIDE)
        ew = orc.quant_error(w, qw, sw, None, orc.PER_ROW, smooth=s, smooth_mode=orc.SMOOTH_MULTIPLY)
        act.append(np.sqrt(ea[0] / ea[1]))
        wgt.append(np.sqrt(ew[0] / ew[1]))
    assert act[0] > act[1] > act[2]
    assert wgt[0] < wgt[1] < wgt[2]


# ------------------------------------------------------------- LLM.int8()
def test_llmint8_outlier_channels_by_numpy(orc):
    x, _, cols = _outlier_layer(41)
    got = orc.llmint8_outlier_cols(x, 6.0)
    np.testing.assert_array_equal(got, np.nonzero(np.abs(x).max(axis=0) > 6.0)[0])
    assert set(cols).issubset(set(got.tolist()))
    assert orc.llmint8_outlier_cols(x, 1e9).size == 0
    np.testing.assert_array_equal(orc.llmint8_outlier_cols(x, -1.0), np.arange(x.shape[1]))


def test_llmint8_decomposition(orc):
    """XW = X_normal W + X_outlier W ([L19] section 10): with no outlier
    channel the layer is the W8A8 layer; with outliers the INT8 part sees
    zeros in those channels, the 16-bit part is an fp64 product with the
    dequantized weight columns, and the result beats plain per-token INT8 on
    outlier inputs."""
    x, w, _ = _outlier_layer(42)
    qw, sw, _ = orc.quantize(w, -127, 127, True, orc.PER_ROW)
    qw8 = qw.astype(np.int8)
    cols, qx, sx, acc, y = orc.llmint8(x, qw8, sw, 1e9)          # no outliers
    assert cols.size == 0
    qx0, sx0, _ = orc.quantize(x, -127, 127, True, orc.PER_ROW)
    np.testing.assert_array_equal(qx, qx0)
    np.testing.assert_array_equal(y, orc.w8a8_out(orc.w8a8_acc(qx0.astype(np.int8), qw8), sx0, sw))
    cols, qx, sx, acc, y = orc.llmint8(x, qw8, sw, 6.0)
    assert cols.size >= 4 and np.all(qx[:, cols] == 0)
    normal = np.setdiff1d(np.arange(x.shape[1]), cols)
    np.testing.assert_array_equal(sx, (np.abs(x[:, normal]).max(axis=1) / np.float32(127)).astype(np.float32))
    wh = sw.astype(np.float64)[:, None] * qw                       # dequantized weight
    xh = x.astype(np.float64).copy()
    xh[:, normal] = sx.astype(np.float64)[:, None] * qx[:, normal]
    np.testing.assert_allclose(y, xh @ wh.T, rtol=1e-12, atol=1e-14)
    exact = x.astype(np.float64) @ w.astype(np.float64).T
    y8 = orc.w8a8_out(orc.w8a8_acc(qx0.astype(np.int8), qw8), sx0, sw)
    assert np.linalg.norm(y - exact) < 0.5 * np.linalg.norm(y8 - exact)


# ------------------------------------------------------------- KV cache
def test_kv_cache_reference_scopes_and_window(orc):
    """[CH11] 11.6.3-11.6.5: K quantized per channel over each group of G
    tokens, V per token (per head), the most recent tokens kept in 16-bit;
    groups are quantized once they have left the window.  Scales against
    numpy min-max, codes in range, the s/2 bound, and exact passthrough."""
    rng = np.random.default_rng(51)
    T, C, D, G, R, bits = 77, 32, 8, 16, 20, 4
    k = rng.standard_normal((T, C)).astype(np.float32)
    k[:, 3] *= 30.0                                                # a K outlier channel
    v = rng.standard_normal((T, C)).astype(np.float32)
    r = orc.kv_cache_reference(k, v, G, R, D, bits)
    assert r["tq"] == 48                                           # 16 * floor((77 - 20) / 16)
    qmax = 15
    for gi in range(3):
        blk = k[gi * G:(gi + 1) * G]
        hi = np.maximum(blk.max(axis=0), 0)
        lo = np.minimum(blk.min(axis=0), 0)
        np.testing.assert_array_equal(r["k_scale"][gi], ((hi - lo) / np.float32(qmax)).astype(np.float32))
    vb = v[:48].reshape(48, C // D, D)
    hi = np.maximum(vb.max(axis=2), 0)
    lo = np.minimum(vb.min(axis=2), 0)
    np.testing.assert_array_equal(r["v_scale"], ((hi - lo) / np.float32(qmax)).astype(np.float32))
    assert r["k_codes"].min() >= 0 and r["k_codes"].max() <= qmax
    assert r["v_codes"].min() >= 0 and r["v_codes"].max() <= qmax
    ks = np.repeat(r["k_scale"], G, axis=0)
    assert np.all(np.abs(r["k_hat"][:48] - k[:48]) <= ks / 2 * (1 + 1e-6))
    vs = np.repeat(r["v_scale"], D, axis=1)
    assert np.all(np.abs(r["v_hat"][:48] - v[:48]) <= vs / 2 * (1 + 1e-6))
    np.testing.assert_array_equal(r["k_hat"][48:], k[48:])
    np.testing.assert_array_equal(r["v_hat"][48:], v[48:])
    # inside the window nothing is quantized; one more group once it has left
    assert orc.kv_cache_reference(k[:R], v[:R], G, R, D, bits)["tq"] == 0
    assert orc.kv_cache_reference(k[:R + G - 1], v[:R + G - 1], G, R, D, bits)["tq"] == 0
    assert orc.kv_cache_reference(k[:R + G], v[:R + G], G, R, D, bits)["tq"] == G
