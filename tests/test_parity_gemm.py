"""GPU parity of the two quantized linear-layer paths against the oracle.

W8A8: INT32 sums bit-exact (acc_out), outputs within GEMM_REL_TOL of the
binary64 oracle sx*sw*acc.  W4A16: the packed blob dequantizes to the
oracle's w^ = bf16(fl(s (q - z))) and outputs are within GEMM_REL_TOL of the
binary64 product with that w^."""
import numpy as np
import pytest
import torch

import oracle
from activation_quantization_quantize_b300 import inputs, qlin
from helpers import GEMM_REL_TOL, codes_to_int, host_f32, oracle_quantize, rel_err, rel_err_out, scales_f32

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------------ W8A8
@pytest.fixture(params=["pair", "tc1"])
def w8_kernel(request, monkeypatch):
    """Each W8A8 case runs on both tensor-core kernels: the CTA-pair kernel
    (the default) and the single-CTA kernel."""
    monkeypatch.setenv("QLIN_W8A8_KERNEL", request.param)
    return request.param


def w8a8_run(x_dev, w_dev, out_dtype=torch.float32, smooth=None):
    """Quantize X per token (optionally smoothed) and W per output channel on
    the GPU, run the GEMM with acc_out; return device results."""
    M, K = x_dev.shape
    N = w_dev.shape[0]
    px = qlin.make_params("s8", "row", smooth_mode=qlin.QLIN_SMOOTH_DIVIDE if smooth is not None else 0)
    pw = qlin.make_params("s8", "row", smooth_mode=qlin.QLIN_SMOOTH_MULTIPLY if smooth is not None else 0)
    qx, sx, _ = qlin.quantize(x_dev, px, smooth=smooth)
    qw, sw, _ = qlin.quantize(w_dev, pw, smooth=smooth)
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    y = qlin.gemm_w8a8(qx, sx, qw, sw, out_dtype=out_dtype, acc_out=acc)
    torch.cuda.synchronize()
    return qx, sx, qw, sw, acc, y


def test_w8a8_tiny_config(w8_kernel):
    """8x128x256 fp32 with outlier channels 3 and 77, fp32 epilogue."""
    cfg = inputs.w8a8_tiny()
    xd = torch.from_numpy(cfg.x).cuda()
    wd = torch.from_numpy(cfg.w).cuda()
    qx, sx, qw, sw, acc, y = w8a8_run(xd, wd, torch.float32)
    p = qlin.make_params("s8", "row")
    qxo, sxo, _ = oracle_quantize(cfg.x, p)
    qwo, swo, _ = oracle_quantize(cfg.w, p)
    np.testing.assert_array_equal(codes_to_int(qx, p, 8, 256), qxo)
    np.testing.assert_array_equal(codes_to_int(qw, p, 128, 256), qwo)
    np.testing.assert_array_equal(sx.cpu().numpy().view(np.uint32), sxo.view(np.uint32))
    acco = oracle.w8a8_acc(qxo, qwo)
    np.testing.assert_array_equal(acc.cpu().numpy(), acco)
    yo = oracle.w8a8_out(acco, sxo, swo)
    assert rel_err(y.cpu().numpy(), yo) < 1e-6            # binary32 epilogue, no bf16 rounding
    # the five-element page-5 vector through the GPU quantizer, per tensor
    v = torch.from_numpy(cfg.vec5.reshape(1, 5).repeat(8, 0)[:1, :].copy())
    v8 = torch.zeros((1, 8), dtype=torch.float32)
    v8[0, :5] = v[0]
    q, s, _ = qlin.quantize(v8.cuda(), qlin.make_params("s8", "tensor"))
    assert list(q.cpu().numpy()[0, :5]) == [30, -73, 127, -48, 103]
    assert int(s.cpu().numpy().view(np.uint32)[0]) == 0x3C877551


@pytest.mark.parametrize("M,N,K", [(1, 1, 16), (3, 5, 32), (17, 33, 80), (130, 129, 208), (64, 256, 1040),
                                   (255, 384, 4096), (128, 128, 2048 + 16)])
def test_w8a8_ragged_exact(M, N, K, w8_kernel):
    rng = np.random.default_rng(M * 1000 + N + K)
    qx = torch.from_numpy(rng.integers(-127, 128, (M, K)).astype(np.int8)).cuda()
    qw = torch.from_numpy(rng.integers(-127, 128, (N, K)).astype(np.int8)).cuda()
    sx = torch.from_numpy(rng.uniform(0.001, 0.1, M).astype(np.float32)).cuda()
    sw = torch.from_numpy(rng.uniform(0.001, 0.1, N).astype(np.float32)).cuda()
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    y = qlin.gemm_w8a8(qx, sx, qw, sw, out_dtype=torch.bfloat16, acc_out=acc)
    acco = oracle.w8a8_acc(qx.cpu().numpy(), qw.cpu().numpy())
    np.testing.assert_array_equal(acc.cpu().numpy(), acco)
    yo = oracle.w8a8_out(acco, sx.cpu().numpy(), sw.cpu().numpy())
    assert rel_err_out(host_f32(y), yo) < GEMM_REL_TOL
    y32 = qlin.gemm_w8a8(qx, sx, qw, sw, out_dtype=torch.float32)
    assert rel_err(y32.cpu().numpy(), yo) < GEMM_REL_TOL    # binary32 output: the plain bound


@pytest.mark.parametrize("K", [1024, 1040, 4096, 28672])
def test_w8a8_extreme_sums(K, w8_kernel):
    """All codes +-127: partial sums reach 16129*K (beyond 2^24 for K > 1040)."""
    M, N = 128, 256
    qx = torch.full((M, K), 127, dtype=torch.int8, device="cuda")
    qx[1::2] = -127
    qw = torch.full((N, K), 127, dtype=torch.int8, device="cuda")
    qw[:, ::3] = -127
    sx = torch.ones(M, device="cuda")
    sw = torch.ones(N, device="cuda")
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    qlin.gemm_w8a8(qx, sx, qw, sw, out_dtype=torch.float32, acc_out=acc)
    acco = oracle.w8a8_acc(qx[:2].cpu().numpy(), qw.cpu().numpy())
    np.testing.assert_array_equal(acc[:2].cpu().numpy(), acco)
    np.testing.assert_array_equal(acc[2:4].cpu().numpy(), acco)


@pytest.mark.parametrize("smooth", [False, True])
def test_w8a8_prefill_config_sampled(smooth, w8_kernel):
    """2048 x 11008 x 4096 SmoothQuant-style prefill; oracle on 64 sampled rows."""
    x, w, _ = inputs.w8a8_prefill()
    xd, wd = x.cuda(), w.cuda()
    sm = None
    if smooth:
        sm = qlin.smooth_factors(qlin.absmax(xd, qlin.QLIN_PER_COL), qlin.absmax(wd, qlin.QLIN_PER_COL), 0.5)
    qx, sx, qw, sw, acc, y = w8a8_run(xd, wd, torch.bfloat16, smooth=sm)
    rows = np.sort(np.random.default_rng(5).choice(2048, 64, replace=False))
    xh = host_f32(x)[rows]
    wh = host_f32(w)
    smh = None if sm is None else sm.cpu().numpy()
    px = qlin.make_params("s8", "row", smooth_mode=qlin.QLIN_SMOOTH_DIVIDE if smooth else 0)
    pw = qlin.make_params("s8", "row", smooth_mode=qlin.QLIN_SMOOTH_MULTIPLY if smooth else 0)
    qxo, sxo, _ = oracle_quantize(xh, px, smooth=smh)
    qwo, swo, _ = oracle_quantize(wh, pw, smooth=smh)
    np.testing.assert_array_equal(codes_to_int(qx, px, 2048, 4096)[rows], qxo)
    np.testing.assert_array_equal(codes_to_int(qw, pw, 11008, 4096), qwo)
    acco = oracle.w8a8_acc(qxo, qwo)
    np.testing.assert_array_equal(acc.cpu().numpy()[rows], acco)
    yo = oracle.w8a8_out(acco, sxo, swo)
    assert rel_err_out(host_f32(y)[rows], yo) < GEMM_REL_TOL


def stratified_rows(M, tile, per_tile, seed):
    """per_tile distinct random rows from every tile of `tile` rows."""
    rng = np.random.default_rng(seed)
    rows = []
    for t0 in range(0, M, tile):
        n = min(tile, M - t0)
        rows.extend(t0 + rng.choice(n, min(per_tile, n), replace=False))
    return np.sort(np.array(rows))


@pytest.mark.parametrize("folded", [False, True])
def test_w8a8_downproj_sampled(folded, w8_kernel):
    """4096 x 8192 x 28672 with outlier channels: two random rows from every
    256-row tile, all 8192 columns (so every output tile, the split-K tail
    tiles of the last wave included, is checked).  folded: the step's input,
    X' = bf16(X / s) with the SmoothQuant factors (alpha = 0.5) folded into
    the previous layer and W smoothed offline (multiply mode), whose larger
    codes make the exact accumulation drain about once per tile."""
    x = inputs.downproj_activation(4096, outliers=True)
    w = inputs.downproj_weight()
    xd, wd = x.cuda(), w.cuda()
    del x, w
    sm = None
    if folded:
        sm = qlin.smooth_factors(qlin.absmax(xd, qlin.QLIN_PER_COL), qlin.absmax(wd, qlin.QLIN_PER_COL), 0.5)
        xd = (xd.float() / sm[None, :]).to(torch.bfloat16)
        pw = qlin.make_params("s8", "row", smooth_mode=qlin.QLIN_SMOOTH_MULTIPLY)
        qw, sw, _ = qlin.quantize(wd, pw, smooth=sm)
        qx, sx, _ = qlin.quantize(xd, qlin.make_params("s8", "row"))
        acc = torch.empty((4096, 8192), dtype=torch.int32, device="cuda")
        y = qlin.gemm_w8a8(qx, sx, qw, sw, out_dtype=torch.bfloat16, acc_out=acc)
        torch.cuda.synchronize()
    else:
        qx, sx, qw, sw, acc, y = w8a8_run(xd, wd, torch.bfloat16)
    rows = stratified_rows(4096, 256, 2, 6 + int(folded))
    acco = oracle.w8a8_acc(qx[torch.from_numpy(rows).cuda()].cpu().numpy(), qw.cpu().numpy())
    np.testing.assert_array_equal(acc.cpu().numpy()[rows], acco)
    yo = oracle.w8a8_out(acco, sx.cpu().numpy()[rows], sw.cpu().numpy())
    assert rel_err_out(host_f32(y)[rows], yo) < GEMM_REL_TOL
    assert qlin.qlin_device_error() == 0


# ------------------------------------------------------------------ W4A16
def w4_prepare(w_dev, group, asym):
    """Quantize W [N x K] group-wise to INT4 with fp16 scales and pack it."""
    N, K = w_dev.shape
    p = qlin.make_params("u4" if asym else "s4", "group", group=group, scale_f16=True)
    q, s, z = qlin.quantize(w_dev, p)
    packed, hdr = qlin.pack_w4(q, s, z, N, K, group)
    return p, q, s, z, packed, hdr


def w4_oracle_weight(q, s, z, p, N, K, group, rows=None):
    """Oracle dequantized weight w^ of the (optionally sampled) rows, from the
    device codes / scales / zero points."""
    if rows is not None:
        idx = torch.from_numpy(np.asarray(rows)).cuda()
        q = q[idx]
        s = s.reshape(N, K // group)[idx]
        z = None if z is None else z.reshape(N, K // group)[idx]
        N = len(rows)
    qi = codes_to_int(q, p, N, K)
    sf = scales_f32(s).reshape(-1)
    zi = None if z is None else z.cpu().numpy().reshape(-1)
    return oracle.w4_dequant(qi, sf, zi, group)


@pytest.mark.parametrize("asym", [False, True])
@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("M", [1, 3, 8, 16, 17, 64, 100])
def test_w4a16_small(asym, group, M):
    N, K = 256, 1024
    w = torch.from_numpy(inputs.normal((N, K), 0.02, 7)).to(torch.bfloat16).cuda()
    x = torch.from_numpy(inputs.normal((M, K), 1.0, 8)).to(torch.bfloat16).cuda()
    p, q, s, z, packed, hdr = w4_prepare(w, group, asym)
    y = qlin.gemm_w4a16(x, packed, hdr)
    # the quantized codes themselves match the oracle quantizer
    qo, so, zo = oracle_quantize(host_f32(w), p)
    np.testing.assert_array_equal(codes_to_int(q, p, N, K), qo)
    np.testing.assert_array_equal(scales_f32(s), so)
    what = w4_oracle_weight(q, s, z, p, N, K, group)
    yo = oracle.matmul_f64(host_f32(x), what)
    assert rel_err_out(host_f32(y), yo) < GEMM_REL_TOL


@pytest.mark.parametrize("M", [1, 4, 16])
def test_w4a16_decode_config(M):
    """4096 x 4096 symmetric INT4, g = 128, fp16 scales (131,072 groups)."""
    x, w = inputs.w4a16_decode(M)
    p, q, s, z, packed, hdr = w4_prepare(w.cuda(), 128, False)
    assert s.numel() == 131072
    y = qlin.gemm_w4a16(x.cuda(), packed, hdr)
    what = w4_oracle_weight(q, s, z, p, 4096, 4096, 128)
    yo = oracle.matmul_f64(host_f32(x), what)
    assert rel_err_out(host_f32(y), yo) < GEMM_REL_TOL


@pytest.mark.parametrize("M", [1, 8, 64, 256])
def test_w4a16_downproj_sampled(M):
    """8192 x 28672 asymmetric UINT4, g = 128: all tokens x 256 sampled output channels."""
    w = inputs.downproj_weight()
    x = inputs.downproj_activation(M)
    p, q, s, z, packed, hdr = w4_prepare(w.cuda(), 128, True)
    y = qlin.gemm_w4a16(x.cuda(), packed, hdr)
    rows = np.sort(np.random.default_rng(9).choice(8192, 256, replace=False))
    what = w4_oracle_weight(q, s, z, p, 8192, 28672, 128, rows=rows)
    yo = oracle.matmul_f64(host_f32(x), what)
    assert rel_err_out(host_f32(y)[:, rows], yo) < GEMM_REL_TOL


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (200, 300, 1056), (64, 512, 28672)])
def test_w8a8_tensor_core_matches_legacy_kernel(M, N, K, w8_kernel, monkeypatch):
    """The fp16-tensor-core kernel and the legacy mma.sync s8 kernel give the
    same INT32 sums and the same outputs."""
    rng = np.random.default_rng(M + N + K)
    qx = torch.from_numpy(rng.integers(-128, 128, (M, K)).astype(np.int8)).cuda()
    qw = torch.from_numpy(rng.integers(-127, 128, (N, K)).astype(np.int8)).cuda()
    sx = torch.from_numpy(rng.uniform(0.001, 0.1, M).astype(np.float32)).cuda()
    sw = torch.from_numpy(rng.uniform(0.001, 0.1, N).astype(np.float32)).cuda()
    a1 = torch.empty((M, N), dtype=torch.int32, device="cuda")
    a2 = torch.empty((M, N), dtype=torch.int32, device="cuda")
    y1 = qlin.gemm_w8a8(qx, sx, qw, sw, out_dtype=torch.float32, acc_out=a1)
    monkeypatch.setenv("QLIN_W8A8_KERNEL", "mma")
    y2 = qlin.gemm_w8a8(qx, sx, qw, sw, out_dtype=torch.float32, acc_out=a2)
    torch.cuda.synchronize()
    assert torch.equal(a1, a2)
    assert torch.equal(y1, y2)
    assert qlin.qlin_device_error() == 0


def test_w8a8_drain_boundary(w8_kernel):
    """Rows whose |code| sums cross the 2^24 / 128 drain threshold at different
    k-blocks: every row's sum stays exact."""
    M, N, K = 128, 256, 8192
    qx = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    for r in range(M):
        qx[r, : 64 * (r + 1)] = 127 if r % 2 == 0 else -128
    qw = torch.full((N, K), -127, dtype=torch.int8, device="cuda")
    qw[::2] = 127
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    qlin.gemm_w8a8(qx, torch.ones(M, device="cuda"), qw, torch.ones(N, device="cuda"), out_dtype=torch.float32,
                   acc_out=acc)
    acco = oracle.w8a8_acc(qx.cpu().numpy(), qw.cpu().numpy())
    np.testing.assert_array_equal(acc.cpu().numpy(), acco)


def test_w8a8_split_tail_tiles(w8_kernel):
    """2560 x 4096 x 1024: 160 tiles of 256 x 256, so the 12 tiles after the
    first 148 are cut into K parts whose INT32 sums are added by a second
    kernel; sampled rows of those tiles and of whole tiles stay exact."""
    M, N, K = 2560, 4096, 1024
    rng = np.random.default_rng(31)
    qx = torch.from_numpy(rng.integers(-127, 128, (M, K)).astype(np.int8)).cuda()
    qw = torch.from_numpy(rng.integers(-127, 128, (N, K)).astype(np.int8)).cuda()
    sx = torch.from_numpy(rng.uniform(0.001, 0.1, M).astype(np.float32)).cuda()
    sw = torch.from_numpy(rng.uniform(0.001, 0.1, N).astype(np.float32)).cuda()
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    y = qlin.gemm_w8a8(qx, sx, qw, sw, out_dtype=torch.bfloat16, acc_out=acc)
    rows = np.sort(np.concatenate([rng.choice(np.arange(2048, 2560), 32, replace=False),
                                   rng.choice(2048, 32, replace=False)]))
    acco = oracle.w8a8_acc(qx.cpu().numpy()[rows], qw.cpu().numpy())
    np.testing.assert_array_equal(acc.cpu().numpy()[rows], acco)
    yo = oracle.w8a8_out(acco, sx.cpu().numpy()[rows], sw.cpu().numpy())
    assert rel_err_out(host_f32(y)[rows], yo) < GEMM_REL_TOL
    assert qlin.qlin_device_error() == 0


@pytest.mark.parametrize("M", [17, 64, 256])
def test_w4a16_tensor_core_vs_legacy_kernel(M, monkeypatch):
    """The tcgen05 GEMM and the mma.sync GEMM agree with the oracle on the
    same packed weights (K = 4096, asymmetric UINT4, g = 128)."""
    N, K = 512, 4096
    w = torch.from_numpy(inputs.normal((N, K), 0.02, 21)).to(torch.bfloat16).cuda()
    x = torch.from_numpy(inputs.normal((M, K), 1.0, 22)).to(torch.bfloat16).cuda()
    p, q, s, z, packed, hdr = w4_prepare(w, 128, True)
    y_tc = qlin.gemm_w4a16(x, packed, hdr)
    monkeypatch.setenv("QLIN_W4A16_KERNEL", "mma")
    y_mma = qlin.gemm_w4a16(x, packed, hdr)
    torch.cuda.synchronize()
    yo = oracle.matmul_f64(host_f32(x), w4_oracle_weight(q, s, z, p, N, K, 128))
    assert rel_err_out(host_f32(y_tc), yo) < GEMM_REL_TOL
    assert rel_err_out(host_f32(y_mma), yo) < GEMM_REL_TOL
    assert qlin.qlin_device_error() == 0


@pytest.mark.parametrize("asym", [False, True])
@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("M", [17, 64, 100, 128])
def test_w4a16_tmem_a_matches_smem_a(M, group, asym, monkeypatch):
    """Up to 128 tokens the converters write the weight tile into TMEM; the
    shared-memory-operand kernel issues the same MMAs in the same order, so the
    two give the same bits (K = 2048: chains of 8 k-blocks and a split)."""
    N, K = 384, 2048
    w = torch.from_numpy(inputs.normal((N, K), 0.02, 41 + group)).to(torch.bfloat16).cuda()
    x = torch.from_numpy(inputs.normal((M, K), 1.0, 42 + M)).to(torch.bfloat16).cuda()
    p, q, s, z, packed, hdr = w4_prepare(w, group, asym)
    y_tm = qlin.gemm_w4a16(x, packed, hdr)
    monkeypatch.setenv("QLIN_W4A16_KERNEL", "smem")
    y_sm = qlin.gemm_w4a16(x, packed, hdr)
    torch.cuda.synchronize()
    assert qlin.qlin_device_error() == 0
    assert torch.equal(y_tm, y_sm)
    yo = oracle.matmul_f64(host_f32(x), w4_oracle_weight(q, s, z, p, N, K, group))
    assert rel_err_out(host_f32(y_tm), yo) < GEMM_REL_TOL


@pytest.mark.parametrize("M", [17, 64])
def test_w4a16_tmem_a_odd_k_block_count(M, monkeypatch):
    """K = 1088 is 17 blocks of 64 k, split 8 + 9: the last 128-k stage of a
    split holds a single block.  Same bits as the shared-memory kernel, which
    steps one 64-k block at a time."""
    N, K = 256, 1088
    w = torch.from_numpy(inputs.normal((N, K), 0.02, 51)).to(torch.bfloat16).cuda()
    x = torch.from_numpy(inputs.normal((M, K), 1.0, 52)).to(torch.bfloat16).cuda()
    p, q, s, z, packed, hdr = w4_prepare(w, 64, True)
    y_tm = qlin.gemm_w4a16(x, packed, hdr)
    monkeypatch.setenv("QLIN_W4A16_KERNEL", "smem")
    y_sm = qlin.gemm_w4a16(x, packed, hdr)
    torch.cuda.synchronize()
    assert qlin.qlin_device_error() == 0
    assert torch.equal(y_tm, y_sm)
    yo = oracle.matmul_f64(host_f32(x), w4_oracle_weight(q, s, z, p, N, K, 64))
    assert rel_err_out(host_f32(y_tm), yo) < GEMM_REL_TOL


def test_w4a16_reproducible():
    """Split-K partial sums are added in a fixed order: two calls agree bit for bit."""
    w = torch.from_numpy(inputs.normal((1024, 8192), 0.02, 23)).to(torch.bfloat16).cuda()
    x = torch.from_numpy(inputs.normal((256, 8192), 1.0, 24)).to(torch.bfloat16).cuda()
    _, _, _, _, packed, hdr = w4_prepare(w, 128, False)
    for m in (1, 16, 256):   # the decode kernels' cross-warp and cross-CTA sums too
        a = qlin.gemm_w4a16(x[:m].contiguous(), packed, hdr)
        b = qlin.gemm_w4a16(x[:m].contiguous(), packed, hdr)
        torch.cuda.synchronize()
        assert torch.equal(a, b)


@pytest.mark.parametrize("N", [96, 4736])
@pytest.mark.parametrize("group", [32, 64])
@pytest.mark.parametrize("M", [1, 5, 16])
def test_w4a16_gemv_odd_chunk_count(N, group, M):
    """K = 1088 (17 chunks of 64): the single-chunk decode kernel, with one
    (N = 96) and two (N = 4736 = 148 x 32) 16-row tiles per CTA."""
    K = 1088
    w = torch.from_numpy(inputs.normal((N, K), 0.02, 11)).to(torch.bfloat16).cuda()
    x = torch.from_numpy(inputs.normal((M, K), 1.0, 12)).to(torch.bfloat16).cuda()
    p, q, s, z, packed, hdr = w4_prepare(w, group, True)
    y = qlin.gemm_w4a16(x, packed, hdr)
    what = w4_oracle_weight(q, s, z, p, N, K, group)
    yo = oracle.matmul_f64(host_f32(x), what)
    assert rel_err_out(host_f32(y), yo) < GEMM_REL_TOL


@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("M", [1, 8, 9, 16])
@pytest.mark.parametrize("asym", [False, True])
def test_w4a16_gemv_two_tiles_per_cta(group, M, asym):
    """N = 9472 (296 CTAs of two 16-row tiles), K = 2048: decode kernel with
    both tiles of a CTA in one loop."""
    N, K = 9472, 2048
    w = torch.from_numpy(inputs.normal((N, K), 0.02, 13)).to(torch.bfloat16).cuda()
    x = torch.from_numpy(inputs.normal((M, K), 1.0, 14)).to(torch.bfloat16).cuda()
    p, q, s, z, packed, hdr = w4_prepare(w, group, asym)
    y = qlin.gemm_w4a16(x, packed, hdr)
    rows = np.sort(np.random.default_rng(15).choice(N, 512, replace=False))
    what = w4_oracle_weight(q, s, z, p, N, K, group, rows=rows)
    yo = oracle.matmul_f64(host_f32(x), what)
    assert rel_err_out(host_f32(y)[:, rows], yo) < GEMM_REL_TOL


@pytest.mark.parametrize("M", [64, 256])
def test_w4a16_back_to_back_calls(M):
    """Many calls queued back to back, alternating two packed copies (as a
    serving loop issues them): no device-side wait runs out and every call
    gives the same bits as a lone call."""
    N, K = 8192, 28672
    w = inputs.downproj_weight()
    x = inputs.downproj_activation(M).cuda()
    copies = []
    for scale in (1.0, 0.5):
        p, q, s, z, packed, hdr = w4_prepare((w.float() * scale).to(torch.bfloat16).cuda(), 128, True)
        copies.append((packed, hdr))
    refs = []
    for packed, hdr in copies:
        refs.append(qlin.gemm_w4a16(x, packed, hdr))
        torch.cuda.synchronize()
    assert qlin.qlin_device_error() == 0
    ys = [None, None]
    for i in range(24):
        packed, hdr = copies[i % 2]
        ys[i % 2] = qlin.gemm_w4a16(x, packed, hdr)
    torch.cuda.synchronize()
    assert qlin.qlin_device_error() == 0
    assert torch.equal(ys[0], refs[0]) and torch.equal(ys[1], refs[1])


def test_w8a8_back_to_back_calls(w8_kernel):
    """W8A8 calls queued back to back (split tail tiles and drains included):
    no device-side wait runs out and the bits match a lone call."""
    M, N, K = 2048, 4096, 28672
    p8 = qlin.make_params("s8", "row")
    qx, sx, _ = qlin.quantize(inputs.downproj_activation(M, outliers=True).cuda(), p8)
    qw, sw, _ = qlin.quantize(inputs.downproj_weight(N=N).cuda(), p8)
    ref = qlin.gemm_w8a8(qx, sx, qw, sw)
    torch.cuda.synchronize()
    for _ in range(24):
        y = qlin.gemm_w8a8(qx, sx, qw, sw)
    torch.cuda.synchronize()
    assert qlin.qlin_device_error() == 0
    assert torch.equal(y, ref)
