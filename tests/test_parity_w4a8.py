"""GPU parity of the W4A8 layer (group-wise INT4 weights x per-token INT8
activations) against the oracle: the exact per-group integer sums (acc_out)
bit for bit, and the outputs within GEMM_REL_TOL of the binary64
sx * sum_g s_g * acc_g."""
import numpy as np
import pytest
import torch

import oracle
from activation_quantization_quantize_b300 import inputs, qlin
from helpers import GEMM_REL_TOL, codes_to_int, host_f32, rel_err, rel_err_out, scales_f32

pytestmark = pytest.mark.gpu


def prepare(N, K, M, group, asym, seed, x_outliers=False):
    """Quantize W [N x K] group-wise (fp16 scales) and pack it; quantize X
    [M x K] per token to INT8.  Returns device and host pieces."""
    w = torch.from_numpy(inputs.normal((N, K), 0.02, seed)).to(torch.bfloat16).cuda()
    xf = inputs.normal((M, K), 1.0, seed + 1)
    if x_outliers:
        inputs.outlier_channels(xf, max(1, K // 100), 20.0, 60.0, seed + 2)
    x = torch.from_numpy(xf).to(torch.bfloat16).cuda()
    pw = qlin.make_params("u4" if asym else "s4", "group", group=group, scale_f16=True)
    q, s, z = qlin.quantize(w, pw)
    packed, hdr = qlin.pack_w4(q, s, z, N, K, group)
    px = qlin.make_params("s8", "row")
    qx, sx, _ = qlin.quantize(x, px)
    torch.cuda.synchronize()
    host = dict(qx=qx.cpu().numpy().astype(np.int8), sx=sx.cpu().numpy(), q=codes_to_int(q, pw, N, K),
                s=scales_f32(s).reshape(-1), z=None if z is None else z.cpu().numpy().reshape(-1))
    return qx, sx, packed, hdr, host


def oracle_out(host, group, rows=None):
    q = host["q"] if rows is None else host["q"][rows]
    N = q.shape[0]
    ngr = q.shape[1] // group
    s = host["s"].reshape(-1, ngr)
    z = None if host["z"] is None else host["z"].reshape(-1, ngr)
    if rows is not None:
        s = s[rows]
        z = None if z is None else z[rows]
    acc = oracle.w4a8_acc(host["qx"], q, None if z is None else z.reshape(-1), group)
    return acc, oracle.w4a8_out(acc, host["sx"], s.reshape(-1))


@pytest.mark.parametrize("asym", [False, True])
@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("M", [1, 2, 3, 8, 9, 16, 17, 40])
def test_w4a8_small_exact_sums(asym, group, M):
    N, K = 256, 1024
    qx, sx, packed, hdr, host = prepare(N, K, M, group, asym, seed=M + group)
    acc = torch.empty((K // group, M, N), dtype=torch.int32, device="cuda")
    y = qlin.gemm_w4a8(qx, sx, packed, hdr, out_dtype=torch.float32, acc_out=acc)
    yb = qlin.gemm_w4a8(qx, sx, packed, hdr, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    acco, yo = oracle_out(host, group)
    np.testing.assert_array_equal(acc.cpu().numpy(), acco)
    assert rel_err(y.cpu().numpy(), yo) < GEMM_REL_TOL
    assert rel_err_out(host_f32(yb), yo) < GEMM_REL_TOL
    assert qlin.qlin_device_error() == 0


@pytest.mark.parametrize("M", [1, 2, 5])
@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("K", [1088 + 64, 2048 + 64 * 3])
def test_w4a8_groups_cut_between_warps(group, K, M):
    """K = 1152 / 2240: the eight warps' K ranges start inside groups of 128,
    so each warp scales its own exact part of a group (M = 1, 2: the dp4a
    kernel; M = 5: the MMA kernel)."""
    if K % group:
        pytest.skip("group does not divide K")
    N = 4736                                            # 148 x 32 rows: two 16-row tiles per CTA
    qx, sx, packed, hdr, host = prepare(N, K, M, group, True, seed=K + group)
    acc = torch.empty((K // group, M, N), dtype=torch.int32, device="cuda")
    y = qlin.gemm_w4a8(qx, sx, packed, hdr, out_dtype=torch.float32, acc_out=acc)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(K).choice(N, 256, replace=False))
    acco, yo = oracle_out(host, group, rows)
    np.testing.assert_array_equal(acc.cpu().numpy()[:, :, rows], acco)
    assert rel_err(y.cpu().numpy()[:, rows], yo) < GEMM_REL_TOL


@pytest.mark.parametrize("M", [1, 8, 16])
def test_w4a8_downproj_sampled(M):
    """8192 x 28672 asymmetric UINT4, g = 128 (the down-projection weight),
    per-token INT8 activations with outlier channels: exact group sums and
    outputs on 256 sampled output channels, all tokens."""
    N, K, g = 8192, 28672, 128
    w = inputs.downproj_weight()
    p4 = qlin.make_params("u4", "group", group=g, scale_f16=True)
    q, s, z = qlin.quantize(w.cuda(), p4)
    packed, hdr = qlin.pack_w4(q, s, z, N, K, g)
    x = inputs.downproj_activation(M, outliers=True).cuda()
    qx, sx, _ = qlin.quantize(x, qlin.make_params("s8", "row"))
    y = qlin.gemm_w4a8(qx, sx, packed, hdr, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(10 + M).choice(N, 256, replace=False))
    idx = torch.from_numpy(rows).cuda()
    host = dict(qx=qx.cpu().numpy().astype(np.int8), sx=sx.cpu().numpy(),
                q=codes_to_int(q[idx], p4, len(rows), K),
                s=scales_f32(s.reshape(N, K // g)[idx]).reshape(-1), z=z.reshape(N, K // g)[idx].cpu().numpy().reshape(-1))
    _, yo = oracle_out(host, g)
    assert rel_err_out(host_f32(y)[:, rows], yo) < GEMM_REL_TOL
    assert qlin.qlin_device_error() == 0


def test_w4a8_reproducible():
    qx, sx, packed, hdr, _ = prepare(1024, 4096, 16, 128, True, seed=5)
    a = qlin.gemm_w4a8(qx, sx, packed, hdr)
    b = qlin.gemm_w4a8(qx, sx, packed, hdr)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_w4a8_matches_w4a16_on_the_same_weights():
    """Both layers read the same packed weight: W4A8 on the per-token codes of
    X equals W4A16 on the dequantized X^ = sx * qx (as bf16 values) within the
    GEMM bound -- the two paths differ only in where the activation scale is
    applied and in their summation order."""
    N, K, M = 512, 2048, 8
    qx, sx, packed, hdr, host = prepare(N, K, M, 128, True, seed=6)
    y8 = qlin.gemm_w4a8(qx, sx, packed, hdr, out_dtype=torch.float32)
    _, yo = oracle_out(host, 128)
    xh = (torch.from_numpy(host["qx"].astype(np.float32) * host["sx"][:, None])).to(torch.bfloat16).cuda()
    y16 = qlin.gemm_w4a16(xh, packed, hdr)
    torch.cuda.synchronize()
    assert rel_err(y8.cpu().numpy(), yo) < GEMM_REL_TOL
    # bf16 activations: X^ itself is rounded (2^-9 relative per element), so
    # the comparison is norm-wise
    d = host_f32(y16) - yo
    assert np.linalg.norm(d) / np.linalg.norm(yo) < 4e-3
