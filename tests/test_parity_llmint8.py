"""GPU parity of the LLM.int8() decomposition against the oracle: the outlier
channel list bit for bit, the output within GEMM_REL_TOL of the binary64
sw * (sx * acc + X_outlier qw_outlier^T), the no-outlier case equal to the
W8A8 layer bit for bit, and the workspace-overflow report."""
import numpy as np
import pytest
import torch

import oracle
from activation_quantization_quantize_b300 import inputs, qlin
from helpers import GEMM_REL_TOL, host_f32, rel_err, rel_err_out

pytestmark = pytest.mark.gpu


def layer(M, N, K, seed, n_out_frac=0.01):
    xf = inputs.normal((M, K), 1.0, seed)
    inputs.outlier_channels(xf, max(1, int(round(n_out_frac * K))), 20.0, 60.0, seed + 1)
    x = torch.from_numpy(xf).to(torch.bfloat16).cuda()
    w = torch.from_numpy(inputs.normal((N, K), 0.02, seed + 2)).to(torch.bfloat16).cuda()
    qw, sw, _ = qlin.quantize(w, qlin.make_params("s8", "row"))
    torch.cuda.synchronize()
    return x, qw, sw


def oracle_rows(xh, qw_h, sw_h, cols, rows):
    xr = xh[rows]
    xn = xr.copy()
    xn[:, cols] = 0.0
    qx, sx, _ = oracle.quantize(xn, -127, 127, True, oracle.PER_ROW)
    acc = oracle.w8a8_acc(qx.astype(np.int8), qw_h)
    return oracle.llmint8_out(xr, qw_h, sw_h, sx, acc, cols)


@pytest.mark.parametrize("M,N,K", [(1, 16, 64), (37, 200, 1024), (130, 384, 4096), (256, 1000, 2048 + 16)])
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_llmint8_small(M, N, K, out):
    x, qw, sw = layer(M, N, K, seed=M + K)
    rep = torch.zeros(1 + K, dtype=torch.int32, device="cuda")
    y = qlin.gemm_llmint8(x, qw, sw, threshold=6.0, out_dtype=out, outliers=rep)
    torch.cuda.synchronize()
    assert qlin.qlin_device_error() == 0
    xh = host_f32(x)
    cols = oracle.llmint8_outlier_cols(xh, 6.0)
    r = rep.cpu().numpy()
    assert r[0] == cols.size
    np.testing.assert_array_equal(r[1:1 + cols.size], cols)
    yo = oracle_rows(xh, qw.cpu().numpy(), sw.cpu().numpy(), cols, np.arange(M))
    err = rel_err(y.cpu().numpy(), yo) if out == torch.float32 else rel_err_out(host_f32(y), yo)
    assert err < GEMM_REL_TOL


def test_llmint8_without_outliers_is_the_w8a8_layer():
    """A threshold no value reaches: no outlier channel, and the layer is the
    W8A8 layer on per-token codes of x, bit for bit."""
    x, qw, sw = layer(300, 512, 2048, seed=7)
    y = qlin.gemm_llmint8(x, qw, sw, threshold=1e30, out_dtype=torch.float32)
    qx, sx, _ = qlin.quantize(x, qlin.make_params("s8", "row"))
    y8 = qlin.gemm_w8a8(qx, sx, qw, sw, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(y, y8)


def test_llmint8_prefill_sampled():
    """2048 x 11008 x 4096 with 1% outlier channels x U[20, 60] (the prefill
    workload): 2 rows from every 128-row tile, all columns."""
    x, qw, sw = layer(2048, 11008, 4096, seed=11)
    rep = torch.zeros(1 + 4096, dtype=torch.int32, device="cuda")
    y = qlin.gemm_llmint8(x, qw, sw, threshold=6.0, outliers=rep)
    torch.cuda.synchronize()
    xh = host_f32(x)
    cols = oracle.llmint8_outlier_cols(xh, 6.0)
    assert rep.cpu().numpy()[0] == cols.size >= 41
    rng = np.random.default_rng(12)
    rows = np.sort(np.concatenate([t + rng.choice(128, 2, replace=False) for t in range(0, 2048, 128)]))
    yo = oracle_rows(xh, qw.cpu().numpy(), sw.cpu().numpy(), cols, rows)
    assert rel_err_out(host_f32(y)[rows], yo) < GEMM_REL_TOL
    assert qlin.qlin_device_error() == 0


def test_llmint8_beats_plain_w8a8_on_outliers():
    """[L19] section 10: keeping the outlier channels out of INT8 protects the
    result -- the decomposition is closer to the exact bf16 product than the
    plain per-token W8A8 layer on the same weight."""
    x, qw, sw = layer(256, 1024, 4096, seed=13)
    y = qlin.gemm_llmint8(x, qw, sw, threshold=6.0, out_dtype=torch.float32).double()
    qx, sx, _ = qlin.quantize(x, qlin.make_params("s8", "row"))
    y8 = qlin.gemm_w8a8(qx, sx, qw, sw, out_dtype=torch.float32).double()
    wh = sw.double()[:, None] * qw.double()
    exact = x.double() @ wh.T
    assert torch.linalg.norm(y - exact) < 0.5 * torch.linalg.norm(y8 - exact)


def test_llmint8_reports_too_many_outliers():
    """More outlier channels than the workspace was sized for: the call
    records QLIN_ERR_WORKSPACE (read by qlin_device_error), the context stays
    usable, and a correctly sized call afterwards is exact."""
    x, qw, sw = layer(64, 256, 1024, seed=15, n_out_frac=0.05)
    qlin.gemm_llmint8(x, qw, sw, threshold=6.0, max_outliers=16)
    assert qlin.qlin_device_error() == qlin.QLIN_ERR_WORKSPACE
    y = qlin.gemm_llmint8(x, qw, sw, threshold=6.0, max_outliers=64, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert qlin.qlin_device_error() == 0
    xh = host_f32(x)
    cols = oracle.llmint8_outlier_cols(xh, 6.0)
    yo = oracle_rows(xh, qw.cpu().numpy(), sw.cpu().numpy(), cols, np.arange(64))
    assert rel_err(y.cpu().numpy(), yo) < GEMM_REL_TOL
