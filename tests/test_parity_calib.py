"""GPU parity of the SmoothQuant calibration pieces against the oracle:
running channel maxima and folded LayerNorm parameters bit for bit, the
quantization-error statistics within binary64 summation-order rounding, and
table 11-4's alpha ordering reproduced from the GPU's own numbers."""
import numpy as np
import pytest
import torch

import oracle
from activation_quantization_quantize_b300 import inputs, qlin
from helpers import codes_to_int, host_f32, oracle_quantize, scales_f32

pytestmark = pytest.mark.gpu

GRAN = {qlin.QLIN_PER_TENSOR: oracle.PER_TENSOR, qlin.QLIN_PER_ROW: oracle.PER_ROW,
        qlin.QLIN_PER_COL: oracle.PER_COL, qlin.QLIN_PER_GROUP: oracle.PER_GROUP}


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("cols", [4096, 1000])
def test_absmax_update_over_batches(dtype, cols):
    """Four calibration batches of the prefill workload's activations (with
    outlier channels); cols = 1000 takes the scalar path."""
    run = torch.zeros(cols, dtype=torch.float32, device="cuda")
    ref = np.zeros(cols, np.float32)
    for b in range(4):
        xf = inputs.normal((96 + 7 * b, cols), 1.0, 60 + b)
        inputs.outlier_channels(xf, max(1, cols // 100), 20.0, 60.0, 70 + b)
        x = torch.from_numpy(xf).to(dtype).cuda()
        qlin.absmax_update(x, run)
        oracle.channel_absmax_update(host_f32(x), ref)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(run.cpu().numpy(), ref)


@pytest.mark.parametrize("with_beta", [True, False])
def test_fold_layernorm(with_beta):
    rng = np.random.default_rng(61)
    K = 4099
    gamma = rng.uniform(0.5, 1.5, K).astype(np.float32)
    beta = rng.uniform(-0.3, 0.3, K).astype(np.float32)
    s = rng.uniform(0.05, 40.0, K).astype(np.float32)
    g2, b2 = qlin.fold_layernorm(torch.from_numpy(gamma).cuda(), torch.from_numpy(beta).cuda() if with_beta else None,
                                 torch.from_numpy(s).cuda())
    go, bo = oracle.fold_layernorm(gamma, beta if with_beta else None, s)
    np.testing.assert_array_equal(g2.cpu().numpy(), go)
    if with_beta:
        np.testing.assert_array_equal(b2.cpu().numpy(), bo)


@pytest.mark.parametrize("code,gran,group,mode", [("s8", "row", 0, qlin.QLIN_SMOOTH_DIVIDE),
                                                  ("s8", "row", 0, qlin.QLIN_SMOOTH_MULTIPLY),
                                                  ("u4", "group", 128, qlin.QLIN_SMOOTH_NONE),
                                                  ("u8", "col", 0, qlin.QLIN_SMOOTH_NONE),
                                                  ("s4", "tensor", 0, qlin.QLIN_SMOOTH_DIVIDE)])
def test_quant_error_statistics(code, gran, group, mode):
    rows, cols = 333, 1024
    xf = inputs.normal((rows, cols), 1.0, 62)
    inputs.outlier_channels(xf, 10, 20.0, 60.0, 63)
    x = torch.from_numpy(xf).to(torch.bfloat16).cuda()
    sm = np.random.default_rng(64).uniform(0.2, 8.0, cols).astype(np.float32) if mode else None
    smd = None if sm is None else torch.from_numpy(sm).cuda()
    p = qlin.make_params(code, gran, group=group, smooth_mode=mode)
    q, s, z = qlin.quantize(x, p, smooth=smd)
    out = qlin.quant_error(x, p, q, s, z, smooth=smd).cpu().numpy()
    eo = oracle.quant_error(host_f32(x), codes_to_int(q, p, rows, cols), scales_f32(s),
                            None if p.symmetric else z.cpu().numpy(), GRAN[p.gran], group, smooth=sm,
                            smooth_mode=mode)
    # binary64 sums of n non-negative terms in two orders differ by at most
    # about n * 2^-53 relative (n = 341k here: 4e-11)
    np.testing.assert_allclose(out[:2], eo[:2], rtol=rows * cols * 2.0 ** -53)
    assert out[2] == eo[2]
    again = qlin.quant_error(x, p, q, s, z, smooth=smd).cpu().numpy()
    np.testing.assert_array_equal(out, again)                   # fixed summation order


def test_alpha_sweep_on_the_prefill_workload():
    """Table 11-4 on the 2048 x 4096 prefill activations (1% outlier channels)
    and the 11008 x 4096 weight: the GPU's activation INT8 error falls and its
    weight INT8 error rises as alpha goes 0.3 -> 0.5 -> 0.7, and every
    number matches the oracle's on the same codes."""
    x, w, _ = inputs.w8a8_prefill()
    xd, wd = x.cuda(), w.cuda()
    xmax = torch.zeros(4096, dtype=torch.float32, device="cuda")
    qlin.absmax_update(xd, xmax)
    wmax = qlin.absmax(wd, qlin.QLIN_PER_COL)
    act, wgt = [], []
    for alpha in (0.3, 0.5, 0.7):
        s = qlin.smooth_factors(xmax, wmax, alpha)
        px = qlin.make_params("s8", "row", smooth_mode=qlin.QLIN_SMOOTH_DIVIDE)
        pw = qlin.make_params("s8", "row", smooth_mode=qlin.QLIN_SMOOTH_MULTIPLY)
        qx, sx, _ = qlin.quantize(xd, px, smooth=s)
        qw, sw, _ = qlin.quantize(wd, pw, smooth=s)
        ea = qlin.quant_error(xd, px, qx, sx, None, smooth=s).cpu().numpy()
        ew = qlin.quant_error(wd, pw, qw, sw, None, smooth=s).cpu().numpy()
        act.append(np.sqrt(ea[0] / ea[1]))
        wgt.append(np.sqrt(ew[0] / ew[1]))
        if alpha == 0.5:
            rows = np.arange(0, 2048, 64)
            sh = s.cpu().numpy()
            qxo, sxo, _ = oracle_quantize(host_f32(x)[rows], px, smooth=sh)
            np.testing.assert_array_equal(codes_to_int(qx, px, 2048, 4096)[rows], qxo)
            eo = oracle.quant_error(host_f32(wd), codes_to_int(qw, pw, 11008, 4096), scales_f32(sw), None,
                                    oracle.PER_ROW, smooth=sh, smooth_mode=oracle.SMOOTH_MULTIPLY)
            np.testing.assert_allclose(ew[:2], eo[:2], rtol=11008 * 4096 * 2.0 ** -53)
    assert act[0] > act[1] > act[2]
    assert wgt[0] < wgt[1] < wgt[2]
