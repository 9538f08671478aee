"""Shared helpers of the parity tests: running the oracle with the same
parameters as a libqlin call, decoding codes, and the relative-error metric."""
import numpy as np
import torch

import oracle
from activation_quantization_quantize_b300 import qlin

# Max relative error of a GEMM output before its final rounding to the output
# type.  A bf16 output also carries that one rounding (up to half a bf16 ulp,
# 2^-8 of |y| at the bottom of a binade), which rel_err_out() allows on top.
GEMM_REL_TOL = 2e-3

_ORC_GRAN = {qlin.QLIN_PER_TENSOR: oracle.PER_TENSOR, qlin.QLIN_PER_ROW: oracle.PER_ROW,
             qlin.QLIN_PER_COL: oracle.PER_COL, qlin.QLIN_PER_GROUP: oracle.PER_GROUP}


def rel_err(y, r):
    """max_i |y_i - r_i| / max(|r_i|, 0.01 * rms(r))."""
    y = np.asarray(y, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    rms = np.sqrt(np.mean(r * r)) if r.size else 0.0
    den = np.maximum(np.abs(r), 0.01 * rms)
    den = np.where(den == 0, 1.0, den)
    return float(np.max(np.abs(y - r) / den)) if r.size else 0.0


def half_ulp(r, mant_bits):
    """Half an ulp of |r| in a binary format with mant_bits fraction bits."""
    r = np.abs(np.asarray(r, dtype=np.float64))
    _, e = np.frexp(np.where(r == 0, 1.0, r))        # r = f * 2^e, f in [0.5, 1)
    return np.ldexp(1.0, e - 2 - mant_bits) * (r != 0)


def rel_err_out(y, r, out="bf16"):
    """rel_err after removing the final rounding of the exact result r to the
    output type: max_i max(|y_i - r_i| - halfulp(r_i), 0) / max(|r_i|, 0.01 rms(r))."""
    y = np.asarray(y, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    if r.size == 0:
        return 0.0
    bits = {"bf16": 7, "f16": 10, "f32": 23}[out]
    rms = np.sqrt(np.mean(r * r))
    den = np.maximum(np.abs(r), 0.01 * rms)
    den = np.where(den == 0, 1.0, den)
    ex = np.maximum(np.abs(y - r) - half_ulp(r, bits) * (1 + 2.0 ** -20), 0.0)
    return float(np.max(ex / den))


def host_f32(t):
    return t.detach().to(torch.float32).cpu().numpy()


def oracle_quantize(x_f32, p, smooth=None, static_s=None, static_z=None):
    return oracle.quantize(x_f32, p.qmin, p.qmax, bool(p.symmetric), _ORC_GRAN[p.gran], p.group,
                           smooth=smooth, smooth_mode=p.smooth_mode, percentile=p.clip_percentile,
                           scale_f16=(p.scale_dtype == qlin.QLIN_F16), static_s=static_s, static_z=static_z)


def codes_to_int(q, p, rows, cols):
    """Device code tensor -> int32 numpy [rows x cols]."""
    a = q.cpu().numpy()
    if p.code in (qlin.QLIN_S4, qlin.QLIN_U4):
        return oracle.unpack_nibbles(a.view(np.uint8).reshape(-1), rows * cols,
                                     p.code == qlin.QLIN_S4).reshape(rows, cols)
    if p.code == qlin.QLIN_S8:
        return a.view(np.int8).astype(np.int32).reshape(rows, cols)
    return a.view(np.uint8).astype(np.int32).reshape(rows, cols)


def scales_f32(s):
    return s.detach().to(torch.float32).cpu().numpy()
