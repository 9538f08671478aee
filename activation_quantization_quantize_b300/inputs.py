"""Seeded synthetic inputs for the quantized linear layer workloads.

This module only draws random numbers and stores them in the workload's
storage type; it holds none of the quantizer's arithmetic, so both the CUDA
path and the CPU oracle can take their inputs from it.

Seeding: base seed 0; tensor number t of a workload uses
``numpy.random.default_rng(seed + t)``.  Values are drawn in binary32 and, for
bf16 workloads, rounded to bf16 by torch's nearest-even conversion.
"""
from dataclasses import dataclass

import numpy as np
import torch


def normal(shape, std, seed):
    """N(0, std^2) samples in binary32."""
    rng = np.random.default_rng(seed)
    out = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    return out


def to_bf16(x):
    """binary32 numpy array -> torch.bfloat16 CPU tensor (nearest-even)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def bf16_values(t):
    """torch.bfloat16 tensor -> binary32 numpy array of the same values."""
    return t.to(torch.float32).cpu().numpy()


def outlier_channels(x, n_channels, lo, hi, seed):
    """Scale n_channels seeded input channels (columns) of x by U[lo, hi]."""
    rng = np.random.default_rng(seed)
    cols = rng.choice(x.shape[1], size=n_channels, replace=False)
    mult = rng.uniform(lo, hi, size=n_channels).astype(np.float32)
    x[:, cols] *= mult[None, :]
    return np.sort(cols)


def outlier_elements(x, fraction, value, seed):
    """Set round(fraction * size) seeded positions of x to +-value."""
    rng = np.random.default_rng(seed)
    n = int(round(fraction * x.size))
    pos = rng.choice(x.size, size=n, replace=False)
    sign = np.where(rng.random(n) < 0.5, -1.0, 1.0).astype(np.float32)
    flat = x.reshape(-1)
    flat[pos] = sign * np.float32(value)
    return n


# --------------------------------------------------------------------------
# Workload recipes.  Shapes and distributions follow the five workloads of
# the quantized linear layer: a tiny W8A8 case, a 4096x4096 W4A16 decode, a
# 2048x11008x4096 SmoothQuant-style prefill, a 16384x4096 quantize sweep and
# a 70B-shaped 8192x28672 down-projection.
# --------------------------------------------------------------------------

@dataclass
class W8A8Tiny:
    x: np.ndarray          # fp32 [8 x 256]
    w: np.ndarray          # fp32 [128 x 256]
    vec5: np.ndarray       # the five-element example vector


def w8a8_tiny(seed=0, M=8, N=128, K=256):
    """Tiny W8A8 case: X ~ N(0,1) with input channels 3 and 77 scaled x50,
    W ~ N(0, 0.02)."""
    x = normal((M, K), 1.0, seed + 0)
    for c in (3, 77):
        if c < K:
            x[:, c] *= np.float32(50.0)
    w = normal((N, K), 0.02, seed + 1)
    vec5 = np.array([0.5, -1.2, 2.1, -0.8, 1.7], dtype=np.float32)
    return W8A8Tiny(x, w, vec5)


def w4a16_decode(M, seed=0, N=4096, K=4096, w_std=0.02):
    """W4A16 decode: W bf16 [N x K] ~ N(0, w_std), X bf16 [M x K] ~ N(0,1)."""
    w = to_bf16(normal((N, K), w_std, seed + 0))
    x = to_bf16(normal((M, K), 1.0, seed + 1))
    return x, w


def w8a8_prefill(seed=0, M=2048, N=11008, K=4096, outlier_frac=0.01, lo=20.0, hi=60.0,
                 w_std=0.02):
    """SmoothQuant-style prefill: X bf16 [M x K] ~ N(0,1) with 1% of input
    channels scaled by U[20, 60]; W bf16 [N x K] ~ N(0, 0.02)."""
    x = normal((M, K), 1.0, seed + 0)
    n_out = max(1, int(round(outlier_frac * K)))
    cols = outlier_channels(x, n_out, lo, hi, seed + 2)
    w = normal((N, K), w_std, seed + 1)
    return to_bf16(x), to_bf16(w), cols


def sweep_tensor(seed=0, rows=16384, cols=4096, frac=0.001, value=100.0):
    """Quantize sweep: bf16 [rows x cols] ~ N(0,1), 0.1% of elements at +-100."""
    x = normal((rows, cols), 1.0, seed + 0)
    outlier_elements(x, frac, value, seed + 1)
    return to_bf16(x)


def downproj_weight(seed=0, N=8192, K=28672, std=0.015):
    """70B-shaped down-projection weight: bf16 [N x K] ~ N(0, 0.015)."""
    return to_bf16(normal((N, K), std, seed + 0))


def downproj_activation(M, seed=0, K=28672, outliers=False, outlier_frac=0.01, lo=20.0,
                        hi=60.0):
    """Down-projection activations: bf16 [M x K] ~ N(0,1), optionally with 1%
    of input channels scaled by U[20, 60]."""
    x = normal((M, K), 1.0, seed + 1)
    if outliers:
        outlier_channels(x, max(1, int(round(outlier_frac * K))), lo, hi, seed + 2)
    return to_bf16(x)
