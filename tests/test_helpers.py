"""The test-side error metric itself (no GPU): a bf16-rounded copy of an exact
result has zero excess error, and a one-ulp-off copy does not."""
import numpy as np
import torch

from helpers import rel_err, rel_err_out


def test_rounding_is_not_counted_as_error():
    r = (np.random.default_rng(0).standard_normal(100000)
         * 10.0 ** np.random.default_rng(1).integers(-3, 4, 100000)).astype(np.float32).astype(np.float64)
    y = torch.from_numpy(r.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert rel_err(y, r) > 2e-3          # one bf16 rounding alone exceeds 2e-3 somewhere
    assert rel_err_out(y, r) == 0.0
    y2 = y.copy()
    i = int(np.argmax(np.abs(r)))
    y2[i] = y2[i] * 1.01
    assert rel_err_out(y2, r) > 2e-3


def test_f32_outputs_use_f32_ulp():
    r = np.array([1.0, -3.0, 1e-3])
    y = r * (1 + 1e-6)
    assert rel_err_out(y, r, "f32") < 2e-6
