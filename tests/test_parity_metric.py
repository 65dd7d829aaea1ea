"""The parity metric itself (CPU): bf16 output rounding is allowed on top of
the 2e-3 bound, a real 3e-3 error is not."""
import numpy as np
import torch

from parity_util import TOL, max_rel_err, max_rel_err_rounded, rel_rmse


def test_bf16_rounding_alone_passes():
    rng = np.random.default_rng(0)
    # fp32 values rounded once to bf16, as the kernel stores o (a float64 ->
    # bf16 conversion in torch goes through fp32 and would round twice)
    y = rng.standard_normal(100000).astype(np.float32).astype(np.float64)
    x = torch.tensor(y, dtype=torch.float32).to(torch.bfloat16).double().numpy()
    assert max_rel_err(x, y) > TOL          # plain relative error exceeds 2e-3 ...
    assert max_rel_err_rounded(x, y, torch.bfloat16) == 0.0  # ... only by rounding
    assert 1.3e-3 < rel_rmse(x, y) < 1.8e-3  # the bf16 floor


def test_real_errors_fail():
    rng = np.random.default_rng(1)
    y = rng.standard_normal(1000)
    bad = y * (1 + 3e-3)
    x = torch.tensor(bad).to(torch.bfloat16).double().numpy()
    assert max_rel_err_rounded(x, y, torch.bfloat16) > TOL * 0.4
    xf = torch.tensor(bad).float().double().numpy()
    assert max_rel_err_rounded(xf, y, torch.float32) > TOL


def test_rms_floor_for_cancelled_elements():
    y = np.array([1.0, -1.0, 1e-9])
    x = np.array([1.0, -1.0, 1e-4])
    assert max_rel_err(x, y) < 2e-4
