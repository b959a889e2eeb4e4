"""Pins for the oracle's AdamW (MatrixFSDP -- Abstract: the packed tail stays on
AdamW).  Checked against its closed-form first step and against
torch.optim.AdamW, an independent library implementation."""
import numpy as np
import pytest
import torch

from oracle import adamw_ref


def test_first_step_closed_form():
    rng = np.random.default_rng(0)
    p0 = rng.standard_normal(4096) * 1e-3
    g = rng.standard_normal(4096) * 1e-3
    lr, b1, b2, eps, wd = 1e-3, 0.9, 0.95, 1e-8, 0.1
    p, m, v = adamw_ref(p0, g, np.zeros_like(g), np.zeros_like(g), lr, b1, b2, eps, wd, 1)
    np.testing.assert_allclose(m, 0.1 * g, rtol=1e-15)
    np.testing.assert_allclose(v, 0.05 * g * g, rtol=1e-14)
    np.testing.assert_allclose(p, p0 * (1 - lr * wd) - lr * g / (np.abs(g) + eps), rtol=1e-12, atol=1e-18)


@pytest.mark.parametrize("steps", [1, 3, 7])
def test_matches_torch_adamw(steps):
    rng = np.random.default_rng(steps)
    n = 1000
    p0 = rng.standard_normal(n)
    lr, b1, b2, eps, wd = 3e-3, 0.9, 0.95, 1e-8, 0.1
    tp = torch.tensor(p0, dtype=torch.float64, requires_grad=True)
    opt = torch.optim.AdamW([tp], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd)
    p, m, v = p0.copy(), np.zeros(n), np.zeros(n)
    for t in range(1, steps + 1):
        g = rng.standard_normal(n)
        tp.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        p, m, v = adamw_ref(p, g, m, v, lr, b1, b2, eps, wd, t)
    st = opt.state[tp]
    np.testing.assert_allclose(p, tp.detach().numpy(), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(m, st["exp_avg"].numpy(), rtol=1e-13, atol=1e-16)
    np.testing.assert_allclose(v, st["exp_avg_sq"].numpy(), rtol=1e-13, atol=1e-16)
