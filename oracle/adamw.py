"""AdamW over the packed non-matrix tail (oracle).

MatrixFSDP: Communication-Free Matrix Optimizers Under ZeRO-3 Parameter
Sharding -- Abstract: non-matrix tensors are packed into tail owners and stay on
AdamW.  The pages give no AdamW variant; the reading is decoupled weight decay
in PyTorch's order (Loshchilov & Hutter), step t counted from 1:
    p <- p * (1 - lr*wd)
    m <- beta1*m + (1-beta1)*g
    v <- beta2*v + (1-beta2)*g^2
    p <- p - (lr / (1-beta1^t)) * m / (sqrt(v) / sqrt(1-beta2^t) + eps)
in float64 from the exact fp32 inputs.
"""
from __future__ import annotations

import numpy as np


def adamw_ref(p, g, m, v, lr: float, beta1: float, beta2: float, eps: float, wd: float,
              step: int):
    p = np.asarray(p, dtype=np.float64) * (1.0 - lr * wd)
    g = np.asarray(g, dtype=np.float64)
    m = beta1 * np.asarray(m, dtype=np.float64) + (1.0 - beta1) * g
    v = beta2 * np.asarray(v, dtype=np.float64) + (1.0 - beta2) * g * g
    bc1 = 1.0 - beta1 ** step
    bc2 = 1.0 - beta2 ** step
    p = p - (lr / bc1) * m / (np.sqrt(v) / np.sqrt(bc2) + eps)
    return p, m, v
