"""Muon momentum and Newton-Schulz orthogonalisation on an owner set (oracle).

MatrixFSDP: Communication-Free Matrix Optimizers Under ZeRO-3 Parameter
Sharding -- Abstract: Muon orthogonalises momentum-smoothed matrix updates with
Newton-Schulz, which needs the complete 2D matrix; under MatrixFSDP the owner
rank holds each matrix's full reduced gradient in its owner shard and runs
Newton-Schulz locally; the update matches full-matrix Muon.  Section 1: a
row-band is not the same optimizer input as the full matrix.

Readings (the pages state no formula):
  * momentum is heavy-ball, M <- beta*M + G, and the Newton-Schulz input is
    U = M; with nesterov, U = G + beta*M (after the update of M);
  * U is scaled to unit Frobenius norm, X0 = U / (||U||_F + eps);
  * Newton-Schulz is Muon's quintic iteration on the short side: X is s x l
    (the stored matrix transposed when rows > cols), and for k = 1..T
        A = X X^T,  B = b A + c A A,  X <- a X + B X;
    the output O = X_T is transposed back to the stored shape;
  * the step returns O itself (no learning-rate or shape scaling: the pages
    give none, and applying the update to weights is the caller's).
Everything is float64; the gradient enters as the exact stored value (fp32, or
bf16 widened exactly).
"""
from __future__ import annotations

from typing import Dict, List, Sequence, Tuple

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def stored_to_f64(buf: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_bits_to_f64(buf)
    if dtype == "f32":
        return np.asarray(buf, dtype=np.float32).astype(np.float64)
    raise ValueError(dtype)


def momentum_ref(G: np.ndarray, M: np.ndarray, beta: float, nesterov: bool
                 ) -> Tuple[np.ndarray, np.ndarray]:
    """Returns (M_new, U): M_new = beta*M + G; U = M_new, or G + beta*M_new."""
    M_new = beta * M + G
    U = G + beta * M_new if nesterov else M_new
    return M_new, U


def newton_schulz_ref(U: np.ndarray, steps: int, a: float, b: float, c: float,
                      eps: float) -> np.ndarray:
    """Quintic Newton-Schulz on the full matrix U (rows x cols), float64."""
    U = np.asarray(U, dtype=np.float64)
    transposed = U.shape[0] > U.shape[1]
    X = U.T if transposed else U
    X = X / (np.sqrt(np.sum(X * X)) + eps)
    for _ in range(steps):
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    return X.T if transposed else X


def muon_matrix_ref(G: np.ndarray, M: np.ndarray, beta: float, nesterov: bool, steps: int,
                    a: float, b: float, c: float, eps: float) -> Tuple[np.ndarray, np.ndarray]:
    """One matrix's owner step: (M_new, O)."""
    M_new, U = momentum_ref(G, M, beta, nesterov)
    return M_new, newton_schulz_ref(U, steps, a, b, c, eps)


def muon_owner_step_ref(shards: Sequence[Dict[str, int]], grad_flat: np.ndarray, grad_dtype: str,
                        momentum_flat: np.ndarray, beta: float, nesterov: bool, steps: int,
                        a: float, b: float, c: float, eps: float,
                        only: Sequence[int] = None) -> Tuple[np.ndarray, Dict[int, np.ndarray]]:
    """The owner-local step over one rank's flat owner buffer.

    Each shard (param_id, offset, rows, cols) views rows*cols elements of the
    flat gradient and momentum buffers at `offset` (row-major).  Returns the new
    momentum buffer (float64, only the shards' elements changed) and
    {param_id: O} for the shards processed (all, or those in `only`)."""
    G_all = stored_to_f64(grad_flat, grad_dtype)
    M_all = np.asarray(momentum_flat, dtype=np.float64).copy()
    out: Dict[int, np.ndarray] = {}
    for sh in shards:
        if only is not None and sh["param_id"] not in only:
            continue
        o, r, c_ = sh["offset"], sh["rows"], sh["cols"]
        G = G_all[o:o + r * c_].reshape(r, c_)
        M = M_all[o:o + r * c_].reshape(r, c_)
        M_new, O = muon_matrix_ref(G, M, beta, nesterov, steps, a, b, c, eps)
        M_all[o:o + r * c_] = M_new.reshape(-1)
        out[sh["param_id"]] = O
    return M_all, out


# ---------------------------------------------------------------------------
# Applying the update to the weights.
#
# The pages stop at the orthogonalised update ("the update matches full-matrix
# Muon").  Applying it is the step right after; the pages give neither the
# learning rate nor a shape-dependent scale, so the reading here is Muon's
# decoupled form W <- W*(1 - lr*wd) - lr*scale*O with three scale choices:
#   mode 0: scale = 1
#   mode 1: scale = sqrt(max(1, rows/cols))        (Muon's reference scaling)
#   mode 2: scale = 0.2*sqrt(max(rows, cols))       (scaling that matches AdamW's
#                                                   update RMS, Liu et al. 2025)
def muon_scale_ref(rows: int, cols: int, mode: int) -> float:
    if mode == 0:
        return 1.0
    if mode == 1:
        return float(np.sqrt(max(1.0, rows / cols)))
    if mode == 2:
        return 0.2 * float(np.sqrt(max(rows, cols)))
    raise ValueError(mode)


def muon_apply_ref(W: np.ndarray, O: np.ndarray, lr: float, wd: float, scale: float) -> np.ndarray:
    """W*(1 - lr*wd) - lr*scale*O in float64."""
    return np.asarray(W, np.float64) * (1.0 - lr * wd) - lr * scale * np.asarray(O, np.float64)
