"""A bf16 emulation of the GPU's Newton-Schulz precision, for deriving test
tolerances.  Test infrastructure: it is neither the oracle (that is the fp64
definition in oracle/) nor the product; nothing outside tests/ uses it.

It follows the precision choices the library documents for its
Newton-Schulz products (bf16 operands and stored A, B and X; fp32
accumulation and fp32 epilogue arithmetic; the Frobenius prescale taken in
fp32 from the unrounded momentum and folded into the first iteration's
epilogues), written with NumPy fp32 matrix products.  Its accumulation order
is BLAS's, not the tensor cores', so it reproduces the error's size, not the
GPU's bits.  Measured against the fp64 oracle it gives the error that bf16
storage alone causes; the tolerances in tests/helpers.py are set from its
maxima (tests/derive_ns_tolerances.py prints them).
"""
from __future__ import annotations

import numpy as np


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even), as float32."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return r.astype(np.uint32).view(np.float32)


def newton_schulz_bf16(U: np.ndarray, steps: int, a: float, b: float, c: float, eps: float,
                       out_bf16: bool = False) -> np.ndarray:
    """Update O (float64, the stored shape of U) of the bf16 pipeline.

    U is the fp32 momentum (the Newton-Schulz input before normalisation)."""
    U = np.asarray(U, dtype=np.float32)
    transposed = U.shape[0] > U.shape[1]
    Uo = U.T if transposed else U
    ss = np.float32(np.sum(np.square(Uo, dtype=np.float32), dtype=np.float32))
    inv = np.float32(1.0) / (np.sqrt(ss, dtype=np.float32) + np.float32(eps))
    fa, fb, fc = np.float32(a), np.float32(b), np.float32(c)
    X = bf16_round(Uo)                        # X0 = bf16(U), unnormalised
    out = None
    for it in range(steps):
        first = it == 0
        acc = X @ X.T
        A = bf16_round(acc * (inv * inv if first else np.float32(1.0)))
        P = bf16_round(fc * (A @ A) + fb * A)
        Xn = (fa * X + P @ X) * (inv if first else np.float32(1.0))
        if it == steps - 1:
            out = bf16_round(Xn) if out_bf16 else Xn.astype(np.float32)
        else:
            X = bf16_round(Xn)
    if out is None:                           # zero steps: the normalised X0
        out = X * inv
    out = out.astype(np.float64)
    return out.T if transposed else out
