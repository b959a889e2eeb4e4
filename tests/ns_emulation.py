"""A bf16 emulation of the GPU's Newton-Schulz precision, for deriving test
tolerances.  Test infrastructure: it is neither the oracle (that is the fp64
definition in oracle/) nor the product; nothing outside tests/ uses it.

It follows the precision choices the library documents for its
Newton-Schulz products (bf16 operands and stored A, B and X; fp32
accumulation and fp32 epilogue arithmetic; the Frobenius prescale taken in
fp32 from the unrounded momentum and folded into the first iteration's
epilogues), written with NumPy fp32 matrix products, and the library's choice
between the direct form and the Gram-space form of the iteration (the shape
rule include/mfsdp.h states; A, P, C and Q stored in bf16 as their 256 x 256
blocks on or above the diagonal, the others their mirror images'
transposes, and each product the true product of the stored matrices).  Its accumulation order
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


def gram_space_shape(s: int, l: int, steps: int) -> bool:
    """The shapes and step counts the library runs in Gram space (include/mfsdp.h)."""
    return s >= 128 and l >= 2 * s and l >= s + 384 and 1 <= steps <= 5


def stored_symmetric(M: np.ndarray, block: int = 256) -> np.ndarray:
    """A symmetric product as the library keeps it: blocks on or above the
    diagonal of block x block blocks as computed (a diagonal block whole), the
    others the transposes of their mirror images."""
    out = M.copy()
    nb = -(-M.shape[0] // block)
    for i in range(nb):
        for j in range(i):
            out[i * block:(i + 1) * block, j * block:(j + 1) * block] = \
                M[j * block:(j + 1) * block, i * block:(i + 1) * block].T
    return out


def newton_schulz_gram_bf16(U: np.ndarray, steps: int, a: float, b: float, c: float, eps: float,
                            out_bf16: bool = False) -> np.ndarray:
    """The Gram-space form in bf16: A_0 = X0 X0^T (prescaled); per iteration
    P = a I + b A + c A A, C = P A, A <- C P, Q <- P Q (Q_0 = P_0); X = Q X0
    (prescaled).  Returns the update like newton_schulz_bf16."""
    U = np.asarray(U, dtype=np.float32)
    transposed = U.shape[0] > U.shape[1]
    Uo = U.T if transposed else U
    ss = np.float32(np.sum(np.square(Uo, dtype=np.float32), dtype=np.float32))
    inv = np.float32(1.0) / (np.sqrt(ss, dtype=np.float32) + np.float32(eps))
    fa, fb, fc = np.float32(a), np.float32(b), np.float32(c)
    X0 = bf16_round(Uo)
    A = stored_symmetric(bf16_round((X0 @ X0.T) * (inv * inv)))
    s = A.shape[0]
    Q = None
    for it in range(steps):
        P = fc * (A @ A) + fb * A
        P[np.diag_indices(s)] += fa
        P = stored_symmetric(bf16_round(P))
        Q = P if Q is None else stored_symmetric(bf16_round(P @ Q))
        if it < steps - 1:
            Cm = stored_symmetric(bf16_round(P @ A))
            A = stored_symmetric(bf16_round(Cm @ P))
    out = (Q @ X0) * inv
    out = bf16_round(out) if out_bf16 else out.astype(np.float32)
    out = out.astype(np.float64)
    return out.T if transposed else out


def newton_schulz_bf16(U: np.ndarray, steps: int, a: float, b: float, c: float, eps: float,
                       out_bf16: bool = False) -> np.ndarray:
    """Update O (float64, the stored shape of U) of the bf16 pipeline, in the
    form the library runs for this shape and step count.

    U is the fp32 momentum (the Newton-Schulz input before normalisation)."""
    U = np.asarray(U, dtype=np.float32)
    if gram_space_shape(min(U.shape), max(U.shape), steps):
        return newton_schulz_gram_bf16(U, steps, a, b, c, eps, out_bf16)
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
