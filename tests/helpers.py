"""Shared test helpers: owner-buffer construction from the seeded workloads,
tolerances, and reading the blocked workspace layout back into dense arrays.
No method arithmetic lives here."""
from __future__ import annotations

import numpy as np

from matrix_optimizers_under_gb300 import workloads as W

# Tolerances (derived from the arithmetic; tests/derive_ns_tolerances.py
# prints the Newton-Schulz ones from a bf16 emulation of the GPU's precision):
NS_REL_FRO = 2e-2      # Newton-Schulz, s >= 64: bf16 operands, fp32 accumulate, 5 iterations
# s < 64: 1.5x the emulated maximum (bf16 rounding of A puts an absolute error
# on the small singular values that the quintic's steep slope near 0
# amplifies, with no averaging over many singular values).  First the shapes
# the tests run (200 seeds of the tests' input each), then, for other shapes,
# per short-side class: (s_lo, s_hi, near-square l < 2s, wide l >= 2s).
NS_TOL_SHAPE = {(1, 1): 0.033, (1, 9): 0.040, (9, 1): 0.041, (7, 300): 0.027, (300, 7): 0.029}
NS_TOL_CLASS = ((1, 1, 0.024, 0.044), (2, 3, 0.226, 0.121), (4, 7, 0.226, 0.092), (8, 15, 0.114, 0.047),
                (16, 31, 0.050, 0.038), (32, 63, 0.027, 0.039))
# Full-size matrices, every 128 x 128 block of the stored update (ragged edge
# blocks included): relative Frobenius error, and the largest elementwise
# error over (block RMS + |reference element|); 1.5x the emulated maxima of
# the standard program over the workloads' shapes (1.33 %, 0.060).  The
# Gram-space program's maxima (1.11 %, 0.077 at 14336 x 4096 with Student-t
# input) stay inside them.
NS_BLOCK_REL = 2e-2
NS_BLOCK_ELEM = 0.091
ADAM_REL = 1e-5        # AdamW: fp32 arithmetic against fp64
ADAM_FLOOR = 1e-2      # relative-error floor: fraction of max |reference|
MOM_REL = 4e-7         # momentum: one fp32 rounding of beta*M + G (2^-23 ~ 1.2e-7, x3 slack)


def rel_fro(x, ref) -> float:
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    nr = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / nr) if nr > 0 else float(np.linalg.norm(x))


def ns_tol(rows: int, cols: int) -> float:
    s, l = min(rows, cols), max(rows, cols)
    if s >= 64:
        return NS_REL_FRO
    if (rows, cols) in NS_TOL_SHAPE:
        return NS_TOL_SHAPE[(rows, cols)]
    for lo, hi, square, wide in NS_TOL_CLASS:
        if lo <= s <= hi:
            return wide if l >= 2 * s else square
    raise AssertionError("unreachable")


def block_errors(O, R, block: int = 128):
    """Per block x block tile of the stored matrix (ragged edge tiles
    included): the relative Frobenius error ||O - R|| / ||R||, and the largest
    elementwise error measured against the block's RMS plus the element's own
    magnitude, max |O - R| / (rms(R) + |R|) -- heavy-tailed inputs give
    updates whose largest entries are tens of RMS and carry their own bf16
    rounding.  Returns two arrays of shape (ceil(rows / block), ceil(cols /
    block))."""
    O = np.asarray(O, np.float64)
    R = np.asarray(R, np.float64)
    rows, cols = R.shape
    nb_r, nb_c = -(-rows // block), -(-cols // block)
    pad = ((0, nb_r * block - rows), (0, nb_c * block - cols))
    D = np.pad(O - R, pad).reshape(nb_r, block, nb_c, block)
    Rp = np.pad(R, pad).reshape(nb_r, block, nb_c, block)
    cnt = np.pad(np.ones_like(R), pad).reshape(nb_r, block, nb_c, block).sum(axis=(1, 3))
    err2 = np.sum(D * D, axis=(1, 3))
    ref2 = np.sum(Rp * Rp, axis=(1, 3))
    rel = np.where(ref2 > 0, np.sqrt(err2 / np.where(ref2 > 0, ref2, 1.0)), np.sqrt(err2))
    rms = np.sqrt(ref2 / cnt)
    den = rms[:, None, :, None] + np.abs(Rp)
    elem = np.max(np.abs(D) / np.where(den > 0, den, 1.0), axis=(1, 3))
    return rel, elem


def check_blocks(O, ref, what="") -> None:
    """Every 128 x 128 block of a full-size update within the block bounds."""
    rel, mx = block_errors(O, ref)
    bad = np.argwhere((rel > NS_BLOCK_REL) | (mx > NS_BLOCK_ELEM))
    assert bad.size == 0, (f"{what}: {len(bad)} blocks out of bounds, first {tuple(bad[0])}: "
                           f"rel {rel[tuple(bad[0])]:.3e}, elementwise {mx[tuple(bad[0])]:.3f}")


def adam_err(x, ref) -> float:
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    floor = ADAM_FLOOR * np.max(np.abs(ref)) if ref.size else 0.0
    den = np.maximum(np.abs(ref), floor)
    den[den == 0] = 1.0
    return float(np.max(np.abs(x - ref) / den)) if ref.size else 0.0


def heaviest_rank(plan) -> int:
    """Largest Newton-Schulz cost, then smallest tail, then lowest id."""
    world = len(plan.rank_matrix_elems)
    cost = [0] * world
    tail = [0] * world
    for s in plan.matrix_shards:
        cost[s.owner] += s.cost
    for s in plan.tail_shards:
        tail[s.owner] += s.numel
    return min(range(world), key=lambda r: (-cost[r], tail[r], r))


def build_grad_buffer(w: W.Workload, shards, numel: int, only=None) -> np.ndarray:
    """Flat gradient buffer of one rank as stored: uint16 bf16 bits or float32.
    Padding between segments is filled with a canary pattern."""
    if w.grad_dtype == "bf16":
        buf = np.full(numel, 0x7FC1, np.uint16)       # a NaN pattern: must never be read
    else:
        buf = np.full(numel, np.nan, np.float32)
    for s in shards:
        if only is not None and s.param_id not in only:
            g = np.zeros(s.rows * s.cols, buf.dtype)
        else:
            g = W.grad_storage(w, s.param_id).reshape(-1)
        buf[s.offset:s.offset + s.rows * s.cols] = g
    return buf


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def unblock(ws_bytes: np.ndarray, off: int, rows_pad: int, cols_pad: int) -> np.ndarray:
    """Dense float32 copy of a blocked, pre-swizzled bf16 matrix in the workspace
    (layout documented in include/mfsdp.h)."""
    raw = ws_bytes[off: off + rows_pad * cols_pad * 2].view(np.uint16)
    atoms = raw.reshape(cols_pad // 64, rows_pad // 8, 8, 8, 8)   # [colblk, rowgrp, r, chunk(swz), e]
    r = np.arange(8)
    out = np.empty((cols_pad // 64, rows_pad // 8, 8, 8, 8), np.uint16)
    for ch in range(8):
        out[:, :, r, ch, :] = atoms[:, :, r, ch ^ r, :]
    dense = out.transpose(1, 2, 0, 3, 4).reshape(rows_pad, cols_pad)
    return bf16_bits_to_f32(dense)


def symmetric_from_upper(m: np.ndarray, block: int = 256) -> np.ndarray:
    """The full symmetric matrix from its blocks on or above the block diagonal
    (block x block blocks), the form in which the workspace keeps A and B: each
    block below the diagonal is the transpose of its mirror image."""
    out = m.copy()
    nb = m.shape[0] // block
    for i in range(nb):
        for j in range(i):
            out[i * block:(i + 1) * block, j * block:(j + 1) * block] = \
                m[j * block:(j + 1) * block, i * block:(i + 1) * block].T
    return out
