"""Shared test helpers: owner-buffer construction from the seeded workloads,
tolerances, and reading the blocked workspace layout back into dense arrays.
No method arithmetic lives here."""
from __future__ import annotations

import numpy as np

from matrix_optimizers_under_gb300 import workloads as W

# Tolerances (derived in the design notes from the arithmetic):
NS_REL_FRO = 2e-2      # Newton-Schulz: bf16 operands, fp32 accumulate, 5 iterations (s >= 64)
NS_REL_FRO_SMALL = 1e-1  # s < 64: bf16 rounding of A puts an absolute error on the small
                         # singular values that the quintic's steep slope near 0
                         # amplifies, with no averaging over many singular values
ADAM_REL = 1e-5        # AdamW: fp32 arithmetic against fp64
ADAM_FLOOR = 1e-2      # relative-error floor: fraction of max |reference|
MOM_REL = 4e-7         # momentum: one fp32 rounding of beta*M + G (2^-23 ~ 1.2e-7, x3 slack)


def rel_fro(x, ref) -> float:
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    nr = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / nr) if nr > 0 else float(np.linalg.norm(x))


def ns_tol(rows: int, cols: int) -> float:
    return NS_REL_FRO if min(rows, cols) >= 64 else NS_REL_FRO_SMALL


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
