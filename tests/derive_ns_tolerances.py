"""Derives the Newton-Schulz tolerances of the GPU tests from the bf16
emulation (tests/ns_emulation.py) against the fp64 oracle, and prints them.

  python tests/derive_ns_tolerances.py small    # per shape (s < 64) and per short-side class
  python tests/derive_ns_tolerances.py blocks   # per 128 x 128 block, workload shapes

small: first, for each shape with s < 64 that the GPU tests use, the largest
relative Frobenius error of the emulated update over 200 seeds of the tests'
input (a second step: U = 0.95 M + G with M, G ~ N(0, 1e-3); fp32 and bf16
gradients alternating); its tolerance is 1.5x that maximum, rounded up to the
next 1e-3, and never below 2e-2.  Then, for shapes the tests do not name,
for every short-side class [1], [2, 3], [4, 7], [8, 15], [16, 31],
[32, 63], split by aspect into near-square (l < 2s) and wide (l >= 2s), the
largest relative Frobenius error of the emulated update over shapes s x l and
l x s of the class (near-square: l in {s, 3s/2}; wide: l in {2s, 2s + 1, 9s,
300}) and 100 seeds each, half with fp32 and half with bf16 gradients, half
from zero momentum and half from a second step (U = 0.95 M + G with M, G ~
N(0, 1e-3)).  The test tolerance of a class is 1.5x its maximum, rounded up
to the next 1e-3, and never below the 2e-2 that holds for s >= 64.  Square
matrices need the split: a random near-square matrix has singular values
close to 0, where the quintic's slope (a^5 ~ 486 at 0) amplifies the bf16
rounding of A; a wide one keeps its smallest singular value near
(1 - sqrt(s / l)) times the typical one.

blocks: for the workloads' matrix shapes, the largest per-block relative
Frobenius error and the largest elementwise error over (block RMS +
|reference element|), over every 128 x 128 block of the emulated update (the 8B shapes with
Student-t(3) gradients, the others with normal ones), one draw per shape.
"""
from __future__ import annotations

import math
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle import newton_schulz_ref  # noqa: E402
from matrix_optimizers_under_gb300 import workloads as W  # noqa: E402
from tests.helpers import block_errors  # noqa: E402
from tests.ns_emulation import bf16_round, newton_schulz_bf16  # noqa: E402

A, B, C = W.NS_COEFFS
CLASSES = ((1, 1), (2, 3), (4, 7), (8, 15), (16, 31), (32, 63))


def rel_fro(x, r):
    n = np.linalg.norm(r)
    return float(np.linalg.norm(x - r) / n) if n > 0 else float(np.linalg.norm(x))


def case_error(rows, cols, seed, bf16_grad, second_step):
    rng = np.random.default_rng([11, rows, cols, seed])
    g = (rng.standard_normal((rows, cols)) * 1e-3).astype(np.float32)
    if bf16_grad:
        g = bf16_round(g)
    m0 = (rng.standard_normal((rows, cols)) * 1e-3).astype(np.float32) if second_step else \
        np.zeros((rows, cols), np.float32)
    U32 = np.float32(0.95) * m0 + g                 # the fp32 momentum the kernels hold
    U64 = 0.95 * m0.astype(np.float64) + g.astype(np.float64)
    O = newton_schulz_bf16(U32, W.NS_STEPS, A, B, C, W.NS_EPS)
    R = newton_schulz_ref(U64, W.NS_STEPS, A, B, C, W.NS_EPS)
    return rel_fro(O, R)


def class_shapes(lo, hi, wide):
    out = []
    for s in sorted({lo, (lo + hi) // 2, hi}):
        ls = {2 * s, 2 * s + 1, 9 * s} | ({300} if 300 >= 2 * s else set()) if wide else \
            {l for l in (s, s + s // 2) if l < 2 * s}
        for l in sorted(ls):
            out.append((s, l))
            if l != s:
                out.append((l, s))
    return out


# The shapes with s < 64 the GPU tests run (the ragged owner set).
TEST_SHAPES = ((1, 1), (1, 9), (9, 1), (7, 300), (300, 7))


def tolerance(worst):
    return max(2e-2, math.ceil(1.5 * worst * 1e3) / 1e3)


def small(seeds=100):
    for shape in TEST_SHAPES:
        worst, at = 0.0, None
        for k in range(2 * seeds):
            e = case_error(shape[0], shape[1], k, bf16_grad=bool(k & 1), second_step=True)
            if e > worst:
                worst, at = e, k
        print(f"shape {shape}: emulated max {worst:.4f} (seed {at}) -> tolerance {tolerance(worst):.3f}", flush=True)
    rows = []
    for lo, hi in CLASSES:
        for wide in (False, True):
            worst, where = 0.0, None
            for shape in class_shapes(lo, hi, wide):
                for k in range(seeds):
                    e = case_error(shape[0], shape[1], k, bf16_grad=bool(k & 1), second_step=bool(k & 2))
                    if e > worst:
                        worst, where = e, (shape, k)
            tol = tolerance(worst)
            rows.append((lo, hi, wide, worst, where, tol))
            print(f"s in [{lo}, {hi}], {'l >= 2s' if wide else 'l < 2s'}: emulated max {worst:.4f} at {where[0]} "
                  f"seed {where[1]} -> tolerance {tol:.3f}", flush=True)
    return rows


def blocks():
    shapes = [("gpt2_block", 768, 2304), ("gpt2_block", 3072, 768), ("llama_1p3b_rank", 5504, 2048),
              ("llama_1p3b_rank", 2048, 2048), ("moe_skewed", 1408, 2048), ("moe_skewed", 2048, 1408),
              ("llama3_8b_rank", 1024, 4096), ("llama3_8b_rank", 4096, 4096), ("llama3_8b_rank", 14336, 4096)]
    worst_rel, worst_max = 0.0, 0.0
    for name, rows, cols in shapes:
        w = W.get(name)
        rng = np.random.default_rng([w.seed, rows, cols, 99])
        if w.grad_dist == "student_t3":
            g = (rng.standard_t(3, size=(rows, cols)) * w.grad_scale).astype(np.float32)
        else:
            g = (rng.standard_normal((rows, cols)) * w.grad_scale).astype(np.float32)
        g = bf16_round(g)
        O = bf16_round(newton_schulz_bf16(g, W.NS_STEPS, A, B, C, W.NS_EPS).astype(np.float32))   # bf16 update
        R = newton_schulz_ref(g.astype(np.float64), W.NS_STEPS, A, B, C, W.NS_EPS)
        rel, mx = block_errors(O, R)
        worst_rel, worst_max = max(worst_rel, rel.max()), max(worst_max, mx.max())
        print(f"{name} {rows}x{cols}: whole {rel_fro(O, R):.4f}, block rel max {rel.max():.4f} "
              f"(median {np.median(rel):.4f}), elementwise max {mx.max():.4f}", flush=True)
    print(f"all shapes: block rel max {worst_rel:.4f}, elementwise max {worst_max:.4f}")


if __name__ == "__main__":
    what = sys.argv[1] if len(sys.argv) > 1 else "small"
    small() if what == "small" else blocks()
