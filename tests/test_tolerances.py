"""The Newton-Schulz tolerances of the GPU tests, checked on the CPU against the
bf16 emulation they were derived from (tests/derive_ns_tolerances.py), and
the block check of the full-size tests against a planted error.

  * every per-shape tolerance is at least 1.5x the emulated error over the
    first 40 of the 200 seeds it was derived from;
  * the emulation rounds like bf16 (ties to even) and, on a workload-like
    shape, lands between 1e-3 and the 2e-2 tolerance of the oracle;
  * a wrong 128 x 128 block in an otherwise exact update is caught by the
    per-block bounds although the whole-matrix error stays within 2e-2.
"""
import numpy as np
import pytest

from oracle import newton_schulz_ref
from matrix_optimizers_under_gb300 import workloads as W
from tests import helpers as H
from tests.derive_ns_tolerances import TEST_SHAPES, case_error
from tests.helpers import block_errors  # noqa: E402
from tests.ns_emulation import bf16_round, newton_schulz_bf16

A, B, C = W.NS_COEFFS


def test_bf16_round_ties_to_even():
    one = np.float32(1.0)
    ulp = np.float32(2.0 ** -7)
    x = np.array([1.0, 1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 1 + 2.0 ** -8 + 2.0 ** -20, -2.5, 0.0], np.float32)
    want = np.array([1.0, 1.0, 1 + 2 * 2.0 ** -7, 1 + 2.0 ** -7, -2.5, 0.0], np.float32)
    assert np.array_equal(bf16_round(x), want)
    assert bf16_round(np.array([one + ulp], np.float32))[0] == one + ulp


@pytest.mark.parametrize("shape", TEST_SHAPES)
def test_small_shape_tolerance_covers_emulation(shape):
    worst = max(case_error(shape[0], shape[1], k, bf16_grad=bool(k & 1), second_step=True) for k in range(40))
    assert worst * 1.5 <= H.NS_TOL_SHAPE[shape] + 1e-12, (shape, worst)
    assert H.ns_tol(*shape) == H.NS_TOL_SHAPE[shape]


def test_tolerance_lookup():
    assert H.ns_tol(64, 64) == H.NS_REL_FRO and H.ns_tol(4096, 14336) == H.NS_REL_FRO
    assert H.ns_tol(8, 8) == 0.114 and H.ns_tol(8, 64) == 0.047 and H.ns_tol(64, 8) == 0.047
    assert all(H.ns_tol(s, l) >= H.NS_REL_FRO for s in range(1, 64) for l in (s, 2 * s, 1000))


def test_emulation_error_size():
    rng = np.random.default_rng(3)
    g = bf16_round((rng.standard_normal((128, 384)) * 1e-3).astype(np.float32))
    O = newton_schulz_bf16(g, 5, A, B, C, W.NS_EPS)
    R = newton_schulz_ref(g.astype(np.float64), 5, A, B, C, W.NS_EPS)
    assert 1e-3 < H.rel_fro(O, R) < H.NS_REL_FRO


def test_block_bound_catches_one_wrong_block():
    """Plant mistakes in the oracle's own update that the whole-matrix bound
    lets through: one 128 x 128 block 10 % too large (a wrong scale in one
    tile's epilogue), and one element off by the block's RMS.  The block
    checks catch each; nothing else is flagged."""
    rng = np.random.default_rng(4)
    g = (rng.standard_normal((512, 1536)) * 1e-3)
    R = newton_schulz_ref(g, 5, A, B, C, W.NS_EPS)
    O = R.copy()
    O[128:256, 384:512] *= 1.1
    rms = np.sqrt(np.mean(R[384:512, 1024:1152] ** 2))
    O[400, 1100] += rms
    assert H.rel_fro(O, R) <= H.NS_REL_FRO
    rel, mx = block_errors(O, R)
    assert rel[1, 3] > H.NS_BLOCK_REL
    assert mx[3, 8] > H.NS_BLOCK_ELEM and rel[3, 8] <= H.NS_BLOCK_REL
    rel[1, 3] = mx[1, 3] = rel[3, 8] = mx[3, 8] = 0.0
    assert rel.max() == 0.0 and mx.max() == 0.0
    # the ragged edge block is measured over its own elements only
    rel, _ = block_errors(R[:300, :200] * (1 + 3e-2), R[:300, :200])
    assert rel.shape == (3, 2) and np.allclose(rel, 3e-2)
