"""The Gram-space form of the Newton-Schulz iteration, checked on the CPU.

One quintic step is X <- a X + b A X + c A A X = P X with A = X X^T and
P = a I + b A + c A A (MatrixFSDP -- Abstract: the owner-local update must
match full-matrix Muon).  So A_{k+1} = P_k A_k P_k and X_T = P_{T-1} ... P_0 X_0:
the library iterates s x s matrices for wide shapes and multiplies X_0 once.

  * in fp64, that sequence of products equals the oracle's iteration (the
    definition, evaluated as written) to rounding, for T = 1 .. 5, wide and
    tall shapes, and a rank-deficient input;
  * the library's choice of form per shape and step count is the rule the
    bf16 emulation (and so the derived tolerances) assumes;
  * the bf16 emulation of the Gram-space form stays within the whole-matrix
    tolerance on a wide shape.
"""
import numpy as np
import pytest

from oracle import newton_schulz_ref
from matrix_optimizers_under_gb300 import workloads as W
from tests import helpers as H
from tests.ns_emulation import bf16_round, gram_space_shape, newton_schulz_bf16

A, B, C = W.NS_COEFFS


def gram_space_f64(U, steps, a, b, c, eps):
    """The product sequence the Gram-space kernels run, in fp64 with dense
    matrices: A_0 = X_0 X_0^T; per step P = a I + b A + c A A, Q <- P Q,
    A <- (P A) P; then X = Q X_0."""
    U = np.asarray(U, np.float64)
    transposed = U.shape[0] > U.shape[1]
    X0 = U.T if transposed else U
    X0 = X0 / (np.linalg.norm(X0) + eps)
    Am = X0 @ X0.T
    s = Am.shape[0]
    Q = np.eye(s)
    for _ in range(steps):
        P = a * np.eye(s) + b * Am + c * (Am @ Am)
        Q = P @ Q
        Am = (P @ Am) @ P
    O = Q @ X0
    return O.T if transposed else O


@pytest.mark.parametrize("rows,cols", [(16, 48), (48, 16), (40, 200), (128, 256)])
@pytest.mark.parametrize("steps", [1, 2, 5])
def test_gram_space_equals_the_iteration(rows, cols, steps):
    rng = np.random.default_rng([rows, cols, steps])
    U = rng.standard_normal((rows, cols)) * 1e-3
    R = newton_schulz_ref(U, steps, A, B, C, W.NS_EPS)
    G = gram_space_f64(U, steps, A, B, C, W.NS_EPS)
    assert H.rel_fro(G, R) < 1e-12


def test_gram_space_rank_deficient():
    """A rank-2 wide input: the Gram matrix is singular, and the form still
    gives the iteration's result (zero singular values stay zero)."""
    rng = np.random.default_rng(9)
    U = rng.standard_normal((24, 2)) @ rng.standard_normal((2, 96))
    R = newton_schulz_ref(U, 5, A, B, C, W.NS_EPS)
    G = gram_space_f64(U, 5, A, B, C, W.NS_EPS)
    assert H.rel_fro(G, R) < 1e-12
    assert np.linalg.matrix_rank(G, tol=1e-9) == 2


def test_library_form_choice_matches_the_emulation(mfsdp):
    shapes = [(s, l) for s in (1, 64, 127, 128, 200, 256, 383, 384, 1000, 1408, 4096)
              for l in (s, s + 383, s + 384, 2 * s - 1, 2 * s, 2 * s + 384, 4 * s)]
    shards = [mfsdp.make_shard(0, s, l) for s, l in shapes] + [mfsdp.make_shard(0, l, s) for s, l in shapes]
    both = shapes + shapes
    for steps in (0, 1, 3, 5, 6):
        got = [g[0] for g in mfsdp.muon_gram_space_layout(shards, steps)]
        want = [1 if gram_space_shape(s, l, steps) else 0 for s, l in both]
        assert got == want, steps


def test_gram_space_emulation_error_size():
    rng = np.random.default_rng(5)
    g = bf16_round((rng.standard_normal((256, 1024)) * 1e-3).astype(np.float32))
    assert gram_space_shape(256, 1024, 5)
    O = newton_schulz_bf16(g, 5, A, B, C, W.NS_EPS)
    R = newton_schulz_ref(g.astype(np.float64), 5, A, B, C, W.NS_EPS)
    assert 1e-3 < H.rel_fro(O, R) < H.NS_REL_FRO
