"""Pins for the oracle's Newton-Schulz and momentum.

MatrixFSDP -- Abstract: Muon orthogonalises momentum-smoothed updates with
Newton-Schulz on the complete 2D matrix.  The iteration X <- a X + b (XX^T) X +
c (XX^T)^2 X acts on each singular value separately through the scalar quintic
f(x) = a x + b x^3 + c x^5, so the whole method has a closed form through the
SVD.  These tests check the matrix iteration against that closed form, against
values of the scalar polynomial, special cases and invariances; none of them
re-calls the oracle's own iteration to produce an expected value.
"""
import numpy as np
import pytest

from oracle import momentum_ref, newton_schulz_ref, muon_matrix_ref

A, B, C = 3.4445, -4.7750, 2.0315
EPS = 1e-7


def phi(x, steps=5, a=A, b=B, c=C):
    """Scalar composition f^(steps)(x), f(x) = a x + b x^3 + c x^5 (Horner form)."""
    x = np.asarray(x, dtype=np.float64)
    for _ in range(steps):
        x2 = x * x
        x = x * (a + x2 * (b + c * x2))
    return x


def svd_closed_form(U, steps, eps, a=A, b=B, c=C):
    P, s, Qt = np.linalg.svd(U, full_matrices=False)
    n = np.linalg.norm(s)   # Frobenius norm = 2-norm of the singular values
    return (P * phi(s / (n + eps), steps, a, b, c)) @ Qt


def test_phi_values_from_hand_evaluation():
    # f(1) = a + b + c = 0.701 exactly; then four more rounds.
    assert phi(1.0, 1) == pytest.approx(0.701, abs=1e-15)
    assert phi(1.0) == pytest.approx(0.6964364094697522, rel=1e-14)
    assert phi(0.0) == 0.0


@pytest.mark.parametrize("shape", [(8, 16), (16, 8), (32, 32), (5, 3), (1, 9), (9, 1)])
@pytest.mark.parametrize("steps", [0, 1, 2, 5])
def test_ns_equals_svd_closed_form(shape, steps):
    rng = np.random.default_rng(shape[0] * 100 + shape[1] + 7 * steps)
    U = rng.standard_normal(shape)
    O = newton_schulz_ref(U, steps, A, B, C, EPS)
    assert O.shape == U.shape
    np.testing.assert_allclose(O, svd_closed_form(U, steps, EPS), atol=1e-12, rtol=0)


def test_ns_small_norm_eps_placement():
    # ||U|| = 1e-6 so eps=1e-7 shifts the normalised spectrum by ~9%: a misplaced
    # eps (inside a square root, or added to each element) fails this.
    rng = np.random.default_rng(3)
    U = rng.standard_normal((12, 20))
    U *= 1e-6 / np.linalg.norm(U)
    O = newton_schulz_ref(U, 5, A, B, C, EPS)
    np.testing.assert_allclose(O, svd_closed_form(U, 5, EPS), atol=1e-12, rtol=0)
    _, s, _ = np.linalg.svd(U, full_matrices=False)
    _, so, _ = np.linalg.svd(O, full_matrices=False)
    np.testing.assert_allclose(np.sort(so), np.sort(phi(s / (1e-6 + EPS))), atol=1e-12)


def test_singular_value_band():
    # For normalised singular values in [1e-2, 1] the quintic keeps the output's
    # singular values inside [0.6818, 1.1344] (the scalar map's range there).
    rng = np.random.default_rng(11)
    for trial in range(20):
        m, n = 24, 40
        P, _ = np.linalg.qr(rng.standard_normal((m, m)))
        Q, _ = np.linalg.qr(rng.standard_normal((n, m)))
        s = rng.uniform(0.06, 1.0, size=m)
        U = (P * s) @ Q.T
        assert (s / np.linalg.norm(s)).min() >= 1e-2
        O = newton_schulz_ref(U, 5, A, B, C, EPS)
        so = np.linalg.svd(O, compute_uv=False)
        assert so.min() >= 0.6818 and so.max() <= 1.1344


def test_rank_one():
    rng = np.random.default_rng(5)
    u = rng.standard_normal(10); u /= np.linalg.norm(u)
    v = rng.standard_normal(30); v /= np.linalg.norm(v)
    O = newton_schulz_ref(np.outer(u, v), 5, A, B, C, 0.0)
    np.testing.assert_allclose(O, 0.6964364094697522 * np.outer(u, v), atol=1e-13)


def test_zero_matrix_gives_exact_zero():
    O = newton_schulz_ref(np.zeros((7, 13)), 5, A, B, C, EPS)
    assert np.all(O == 0.0) and np.all(np.isfinite(O))


def test_orthonormal_rows():
    rng = np.random.default_rng(9)
    s, l = 16, 48
    Q, _ = np.linalg.qr(rng.standard_normal((l, s)))
    X = Q.T   # s x l, orthonormal rows, every singular value 1
    O = newton_schulz_ref(X, 5, A, B, C, 0.0)
    np.testing.assert_allclose(O, phi(1.0 / np.sqrt(s)) * X, atol=1e-13)


def test_invariances():
    rng = np.random.default_rng(21)
    U = rng.standard_normal((12, 18))
    O = newton_schulz_ref(U, 5, A, B, C, 0.0)
    # scale
    np.testing.assert_allclose(newton_schulz_ref(37.5 * U, 5, A, B, C, 0.0), O, atol=1e-12)
    # transpose
    np.testing.assert_array_equal(newton_schulz_ref(U.T, 5, A, B, C, 0.0), O.T)
    S = rng.standard_normal((15, 15))
    np.testing.assert_allclose(newton_schulz_ref(S.T, 5, A, B, C, 0.0),
                               newton_schulz_ref(S, 5, A, B, C, 0.0).T, atol=1e-12)
    # orthogonal equivariance
    P, _ = np.linalg.qr(rng.standard_normal((12, 12)))
    Q, _ = np.linalg.qr(rng.standard_normal((18, 18)))
    np.testing.assert_allclose(newton_schulz_ref(P @ U @ Q, 5, A, B, C, 0.0), P @ O @ Q, atol=1e-12)


def test_distance_to_polar_factor_bounded():
    # ||O - U V^T||_2 = max_i |phi(sigma_i) - 1| for well-conditioned input.
    rng = np.random.default_rng(31)
    P, _ = np.linalg.qr(rng.standard_normal((8, 8)))
    Q, _ = np.linalg.qr(rng.standard_normal((20, 8)))
    s = np.linspace(1.0, 3.0, 8)
    U = (P * s) @ Q.T
    O = newton_schulz_ref(U, 5, A, B, C, 0.0)
    polar = P @ Q.T
    bound = np.max(np.abs(phi(s / np.linalg.norm(s)) - 1.0))
    assert np.linalg.norm(O - polar, 2) <= bound + 1e-12


def test_momentum_closed_forms():
    rng = np.random.default_rng(2)
    G1, G2 = rng.standard_normal((2, 6, 4)).astype(np.float32).astype(np.float64)
    beta = 0.95
    M1, U1 = momentum_ref(G1, np.zeros_like(G1), beta, False)
    assert np.array_equal(M1, G1) and np.array_equal(U1, G1)
    M2, U2 = momentum_ref(G2, M1, beta, False)
    np.testing.assert_allclose(M2, beta * G1 + G2, rtol=0, atol=1e-15)
    np.testing.assert_array_equal(U2, M2)
    _, U1n = momentum_ref(G1, np.zeros_like(G1), beta, True)
    np.testing.assert_allclose(U1n, (1 + beta) * G1, rtol=1e-15)
    _, U2n = momentum_ref(G2, M1, beta, True)
    np.testing.assert_allclose(U2n, G2 + beta * (beta * G1 + G2), rtol=1e-14)


def test_step_one_nesterov_and_heavy_ball_agree_after_normalisation():
    # From zero momentum every variant gives U proportional to G, and the
    # normalisation makes O identical up to eps.
    rng = np.random.default_rng(4)
    G = rng.standard_normal((8, 12))
    _, O1 = muon_matrix_ref(G, np.zeros_like(G), 0.95, False, 5, A, B, C, 0.0)
    _, O2 = muon_matrix_ref(G, np.zeros_like(G), 0.95, True, 5, A, B, C, 0.0)
    np.testing.assert_allclose(O1, O2, atol=1e-12)


def test_apply_scale_forms():
    from oracle import muon_scale_ref
    assert muon_scale_ref(4096, 1024, 0) == 1.0
    assert muon_scale_ref(4096, 1024, 1) == 2.0          # sqrt(4096/1024)
    assert muon_scale_ref(1024, 4096, 1) == 1.0          # wide matrices are not scaled down
    assert muon_scale_ref(4096, 1024, 2) == pytest.approx(12.8)   # 0.2 * sqrt(4096)
    assert muon_scale_ref(100, 2500, 2) == pytest.approx(10.0)    # 0.2 * sqrt(2500)


def test_apply_special_cases():
    from oracle import muon_apply_ref
    rng = np.random.default_rng(8)
    W, O = rng.standard_normal((2, 6, 9))
    np.testing.assert_array_equal(muon_apply_ref(W, O, 0.0, 0.1, 3.0), W)          # lr = 0
    np.testing.assert_allclose(muon_apply_ref(W, O, 0.02, 0.0, 1.0), W - 0.02 * O, rtol=0, atol=1e-15)
    np.testing.assert_allclose(muon_apply_ref(W, np.zeros_like(O), 0.02, 0.5, 7.0), 0.99 * W, rtol=1e-15)
    # one step on W = O with lr*wd = 0 and scale = 1/lr cancels exactly
    np.testing.assert_allclose(muon_apply_ref(O, O, 0.5, 0.0, 2.0), 0 * O, atol=1e-15)


def test_bf16_bits_to_f64_ieee_values():
    """bf16 is the top half of an IEEE binary32: sign, 8 exponent bits, 7
    fraction bits.  Values fixed by that definition, including the smallest
    subnormal and the largest finite value."""
    from oracle import bf16_bits_to_f64
    bits = np.array([0x0000, 0x8000, 0x3F80, 0xBF80, 0x4049, 0x3F81, 0x0001, 0x0080, 0x7F7F, 0x7F80, 0xFF80],
                    np.uint16)
    want = np.array([0.0, -0.0, 1.0, -1.0, 3.140625, 1 + 2.0 ** -7, 2.0 ** -133, 2.0 ** -126,
                     (2 - 2.0 ** -7) * 2.0 ** 127, np.inf, -np.inf])
    got = bf16_bits_to_f64(bits)
    assert got.dtype == np.float64
    assert np.array_equal(got, want) and np.signbit(got[1])
    assert np.isnan(bf16_bits_to_f64(np.array([0x7FC1], np.uint16)))[0]


def test_owner_step_over_a_flat_buffer():
    """The flat-buffer owner step: two matrices (one wide, one tall) at ragged
    offsets of one buffer, with padding between and after them.  Each matrix's
    update is the SVD closed form of its own momentum-smoothed slice, its
    momentum is beta M + G on that slice, and every padding element of the
    momentum buffer comes back unchanged; `only` restricts the work."""
    from oracle.muon import muon_owner_step_ref, stored_to_f64
    rng = np.random.default_rng(21)
    shapes, offsets = [(6, 10), (12, 5)], [3, 3 + 60 + 4]
    numel = offsets[1] + 60 + 7
    G32 = (rng.standard_normal(numel) * 1e-2).astype(np.float32)
    bits = (G32.view(np.uint32) >> 16).astype(np.uint16)        # truncated to bf16: exact bf16 values
    M0 = rng.standard_normal(numel)
    shards = [dict(param_id=i, offset=o, rows=r, cols=c) for i, ((r, c), o) in enumerate(zip(shapes, offsets))]
    beta = 0.9
    for dtype, buf in (("f32", G32), ("bf16", bits)):
        Gall = stored_to_f64(buf, dtype)
        if dtype == "bf16":
            assert np.array_equal(Gall, ((bits.astype(np.uint32) << 16).view(np.float32)).astype(np.float64))
        else:
            assert np.array_equal(Gall, G32.astype(np.float64))
        M, out = muon_owner_step_ref(shards, buf, dtype, M0, beta, False, 5, A, B, C, EPS)
        used = np.zeros(numel, bool)
        for sh in shards:
            o, r, c = sh["offset"], sh["rows"], sh["cols"]
            used[o:o + r * c] = True
            G = Gall[o:o + r * c].reshape(r, c)
            Mi = beta * M0[o:o + r * c].reshape(r, c) + G
            np.testing.assert_allclose(M[o:o + r * c].reshape(r, c), Mi, rtol=1e-15, atol=0)
            assert out[sh["param_id"]].shape == (r, c)
            np.testing.assert_allclose(out[sh["param_id"]], svd_closed_form(Mi, 5, EPS), atol=1e-12, rtol=0)
        assert np.array_equal(M[~used], M0[~used])
    M, out = muon_owner_step_ref(shards, G32, "f32", M0, beta, False, 5, A, B, C, EPS, only=[1])
    assert list(out) == [1]
    o = offsets[0]
    assert np.array_equal(M[o:o + 60], M0[o:o + 60])
    with pytest.raises(ValueError):
        stored_to_f64(G32, "f16")
