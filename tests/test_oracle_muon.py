"""Pins for the fp64 Muon oracle: closed forms, textbook limits, special cases, invariants.

None of these re-types the oracle's formula: Newton-Schulz is checked through the
scalar map it induces on singular values (NumPy SVD), through the textbook cubic
iteration's limit (the polar factor), through symmetry properties, and the matmul
primitive through an explicit triple loop.
"""

import numpy as np
import pytest
import torch

from oracle import muon as M
from zero_sharded_gb300 import workloads as wl


def _svd_closed_form(X0, steps, coeffs):
    U, s, Vt = np.linalg.svd(X0, full_matrices=False)
    fs = np.array([M.ns_poly_scalar(x, coeffs, steps) for x in s])
    return (U * fs) @ Vt


def test_triple_loop_matmul_matches_numpy():
    rng = np.random.default_rng(1)
    A = rng.standard_normal((4, 6))
    B = rng.standard_normal((6, 5))
    C = np.zeros((4, 5))
    for i in range(4):
        for j in range(5):
            acc = 0.0
            for k in range(6):
                acc += A[i, k] * B[k, j]
            C[i, j] = acc
    assert np.allclose(A @ B, C, rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("shape", [(8, 12), (12, 12), (5, 16), (1, 7)])
@pytest.mark.parametrize("coeffs", [M.QUINTIC, M.CUBIC, (2.0, -1.5, 0.5)])
def test_ns_is_the_scalar_map_on_singular_values(shape, coeffs):
    """NS is an odd matrix polynomial: X_K = U f^K(Sigma) V^T for X_0 = U Sigma V^T."""
    rng = np.random.default_rng(sum(shape))
    X0 = rng.standard_normal(shape)
    X0 /= np.linalg.norm(X0)
    got = M.newton_schulz(X0, 5, coeffs)
    want = _svd_closed_form(X0, 5, coeffs)
    assert np.linalg.norm(got - want) <= 1e-10 * max(1.0, np.linalg.norm(want))


def test_cubic_converges_to_polar_factor():
    """(a,b,c) = (1.5,-0.5,0) is the textbook Newton-Schulz polar iteration (quadratic
    convergence for ||X||_2 < sqrt(3)); started from X/||X||_F it reaches U V^T."""
    for (r, c) in [(6, 9), (9, 9), (3, 11)]:
        k = min(r, c)
        sig = np.linspace(1.0, 0.05, k)
        X, U, s, V = wl.spectrum_matrix(r, c, sig, seed=r * c)
        X = X.numpy()
        polar = U.numpy() @ V.numpy().T
        out = M.orthogonalise(X, 60, M.CUBIC, eps=0.0)
        assert np.linalg.norm(out - polar) <= 1e-10 * np.linalg.norm(polar)


def test_quintic_band_and_singular_vectors():
    """Quintic K=5: for normalised singular values >= 2e-3 the outputs lie in [0.5, 1.3]
    and the singular vectors are those of the input (SVD)."""
    rng = np.random.default_rng(3)
    for (r, c) in [(16, 24), (24, 16), (20, 20)]:
        k = min(r, c)
        sig = np.exp(rng.uniform(np.log(0.004), 0.0, size=k))
        sig /= np.linalg.norm(sig)
        assert sig.min() >= 2e-3
        X, U, s, V = wl.spectrum_matrix(r, c, sig, seed=k)
        out = M.orthogonalise(X.numpy(), 5, M.QUINTIC, eps=0.0)
        so = np.linalg.svd(out, compute_uv=False)
        assert so.min() >= 0.5 and so.max() <= 1.3
        # singular vectors: U^T out V is diagonal with entries f^5(sigma)
        D = U.numpy().T @ out @ V.numpy()
        fs = np.array([M.ns_poly_scalar(x) for x in s.numpy()])
        assert np.allclose(np.diag(D), fs, atol=1e-12)
        assert np.linalg.norm(D - np.diag(np.diag(D))) <= 1e-12


def test_quintic_scalar_facts():
    assert M.ns_poly_scalar(1.0) == pytest.approx(0.6964364, abs=1e-7)
    a, b, c = M.QUINTIC
    assert a + b + c == pytest.approx(0.701, abs=1e-12)          # f(1)
    assert M.ns_poly_scalar(1.068e-3) >= 0.5                    # band threshold
    assert M.ns_poly_scalar(1.066e-3) < 0.5


def test_rank_one_closed_form():
    rng = np.random.default_rng(5)
    u = rng.standard_normal(7); u /= np.linalg.norm(u)
    v = rng.standard_normal(11); v /= np.linalg.norm(v)
    s = 3.0
    G = s * np.outer(u, v)
    out = M.orthogonalise(G, 5)
    sigma = s / (s + M.EPS)
    assert np.allclose(out, M.ns_poly_scalar(sigma) * np.outer(u, v), atol=1e-13)


def test_invariances():
    rng = np.random.default_rng(9)
    G = rng.standard_normal((10, 14))
    base = M.orthogonalise(G, 5, eps=0.0)
    assert np.allclose(M.orthogonalise(7.5 * G, 5, eps=0.0), base, atol=1e-12)       # scale
    assert np.allclose(M.orthogonalise(G.T, 5, eps=0.0), base.T, atol=1e-12)         # transpose
    Pm, _ = np.linalg.qr(rng.standard_normal((10, 10)))
    Qm, _ = np.linalg.qr(rng.standard_normal((14, 14)))
    assert np.allclose(M.orthogonalise(Pm @ G @ Qm, 5, eps=0.0), Pm @ base @ Qm, atol=1e-11)


def test_momentum_nesterov_two_steps():
    rng = np.random.default_rng(11)
    mu = 0.95
    g1 = rng.standard_normal(50).astype(np.float32)
    g2 = rng.standard_normal(50).astype(np.float32)
    m1, u1 = M.momentum(g1, np.zeros(50, np.float32), mu)
    assert np.array_equal(m1, g1)                              # m = mu*0 + g
    assert np.allclose(u1, (1 + mu) * g1.astype(np.float64), rtol=1e-7)
    m2, u2 = M.momentum(g2, m1, mu)
    assert np.allclose(m2, mu * g1.astype(np.float64) + g2, rtol=1e-6)
    assert np.allclose(u2, g2 + mu * (mu * g1.astype(np.float64) + g2), rtol=1e-6)


def test_shape_scale_and_full_step_rank_one():
    assert M.shape_scale(4, 2) == pytest.approx(np.sqrt(2))
    assert M.shape_scale(2, 4) == 1.0
    rng = np.random.default_rng(13)
    for (r, c) in [(6, 3), (3, 6)]:
        # integer factors: the outer product is exact in fp32, so g is exactly rank one
        u = rng.integers(-4, 5, size=r).astype(np.float64); u[0] = 3.0
        v = rng.integers(-4, 5, size=c).astype(np.float64); v[0] = 2.0
        g = np.outer(u, v).astype(np.float32)
        W = (0.02 * rng.standard_normal((r, c))).astype(np.float32)
        m0 = np.zeros((r, c), np.float32)
        lr, mu = 0.02, 0.95
        W1, m1, b1, delta = M.muon_step_tensor(W, g, m0, lr, mu)
        unorm = np.linalg.norm((1 + mu) * g.astype(np.float64))
        sigma = unorm / (unorm + M.EPS)
        gn = g.astype(np.float64) / np.linalg.norm(g.astype(np.float64))
        expect = lr * np.sqrt(max(1.0, r / c)) * M.ns_poly_scalar(sigma) * gn
        assert np.allclose(delta, expect, atol=1e-7 * lr)
        assert np.array_equal(W1, (W.astype(np.float64) - delta).astype(np.float32))
        assert np.array_equal(m1, g)


def test_bf16_rne_matches_known_values_and_torch():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0, 3.0e38, 1e-40], np.float32)
    bits = M.bf16_rne(vals)
    assert bits[0] == 0x3F80
    assert bits[1] == 0x3F80      # halfway, ties to even
    assert bits[2] == 0x3F82      # halfway, ties to even (up)
    assert bits[3] == 0xC020
    x = torch.randn(10000, generator=torch.Generator().manual_seed(0)) * 10
    want = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(M.bf16_rne(x.numpy()), want)
    assert np.array_equal(M.bf16_rne(vals), torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))


def test_flat_step_touches_only_owned():
    w = wl.tiny()
    p, g, m = wl.make_state(w, seed=0)
    owned = [True, False, True, False, False, True]
    P2, M2, B2, d = M.muon_step_flat(p.numpy(), g.numpy(), m.numpy(), w.offsets, w.shapes, owned, 0.02, 0.95)
    for i, (off, (r, c)) in enumerate(zip(w.offsets, w.shapes)):
        sl = slice(off, off + r * c)
        if owned[i]:
            assert not np.array_equal(P2[sl], p.numpy()[sl])
        else:
            assert np.array_equal(P2[sl], p.numpy()[sl])
            assert np.array_equal(M2[sl], m.numpy()[sl])


def test_ns_flops_formula():
    # q/k/v/o/gate/up/down of one Qwen3-1.7B layer: 2.43 TFLOP for 5 steps
    tot = sum(M.ns_flops(r, c) for r, c in wl.qwen3_1p7b_layers(1).shapes)
    assert tot == pytest.approx(2.43e12, rel=0.01)


def test_bf16_model_without_rounding_is_the_oracle_iteration():
    """The rounding model runs the oracle's iteration (only storage precision differs):
    with rounding off it matches the fp64 oracle to 1e-12 on ragged, tall and wide shapes."""
    from tests.bf16_model import orthogonalise_bf16
    rng = np.random.default_rng(11)
    for r, c in [(3, 256), (40, 17), (64, 64), (7, 1)]:
        u = rng.standard_normal((r, c))
        for steps in (1, 5):
            want = M.orthogonalise(u, steps)
            got = orthogonalise_bf16(u, steps, rounding=False)
            assert np.linalg.norm(got - want) <= 1e-12 * np.linalg.norm(want)


def test_bf16_storage_alone_can_exceed_the_update_bar():
    """A Gaussian 3 x 256 gradient: its normalised singular values all sit near 1/sqrt(3),
    f maps them near 1.2 where f' ~ 3.9, and bf16 storage alone (the rounding model)
    lands more than 2e-2 from the fp64 oracle after 5 steps, while 1 step stays well inside."""
    from tests.bf16_model import orthogonalise_bf16
    a, b, c = M.QUINTIC
    x = M.ns_poly_scalar(1 / np.sqrt(3), steps=1)
    assert 1.15 < x < 1.25 and a + 3 * b * x * x + 5 * c * x ** 4 > 3.0
    rng = np.random.default_rng(5)
    u = rng.standard_normal((3, 256))
    e5 = np.linalg.norm(orthogonalise_bf16(u, 5) - M.orthogonalise(u, 5)) / np.linalg.norm(M.orthogonalise(u, 5))
    e1 = np.linalg.norm(orthogonalise_bf16(u, 1) - M.orthogonalise(u, 1)) / np.linalg.norm(M.orthogonalise(u, 1))
    assert e1 < 1e-2
    assert e5 > 1.5e-2


def test_apply_update_hand_worked_values():
    """Step 5 on dyadic values (exact in fp32 and fp64): tall 8 x 2 has scale 2, wide 2 x 8 scale 1."""
    W = np.full((8, 2), 1.0, np.float32)
    X = np.full((8, 2), 0.5)
    assert np.array_equal(M.apply_update(W, X, 0.25), np.full((8, 2), 0.75, np.float32))      # 1 - 0.25*2*0.5
    Wt = np.full((2, 8), 1.0, np.float32)
    assert np.array_equal(M.apply_update(Wt, X.T, 0.25), np.full((2, 8), 0.875, np.float32))  # 1 - 0.25*0.5
    # no shape scale, lr = -1: the TP local add P + Delta W
    assert np.array_equal(M.apply_update(W, X, -1.0, False), np.full((8, 2), 1.5, np.float32))
    # X = 0 leaves W unchanged
    Wr = np.random.default_rng(0).standard_normal((5, 3)).astype(np.float32)
    assert np.array_equal(M.apply_update(Wr, np.zeros((5, 3)), 0.02), Wr)


def test_apply_update_rounds_once():
    """The fp64 result is rounded to fp32 once: 1 - 2^-25 is a tie between 1 - 2^-24 and 1
    (goes to 1, even mantissa); 1 - 3*2^-26 is nearer to 1 - 2^-24."""
    one = np.ones((1, 1), np.float32)
    assert M.apply_update(one, np.full((1, 1), 2.0 ** -25), 1.0, False)[0, 0] == np.float32(1.0)
    assert M.apply_update(one, np.full((1, 1), 3 * 2.0 ** -26), 1.0, False)[0, 0] == np.float32(1.0 - 2.0 ** -24)
