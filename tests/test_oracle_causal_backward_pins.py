"""Pins of the float64 causal backward oracle against what the mathematics fixes.

None of these compares an oracle function with itself: central finite
differences of the (separately pinned) causal forward; the blocked reverse walk
against the matrix-form derivative of the explicit causal N x N form (two
independent derivations); causality of the gradients; zero gradient for the
entries of W above the diagonal; Euler's identities of the forward's
homogeneity; linearity in dout.  A dropped own-block term, a prefix sum taken
over the wrong side (t <= s instead of t >= s), a transposed W or a missing
W[i, i] fails at least one of them.
"""

import numpy as np
import pytest

import oracle
from oracle.mhla_causal_backward import backward_causal, backward_causal_dense


def away_from_zero(shape, rng, margin=0.05):
    x = rng.standard_normal(shape)
    return np.where(np.abs(x) < margin, np.sign(x + 1e-300) * margin, x)


CASES = [
    # (B, N, H, d, grid, block): contiguous blocks only
    (1, 12, 2, 3, (1, 12), (1, 4)),        # a 1-D sequence in three chunks
    (2, 16, 1, 2, (4, 4), (1, 4)),          # whole rows of a grid
    (1, 16, 1, 3, (2, 2, 4), (1, 2, 4)),    # whole frames of a 3-D grid
    (1, 8, 1, 2, (1, 8), (1, 8)),           # M = 1: causal linear attention
]


def setup(case, seed):
    B, N, H, d, grid, block = case
    M = oracle.num_blocks(grid, block)
    rng = np.random.default_rng(seed)
    q, k, v = (away_from_zero((B, N, H, d), rng) for _ in range(3))
    W = rng.uniform(0.1, 1.0, (M, M))           # asymmetric, with entries above the diagonal
    g = rng.standard_normal((B, N, H, d))
    return q, k, v, W, g, grid, block


def loss(q, k, v, W, g, grid, block, phi_kind, eps):
    return float((oracle.forward_causal(q, k, v, W, grid, block, phi_kind, eps) * g).sum())


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[4]}-{c[5]}")
@pytest.mark.parametrize("phi_kind", [oracle.PHI_RELU, oracle.PHI_RELU_EPS])
def test_causal_backward_matches_central_differences(case, phi_kind):
    q, k, v, W, g, grid, block = setup(case, 31 + phi_kind + case[1])
    eps = 1e-3                                  # large enough that a dropped eps shows
    grads = backward_causal(q, k, v, W, g, grid, block, phi_kind, eps)
    h = 1e-6
    for name, x, gx in zip(("q", "k", "v", "W"), (q, k, v, W), grads):
        assert gx.shape == x.shape
        fd = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            old = x[idx]
            x[idx] = old + h
            lp = loss(q, k, v, W, g, grid, block, phi_kind, eps)
            x[idx] = old - h
            lm = loss(q, k, v, W, g, grid, block, phi_kind, eps)
            x[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        err = np.abs(fd - gx).max() / max(np.abs(fd).max(), 1e-12)
        assert err < 1e-6, f"d{name}: {err:.2e}"


@pytest.mark.parametrize("case", CASES + [(2, 64, 2, 4, (8, 8), (2, 8)), (1, 48, 3, 5, (3, 4, 4), (1, 4, 4))],
                         ids=lambda c: f"{c[4]}-{c[5]}")
@pytest.mark.parametrize("phi_kind", [oracle.PHI_RELU, oracle.PHI_RELU_EPS])
def test_blocked_walk_equals_the_matrix_form(case, phi_kind):
    q, k, v, W, g, grid, block = setup(case, 5 + case[1])
    a = backward_causal(q, k, v, W, g, grid, block, phi_kind, 1e-6)
    b = backward_causal_dense(q, k, v, W, g, grid, block, phi_kind, 1e-6)
    for name, x, y in zip(("dq", "dk", "dv", "dW"), a, b):
        assert np.abs(x - y).max() <= 1e-10 * max(np.abs(y).max(), 1.0), name


def test_gradients_are_causal():
    """A loss on the first T outputs only: no input after T has any gradient,
    and the outputs after T never feed back."""
    case = (1, 24, 1, 3, (1, 24), (1, 6))
    q, k, v, W, g, grid, block = setup(case, 77)
    T = 10
    g[:, T:] = 0.0
    dq, dk, dv, dW = backward_causal(q, k, v, W, g, grid, block)
    assert np.all(dq[:, T:] == 0) and np.all(dk[:, T:] == 0) and np.all(dv[:, T:] == 0)
    assert np.abs(dq[:, :T]).max() > 0 and np.abs(dk[:, :T]).max() > 0
    # blocks 2 and 3 (tokens 12..23) have no dout at all, so no row of W that
    # mixes into them has a gradient
    assert np.all(dW[2:] == 0)


def test_w_above_the_diagonal_gets_no_gradient():
    case = (2, 16, 2, 3, (4, 4), (1, 4))
    q, k, v, W, g, grid, block = setup(case, 12)
    dW = backward_causal(q, k, v, W, g, grid, block)[3]
    assert np.all(np.triu(dW, 1) == 0)
    assert np.all(np.abs(np.diag(dW)) > 0) and np.all(np.abs(np.tril(dW, -1))[np.tril_indices(4, -1)] > 0)


def test_euler_identities_of_the_forward_homogeneity():
    """With eps = 0 and pure ReLU, o is homogeneous of degree 1 in v and of
    degree 0 in q, in k and in W, so <dv, v> = <dout, o> and <dq, q> =
    <dk, k> = <dW, W> = 0."""
    case = (2, 32, 2, 4, (4, 8), (1, 8))
    q, k, v, W, g, grid, block = setup(case, 5)
    q[..., 0] = np.abs(q[..., 0]) + 0.1         # every den > 0 with eps = 0
    k[..., 0] = np.abs(k[..., 0]) + 0.1
    o = oracle.forward_causal(q, k, v, W, grid, block, oracle.PHI_RELU, 0.0)
    dq, dk, dv, dW = backward_causal(q, k, v, W, g, grid, block, oracle.PHI_RELU, 0.0)
    scale = np.abs(g * o).sum()
    assert abs(np.sum(dv * v) - np.sum(g * o)) < 1e-10 * scale
    for name, dx, x in (("q", dq, q), ("k", dk, k), ("W", dW, W)):
        assert abs(np.sum(dx * x)) < 1e-10 * scale, name


def test_gradients_are_linear_in_dout():
    case = (1, 16, 2, 3, (1, 16), (1, 4))
    q, k, v, W, g, grid, block = setup(case, 9)
    g2 = np.random.default_rng(10).standard_normal(g.shape)
    a = backward_causal(q, k, v, W, g, grid, block)
    b = backward_causal(q, k, v, W, g2, grid, block)
    c = backward_causal(q, k, v, W, 2.0 * g - 3.0 * g2, grid, block)
    for x, y, z in zip(a, b, c):
        assert np.allclose(z, 2.0 * x - 3.0 * y, rtol=1e-10, atol=1e-12)


def test_non_contiguous_blocks_are_refused():
    q = np.zeros((1, 16, 1, 2))
    with pytest.raises(ValueError):
        backward_causal(q, q, q, np.ones((4, 4)), q, (4, 4), (2, 2))
