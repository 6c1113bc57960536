"""Pins of the float64 backward oracle against what the mathematics fixes.

None of these compares the backward with itself: central finite differences of
the (separately pinned) forward; Euler's identities of the forward's
homogeneity in v, k, q and in each row of W; a closed form of dv from the
explicit N x N two-stage form; linearity in dout; zero gradients where phi is
flat.  A plausible mistake (a dropped term, a transposed W, a wrong sign, the
derivative mask on the wrong operand) fails at least one of them.
"""

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(20240607)


def away_from_zero(shape, rng, margin=0.05):
    x = rng.standard_normal(shape)
    return np.where(np.abs(x) < margin, np.sign(x + 1e-300) * margin, x)


CASES = [
    # (B, N, H, d, grid, block)
    (1, 16, 2, 3, (4, 4), (2, 2)),
    (2, 12, 1, 4, (3, 4), (1, 2)),
    (1, 16, 1, 2, (2, 2, 4), (1, 2, 2)),
    (1, 8, 1, 3, (2, 4), (2, 4)),        # M = 1
]


def loss(q, k, v, W, g, grid, block, phi_kind, eps):
    return float((oracle.forward(q, k, v, W, grid, block, phi_kind, eps) * g).sum())


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[4]}-{c[5]}")
@pytest.mark.parametrize("phi_kind", [oracle.PHI_RELU, oracle.PHI_RELU_EPS])
def test_backward_matches_central_differences(case, phi_kind):
    B, N, H, d, grid, block = case
    M = oracle.num_blocks(grid, block)
    rng = np.random.default_rng(7 + N + phi_kind)
    q, k, v = (away_from_zero((B, N, H, d), rng) for _ in range(3))
    W = rng.uniform(0.1, 1.0, (M, M))           # asymmetric
    g = rng.standard_normal((B, N, H, d))
    eps = 1e-3                                  # large enough that a dropped eps shows
    grads = oracle.backward(q, k, v, W, g, grid, block, phi_kind, eps)
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


def euler_setup(seed):
    B, N, H, d, grid, block = 2, 32, 2, 5, (4, 8), (2, 4)
    M = oracle.num_blocks(grid, block)
    rng = np.random.default_rng(seed)
    q, k, v, g = (rng.standard_normal((B, N, H, d)) for _ in range(4))
    q[..., 0] = np.abs(q[..., 0]) + 0.1        # every phi(q_t) != 0: den > 0 even with eps = 0
    k[:, :, :, 0] = np.abs(k[:, :, :, 0]) + 0.1
    W = rng.uniform(0.05, 1.0, (M, M))
    return q, k, v, W, g, grid, block


def test_euler_identities_of_the_forward_homogeneity():
    # eps = 0, phi = ReLU: o is linear (degree 1) in v, degree 0 in k, in q and in
    # each row of W (scaling a row of W scales S~_i and z~_i alike).
    q, k, v, W, g, grid, block = euler_setup(11)
    dq, dk, dv, dW = oracle.backward(q, k, v, W, g, grid, block, oracle.PHI_RELU, 0.0)
    o = oracle.forward(q, k, v, W, grid, block, oracle.PHI_RELU, 0.0)
    scale = np.abs(g * o).sum()
    assert abs((dv * v).sum() - (g * o).sum()) < 1e-12 * scale
    assert abs((dk * k).sum()) < 1e-12 * scale
    assert abs((dq * q).sum()) < 1e-12 * scale
    assert np.abs((W * dW).sum(axis=1)).max() < 1e-12 * scale
    # ... but not in the columns of W: a transposed dW would pass the row test
    assert np.abs((W * dW).sum(axis=0)).max() > 1e-6 * scale


def test_dv_closed_form_of_the_two_stage_form():
    # o_t = sum_s A[t, s] v_s / (sum_s A[t, s] + eps) gives dv_s = sum_t A[t, s] g_t / den_t.
    q, k, v, W, g, grid, block = euler_setup(12)
    eps = 1e-3
    _, _, dv, _ = oracle.backward(q, k, v, W, g, grid, block, oracle.PHI_RELU, eps)
    ids = oracle.block_of_token(grid, block)
    Wexp = W[np.ix_(ids, ids)]
    B, N, H, d = q.shape
    for b in range(B):
        for h in range(H):
            A = Wexp * (np.maximum(q[b, :, h], 0) @ np.maximum(k[b, :, h], 0).T)
            den = A.sum(axis=1) + eps
            ref = A.T @ (g[b, :, h] / den[:, None])
            assert np.abs(dv[b, :, h] - ref).max() < 1e-12 * np.abs(ref).max()


def test_gradients_are_linear_in_dout():
    q, k, v, W, g, grid, block = euler_setup(13)
    g2 = np.random.default_rng(14).standard_normal(g.shape)
    a = oracle.backward(q, k, v, W, g, grid, block)
    b = oracle.backward(q, k, v, W, g2, grid, block)
    c = oracle.backward(q, k, v, W, g + 2.0 * g2, grid, block)
    for x, y, z in zip(a, b, c):
        assert np.abs(z - (x + 2.0 * y)).max() < 1e-10 * np.abs(z).max()


def test_flat_phi_gives_zero_gradient_and_zero_dout_gives_zero():
    q, k, v, W, g, grid, block = euler_setup(15)
    dq, dk, dv, dW = oracle.backward(q, k, v, W, g, grid, block)
    assert np.all(dq[q < 0] == 0.0) and np.all(dk[k < 0] == 0.0)
    assert np.abs(dq[q > 0]).min() > 0.0 and np.abs(dk[k > 0]).min() > 0.0
    for x in oracle.backward(q, k, v, W, np.zeros_like(g), grid, block):
        assert np.all(x == 0.0)


def test_single_block_w_gradient_vanishes_without_eps():
    # M = 1: o does not depend on the scalar W at all when eps = 0.
    rng = np.random.default_rng(16)
    q, k, v, g = (rng.standard_normal((1, 16, 2, 4)) for _ in range(4))
    q[..., 0] = np.abs(q[..., 0]) + 0.1
    k[..., 0] = np.abs(k[..., 0]) + 0.1
    W = np.array([[0.7]])
    _, _, _, dW = oracle.backward(q, k, v, W, g, (4, 4), (4, 4), oracle.PHI_RELU, 0.0)
    _, _, _, dW_eps = oracle.backward(q, k, v, W, g, (4, 4), (4, 4), oracle.PHI_RELU, 1e-2)
    assert abs(dW[0, 0]) < 1e-12 and abs(dW_eps[0, 0]) > 1e-8
