"""Pins of the causal float64 oracle against what the mathematics fixes.

The blocked form (mixed past summaries plus the running prefix of the own
block) against the explicit causal N x N form; one block against causal linear
attention written as a running sum; causality itself (later tokens change
nothing before them); irrelevance of W above the diagonal; the first token and,
with an all-ones W, the last token in closed form; a lower-triangular W at the
last token of every block against the separately pinned non-causal oracle.
"""

import numpy as np
import pytest

import oracle

CASES = [
    # (B, H, d, grid, block): blocks that are contiguous token ranges
    (1, 2, 3, (1, 24), (1, 4)),
    (2, 1, 4, (6, 5), (2, 5)),
    (1, 2, 2, (4, 2, 3), (2, 2, 3)),
    (1, 1, 5, (1, 16), (1, 16)),      # M = 1
]


def draw(B, N, H, d, seed):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal((B, N, H, d)) for _ in range(3)]


def causal_linear_attention(q, k, v, eps):
    """o_t = phi(q_t) sum_{s<=t} phi(k_s) v_s^T / (phi(q_t) . sum_{s<=t} phi(k_s) + eps), running sums."""
    B, N, H, d = q.shape
    o = np.empty_like(q)
    for b in range(B):
        for h in range(H):
            kv, ks = np.zeros((d, d)), np.zeros(d)
            for t in range(N):
                pk = np.maximum(k[b, t, h], 0)
                kv += np.outer(pk, v[b, t, h])
                ks += pk
                pq = np.maximum(q[b, t, h], 0)
                o[b, t, h] = pq @ kv / (pq @ ks + eps)
    return o


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[3]}-{c[4]}")
@pytest.mark.parametrize("phi_kind", [oracle.PHI_RELU, oracle.PHI_RELU_EPS])
def test_blocked_causal_form_equals_causal_two_stage_form(case, phi_kind):
    B, H, d, grid, block = case
    N = int(np.prod(grid))
    q, k, v = draw(B, N, H, d, 1 + N)
    M = oracle.num_blocks(grid, block)
    W = np.random.default_rng(2).uniform(0.1, 1.0, (M, M))
    a = oracle.forward_causal(q, k, v, W, grid, block, phi_kind, 1e-3)
    b = oracle.forward_causal_dense(q, k, v, W, grid, block, phi_kind, 1e-3)
    assert np.abs(a - b).max() < 1e-12 * np.abs(b).max()


def test_one_block_is_causal_linear_attention():
    q, k, v = draw(2, 20, 2, 4, 3)
    a = oracle.forward_causal(q, k, v, np.array([[0.6]]), (1, 20), (1, 20), oracle.PHI_RELU, 1e-3)
    # a lone W scales numerator and denominator alike except against eps
    b = causal_linear_attention(q, k, v, 1e-3 / 0.6)
    assert np.abs(a - b).max() < 1e-12 * np.abs(b).max()


def test_causality_later_tokens_change_nothing_before_them():
    q, k, v = draw(1, 32, 2, 3, 4)
    W = np.random.default_rng(5).uniform(0.1, 1.0, (8, 8))
    a = oracle.forward_causal(q, k, v, W, (1, 32), (1, 4))
    t = 13
    rng = np.random.default_rng(6)
    for x in (q, k, v):
        x[:, t + 1:] = rng.standard_normal(x[:, t + 1:].shape)
    b = oracle.forward_causal(q, k, v, W, (1, 32), (1, 4))
    assert np.array_equal(a[:, : t + 1], b[:, : t + 1])
    assert not np.allclose(a[:, t + 1:], b[:, t + 1:])


def test_w_above_the_diagonal_never_enters():
    q, k, v = draw(1, 24, 1, 3, 7)
    W = np.random.default_rng(8).uniform(0.1, 1.0, (6, 6))
    W2 = W.copy()
    W2[np.triu_indices(6, 1)] = np.random.default_rng(9).uniform(5.0, 9.0, 15)
    a = oracle.forward_causal(q, k, v, W, (1, 24), (1, 4))
    b = oracle.forward_causal(q, k, v, W2, (1, 24), (1, 4))
    assert np.array_equal(a, b)


def test_first_token_and_all_ones_last_token_closed_forms():
    q, k, v = draw(1, 16, 1, 4, 10)
    q[0, 0, 0, 0] = abs(q[0, 0, 0, 0]) + 0.5
    k[0, 0, 0, 0] = abs(k[0, 0, 0, 0]) + 0.5
    eps = 1e-3
    W = np.random.default_rng(11).uniform(0.1, 1.0, (4, 4))
    o = oracle.forward_causal(q, k, v, W, (1, 16), (1, 4), oracle.PHI_RELU, eps)
    a = W[0, 0] * (np.maximum(q[0, 0, 0], 0) @ np.maximum(k[0, 0, 0], 0))
    assert np.allclose(o[0, 0, 0], a * v[0, 0, 0] / (a + eps), rtol=1e-13, atol=0)
    ones = oracle.forward_causal(q, k, v, np.ones((4, 4)), (1, 16), (1, 4), oracle.PHI_RELU, eps)
    glob = oracle.linear_attention(q, k, v, oracle.PHI_RELU, eps)
    assert np.allclose(ones[0, -1], glob[0, -1], rtol=1e-12, atol=0)


def test_lower_triangular_w_matches_noncausal_oracle_at_each_blocks_last_token():
    q, k, v = draw(2, 30, 2, 3, 12)
    W = np.tril(np.random.default_rng(13).uniform(0.1, 1.0, (5, 5)))
    a = oracle.forward_causal(q, k, v, W, (5, 6), (1, 6))
    b = oracle.forward(q, k, v, W, (5, 6), (1, 6))
    last = np.arange(5) * 6 + 5
    assert np.abs(a[:, last] - b[:, last]).max() < 1e-12 * np.abs(b[:, last]).max()
    assert np.abs(a[:, last - 1] - b[:, last - 1]).max() > 1e-6       # not at earlier tokens


def test_non_contiguous_blocks_are_refused():
    q, k, v = draw(1, 16, 1, 2, 14)
    assert oracle.blocks_are_contiguous((4, 4), (1, 4)) and oracle.blocks_are_contiguous((1, 32), (1, 8))
    assert oracle.blocks_are_contiguous((3, 8), (1, 4)) and oracle.blocks_are_contiguous((4, 2, 3), (2, 2, 3))
    assert not oracle.blocks_are_contiguous((4, 4), (2, 2)) and not oracle.blocks_are_contiguous((2, 4, 4), (2, 2, 4))
    assert oracle.blocks_are_contiguous((2, 4, 4), (1, 2, 4))          # two whole rows of one frame
    with pytest.raises(ValueError):
        oracle.forward_causal(q, k, v, np.ones((4, 4)), (4, 4), (2, 2))
