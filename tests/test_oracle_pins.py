"""Pins of the CPU oracle against what the MHLA pages and the mathematics fix.

None of these compare the oracle with itself: each case is a hand-enumerated
table, a closed form worked out by hand from the definitions, a special case that
reduces to a textbook routine (global linear attention), or an invariant of the
method.  Sources: the MHLA module walkthrough (171host.com/767426.html) §五 and
§七 (BlockDistanceConv, MHLA.forward), and the paperlayer.ai summary of arXiv
2601.07832v2 §3-§4.
"""

import math

import numpy as np
import pytest

import oracle as orc

RNG = np.random.default_rng(20260112)


def rand_qkv(B, N, H, d, rng=RNG):
    return tuple(rng.standard_normal((B, N, H, d)) for _ in range(3))


# ---------------------------------------------------------------- block ids

def test_block_ids_2d_hand_table():
    # 4x4 grid, 2x2 blocks: raster tokens row by row.
    assert orc.block_of_token((4, 4), (2, 2)).tolist() == [
        0, 0, 1, 1, 0, 0, 1, 1, 2, 2, 3, 3, 2, 2, 3, 3]


def test_block_ids_rectangular_hand_table():
    # 2x6 grid, 1x3 blocks -> 2x2 block grid.
    assert orc.block_of_token((2, 6), (1, 3)).tolist() == [0, 0, 0, 1, 1, 1, 2, 2, 2, 3, 3, 3]


def test_block_ids_3d_hand_tables():
    # (T, Y, X) = (2, 2, 2); blocks (1, 1, 2): block = t*2 + y.
    assert orc.block_of_token((2, 2, 2), (1, 1, 2)).tolist() == [0, 0, 1, 1, 2, 2, 3, 3]
    # blocks (2, 1, 1): block = y*2 + x, shared by both frames.
    assert orc.block_of_token((2, 2, 2), (2, 1, 1)).tolist() == [0, 1, 2, 3, 0, 1, 2, 3]


def test_block_centres_hand_table():
    c = orc.block_centres((4, 4), (2, 2))
    assert c.tolist() == [[0.5, 0.5], [0.5, 1.5], [1.5, 0.5], [1.5, 1.5]]


def test_bad_tiling_rejected():
    with pytest.raises(ValueError):
        orc.block_of_token((14, 14), (4, 4))


# ------------------------------------------------------------- W builder

R2 = math.sqrt(2.0)


def _two_by_two_closed_form(f):
    """2x2 block grid: every column is a permutation of distances (0, 1, 1, sqrt 2)."""
    D = [[0, 1, 1, R2], [1, 0, R2, 1], [1, R2, 0, 1], [R2, 1, 1, 0]]
    s = f(0.0) + 2 * f(1.0) + f(R2)
    return np.array([[f(D[i][j]) / s for j in range(4)] for i in range(4)])


@pytest.mark.parametrize("transform,f", [
    ("linear", lambda x: 1.0 - x / R2),
    ("cos", lambda x: math.cos(x / R2 * math.pi / 4)),
    ("exp", lambda x: math.exp(-x / 3.0)),
    ("gaussian", lambda x: math.exp(-x * x * 9.0 / (2.0 * 2.0))),  # sigma = sqrt2/3
    ("local", lambda x: 1.0 if x <= 1.5 else 0.0),
])
def test_w_two_by_two_closed_forms(transform, f):
    W = orc.mixing_matrix((4, 4), (2, 2), transform, local_thres=1.5, exp_sigma=3.0)
    ref = _two_by_two_closed_form(f)
    np.testing.assert_allclose(W, ref.astype(np.float32), rtol=2 ** -23, atol=0)


def test_w_two_by_two_printed_values():
    # Column 0 written out for the linear and exp (sigma=3) transforms.
    lin = orc.mixing_matrix((4, 4), (2, 2), "linear")[:, 0]
    np.testing.assert_allclose(lin, [0.63060194, 0.18469903, 0.18469903, 0.0], atol=2e-8)
    ex = orc.mixing_matrix((4, 4), (2, 2), "exp", exp_sigma=3.0)[:, 0]
    np.testing.assert_allclose(ex, [0.32709801, 0.23437596, 0.23437596, 0.20415006], atol=2e-8)


def test_w_four_by_four_linear():
    W = orc.apply_transform(orc.block_distances((16, 16), (4, 4)), "linear")
    # Columns sum to one (mat / mat.sum(dim=0)).
    np.testing.assert_allclose(W.sum(axis=0), np.ones(16), rtol=1e-14)
    # Zero only between a corner and its opposite corner (distance = max = 3 sqrt 2).
    zeros = sorted(map(tuple, np.argwhere(W == 0.0).tolist()))
    assert zeros == [(0, 15), (3, 12), (12, 3), (15, 0)]
    # W[0][0] = 1 / sum over the 16 blocks of (1 - dist / (3 sqrt 2)).
    s = sum(1 - math.hypot(a, b) / (3 * R2) for a in range(4) for b in range(4))
    assert abs(W[0, 0] - 1 / s) < 1e-15
    assert abs(W[0, 0] - 0.144361) < 1e-6
    assert abs(W[0].sum() - 0.82819) < 1e-5


def test_w_four_by_four_local_neighbourhoods():
    W = orc.mixing_matrix((16, 16), (4, 4), "local", local_thres=1.5)
    # sqrt 2 <= 1.5 < 2: the 8-neighbourhood plus the block itself.
    counts = (W > 0).sum(axis=0).tolist()
    assert counts[5] == 9 and counts[0] == 4 and counts[1] == 6
    np.testing.assert_allclose(W[W[:, 5] > 0, 5], np.full(9, 1 / 9, dtype=np.float32), rtol=1e-7)


@pytest.mark.parametrize("transform", orc.TRANSFORMS)
def test_w_single_block_is_one(transform):
    assert orc.mixing_matrix((8, 8), (8, 8), transform).tolist() == [[1.0]]


def test_w_3d_video_block_grid():
    # 20x32x32 grid with 4x8x8 blocks -> 5x4x4 block grid, centres in block units.
    D = orc.block_distances((20, 32, 32), (4, 8, 8))
    assert D.shape == (80, 80)
    assert D.max() == math.sqrt(4 ** 2 + 3 ** 2 + 3 ** 2)
    W = orc.apply_transform(D, "linear")
    np.testing.assert_allclose(W.sum(axis=0), np.ones(80), rtol=1e-14)
    assert (W == 0).sum() == 8          # 4 pairs of opposite corners, both orders


def test_w_columns_normalised_not_rows_on_rectangular_grid():
    W = orc.mixing_matrix((8, 12), (4, 4), "linear")   # 2x3 block grid
    np.testing.assert_allclose(W.sum(axis=0), np.ones(6), rtol=1e-6)
    assert not np.allclose(W.sum(axis=1), 1.0)
    assert not np.allclose(W, W.T)       # so a transposed W is detectable


# ---------------------------------------------------------------- forward

def test_hand_worked_two_token_example():
    # Two tokens, one per block (grid 1x2, blocks 1x1), d = 1, asymmetric W.
    q = np.array([2.0, 0.5]).reshape(1, 2, 1, 1)
    k = np.array([1.5, 3.0]).reshape(1, 2, 1, 1)
    v = np.array([-1.0, 4.0]).reshape(1, 2, 1, 1)
    W = np.array([[0.7, 0.2], [0.1, 0.9]])
    eps = 1e-6
    o = orc.forward(q, k, v, W, (1, 2), (1, 1), eps=eps).reshape(2)
    # o_0 = (0.7*2*1.5*(-1) + 0.2*2*3*4) / (0.7*2*1.5 + 0.2*2*3 + eps)
    assert abs(o[0] - (-2.1 + 4.8) / (2.1 + 1.2 + eps)) < 1e-14
    # o_1 = (0.1*0.5*1.5*(-1) + 0.9*0.5*3*4) / (0.1*0.5*1.5 + 0.9*0.5*3 + eps)
    assert abs(o[1] - (-0.075 + 5.4) / (0.075 + 1.35 + eps)) < 1e-14


def test_hand_worked_negative_key_is_dropped():
    # phi = ReLU on keys: a negative key contributes nothing, whatever its value.
    q = np.array([1.0, 1.0]).reshape(1, 2, 1, 1)
    k = np.array([2.0, -5.0]).reshape(1, 2, 1, 1)
    v = np.array([3.0, 100.0]).reshape(1, 2, 1, 1)
    W = np.array([[1.0, 1.0], [1.0, 1.0]])
    o = orc.forward(q, k, v, W, (1, 2), (1, 1), eps=0.0).reshape(2)
    assert o.tolist() == [3.0, 3.0]
    # ... and a negative query value v is not rectified: v passes through.
    v2 = np.array([-3.0, 100.0]).reshape(1, 2, 1, 1)
    assert orc.forward(q, k, v2, W, (1, 2), (1, 1), eps=0.0).reshape(2).tolist() == [-3.0, -3.0]


@pytest.mark.parametrize("grid,block", [
    ((4, 4), (2, 2)), ((6, 8), (3, 2)), ((2, 4, 4), (1, 2, 2)), ((4, 2, 6), (2, 1, 3)), ((8, 8), (8, 8)),
])
@pytest.mark.parametrize("phi_kind", [orc.PHI_RELU, orc.PHI_RELU_EPS])
def test_blocked_equals_dense_two_stage_form(grid, block, phi_kind):
    N = int(np.prod(grid))
    M = orc.num_blocks(grid, block)
    q, k, v = rand_qkv(2, N, 3, 5)
    W = RNG.uniform(0.0, 1.0, size=(M, M))           # asymmetric on purpose
    a = orc.forward(q, k, v, W, grid, block, phi_kind, eps=1e-3)
    b = orc.forward_dense(q, k, v, W, grid, block, phi_kind, eps=1e-3)
    np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("phi_kind", [orc.PHI_RELU, orc.PHI_RELU_EPS])
def test_single_block_is_global_linear_attention(phi_kind):
    q, k, v = rand_qkv(2, 16, 2, 4)
    W = orc.mixing_matrix((4, 4), (4, 4), "linear")
    a = orc.forward(q, k, v, W, (4, 4), (4, 4), phi_kind, eps=1e-6)
    b = orc.linear_attention(q, k, v, phi_kind, eps=1e-6)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)


def test_identity_mixing_is_blockwise_linear_attention():
    grid, block = (4, 6), (2, 3)
    q, k, v = rand_qkv(1, 24, 2, 4)
    M = orc.num_blocks(grid, block)
    o = orc.forward(q, k, v, np.eye(M), grid, block, eps=1e-6)
    ids = orc.block_of_token(grid, block)
    for j in range(M):
        sel = np.nonzero(ids == j)[0]
        ref = orc.linear_attention(q[:, sel], k[:, sel], v[:, sel], eps=1e-6)
        np.testing.assert_allclose(o[:, sel], ref, rtol=1e-12, atol=1e-13)


def test_all_ones_mixing_is_global_linear_attention():
    grid, block = (4, 4), (2, 2)
    q, k, v = rand_qkv(1, 16, 1, 3)
    o = orc.forward(q, k, v, np.ones((4, 4)), grid, block, eps=1e-6)
    np.testing.assert_allclose(o, orc.linear_attention(q, k, v, eps=1e-6), rtol=1e-12, atol=1e-13)


def test_linear_in_v():
    grid, block = (4, 4), (2, 2)
    q, k, v1 = rand_qkv(1, 16, 2, 4)
    v2 = RNG.standard_normal(v1.shape)
    W = orc.mixing_matrix(grid, block, "cos")
    f = lambda v: orc.forward(q, k, v, W, grid, block)
    np.testing.assert_allclose(f(v1 + 2.5 * v2), f(v1) + 2.5 * f(v2), rtol=1e-11, atol=1e-12)


def test_constant_v_and_eps_in_denominator():
    grid, block = (4, 4), (2, 2)
    q, k, _ = rand_qkv(1, 16, 1, 4)
    q = np.abs(q)                                    # every phi(q_t) non-zero
    W = orc.mixing_matrix(grid, block, "exp")
    ones = np.ones_like(q)
    # eps = 0: a weighted mean of a constant is that constant.
    np.testing.assert_allclose(orc.forward(q, k, 7.0 * ones, W, grid, block, eps=0.0), 7.0, rtol=1e-13)
    # eps > 0: o = den / (den + eps) for v = 1, the same den at every eps.
    o1 = orc.forward(q, k, ones, W, grid, block, eps=0.5)
    den = 0.5 * o1 / (1.0 - o1)
    o2 = orc.forward(q, k, ones, W, grid, block, eps=2.0)
    np.testing.assert_allclose(o2, den / (den + 2.0), rtol=1e-12)


def test_row_scaling_of_w_cancels_column_scaling_does_not():
    grid, block = (4, 4), (2, 2)
    q, k, v = rand_qkv(1, 16, 1, 4)
    q = np.abs(q)
    W = RNG.uniform(0.1, 1.0, size=(4, 4))
    s = np.array([0.5, 2.0, 3.0, 7.0])
    o = orc.forward(q, k, v, W, grid, block, eps=0.0)
    np.testing.assert_allclose(orc.forward(q, k, v, s[:, None] * W, grid, block, eps=0.0), o, rtol=1e-12)
    assert not np.allclose(orc.forward(q, k, v, W * s[None, :], grid, block, eps=0.0), o, rtol=1e-6)


def test_permuting_tokens_inside_a_block_permutes_outputs():
    grid, block = (4, 4), (2, 2)
    q, k, v = rand_qkv(1, 16, 2, 4)
    W = orc.mixing_matrix(grid, block, "linear")
    perm = np.arange(16)
    perm[[0, 5]] = perm[[5, 0]]                     # tokens 0 and 5 share block 0
    perm[[10, 11]] = perm[[11, 10]]                 # tokens 10 and 11 share block 3
    o = orc.forward(q, k, v, W, grid, block)
    op = orc.forward(q[:, perm], k[:, perm], v[:, perm], W, grid, block)
    np.testing.assert_allclose(op, o[:, perm], rtol=1e-12, atol=1e-13)


def test_batch_and_head_independence():
    grid, block = (4, 4), (2, 2)
    q, k, v = rand_qkv(3, 16, 4, 4)
    W = orc.mixing_matrix(grid, block, "gaussian")
    o = orc.forward(q, k, v, W, grid, block)
    one = orc.forward(q[1:2, :, 2:3], k[1:2, :, 2:3], v[1:2, :, 2:3], W, grid, block)
    np.testing.assert_allclose(one, o[1:2, :, 2:3], rtol=1e-13, atol=0)


def test_zero_query_gives_zero_output():
    grid, block = (4, 4), (2, 2)
    q, k, v = rand_qkv(1, 16, 1, 4)
    q[0, 6, 0, :] = -np.abs(q[0, 6, 0, :]) - 0.1    # phi(q_6) = 0 exactly
    o = orc.forward(q, k, v, orc.mixing_matrix(grid, block, "linear"), grid, block)
    assert np.all(o[0, 6, 0] == 0.0)


def test_relu_eps_closed_form_for_negative_inputs():
    # phi(x) = relu(x) + eps = eps for x < 0, so phi(q_t).phi(k_s) = d eps^2.
    grid, block = (2, 4), (2, 2)
    d, eps = 3, 1e-2
    q = -np.ones((1, 8, 1, d))
    k = -np.ones((1, 8, 1, d))
    v = RNG.standard_normal((1, 8, 1, d))
    W = np.array([[0.6, 0.3], [0.2, 0.9]])
    ids = [0, 0, 1, 1, 0, 0, 1, 1]
    o = orc.forward(q, k, v, W, grid, block, orc.PHI_RELU_EPS, eps)
    for t in range(8):
        a = [W[ids[t], ids[s]] * d * eps * eps for s in range(8)]
        ref = sum(a[s] * v[0, s, 0] for s in range(8)) / (sum(a) + eps)
        np.testing.assert_allclose(o[0, t, 0], ref, rtol=1e-13)


def test_listing_normaliser_variant_agrees_only_for_one_block():
    q, k, v = rand_qkv(1, 16, 1, 4)
    W1 = np.ones((1, 1))
    np.testing.assert_allclose(
        orc.forward_listing_normaliser(q, k, v, W1, (4, 4), (4, 4), orc.PHI_RELU_EPS),
        orc.forward(q, k, v, W1, (4, 4), (4, 4), orc.PHI_RELU_EPS), rtol=1e-12)
    W = orc.mixing_matrix((4, 4), (2, 2), "linear")
    assert not np.allclose(orc.forward_listing_normaliser(q, k, v, W, (4, 4), (2, 2)),
                           orc.forward(q, k, v, W, (4, 4), (2, 2), orc.PHI_RELU_EPS))
