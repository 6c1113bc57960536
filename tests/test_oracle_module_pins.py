"""Pins of the module oracle (LayerNorm, the projections, the 5 x 5 depthwise
positional term and their composition) against closed forms, brute force and
the rearrangement the listing states.
"""

import numpy as np
import pytest

import oracle


def test_layer_norm_two_element_closed_form():
    # row (a, b): mean (a + b) / 2, biased variance ((a - b) / 2)^2
    a, b = 3.0, -1.0
    half = (a - b) / 2
    expect = np.array([half, -half]) / np.sqrt(half * half + oracle.LN_EPS)
    got = oracle.layer_norm(np.array([[a, b]]), np.ones(2), np.zeros(2))
    assert np.allclose(got[0], expect, rtol=0, atol=1e-15)
    # eps matters when the spread is tiny
    tiny = oracle.layer_norm(np.array([[1.0, 1.0 + 2e-3]]), np.ones(2), np.zeros(2))
    assert np.allclose(tiny[0], np.array([-1e-3, 1e-3]) / np.sqrt(1e-6 + oracle.LN_EPS), rtol=1e-12)


def test_layer_norm_moments_and_affine():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 7, 48)) * 5 + 2
    g, b = rng.standard_normal(48), rng.standard_normal(48)
    plain = oracle.layer_norm(x, np.ones(48), np.zeros(48))
    var = x.var(axis=-1, keepdims=True)
    assert np.allclose(plain.mean(axis=-1), 0, atol=1e-13)
    assert np.allclose((plain ** 2).mean(axis=-1, keepdims=True), var / (var + oracle.LN_EPS), rtol=1e-12)
    assert np.allclose(oracle.layer_norm(x, g, b), plain * g + b, rtol=1e-13, atol=1e-13)


def test_linear_brute_force():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((2, 3, 5))
    w = rng.standard_normal((4, 5))       # out 4, in 5
    bias = rng.standard_normal(4)
    got = oracle.linear(x, w, bias)
    assert got.shape == (2, 3, 4)
    for i in range(2):
        for t in range(3):
            for o in range(4):
                s = bias[o]
                for c in range(5):
                    s += x[i, t, c] * w[o, c]
                assert abs(got[i, t, o] - s) < 1e-12


def _image(v, Y, X):
    return v.reshape(v.shape[0], Y, X, v.shape[-1])


@pytest.mark.parametrize("tap", [(2, 2), (0, 0), (4, 1), (1, 3)])
def test_lepe_single_tap_is_a_shift(tap):
    # cross-correlation: out[y, x] = w[i, j] * v[y + i - 2, x + j - 2], zero outside
    rng = np.random.default_rng(5)
    B, Y, X, C = 2, 6, 7, 3
    v = rng.standard_normal((B, Y * X, C))
    w = np.zeros((C, 5, 5))
    w[:, tap[0], tap[1]] = [1.0, 2.0, -0.5]
    bias = np.array([0.25, 0.0, -1.0])
    got = _image(oracle.lepe(v, (Y, X), w, bias), Y, X)
    img = _image(v, Y, X)
    for y in range(Y):
        for x in range(X):
            sy, sx = y + tap[0] - 2, x + tap[1] - 2
            src = img[:, sy, sx, :] if (0 <= sy < Y and 0 <= sx < X) else np.zeros((B, C))
            assert np.allclose(got[:, y, x, :], src * np.array([1.0, 2.0, -0.5]) + bias, rtol=0, atol=1e-14)


def test_lepe_box_filter_by_prefix_sums():
    rng = np.random.default_rng(6)
    B, Y, X, C = 1, 9, 8, 2
    v = rng.standard_normal((B, Y * X, C))
    got = _image(oracle.lepe(v, (Y, X), np.ones((C, 5, 5)), np.zeros(C)), Y, X)
    img = _image(v, Y, X)[0]
    P = np.zeros((Y + 1, X + 1, C))
    P[1:, 1:] = img.cumsum(axis=0).cumsum(axis=1)
    for y in range(Y):
        for x in range(X):
            y0, y1 = max(0, y - 2), min(Y, y + 3)
            x0, x1 = max(0, x - 2), min(X, x + 3)
            box = P[y1, x1] - P[y0, x1] - P[y1, x0] + P[y0, x0]
            assert np.allclose(got[0, y, x], box, atol=1e-12)


def test_lepe_frames_of_a_3d_grid_are_independent():
    rng = np.random.default_rng(7)
    B, T, Y, X, C = 2, 3, 5, 6, 4
    v = rng.standard_normal((B, T * Y * X, C))
    w, bias = rng.standard_normal((C, 5, 5)), rng.standard_normal(C)
    got = oracle.lepe(v, (T, Y, X), w, bias).reshape(B, T, Y * X, C)
    for t in range(T):
        frame = v.reshape(B, T, Y * X, C)[:, t]
        assert np.allclose(got[:, t], oracle.lepe(frame, (Y, X), w, bias), atol=1e-13)


def test_listing_rearrangement_is_the_raster_image():
    # The listing holds tokens as (piece, position in piece) and forms the image
    # by "b (h w) (p1 p2) d -> b d (h p1) (w p2)".  Starting from raster tokens,
    # putting them in that order and applying the rearrangement gives back the
    # raster image.
    Y = X = 8
    p = 4                                    # 4 x 4 pieces, 2 x 2 of them
    n_side = Y // p
    raster = np.arange(Y * X).reshape(Y, X)
    pieces = np.empty((n_side * n_side, p * p), dtype=int)
    for hh in range(n_side):
        for ww in range(n_side):
            for p1 in range(p):
                for p2 in range(p):
                    pieces[hh * n_side + ww, p1 * p + p2] = raster[hh * p + p1, ww * p + p2]
    img = pieces.reshape(n_side, n_side, p, p).transpose(0, 2, 1, 3).reshape(Y, X)
    assert np.array_equal(img, raster)


def _params(rng, C, lepe=True, biases=True):
    p = {
        "ln_weight": 1 + 0.1 * rng.standard_normal(C),
        "ln_bias": 0.1 * rng.standard_normal(C),
        "qkv_weight": rng.standard_normal((3 * C, C)) / np.sqrt(C),
        "out_weight": rng.standard_normal((C, C)) / np.sqrt(C),
    }
    if biases:
        p["qkv_bias"] = 0.1 * rng.standard_normal(3 * C)
        p["out_bias"] = 0.1 * rng.standard_normal(C)
    if lepe:
        p["lepe_weight"] = 0.2 * rng.standard_normal((C, 5, 5))
        p["lepe_bias"] = 0.1 * rng.standard_normal(C)
    return p


def test_module_one_block_is_linear_attention_through_the_projections():
    # M = 1 and identity projections: y = linear attention of the normalised input
    rng = np.random.default_rng(8)
    B, Y, X, heads, d = 1, 4, 4, 2, 3
    C = heads * d
    x = rng.standard_normal((B, Y * X, C))
    eye = np.eye(C)
    params = {"ln_weight": np.ones(C), "ln_bias": np.zeros(C), "qkv_weight": np.vstack([eye, eye, eye]),
              "out_weight": eye}
    W = oracle.mixing_matrix((Y, X), (Y, X))
    got = oracle.module_forward(x, params, W, (Y, X), (Y, X), heads, oracle.PHI_RELU_EPS, 1e-6)
    xn = oracle.layer_norm(x, np.ones(C), np.zeros(C)).reshape(B, Y * X, heads, d)
    expect = oracle.linear_attention(xn, xn, xn, oracle.PHI_RELU_EPS, 1e-6).reshape(B, Y * X, C)
    assert np.allclose(got, expect, rtol=1e-12, atol=1e-12)


def test_module_output_projection_and_positional_term_are_additive():
    # y is affine in (o + lepe): doubling the positional weights and bias adds
    # lepe(v) W_out^T once more, and the out bias shifts every token alike
    rng = np.random.default_rng(9)
    B, Y, X, heads, d = 2, 8, 8, 2, 4
    C = heads * d
    grid, block = (Y, X), (4, 4)
    x = rng.standard_normal((B, Y * X, C))
    W = oracle.mixing_matrix(grid, block, "exp")
    p = _params(rng, C)
    base = oracle.module_forward(x, p, W, grid, block, heads)
    p2 = dict(p, lepe_weight=2 * p["lepe_weight"], lepe_bias=2 * p["lepe_bias"])
    twice = oracle.module_forward(x, p2, W, grid, block, heads)
    xn = oracle.layer_norm(x, p["ln_weight"], p["ln_bias"])
    v = oracle.linear(xn, p["qkv_weight"], p["qkv_bias"])[..., 2 * C:]
    extra = oracle.lepe(v, grid, p["lepe_weight"], p["lepe_bias"]) @ p["out_weight"].T
    assert np.allclose(twice - base, extra, rtol=1e-11, atol=1e-11)
    p3 = dict(p, out_bias=p["out_bias"] + 1.5)
    assert np.allclose(oracle.module_forward(x, p3, W, grid, block, heads) - base, 1.5, atol=1e-12)
