"""Plain float64 CPU oracle of the whole MHLA module: the projections and the
locally-enhanced positional encoding around the MHLA core.

TEST INFRASTRUCTURE ONLY, like ``mhla_oracle``: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may import or run it,
and the library shares no code with it.

Source: [P1] "MHLA：通过令牌级多头机制恢复线性注意力机制的表达能力"
(171host.com/767426.html), §七 "即插即用模块代码", class MHLA: ``__init__``
(``norm``, ``to_qkv``, ``lepe``, ``to_out``), ``_mlp_lepe``,
``_process_qkv_impl`` and ``forward``.  In order, for an input x of C = dim
channels per token:

    xn       = LayerNorm(x)                      (per token over C, affine, eps 1e-5)
    q, k, v  = split(xn W_qkv^T (+ b_qkv), 3)    (C channels each, head-major (h d))
    lepe     = depthwise 5 x 5 convolution of v over the token image, zero
               padding 2, plus its bias (one 5 x 5 kernel per channel)
    o        = MHLA(q, k, v)                     (phi = ReLU + eps, mixing W, eps)
    y        = (o + lepe) W_out^T + b_out

Readings taken (listed in the design notes):
  * Tokens are in raster order over the grid.  The listing holds them as
    (piece, position in piece) and rearranges "b (h w) (p1 p2) d -> b d (h p1)
    (w p2)" to reach the image; that image is the raster grid, so the
    convolution runs over the grid's (Y, X) axes directly.  On a 3-D (T, Y, X)
    grid the 2-D convolution runs over each frame.
  * The listing's convolution has C input channels and is applied to v, which
    has inner_dim = heads * dim_head channels: the module is read with
    inner_dim = C.
  * q_norm and k_norm are identities (``qk_norm=False``, the listing's
    default); Dropout is the identity (inference).
  * LayerNorm uses the biased variance and eps = 1e-5 (``nn.LayerNorm``
    defaults); a Linear weight is ``[out_features, in_features]``.
"""

from __future__ import annotations

import numpy as np

from .mhla_oracle import PHI_RELU_EPS, _as_f64, forward

LN_EPS = 1e-5
LEPE_K = 5


def layer_norm(x, gamma, beta, eps=LN_EPS):
    """Normalise each token over its last axis: (x - mean) / sqrt(var + eps) * gamma + beta."""
    x = _as_f64(x)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * _as_f64(gamma) + _as_f64(beta)


def linear(x, weight, bias=None):
    """x W^T + b with W of shape [out_features, in_features]."""
    y = _as_f64(x) @ _as_f64(weight).T
    if bias is not None:
        y = y + _as_f64(bias)
    return y


def lepe(v, grid, weight, bias):
    """Depthwise 5 x 5 convolution (zero padding 2, cross-correlation as in a
    convolution layer) of v [B, N, C] over the token image, plus the bias.

    weight [C, 5, 5], bias [C]; the image is the raster (Y, X) grid, one image
    per frame of a 3-D grid."""
    v = _as_f64(v)
    weight, bias = _as_f64(weight), _as_f64(bias)
    B, N, C = v.shape
    grid = tuple(grid)
    T = 1 if len(grid) == 2 else grid[0]
    Y, X = grid[-2], grid[-1]
    if T * Y * X != N:
        raise ValueError("grid does not hold N tokens")
    img = v.reshape(B * T, Y, X, C)
    pad = LEPE_K // 2
    padded = np.zeros((B * T, Y + 2 * pad, X + 2 * pad, C))
    padded[:, pad:pad + Y, pad:pad + X, :] = img
    out = np.zeros_like(img)
    for i in range(LEPE_K):
        for j in range(LEPE_K):
            out += padded[:, i:i + Y, j:j + X, :] * weight[:, i, j]
    out += bias
    return out.reshape(B, N, C)


def module_forward(x, params, W, grid, block, heads, phi_kind=PHI_RELU_EPS, eps=1e-6):
    """The MHLA module on x [B, N, C] (float64 result [B, N, C]).

    ``params``: dict with ln_weight, ln_bias [C]; qkv_weight [3C, C] and
    optional qkv_bias [3C]; optional lepe_weight [C, 5, 5] and lepe_bias [C]
    (absent: no positional term); out_weight [C, C] and optional out_bias [C].
    """
    x = _as_f64(x)
    B, N, C = x.shape
    if C % heads:
        raise ValueError("C must be a multiple of heads")
    d = C // heads
    xn = layer_norm(x, params["ln_weight"], params["ln_bias"])
    qkv = linear(xn, params["qkv_weight"], params.get("qkv_bias"))
    q, k, v = (qkv[..., s * C:(s + 1) * C] for s in range(3))
    o = forward(q.reshape(B, N, heads, d), k.reshape(B, N, heads, d), v.reshape(B, N, heads, d), W, grid, block,
                phi_kind, eps).reshape(B, N, C)
    if params.get("lepe_weight") is not None:
        o = o + lepe(v, grid, params["lepe_weight"], params["lepe_bias"])
    return linear(o, params["out_weight"], params.get("out_bias"))
