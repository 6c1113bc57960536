"""Plain float64 CPU oracle of the MHLA forward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
this module.  The library (``token_level_head_block_gb300``) never imports it
and shares no code with it: it is the independent restatement the CUDA path is
checked against.

What it follows (the sources are web pages; cited by title and section):

[P1] "MHLA：通过令牌级多头机制恢复线性注意力机制的表达能力" module walkthrough
     (171host.com/767426.html): §五 "MHLA模块的原理" (token-dimension heads,
     local KV summaries, multi-head mixing, two-stage selection) and §七
     "即插即用模块代码" (the BlockDistanceConv / MHLA PyTorch module:
     ``_compute_block_distances``, ``_apply_transform``,
     ``_process_qkv_impl``, ``forward``).
[P2] "MHLA: Restoring Expressivity of Linear Attention via Token-Level
     Multi-Head", paperlayer.ai summary of arXiv 2601.07832v2: §3 "Linear
     Attention Formulation", §4 "Architecture", "Multi-Head Mixing",
     "Token-Level Adaptivity", "Efficiency"; App. B "Global Linear Attention".

Notation: B batch, N tokens, H heads, d head dim, M token blocks ("token-level
heads"), w = N / M tokens per block.  Tensors are ``[B, N, H, d]`` with the N
tokens in raster order over a 2-D ``(Y, X)`` or 3-D ``(T, Y, X)`` grid.

Readings taken where the pages are silent or disagree (each one is listed in
the design notes as well):
  * phi is ReLU; ``PHI_RELU_EPS`` adds eps to ReLU as the [P1 §七] module does.
    The denominator always adds eps.
  * The normaliser of token t in query block i is phi(q_t) . z~_i + eps with
    z~_i = sum_j W[i, j] z_j (the row-normalised two-stage form of [P1 §五(4)],
    [P2 §4 Token-Level Adaptivity]).  The [P1 §七] listing instead mixes
    phi(q) . z over blocks at a fixed in-block slot; that variant is kept below
    as ``forward_listing_normaliser`` for information only (parity unpinned).
  * W[i, j]: i is the query (output) block, j the source block, as the 1x1
    convolution weight ``weight[out, in]`` of [P1 §七]; columns sum to one
    (``mat.sum(dim=0)``).
  * Block centres are at (index + 0.5) in block units, block ids row-major with
    the slowest grid axis first; the same rule extends to rectangular and 3-D
    grids.  A single block (M = 1) gets W = [[1]] for every transform (the
    listing's 0/0 there is undefined), which makes M = 1 plain linear attention.
  * W is built in float64 and rounded once to float32.
  * No 1/sqrt(d) scale: the listing defines ``self.scale`` but never applies it,
    and the normaliser would cancel it anyway.
"""

from __future__ import annotations

import math

import numpy as np

PHI_RELU = 0
PHI_RELU_EPS = 1

TRANSFORMS = ("linear", "cos", "exp", "gaussian", "local")


# --------------------------------------------------------------------------
# Token blocks and block geometry  ([P1 §七] BlockDistanceConv, rearrange of
# "b (h w) (p1 p2) d -> b d (h p1) (w p2)"; [P2 §4 Architecture])
# --------------------------------------------------------------------------

def _check_grid(grid, block):
    grid = tuple(int(g) for g in grid)
    block = tuple(int(b) for b in block)
    if len(grid) != len(block) or len(grid) not in (2, 3):
        raise ValueError("grid and block must both be 2-D (Y, X) or 3-D (T, Y, X)")
    for g, b in zip(grid, block):
        if b <= 0 or g <= 0 or g % b:
            raise ValueError(f"block extent {b} does not tile grid extent {g}")
    return grid, block


def blocks_per_axis(grid, block):
    grid, block = _check_grid(grid, block)
    return tuple(g // b for g, b in zip(grid, block))


def num_blocks(grid, block):
    return int(np.prod(blocks_per_axis(grid, block)))


def block_of_token(grid, block):
    """Block id of every token, tokens in raster order (last axis fastest).

    A token at grid coordinates (.., y, x) belongs to the block whose
    coordinates are (.., y // by, x // bx); block ids are row-major over the
    block grid, slowest axis first, as the listing enumerates block centres
    (outer loop over block rows, inner over block columns).
    """
    grid, block = _check_grid(grid, block)
    nb = blocks_per_axis(grid, block)
    coords = np.indices(grid).reshape(len(grid), -1)
    ids = np.zeros(coords.shape[1], dtype=np.int64)
    for axis in range(len(grid)):
        ids = ids * nb[axis] + coords[axis] // block[axis]
    return ids


def block_centres(grid, block):
    """Centres of the M blocks in block-index units: (index + 0.5) per axis."""
    nb = blocks_per_axis(grid, block)
    idx = np.indices(nb).reshape(len(nb), -1).T.astype(np.float64)
    return idx + 0.5


def block_distances(grid, block):
    """Euclidean distance between every pair of block centres, float64 (M x M)."""
    c = block_centres(grid, block)
    diff = c[:, None, :] - c[None, :, :]
    return np.sqrt((diff * diff).sum(axis=-1))


def _libm(fn, x):
    # C libm through the math module, element by element: the same routines a
    # C implementation calls, so the float64 values agree to the last bit.
    out = np.empty_like(x)
    flat_in, flat_out = x.reshape(-1), out.reshape(-1)
    for n in range(flat_in.size):
        flat_out[n] = fn(float(flat_in[n]))
    return out


def apply_transform(D, transform, local_thres=1.5, exp_sigma=3.0):
    """Distance matrix -> column-normalised mixing weights ([P1 §七] _apply_transform).

    linear:   1 - D / max D
    cos:      cos(D / max D * pi / 4)
    exp:      exp(-D / exp_sigma)
    gaussian: exp(-D^2 / (2 sigma^2)),  sigma = max D / 3
    local:    1 where D <= local_thres, else 0
    then every column is divided by its sum (Σ_i W[i, j] = 1).
    """
    D = np.asarray(D, dtype=np.float64)
    M = D.shape[0]
    if transform not in TRANSFORMS:
        raise ValueError(f"unknown transform {transform!r}")
    if M == 1:
        return np.ones((1, 1))
    if transform == "linear":
        mat = 1.0 - D / D.max()
    elif transform == "cos":
        mat = _libm(math.cos, D / D.max() * math.pi / 4)
    elif transform == "exp":
        mat = _libm(math.exp, -D / float(exp_sigma))
    elif transform == "gaussian":
        sigma = D.max() / 3
        mat = _libm(math.exp, -(D * D) / (2 * sigma * sigma))
    else:
        mat = (D <= float(local_thres)).astype(np.float64)
    col = np.zeros(M)
    for i in range(M):            # sequential column sums, top row first
        col = col + mat[i]
    return mat / col[None, :]


def mixing_matrix(grid, block, transform="linear", local_thres=1.5, exp_sigma=3.0):
    """M x M float32 W, W[i, j] = weight of source block j for query block i."""
    W = apply_transform(block_distances(grid, block), transform, local_thres, exp_sigma)
    return W.astype(np.float32)


# --------------------------------------------------------------------------
# The forward pass ([P1 §五], [P1 §七] MHLA.forward, [P2 §4])
# --------------------------------------------------------------------------

def phi(x, kind=PHI_RELU, eps=1e-6):
    """Positive feature map: ReLU, or ReLU + eps as in the listing's _process_qkv_impl."""
    x = np.asarray(x, dtype=np.float64)
    out = np.maximum(x, 0.0)
    if kind == PHI_RELU_EPS:
        out = out + eps
    elif kind != PHI_RELU:
        raise ValueError(f"unknown phi kind {kind}")
    return out


def _as_f64(t):
    a = np.asarray(t)
    if a.dtype != np.float64:
        a = a.astype(np.float64)
    return a


def _tokens_by_block(grid, block, N):
    ids = block_of_token(grid, block)
    if ids.size != N:
        raise ValueError(f"grid holds {ids.size} tokens, tensors hold {N}")
    M = num_blocks(grid, block)
    order = np.argsort(ids, kind="stable")      # block 0's tokens, then block 1's, ...
    return ids, order, M, N // M


def summaries(k, v, grid, block, phi_kind=PHI_RELU, eps=1e-6):
    """Local KV summaries S_j = phi(K_j)^T V_j (d x d) and key sums z_j = Σ phi(k_s).

    Returns S [B, H, M, d, d] and z [B, H, M, d] in float64.
    ([P1 §七] ``kv = k @ v`` after ``k.transpose(-2, -1)``, ``k_sum``;
    [P2 §4 Architecture] "local key-value summaries for each block".)
    """
    k, v = _as_f64(k), _as_f64(v)
    B, N, H, d = k.shape
    _, order, M, w = _tokens_by_block(grid, block, N)
    S = np.empty((B, H, M, d, d))
    z = np.empty((B, H, M, d))
    for b in range(B):
        for h in range(H):
            Kb = phi(k[b, order, h, :], phi_kind, eps).reshape(M, w, d)
            Vb = v[b, order, h, :].reshape(M, w, d)
            S[b, h] = np.matmul(Kb.transpose(0, 2, 1), Vb)
            z[b, h] = Kb.sum(axis=1)
    return S, z


def mix(W, S, z):
    """Multi-head mixing: S~_i = Σ_j W[i, j] S_j and z~_i = Σ_j W[i, j] z_j.

    ([P1 §七] ``piece_attn``, a bias-free 1x1 convolution over the block axis;
    [P2 §4 Multi-Head Mixing]: each row of the coefficient matrix is the mixture
    for one query block.)
    """
    W = _as_f64(W)
    St = np.einsum("ij,bhjrc->bhirc", W, S)
    zt = np.einsum("ij,bhjr->bhir", W, z)
    return St, zt


def readout(q, St, zt, grid, block, phi_kind=PHI_RELU, eps=1e-6):
    """o_t = phi(q_t) S~_{b(t)} / (phi(q_t) . z~_{b(t)} + eps) for every token."""
    q = _as_f64(q)
    B, N, H, d = q.shape
    _, order, M, w = _tokens_by_block(grid, block, N)
    o = np.empty((B, N, H, d))
    for b in range(B):
        for h in range(H):
            Qb = phi(q[b, order, h, :], phi_kind, eps).reshape(M, w, d)
            num = np.matmul(Qb, St[b, h])                        # (M, w, d)
            den = (Qb * zt[b, h][:, None, :]).sum(axis=-1) + eps  # (M, w)
            o[b, order, h, :] = (num / den[..., None]).reshape(N, d)
    return o


def forward(q, k, v, W, grid, block, phi_kind=PHI_RELU, eps=1e-6):
    """MHLA forward in the blocked, linear-time order (float64 [B, N, H, d])."""
    S, z = summaries(k, v, grid, block, phi_kind, eps)
    St, zt = mix(W, S, z)
    return readout(q, St, zt, grid, block, phi_kind, eps)


def forward_dense(q, k, v, W, grid, block, phi_kind=PHI_RELU, eps=1e-6):
    """The same output through the explicit N x N two-stage form (tiny inputs only).

    A[t, s] = W[b(t), b(s)] * phi(q_t) . phi(k_s): block selection by the
    coefficient row, then token reweighting inside each block ([P1 §五(4)],
    [P2 §4 Token-Level Adaptivity]); o_t = Σ_s A[t, s] v_s / (Σ_s A[t, s] + eps).
    """
    q, k, v, W = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(W)
    B, N, H, d = q.shape
    if N > 4096:
        raise ValueError("the N x N form is for tiny inputs")
    ids = block_of_token(grid, block)
    Wexp = W[np.ix_(ids, ids)]
    o = np.empty((B, N, H, d))
    for b in range(B):
        for h in range(H):
            A = Wexp * (phi(q[b, :, h, :], phi_kind, eps) @ phi(k[b, :, h, :], phi_kind, eps).T)
            o[b, :, h, :] = (A @ v[b, :, h, :]) / (A.sum(axis=1) + eps)[:, None]
    return o


def linear_attention(q, k, v, phi_kind=PHI_RELU, eps=1e-6):
    """Vanilla (global) linear attention, one shared summary ([P2 §3], App. B).

    o_t = phi(q_t)^T (Σ_s phi(k_s) v_s^T) / (phi(q_t) . Σ_s phi(k_s) + eps), written
    as explicit loops over tokens so that it shares nothing with ``forward``.
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, N, H, d = q.shape
    o = np.empty((B, N, H, d))
    for b in range(B):
        for h in range(H):
            kv = np.zeros((d, d))
            ks = np.zeros(d)
            for s in range(N):
                pk = phi(k[b, s, h], phi_kind, eps)
                kv += np.outer(pk, v[b, s, h])
                ks += pk
            for t in range(N):
                pq = phi(q[b, t, h], phi_kind, eps)
                o[b, t, h] = (pq @ kv) / (pq @ ks + eps)
    return o


def forward_listing_normaliser(q, k, v, W, grid, block, phi_kind=PHI_RELU_EPS, eps=1e-6):
    """Information only, parity unpinned: the [P1 §七] listing's own normaliser.

    The listing forms ``piece_attn(q @ k_sum) + eps``: for query slot t of block i
    the denominator is Σ_j W[i, j] phi(q_{j,t}) . z_j, mixing the queries that sit
    at the same in-block slot of other blocks.  The numerator is the same as in
    ``forward``.  Not computed by the library; kept to document the difference.
    """
    q = _as_f64(q)
    B, N, H, d = q.shape
    S, z = summaries(k, v, grid, block, phi_kind, eps)
    St, _ = mix(W, S, z)
    _, order, M, w = _tokens_by_block(grid, block, N)
    W64 = _as_f64(W)
    o = np.empty((B, N, H, d))
    for b in range(B):
        for h in range(H):
            Qb = phi(q[b, order, h, :], phi_kind, eps).reshape(M, w, d)
            own = np.einsum("jtr,jr->jt", Qb, z[b, h])          # phi(q_{j,t}) . z_j
            den = W64 @ own + eps                                  # (M, w)
            num = np.matmul(Qb, St[b, h])
            o[b, order, h, :] = (num / den[..., None]).reshape(N, d)
    return o
