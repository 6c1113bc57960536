"""Plain float64 CPU oracle of causal (chunkwise) MHLA.

TEST INFRASTRUCTURE ONLY, like ``mhla_oracle``: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may import or run it,
and the library shares no code with it.

Source: [P2] "MHLA: Restoring Expressivity of Linear Attention via Token-Level
Multi-Head", App. B "Query-Conditioned Selectivity in Softmax Attention",
"Causal MHLA": in causal chunkwise training MHLA forms block-specific mixed
summaries and reuses each block's mixture, preserving causality at the
asymptotic cost of chunkwise linear attention.  The page gives no formula; the
reading taken here (listed in the design notes) is the causal restriction of
the two-stage form of [P1] section 5(4) / [P2] section 4:

    A[t, s] = W[b(t), b(s)] * (phi(q_t) . phi(k_s)) * [s <= t]
    o_t     = sum_s A[t, s] v_s / (sum_s A[t, s] + eps)

Tokens are in raster order and every block must be a contiguous range of
tokens (a 1-D sequence cut into chunks, or whole rows or frames of a grid), so
"past" is well defined.  In blocked form,
for token t of query block i:

    S<_i = sum_{j < i} W[i, j] S_j,      z<_i = sum_{j < i} W[i, j] z_j
    P_t  = sum_{s in i, s <= t} phi(k_s) v_s^T,   y_t = sum_{s in i, s <= t} phi(k_s)
    o_t  = phi(q_t)^T (S<_i + W[i, i] P_t) / (phi(q_t) . (z<_i + W[i, i] y_t) + eps)

Entries W[i, j] with j > i never enter.
"""

from __future__ import annotations

import numpy as np

from .mhla_oracle import PHI_RELU, _as_f64, block_of_token, num_blocks, phi, summaries


def blocks_are_contiguous(grid, block):
    """True when every block is a contiguous range of raster-order tokens: for
    some axis k, the block is one unit long on every slower axis and covers
    every faster axis whole (a 1-D sequence (1, N) in blocks (1, w), or whole
    rows, or whole frames)."""
    grid, block = tuple(grid), tuple(block)
    n = len(grid)
    return any(all(block[a] == 1 for a in range(k)) and all(block[a] == grid[a] for a in range(k + 1, n))
               for k in range(n))


def _check(grid, block):
    if not blocks_are_contiguous(grid, block):
        raise ValueError("causal MHLA needs blocks that are contiguous token ranges")


def forward_causal(q, k, v, W, grid, block, phi_kind=PHI_RELU, eps=1e-6):
    """Causal MHLA in the blocked order: mixed past summaries plus the running
    prefix of the query's own block (float64 [B, N, H, d])."""
    _check(grid, block)
    q, k, v, W = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(W)
    B, N, H, d = q.shape
    M = num_blocks(grid, block)
    w = N // M
    S, z = summaries(k, v, grid, block, phi_kind, eps)          # blocks of contiguous tokens
    o = np.empty((B, N, H, d))
    for b in range(B):
        for h in range(H):
            for i in range(M):
                Sp = np.zeros((d, d))
                zp = np.zeros(d)
                for j in range(i):                              # past blocks only
                    Sp += W[i, j] * S[b, h, j]
                    zp += W[i, j] * z[b, h, j]
                P = np.zeros((d, d))
                y = np.zeros(d)
                for s in range(i * w, (i + 1) * w):             # the block's tokens, in order
                    pk = phi(k[b, s, h], phi_kind, eps)
                    P += np.outer(pk, v[b, s, h])
                    y += pk
                    pq = phi(q[b, s, h], phi_kind, eps)
                    o[b, s, h] = (pq @ (Sp + W[i, i] * P)) / (pq @ (zp + W[i, i] * y) + eps)
    return o


def forward_causal_dense(q, k, v, W, grid, block, phi_kind=PHI_RELU, eps=1e-6):
    """The same output through the explicit causal N x N two-stage form (tiny inputs)."""
    _check(grid, block)
    q, k, v, W = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(W)
    B, N, H, d = q.shape
    if N > 4096:
        raise ValueError("the N x N form is for tiny inputs")
    ids = block_of_token(grid, block)
    mask = np.tril(np.ones((N, N)))
    Wexp = W[np.ix_(ids, ids)] * mask
    o = np.empty((B, N, H, d))
    for b in range(B):
        for h in range(H):
            A = Wexp * (phi(q[b, :, h], phi_kind, eps) @ phi(k[b, :, h], phi_kind, eps).T)
            o[b, :, h] = (A @ v[b, :, h]) / (A.sum(axis=1) + eps)[:, None]
    return o
