"""Plain float64 CPU oracle of the causal MHLA backward pass.

TEST INFRASTRUCTURE ONLY, like ``mhla_oracle``: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may import or run it,
and the library shares no code with it.

The pages print no backward pass; [P2] "MHLA: Restoring Expressivity of Linear
Attention via Token-Level Multi-Head", App. B "Causal MHLA" uses causal MHLA for
chunkwise training, and section 4 "Multi-Head Mixing" makes W learnable, so
training needs the derivatives of ``mhla_causal.forward_causal`` with respect to
q, k, v and W.  They are written out here for the loss L = sum(dout * o), twice:

``backward_causal`` follows the blocked forward in reverse.  Per batch b and
head h, for token t of query block i (blocks are contiguous token ranges):

    S<_i  = sum_{j < i} W[i, j] S_j,            z<_i = sum_{j < i} W[i, j] z_j
    P_t   = sum_{s in i, s <= t} kp_s v_s^T,    y_t  = sum_{s in i, s <= t} kp_s
    C_t   = S<_i + W[i, i] P_t,                 c_t  = z<_i + W[i, i] y_t
    num_t = qp_t^T C_t,   den_t = qp_t . c_t + eps,   o_t = num_t / den_t

Reverse, with g_t = dout_t:

    dnum_t = g_t / den_t,   dden_t = -(g_t . o_t) / den_t
    dqp_t  = C_t dnum_t + dden_t c_t
    dS<_i  = sum_{t in i} qp_t dnum_t^T,        dz<_i = sum_{t in i} dden_t qp_t
    dW[i, i] = sum_{t in i} qp_t^T P_t dnum_t + dden_t (qp_t . y_t)
    dW[i, j] = <dS<_i, S_j> + dz<_i . z_j      (j < i; entries above the diagonal get 0)
    the own block reaches source token s through every t >= s of its block:
    R_s = W[i, i] sum_{t in i, t >= s} qp_t dnum_t^T,   r_s = W[i, i] sum_{t in i, t >= s} dden_t qp_t
    the past blocks through the mixing: dS_j = sum_{i > j} W[i, j] dS<_i, dz_j likewise
    dv_s  = (dS_j + R_s)^T kp_s,   dkp_s = (dS_j + R_s) v_s + dz_j + r_s
    dq_t  = dqp_t * [q_t > 0],     dk_s  = dkp_s * [k_s > 0]

``backward_causal_dense`` differentiates the explicit causal N x N form
instead, A = (W expanded to tokens, lower triangle) * (Qp Kp^T),
o = A V / (A 1 + eps), as matrix products: an independent derivation for tiny
inputs.  phi'(x) is 1 for x > 0 and 0 otherwise in both phi modes, as in
``mhla_backward``.
"""

from __future__ import annotations

import numpy as np

from .mhla_backward import phi_derivative
from .mhla_causal import _check
from .mhla_oracle import PHI_RELU, _as_f64, block_of_token, num_blocks, phi, summaries


def backward_causal(q, k, v, W, dout, grid, block, phi_kind=PHI_RELU, eps=1e-6):
    """Gradients (dq, dk, dv, dW) of L = sum(dout * forward_causal(q, k, v, W)),
    in the blocked order: each query block's causal states walked in reverse.

    q, k, v, dout: [B, N, H, d]; W: M x M.  dW sums over every batch and head."""
    _check(grid, block)
    q, k, v, dout, W = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout), _as_f64(W)
    B, N, H, d = q.shape
    M = num_blocks(grid, block)
    w = N // M
    S, z = summaries(k, v, grid, block, phi_kind, eps)
    dq = np.empty((B, N, H, d))
    dk = np.empty((B, N, H, d))
    dv = np.empty((B, N, H, d))
    dW = np.zeros((M, M))
    for b in range(B):
        for h in range(H):
            Qp = phi(q[b, :, h], phi_kind, eps)
            Kp = phi(k[b, :, h], phi_kind, eps)
            V = v[b, :, h]
            G = dout[b, :, h]
            dQp = np.empty((N, d))
            dSp = np.zeros((M, d, d))          # d L / d S<_i
            dzp = np.zeros((M, d))             # d L / d z<_i
            R = np.empty((N, d, d))            # own-block gradient of kp_s v_s^T
            r = np.empty((N, d))               # own-block gradient of kp_s
            for i in range(M):
                Sp = np.zeros((d, d))
                zp = np.zeros(d)
                for j in range(i):
                    Sp += W[i, j] * S[b, h, j]
                    zp += W[i, j] * z[b, h, j]
                toks = range(i * w, (i + 1) * w)
                # the block's running prefixes P_t, y_t, as in the forward
                P = np.zeros((w, d, d))
                y = np.zeros((w, d))
                acc_P = np.zeros((d, d))
                acc_y = np.zeros(d)
                for n, s in enumerate(toks):
                    acc_P = acc_P + np.outer(Kp[s], V[s])
                    acc_y = acc_y + Kp[s]
                    P[n], y[n] = acc_P, acc_y
                # the readout in reverse; suffix sums over t >= s give R_s, r_s
                suf_R = np.zeros((d, d))
                suf_r = np.zeros(d)
                for n in reversed(range(w)):
                    t = i * w + n
                    C = Sp + W[i, i] * P[n]
                    c = zp + W[i, i] * y[n]
                    den = Qp[t] @ c + eps
                    o = (Qp[t] @ C) / den
                    dnum = G[t] / den
                    dden = -(G[t] @ o) / den
                    dQp[t] = C @ dnum + dden * c
                    dSp[i] += np.outer(Qp[t], dnum)
                    dzp[i] += dden * Qp[t]
                    dW[i, i] += Qp[t] @ P[n] @ dnum + dden * (Qp[t] @ y[n])
                    suf_R += W[i, i] * np.outer(Qp[t], dnum)
                    suf_r += W[i, i] * dden * Qp[t]
                    R[t], r[t] = suf_R, suf_r
            # the past mixing in reverse
            dS = np.zeros((M, d, d))
            dz = np.zeros((M, d))
            for i in range(M):
                for j in range(i):
                    dS[j] += W[i, j] * dSp[i]
                    dz[j] += W[i, j] * dzp[i]
                    dW[i, j] += np.sum(dSp[i] * S[b, h, j]) + dzp[i] @ z[b, h, j]
            # source tokens: past-block and own-block parts
            for s in range(N):
                j = s // w
                Gs = dS[j] + R[s]
                dv[b, s, h] = Gs.T @ Kp[s]
                dKp = Gs @ V[s] + dz[j] + r[s]
                dk[b, s, h] = dKp * phi_derivative(k[b, s, h])
            dq[b, :, h] = dQp * phi_derivative(q[b, :, h])
    return dq, dk, dv, dW


def backward_causal_dense(q, k, v, W, dout, grid, block, phi_kind=PHI_RELU, eps=1e-6):
    """The same gradients from the explicit causal N x N form (tiny inputs)."""
    _check(grid, block)
    q, k, v, dout, W = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout), _as_f64(W)
    B, N, H, d = q.shape
    if N > 4096:
        raise ValueError("the N x N form is for tiny inputs")
    M = num_blocks(grid, block)
    ids = block_of_token(grid, block)
    onehot = np.zeros((N, M))
    onehot[np.arange(N), ids] = 1.0
    mask = np.tril(np.ones((N, N)))
    Wt = W[np.ix_(ids, ids)] * mask
    dq = np.empty((B, N, H, d))
    dk = np.empty((B, N, H, d))
    dv = np.empty((B, N, H, d))
    dW = np.zeros((M, M))
    for b in range(B):
        for h in range(H):
            Qp = phi(q[b, :, h], phi_kind, eps)
            Kp = phi(k[b, :, h], phi_kind, eps)
            V = v[b, :, h]
            G = dout[b, :, h]
            E = Qp @ Kp.T
            A = Wt * E
            den = A.sum(axis=1) + eps
            o = (A @ V) / den[:, None]
            dnum = G / den[:, None]
            dden = -(G * o).sum(axis=1) / den
            dA = dnum @ V.T + dden[:, None]            # d L / d A[t, s]
            dv[b, :, h] = A.T @ dnum
            dE = Wt * dA
            dq[b, :, h] = (dE @ Kp) * phi_derivative(q[b, :, h])
            dk[b, :, h] = (dE.T @ Qp) * phi_derivative(k[b, :, h])
            dW += onehot.T @ (E * dA * mask) @ onehot  # W[b(t), b(s)] enters A[t, s] for s <= t
    return dq, dk, dv, dW
