"""Plain float64 CPU oracle of the MHLA backward pass.

TEST INFRASTRUCTURE ONLY, like ``mhla_oracle``: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may import or run it, and
the library shares no code with it.

The pages print no backward pass.  They make the mixing coefficients learnable
([P2] "MHLA: Restoring Expressivity of Linear Attention via Token-Level
Multi-Head", section 4 "Multi-Head Mixing": the coefficient matrix is learned,
initialised from block distances; [P1] 171host.com/767426.html, section 7: W is
the weight of a 1x1 convolution inside an ``nn.Module``), so training needs the
derivatives of the forward of ``mhla_oracle.forward`` with respect to q, k, v
and W.  This module writes them out by the chain rule, step by step in the
reverse order of the forward, for the loss L = sum(dout * o).

Forward, per batch b and head h (``mhla_oracle``):
    kp_s = phi(k_s),  qp_t = phi(q_t)
    S_j  = sum_{s in j} kp_s v_s^T,      z_j  = sum_{s in j} kp_s
    S~_i = sum_j W[i, j] S_j,            z~_i = sum_j W[i, j] z_j
    num_t = qp_t^T S~_{b(t)},            den_t = qp_t . z~_{b(t)} + eps
    o_t  = num_t / den_t
Reverse, with g_t = dout_t:
    dnum_t = g_t / den_t,                dden_t = -(g_t . o_t) / den_t
    dqp_t  = S~_{b(t)} dnum_t + dden_t z~_{b(t)}
    dS~_i  = sum_{t in i} qp_t dnum_t^T, dz~_i  = sum_{t in i} dden_t qp_t
    dS_j   = sum_i W[i, j] dS~_i,        dz_j   = sum_i W[i, j] dz~_i
    dW[i, j] = sum_{b, h} <dS~_i, S_j> + dz~_i . z_j
    dv_s   = dS_{b(s)}^T kp_s,           dkp_s  = dS_{b(s)} v_s + dz_{b(s)}
    dq_t   = dqp_t * [q_t > 0],          dk_s   = dkp_s * [k_s > 0]
phi'(x) is taken as 1 for x > 0 and 0 otherwise (ReLU's derivative at 0 is
undefined; 0 is the usual convention), in both phi modes: the eps that
``PHI_RELU_EPS`` adds is a constant.
"""

from __future__ import annotations

import numpy as np

from .mhla_oracle import PHI_RELU, _as_f64, _tokens_by_block, mix, phi, summaries


def phi_derivative(x):
    """d phi / dx elementwise: 1 where x > 0, else 0."""
    return (np.asarray(x, dtype=np.float64) > 0.0).astype(np.float64)


def backward(q, k, v, W, dout, grid, block, phi_kind=PHI_RELU, eps=1e-6):
    """Gradients (dq, dk, dv, dW) of L = sum(dout * forward(q, k, v, W)).

    q, k, v, dout: [B, N, H, d]; W: M x M.  Returns float64 arrays of the same
    shapes; dW sums over every batch and head (one W is shared by all).
    """
    q, k, v, dout, W = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout), _as_f64(W)
    B, N, H, d = q.shape
    _, order, M, w = _tokens_by_block(grid, block, N)
    S, z = summaries(k, v, grid, block, phi_kind, eps)
    St, zt = mix(W, S, z)
    dq = np.empty((B, N, H, d))
    dk = np.empty((B, N, H, d))
    dv = np.empty((B, N, H, d))
    dW = np.zeros((M, M))
    for b in range(B):
        for h in range(H):
            # readout, reversed (per query block i, its w tokens t)
            Qraw = q[b, order, h, :].reshape(M, w, d)
            Qp = phi(Qraw, phi_kind, eps)
            G = dout[b, order, h, :].reshape(M, w, d)
            num = np.matmul(Qp, St[b, h])                               # (M, w, d)
            den = (Qp * zt[b, h][:, None, :]).sum(axis=-1) + eps         # (M, w)
            o = num / den[..., None]
            dnum = G / den[..., None]
            dden = -(G * o).sum(axis=-1) / den                            # (M, w)
            dQp = np.matmul(dnum, St[b, h].transpose(0, 2, 1)) + dden[..., None] * zt[b, h][:, None, :]
            dSt = np.matmul(Qp.transpose(0, 2, 1), dnum)                  # (M, d, d)
            dzt = (Qp * dden[..., None]).sum(axis=1)                      # (M, d)
            # mixing, reversed: S~ = W S
            dS = np.einsum("ij,irc->jrc", W, dSt)
            dz = np.einsum("ij,ir->jr", W, dzt)
            dW += np.einsum("irc,jrc->ij", dSt, S[b, h]) + np.einsum("ir,jr->ij", dzt, z[b, h])
            # summaries, reversed (per source block j, its w tokens s)
            Kraw = k[b, order, h, :].reshape(M, w, d)
            Kp = phi(Kraw, phi_kind, eps)
            V = v[b, order, h, :].reshape(M, w, d)
            dV = np.matmul(Kp, dS)                                        # (M, w, d)
            dKp = np.matmul(V, dS.transpose(0, 2, 1)) + dz[:, None, :]
            dq[b, order, h, :] = (dQp * phi_derivative(Qraw)).reshape(N, d)
            dk[b, order, h, :] = (dKp * phi_derivative(Kraw)).reshape(N, d)
            dv[b, order, h, :] = dV.reshape(N, d)
    return dq, dk, dv, dW
