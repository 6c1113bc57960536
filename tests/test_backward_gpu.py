"""Parity of the CUDA backward pass (mhla_backward) with the float64 backward oracle.

Same normwise metric and bars as the forward: max |x - x_ref| / max |x_ref| at
most 1e-4 for float32 inputs and 2e-2 for bf16 inputs (dq, dk, dv are rounded
to the input dtype; dW is float32), for each of dq, dk, dv and dW.  dout is a
seeded N(0, 1) tensor in the input dtype.
"""

import json
import os

import numpy as np
import pytest
import torch

import oracle
import token_level_head_block_gb300 as mhla
from token_level_head_block_gb300.synth import as_f64, draw_matrix, draw_qkv, draw_workload
from token_level_head_block_gb300.workloads import WORKLOADS

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f32": 1e-4}
DEV = torch.device("cuda:0")
PHI = {"relu": oracle.PHI_RELU, "relu_eps": oracle.PHI_RELU_EPS}


def normwise(got, ref):
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


def log(case, **kw):
    path = os.environ.get("MHLA_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": case, **kw}) + "\n")


def dw_term_scale(q, k, v, W, g, grid, block, phi_kind, eps):
    """max over (i, j) of sum_{b,h} sum |dS~_i| |S_j| + |dz~_i| |z_j|: the size of
    the terms dW[i][j] adds up.  With one block dW is O(eps) times this (o does
    not depend on a lone W except through eps), so bf16 operands are measured
    against the terms, not against dW's own near-zero value."""
    S, z = oracle.summaries(k, v, grid, block, phi_kind, eps)
    St, zt = oracle.mix(W, S, z)
    B, N, H, d = q.shape
    _, order, M, w = oracle.mhla_oracle._tokens_by_block(grid, block, N)
    scale = np.zeros((M, M))
    for b in range(B):
        for h in range(H):
            Qp = oracle.phi(q[b, order, h], phi_kind, eps).reshape(M, w, d)
            G = g[b, order, h].reshape(M, w, d)
            den = (Qp * zt[b, h][:, None, :]).sum(-1) + eps
            o = np.matmul(Qp, St[b, h]) / den[..., None]
            dnum = G / den[..., None]
            dden = -(G * o).sum(-1) / den
            dSt = np.abs(np.matmul(Qp.transpose(0, 2, 1), dnum))
            dzt = np.abs((Qp * dden[..., None]).sum(1))
            scale += np.einsum("irc,jrc->ij", dSt, np.abs(S[b, h])) + np.einsum("ir,jr->ij", dzt, np.abs(z[b, h]))
    return float(scale.max())


def draw_dout(shape, seed, dtype):
    return draw_qkv(*shape, seed=seed, dtype=dtype)[0]


def run_backward(q, k, v, W, g, grid, block, phi="relu", eps=1e-6, path="auto", workspace=None):
    dq, dk, dv, dW = mhla.backward(q.to(DEV), k.to(DEV), v.to(DEV), torch.as_tensor(W).to(DEV), g.to(DEV),
                                   grid, block, phi=phi, eps=eps, path=path, workspace=workspace)
    torch.cuda.synchronize()
    assert mhla.device_status() == 0
    return [as_f64(x.cpu()) for x in (dq, dk, dv, dW)]


def check(case, q, k, v, W, g, grid, block, dtype, phi="relu", eps=1e-6):
    got = run_backward(q, k, v, W, g, grid, block, phi, eps)
    ref = oracle.backward(as_f64(q), as_f64(k), as_f64(v), W, as_f64(g), grid, block, PHI[phi], eps)
    errs = {name: normwise(a, b) for name, a, b in zip(("dq", "dk", "dv", "dW"), got, ref)}
    log(f"bwd/{case}", **errs)
    for name, err in errs.items():
        assert err <= TOL[dtype], f"{case} {name}: normwise error {err:.3e}"
    return got


CASES = {
    # (B, H, d, grid, block, dtype)
    "tiny_f32": (1, 1, 32, (16, 16), (4, 4), "f32"),
    "d48_block3x5_f32": (2, 2, 48, (9, 10), (3, 5), "f32"),
    "d7_3d_f32": (1, 3, 7, (2, 6, 4), (1, 3, 2), "f32"),
    "d128_f32": (1, 1, 128, (8, 8), (2, 2), "f32"),
    # d = 1: dq_t = (g_t / den_t) S~ eps / den_t is the difference of two terms
    # equal to 1 part in den / eps; float32 resolves it only for a larger eps.
    "d1_f32_eps1e-2": (1, 2, 1, (4, 4), (2, 2), "f32", 1e-2),
    "deit_like_bf16": (4, 3, 64, (14, 14), (2, 2), "bf16"),
    "w256_bf16": (2, 2, 64, (32, 32), (16, 16), "bf16"),
    "3d_d32_bf16": (2, 2, 32, (4, 16, 16), (2, 8, 8), "bf16"),
    "m70_bf16": (1, 2, 64, (10, 28), (1, 4), "bf16"),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("phi", ["relu", "relu_eps"])
def test_backward_small(name, phi):
    B, H, d, grid, block, dtype = CASES[name][:6]
    eps = CASES[name][6] if len(CASES[name]) > 6 else 1e-6
    N = int(np.prod(grid))
    q, k, v = draw_qkv(B, N, H, d, seed=51, dtype=dtype)
    g = draw_dout((B, N, H, d), 52, dtype)
    W = draw_matrix(oracle.num_blocks(grid, block), seed=53)      # asymmetric
    check(f"{name}/{phi}", q, k, v, W, g, grid, block, dtype, phi, eps)


# Tensor-core backward: bf16, d in {32, 64}, tokens per block a multiple of 128.
# Odd head counts leave part of the last head group empty; M > 256 takes the
# general mixing GEMM and several dW tiles.
TC_CASES = {
    "2d_h3_d64": (2, 3, 64, (32, 48), (16, 8)),
    "2d_h5_d32": (2, 5, 32, (32, 32), (8, 16)),
    "3d_h2_d64": (2, 2, 64, (4, 16, 16), (2, 8, 8)),
    "3d_frames_d32": (1, 3, 32, (8, 8, 16), (4, 4, 8)),
    "w256_d64": (2, 2, 64, (32, 32), (16, 16)),
    "m300_d64": (1, 2, 64, (240, 160), (16, 8)),
    "one_block": (1, 2, 64, (16, 16), (16, 16)),
}


@pytest.mark.parametrize("name", sorted(TC_CASES))
@pytest.mark.parametrize("phi", ["relu", "relu_eps"])
def test_backward_tensor_core_path(name, phi):
    B, H, d, grid, block = TC_CASES[name]
    N = int(np.prod(grid))
    q, k, v = draw_qkv(B, N, H, d, seed=61, dtype="bf16")
    g = draw_dout((B, N, H, d), 62, "bf16")
    W = draw_matrix(oracle.num_blocks(grid, block), seed=63)      # asymmetric
    got = run_backward(q, k, v, W, g, grid, block, phi, 1e-6, path="tc")
    args = (as_f64(q), as_f64(k), as_f64(v), W, as_f64(g), grid, block, PHI[phi], 1e-6)
    ref = oracle.backward(*args)
    errs = {gname: normwise(a, b) for gname, a, b in zip(("dq", "dk", "dv", "dW"), got, ref)}
    if W.shape[0] == 1:
        errs["dW"] = float(np.abs(got[3] - ref[3]).max()) / dw_term_scale(*args)
    log(f"bwd_tc/{name}/{phi}", **errs)
    for gname, err in errs.items():
        assert err <= TOL["bf16"], f"tc/{name}/{phi} {gname}: normwise error {err:.3e}"


def test_backward_paths_agree_and_tensor_core_path_is_deterministic():
    B, H, d, grid, block = 2, 3, 64, (32, 32), (16, 8)
    q, k, v = draw_qkv(B, 1024, H, d, seed=64)
    g = draw_dout((B, 1024, H, d), 65, "bf16")
    W = mhla.init_mixing(grid, block, "cos")
    a = run_backward(q, k, v, W, g, grid, block, path="tc")
    b = run_backward(q, k, v, W, g, grid, block, path="tc")
    c = run_backward(q, k, v, W, g, grid, block, path="simt")
    for x, y, z in zip(a, b, c):
        assert np.array_equal(x, y)
        assert normwise(x, z) <= TOL["bf16"]


def test_backward_tensor_core_strided_slices():
    B, N, H, d, grid, block = 2, 512, 3, 64, (16, 32), (16, 8)
    qkv = draw_qkv(B, N, 3 * H, d, seed=66)[0].view(B, N, 3, H, d)
    g = draw_dout((B, N, H, d), 67, "bf16")
    W = draw_matrix(oracle.num_blocks(grid, block), seed=68)
    qd = qkv.to(DEV)
    got = mhla.backward(qd[:, :, 0], qd[:, :, 1], qd[:, :, 2], torch.from_numpy(W).to(DEV), g.to(DEV), grid, block,
                        path="tc")
    torch.cuda.synchronize()
    assert mhla.device_status() == 0
    ref = oracle.backward(as_f64(qkv[:, :, 0]), as_f64(qkv[:, :, 1]), as_f64(qkv[:, :, 2]), W, as_f64(g), grid, block)
    for a, b in zip(got, ref):
        assert normwise(as_f64(a.cpu()), b) <= TOL["bf16"]


def test_backward_of_strided_slices_and_determinism():
    B, N, H, d, grid, block = 2, 256, 3, 64, (16, 16), (4, 8)
    qkv = draw_qkv(B, N, 3 * H, d, seed=54)[0].view(B, N, 3, H, d)
    g = draw_dout((B, N, H, d), 55, "bf16")
    W = draw_matrix(oracle.num_blocks(grid, block), seed=56)
    qd, Wd, gd = qkv.to(DEV), torch.from_numpy(W).to(DEV), g.to(DEV)
    outs = [mhla.backward(qd[:, :, 0], qd[:, :, 1], qd[:, :, 2], Wd, gd, grid, block) for _ in range(2)]
    torch.cuda.synchronize()
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    ref = oracle.backward(as_f64(qkv[:, :, 0]), as_f64(qkv[:, :, 1]), as_f64(qkv[:, :, 2]), W, as_f64(g), grid, block)
    for a, b in zip(outs[0], ref):
        assert normwise(as_f64(a.cpu()), b) <= TOL["bf16"]


def test_backward_explicit_workspace_and_empty_batch():
    B, H, d, grid, block = 1, 2, 32, (16, 16), (8, 8)
    q, k, v = draw_qkv(B, 256, H, d, seed=57, dtype="f32")
    g = draw_dout((B, 256, H, d), 58, "f32")
    W = draw_matrix(4, seed=59)
    need = mhla.backward_workspace_size(q, grid, block)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    a = run_backward(q, k, v, W, g, grid, block, workspace=ws)
    b = run_backward(q, k, v, W, g, grid, block)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    e = torch.empty(0, 256, 2, 32, device=DEV)
    dW = torch.full((4, 4), 5.0, device=DEV)
    mhla.backward(e, e, e, torch.from_numpy(W).to(DEV), e, grid, block, dW=dW)
    torch.cuda.synchronize()
    assert torch.all(dW == 0)


def test_backward_workload_deit_all_slices():
    wl = WORKLOADS["deit_t_14x14"]
    q, k, v = draw_workload(wl)
    g = draw_dout((wl.B, wl.N, wl.H, wl.d), wl.seed + 100, wl.dtype)
    W = mhla.init_mixing(wl.grid, wl.block, wl.transform, wl.local_thres, wl.exp_sigma)
    check("workload/deit", q, k, v, W, g, wl.grid, wl.block, wl.dtype)


def test_backward_workload_dit_all_slices():
    wl = WORKLOADS["dit_s2_4096px"]
    q, k, v = draw_workload(wl)
    g = draw_dout((wl.B, wl.N, wl.H, wl.d), wl.seed + 100, wl.dtype)
    W = mhla.init_mixing(wl.grid, wl.block, wl.transform, wl.local_thres, wl.exp_sigma)
    check("workload/dit", q, k, v, W, g, wl.grid, wl.block, wl.dtype)
