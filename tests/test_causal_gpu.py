"""Parity of causal MHLA (mhla_forward_causal) with the float64 causal oracle.

Same normwise metric and bars as the forward: 1e-4 for float32 inputs, 2e-2
for bf16 inputs.  Blocks are contiguous token ranges: 1-D sequences cut into
chunks, whole rows, whole frames.
"""

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
    return float(np.abs(got - ref).max() / np.abs(ref).max())


def run(q, k, v, W, grid, block, phi="relu", eps=1e-6, path="auto"):
    out = mhla.forward_causal(q.to(DEV), k.to(DEV), v.to(DEV), torch.as_tensor(W).to(DEV), grid, block, phi=phi,
                              eps=eps, path=path)
    torch.cuda.synchronize()
    assert mhla.device_status() == 0
    return as_f64(out.cpu())


CASES = {
    # (B, H, d, grid, block, dtype)
    "seq_d64_bf16": (2, 3, 64, (1, 512), (1, 64), "bf16"),
    "seq_ragged_chunk_d32_bf16": (1, 2, 32, (1, 300), (1, 50), "bf16"),   # 50 = 32 + 18 tokens per block
    "seq_d64_f32": (1, 2, 64, (1, 256), (1, 32), "f32"),
    "rows_d48_f32": (2, 2, 48, (12, 10), (3, 10), "f32"),
    "frames_d16_f32": (1, 3, 16, (6, 4, 4), (2, 4, 4), "f32"),
    "one_block_d128_f32": (1, 1, 128, (1, 96), (1, 96), "f32"),
    "token_blocks_d7_f32": (1, 2, 7, (1, 40), (1, 1), "f32"),              # w = 1: mixing only
    "seq_d1_f32": (2, 1, 1, (1, 64), (1, 8), "f32"),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("phi", ["relu", "relu_eps"])
def test_causal_matches_oracle(name, phi):
    B, H, d, grid, block, dtype = CASES[name]
    N = int(np.prod(grid))
    q, k, v = draw_qkv(B, N, H, d, seed=71, dtype=dtype)
    W = draw_matrix(oracle.num_blocks(grid, block), seed=72)     # asymmetric, upper triangle must not matter
    got = run(q, k, v, W, grid, block, phi)
    ref = oracle.forward_causal(as_f64(q), as_f64(k), as_f64(v), W, grid, block, PHI[phi], 1e-6)
    err = normwise(got, ref)
    assert err <= TOL[dtype], f"{name}/{phi}: normwise error {err:.3e}"


# Tensor-core causal path: bf16, d in {32, 64}, N a multiple of 128, blocks of
# 64 tokens (two units per tile) or a multiple of 128 (one unit per tile, one
# or more units per block); M_u = 512 takes the streaming mixing GEMM.
TC_CASES = {
    "w64_d64": (2, 3, 64, (1, 512), (1, 64)),
    "w64_d32": (1, 2, 32, (1, 1024), (1, 64)),
    "w128_d64": (2, 2, 64, (1, 768), (1, 128)),
    "w256_d64": (1, 3, 64, (1, 1024), (1, 256)),
    "w384_d32": (1, 2, 32, (1, 768), (1, 384)),
    "rows_w128_d64": (1, 2, 64, (8, 128), (1, 128)),
    "frames_w256_d32": (1, 2, 32, (4, 8, 16), (2, 8, 16)),
    "mu512_d64": (1, 1, 64, (1, 32768), (1, 64)),
}


@pytest.mark.parametrize("name", sorted(TC_CASES))
@pytest.mark.parametrize("phi", ["relu", "relu_eps"])
def test_causal_tensor_core_path(name, phi):
    B, H, d, grid, block = TC_CASES[name]
    N = int(np.prod(grid))
    q, k, v = draw_qkv(B, N, H, d, seed=76, dtype="bf16")
    W = draw_matrix(oracle.num_blocks(grid, block), seed=77)
    got = run(q, k, v, W, grid, block, phi, path="tc")
    if N <= 4096:
        ref = oracle.forward_causal(as_f64(q), as_f64(k), as_f64(v), W, grid, block, PHI[phi], 1e-6)
        err = normwise(got, ref)
    else:   # the python-loop oracle on a sample of tokens: the first, a middle and the last block
        M = oracle.num_blocks(grid, block)
        w = N // M
        cut = [slice(0, 2 * w), slice(N // 2 - w, N // 2 + w), slice(N - 2 * w, N)]
        ref_all = oracle.forward_causal(as_f64(q), as_f64(k), as_f64(v), W, grid, block, PHI[phi], 1e-6)
        err = max(normwise(got[:, c], ref_all[:, c]) for c in cut)
    assert err <= TOL["bf16"], f"tc/{name}/{phi}: normwise error {err:.3e}"


def test_causal_paths_agree():
    B, H, d, grid, block = 2, 3, 64, (1, 1024), (1, 64)
    q, k, v = draw_qkv(B, 1024, H, d, seed=78)
    W = mhla.init_mixing(grid, block, "linear")
    a = run(q, k, v, W, grid, block, path="tc")
    b = run(q, k, v, W, grid, block, path="simt")
    c = run(q, k, v, W, grid, block, path="tc")
    assert np.array_equal(a, c)
    assert normwise(a, b) <= TOL["bf16"]


def test_causal_ignores_w_above_the_diagonal_and_is_deterministic():
    B, H, d, grid, block = 2, 2, 64, (1, 256), (1, 32)
    q, k, v = draw_qkv(B, 256, H, d, seed=73)
    W = draw_matrix(8, seed=74)
    W2 = W.copy()
    W2[np.triu_indices(8, 1)] = 7.0
    a = run(q, k, v, W, grid, block)
    b = run(q, k, v, W2, grid, block)
    c = run(q, k, v, W, grid, block)
    assert np.array_equal(a, b) and np.array_equal(a, c)


@pytest.mark.parametrize("grid,block", [((1, 384), (1, 48)), ((1, 512), (1, 64))], ids=["simt", "tc"])
def test_causal_strided_slices_of_one_projection(grid, block):
    B, H, d = 2, 3, 64
    N = int(np.prod(grid))
    qkv = draw_qkv(B, N, 3 * H, d, seed=75)[0].view(B, N, 3, H, d)
    W = mhla.init_mixing(grid, block, "linear")
    qd = qkv.to(DEV)
    out = mhla.forward_causal(qd[:, :, 0], qd[:, :, 1], qd[:, :, 2], torch.from_numpy(W).to(DEV), grid, block)
    torch.cuda.synchronize()
    ref = oracle.forward_causal(as_f64(qkv[:, :, 0]), as_f64(qkv[:, :, 1]), as_f64(qkv[:, :, 2]), W, grid, block)
    assert normwise(as_f64(out.cpu()), ref) <= TOL["bf16"]


def test_causal_workload_sampled_slices():
    wl = WORKLOADS["lm_causal_4096"]
    q, k, v = draw_workload(wl)
    W = mhla.init_mixing(wl.grid, wl.block, wl.transform, wl.local_thres, wl.exp_sigma)
    out = run(q, k, v, W, wl.grid, wl.block, wl.phi, wl.eps)
    for b, h in [(0, 0), (wl.B - 1, wl.H - 1), (wl.B // 2, wl.H // 2)]:
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1), slice(None))
        ref = oracle.forward_causal(as_f64(q[sl]), as_f64(k[sl]), as_f64(v[sl]), W, wl.grid, wl.block,
                                    PHI[wl.phi], wl.eps)
        assert normwise(out[sl], ref) <= TOL[wl.dtype], (b, h)
