"""Parity of the causal backward pass (mhla_backward_causal) with the float64
causal backward oracle.

Same normwise metric and bars as the other backward tests: max |x - x_ref| /
max |x_ref| at most 1e-4 for float32 inputs and 2e-2 for bf16 inputs, for each
of dq, dk, dv and dW.  Blocks are contiguous token ranges as for the causal
forward: 1-D sequences cut into chunks (some not a multiple of the kernels'
32-token chunk), whole rows, whole frames, one token per block, one block.
"""

import numpy as np
import pytest
import torch

import oracle
import token_level_head_block_gb300 as mhla
from token_level_head_block_gb300.synth import as_f64, draw_matrix, draw_qkv

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f32": 1e-4}
DEV = torch.device("cuda:0")
PHI = {"relu": oracle.PHI_RELU, "relu_eps": oracle.PHI_RELU_EPS}
NAMES = ("dq", "dk", "dv", "dW")


def normwise(got, ref):
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


def draw_dout(shape, seed, dtype):
    return draw_qkv(*shape, seed=seed, dtype=dtype)[0]


def run(q, k, v, W, g, grid, block, phi="relu", eps=1e-6, workspace=None, path="auto"):
    out = mhla.backward_causal(q.to(DEV), k.to(DEV), v.to(DEV), torch.as_tensor(W).to(DEV), g.to(DEV), grid, block,
                               phi=phi, eps=eps, workspace=workspace, path=path)
    torch.cuda.synchronize()
    assert mhla.device_status() == 0
    return [as_f64(x.cpu()) for x in out]


def dw_term_scale(q, k, v, W, g, grid, block, phi_kind, eps):
    """max over (i, j) of the sum of |terms| dW[i][j] adds up, from the explicit
    causal form: sum over t in i, s in j, s <= t of |phi(q_t).phi(k_s)| |dA_ts|.
    With a single block, o does not depend on W but through eps, so dW is a
    near-cancelling sum; it is measured against the size of its terms."""
    B, N, H, d = q.shape
    ids = oracle.block_of_token(grid, block)
    M = oracle.num_blocks(grid, block)
    onehot = np.zeros((N, M))
    onehot[np.arange(N), ids] = 1.0
    mask = np.tril(np.ones((N, N)))
    Wt = W[np.ix_(ids, ids)] * mask
    scale = np.zeros((M, M))
    for b in range(B):
        for h in range(H):
            Qp = oracle.phi(q[b, :, h], phi_kind, eps)
            Kp = oracle.phi(k[b, :, h], phi_kind, eps)
            E = Qp @ Kp.T
            A = Wt * E
            den = A.sum(axis=1) + eps
            o = (A @ v[b, :, h]) / den[:, None]
            dnum = g[b, :, h] / den[:, None]
            dden = -(g[b, :, h] * o).sum(axis=1) / den
            dA = dnum @ v[b, :, h].T + dden[:, None]
            scale += onehot.T @ (np.abs(E) * np.abs(dA) * mask) @ onehot
    return float(scale.max())


def check(case, q, k, v, W, g, grid, block, dtype, phi="relu", eps=1e-6, path="auto"):
    got = run(q, k, v, W, g, grid, block, phi, eps, path=path)
    args = (as_f64(q), as_f64(k), as_f64(v), W, as_f64(g), grid, block, PHI[phi], eps)
    ref = oracle.backward_causal(*args)
    errs = {name: normwise(a, b) for name, a, b in zip(NAMES, got, ref)}
    if W.shape[0] == 1:
        errs["dW"] = float(np.abs(got[3] - ref[3]).max()) / dw_term_scale(*args)
    for name, err in errs.items():
        assert err <= TOL[dtype], f"{case} {name}: normwise error {err:.3e}"
    return got


CASES = {
    # (B, H, d, grid, block, dtype[, eps])
    "seq_d64_bf16": (2, 3, 64, (1, 512), (1, 64), "bf16"),
    "seq_ragged_chunk_d32_bf16": (1, 2, 32, (1, 300), (1, 50), "bf16"),   # 50 = 32 + 18 tokens per block
    "seq_long_blocks_d64_bf16": (1, 2, 64, (1, 1024), (1, 256), "bf16"),  # 8 chunks per block
    "seq_ragged_chunk_d64_f32": (1, 2, 64, (1, 280), (1, 70), "f32"),     # 70 = 2 x 32 + 6 tokens per block
    "seq_short_blocks_d64_bf16": (2, 2, 64, (1, 200), (1, 20), "bf16"),  # one part-filled chunk per block
    "frames_d32_bf16": (1, 2, 32, (4, 8, 8), (1, 8, 8), "bf16"),         # whole 64-token frames
    "seq_d64_f32": (1, 2, 64, (1, 256), (1, 32), "f32"),
    "rows_d48_f32": (2, 2, 48, (12, 10), (3, 10), "f32"),
    "rows_d128_bf16": (1, 2, 128, (8, 16), (2, 16), "bf16"),
    "frames_d16_f32": (1, 3, 16, (6, 4, 4), (2, 4, 4), "f32"),
    "one_block_d128_f32": (1, 1, 128, (1, 96), (1, 96), "f32"),
    "token_blocks_d7_f32": (1, 2, 7, (1, 40), (1, 1), "f32"),             # w = 1: mixing only
    # d = 1: dq is a difference of two terms equal to 1 part in den / eps, as
    # in the non-causal backward; float32 resolves it only for a larger eps.
    "seq_d1_f32_eps1e-2": (2, 1, 1, (1, 64), (1, 8), "f32", 1e-2),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("phi", ["relu", "relu_eps"])
def test_causal_backward_matches_oracle(name, phi):
    B, H, d, grid, block, dtype = CASES[name][:6]
    eps = CASES[name][6] if len(CASES[name]) > 6 else 1e-6
    N = int(np.prod(grid))
    q, k, v = draw_qkv(B, N, H, d, seed=81, dtype=dtype)
    g = draw_dout((B, N, H, d), 82, dtype)
    W = draw_matrix(oracle.num_blocks(grid, block), seed=83)      # asymmetric; the upper triangle must not matter
    check(f"{name}/{phi}", q, k, v, W, g, grid, block, dtype, phi, eps)


@pytest.mark.parametrize("path", ["simt", "tc"])
@pytest.mark.parametrize("grid,block", [((1, 512), (1, 64)), ((1, 768), (1, 128)), ((4, 8, 8), (1, 8, 8))])
def test_causal_backward_both_ways_to_the_states(path, grid, block):
    """The summaries and the mixed past formed on CUDA cores (SIMT) or by the
    tensor-core causal forward's kernels (TC: bf16 operands), each against the
    oracle, on the shapes TC takes: blocks of 64 and 128 tokens, whole frames."""
    B, H, d = 2, 3, 64
    N = int(np.prod(grid))
    q, k, v = draw_qkv(B, N, H, d, seed=96, dtype="bf16")
    g = draw_dout((B, N, H, d), 97, "bf16")
    W = draw_matrix(oracle.num_blocks(grid, block), seed=98)
    check(f"{path}/{grid}/{block}", q, k, v, W, g, grid, block, "bf16", "relu_eps", 1e-6, path=path)


def test_causal_backward_tc_path_padding_columns_and_repeatability():
    """B H = 3 at d = 64: the summary layout's last 128-column group is half
    padding, which the dW product reads and must see as zero; and the TC path's
    reductions run in a fixed order, so two calls agree bit for bit."""
    B, N, H, d, grid, block = 1, 512, 3, 64, (1, 512), (1, 64)
    q, k, v = draw_qkv(B, N, H, d, seed=102, dtype="bf16")
    g = draw_dout((B, N, H, d), 103, "bf16")
    W = draw_matrix(8, seed=104)
    a = check("tc/BH3", q, k, v, W, g, grid, block, "bf16", path="tc")
    b = run(q, k, v, W, g, grid, block, path="tc")
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_causal_backward_tc_states_past_the_resident_mixing():
    """M = 320 blocks: the tensor-core mixing streams W instead of holding it in
    shared memory; the summaries it reads must survive it for dW."""
    B, N, H, d, grid, block = 1, 20480, 1, 64, (1, 20480), (1, 64)
    q, k, v = draw_qkv(B, N, H, d, seed=99, dtype="bf16")
    g = draw_dout((B, N, H, d), 100, "bf16")
    W = draw_matrix(320, seed=101)
    check("tc/M320", q, k, v, W, g, grid, block, "bf16", path="tc")


def test_causal_backward_ignores_w_above_the_diagonal_and_is_deterministic():
    B, H, d, grid, block = 2, 2, 32, (1, 256), (1, 32)
    q, k, v = draw_qkv(B, 256, H, d, seed=84, dtype="f32")
    g = draw_dout((B, 256, H, d), 85, "f32")
    W = draw_matrix(8, seed=86)
    W2 = W.copy()
    W2[np.triu_indices(8, 1)] = 123.0
    a = run(q, k, v, W, g, grid, block)
    b = run(q, k, v, W, g, grid, block)
    c = run(q, k, v, W2, g, grid, block)
    for x, y, z in zip(a, b, c):
        assert np.array_equal(x, y)            # fixed reduction orders: bitwise repeatable
        assert np.array_equal(x, z)            # W above the diagonal is never read
    assert not np.any(a[3][np.triu_indices(8, 1)])   # and dW is zero there


def test_causal_backward_of_strided_slices():
    B, N, H, d, grid, block = 2, 512, 3, 64, (1, 512), (1, 128)
    qkv = draw_qkv(B, N, 3 * H, d, seed=87)[0].view(B, N, 3, H, d)
    g = draw_dout((B, N, H, d), 88, "bf16")
    W = draw_matrix(4, seed=89)
    qd = qkv.to(DEV)
    got = mhla.backward_causal(qd[:, :, 0], qd[:, :, 1], qd[:, :, 2], torch.from_numpy(W).to(DEV), g.to(DEV), grid,
                               block)
    torch.cuda.synchronize()
    assert mhla.device_status() == 0
    ref = oracle.backward_causal(as_f64(qkv[:, :, 0]), as_f64(qkv[:, :, 1]), as_f64(qkv[:, :, 2]), W, as_f64(g),
                                 grid, block)
    for name, a, b in zip(NAMES, got, ref):
        assert normwise(as_f64(a.cpu()), b) <= TOL["bf16"], name


def test_causal_backward_explicit_workspace_and_empty_batch():
    B, H, d, grid, block = 1, 2, 32, (1, 256), (1, 64)
    q, k, v = draw_qkv(B, 256, H, d, seed=90, dtype="f32")
    g = draw_dout((B, 256, H, d), 91, "f32")
    W = draw_matrix(4, seed=92)
    need = mhla.backward_causal_workspace_size(q, grid, block)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    a = run(q, k, v, W, g, grid, block, workspace=ws)
    b = run(q, k, v, W, g, grid, block)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    e = torch.empty(0, 256, 2, 32, device=DEV)
    dW = torch.full((4, 4), 7.0, device=DEV)
    mhla.backward_causal(e, e, e, torch.from_numpy(W).to(DEV), e, grid, block, dW=dW)
    torch.cuda.synchronize()
    assert not dW.any()


def test_causal_backward_matches_autograd_of_the_dense_form():
    """The float32 CUDA result against torch autograd of the explicit causal
    N x N form (float64, CPU): a derivation independent of both."""
    B, H, d, grid, block = 1, 2, 16, (1, 96), (1, 24)
    q, k, v = draw_qkv(B, 96, H, d, seed=93, dtype="f32")
    g = draw_dout((B, 96, H, d), 94, "f32")
    W = draw_matrix(4, seed=95)
    got = run(q, k, v, W, g, grid, block)
    qt, kt, vt = (torch.tensor(as_f64(x), requires_grad=True) for x in (q, k, v))
    Wt = torch.tensor(W, dtype=torch.float64, requires_grad=True)
    ids = torch.as_tensor(oracle.block_of_token(grid, block))
    mask = torch.tril(torch.ones(96, 96, dtype=torch.float64))
    Wtok = Wt[ids][:, ids] * mask
    Qp, Kp = torch.relu(qt), torch.relu(kt)
    A = Wtok[None, None] * torch.einsum("bnhd,bmhd->bhnm", Qp, Kp)
    o = torch.einsum("bhnm,bmhd->bnhd", A, vt) / (A.sum(-1).permute(0, 2, 1)[..., None] + 1e-6)
    (o * torch.tensor(as_f64(g))).sum().backward()
    for name, a, b in zip(NAMES, got, (qt.grad, kt.grad, vt.grad, Wt.grad)):
        assert normwise(a, b.numpy()) <= TOL["f32"], name


def test_causal_backward_workload_sampled_slices():
    """The causal LM workload at full size (B=4, H=12, N=4096, 64-token blocks), as
    the backward bench runs it: dq, dk, dv of three (b, h) slices against the
    oracle on those slices (a slice's gradients depend on that slice alone); dW,
    which sums over every slice, is checked for its zero upper triangle."""
    from token_level_head_block_gb300.synth import draw_workload
    from token_level_head_block_gb300.workloads import WORKLOADS
    wl = WORKLOADS["lm_causal_4096"]
    q, k, v = draw_workload(wl)
    g = draw_dout((wl.B, wl.N, wl.H, wl.d), wl.seed + 100, wl.dtype)
    W = mhla.init_mixing(wl.grid, wl.block, wl.transform, wl.local_thres, wl.exp_sigma)
    dq, dk, dv, dW = run(q, k, v, W, g, wl.grid, wl.block, wl.phi, wl.eps)
    assert np.all(np.isfinite(dW)) and not np.any(dW[np.triu_indices(wl.M, 1)])
    for b, h in [(0, 0), (wl.B - 1, wl.H - 1), (wl.B // 2, wl.H // 2)]:
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1), slice(None))
        ref = oracle.backward_causal(as_f64(q[sl]), as_f64(k[sl]), as_f64(v[sl]), W, as_f64(g[sl]), wl.grid,
                                     wl.block, PHI[wl.phi], wl.eps)
        for name, a, r in zip(NAMES[:3], (dq, dk, dv), ref[:3]):
            assert normwise(a[sl], r) <= TOL[wl.dtype], (name, b, h)
