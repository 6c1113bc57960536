"""Parity of the CUDA path with the CPU oracle, through the C ABI.

Error metric (elementwise relative error is ill-posed: outputs are weighted
means of zero-mean values, many near 0): normwise
    max |o_gpu - o_oracle| / max |o_oracle|
at most 1e-4 for float32 inputs and 2e-2 for bf16 inputs with float32
accumulation.  Small problems are compared element by element in full; the
full-size workloads run in the launch configuration the benchmark times and are
compared on every output of a sample of (batch, head) slices (each slice is an
independent problem the oracle can solve alone).
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
    return float(np.abs(got - ref).max() / np.abs(ref).max())


def error_report(got, ref):
    """The bar (normwise) with two views of the whole error distribution: the
    relative Frobenius error and the elementwise 99.9th percentile of
    |got - ref|, both against the same scale max |ref|."""
    diff = np.abs(got - ref)
    scale = np.abs(ref).max()
    return {"normwise": float(diff.max() / scale),
            "frobenius": float(np.linalg.norm(diff.ravel()) / np.linalg.norm(ref.ravel())),
            "p999": float(np.percentile(diff, 99.9) / scale)}


def log(case, **kw):
    path = os.environ.get("MHLA_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": case, **kw}) + "\n")


def run(q, k, v, W, grid, block, phi="relu", eps=1e-6, path="auto", workspace=None):
    out = mhla.forward(q.to(DEV), k.to(DEV), v.to(DEV), torch.as_tensor(W).to(DEV), grid, block, phi=phi,
                       eps=eps, path=path, workspace=workspace)
    torch.cuda.synchronize()
    assert mhla.device_status() == 0
    return out


def check_full(case, q, k, v, W, grid, block, dtype, phi="relu", eps=1e-6, path="auto"):
    out = run(q, k, v, W, grid, block, phi, eps, path)
    assert out.dtype == q.dtype
    ref = oracle.forward(as_f64(q), as_f64(k), as_f64(v), W, grid, block, PHI[phi], eps)
    rep = error_report(as_f64(out), ref)
    err = rep["normwise"]
    log(case, err=err, path=path, dtype=dtype, **rep)
    assert err <= TOL[dtype], f"{case}: normwise error {err:.3e}"
    return err


# ------------------------------------------------------------------ small cases
# (B, H, d, grid, block): tokens per block a multiple of 128 so both paths apply;
# odd head counts leave part of the last head group of the summary kernel empty,
# M > 256 needs two query-block tiles in the mixing GEMM, M not a multiple of 64
# leaves a ragged source-block chunk; d = 32 with an even head count reads out
# head pairs as 64-channel rows (block-diagonal operand), odd counts one head at
# a time.
TC_CASES = {
    "2d_h3_d64": (2, 3, 64, (32, 48), (16, 8)),
    "2d_h5_d32": (2, 5, 32, (32, 32), (8, 16)),
    "2d_h4_d32_pairs": (2, 4, 32, (32, 32), (8, 16)),
    "3d_h6_d32_pairs": (1, 6, 32, (8, 8, 16), (4, 4, 8)),
    "3d_h2_d64": (2, 2, 64, (4, 16, 16), (2, 8, 8)),
    "3d_frames_d32": (1, 3, 32, (8, 8, 16), (4, 4, 8)),
    "w256_d64": (2, 2, 64, (32, 32), (16, 16)),
    "m300_d64": (1, 2, 64, (240, 160), (16, 8)),
    "one_block": (1, 2, 64, (16, 16), (16, 16)),
}


@pytest.mark.parametrize("name", sorted(TC_CASES))
@pytest.mark.parametrize("phi", ["relu", "relu_eps"])
def test_tensor_core_path_small(name, phi):
    B, H, d, grid, block = TC_CASES[name]
    N = int(np.prod(grid))
    q, k, v = draw_qkv(B, N, H, d, seed=11, dtype="bf16")
    M = oracle.num_blocks(grid, block)
    W = draw_matrix(M, seed=12)                  # asymmetric: a transposed W would show
    check_full(f"tc/{name}/{phi}", q, k, v, W, grid, block, "bf16", phi, 1e-6, "tc")


@pytest.mark.parametrize("name", sorted(TC_CASES))
def test_tensor_core_single_launch_small(name):
    """The same cases in one persistent launch (where M <= 256)."""
    B, H, d, grid, block = TC_CASES[name]
    N = int(np.prod(grid))
    q, k, v = draw_qkv(B, N, H, d, seed=11, dtype="bf16")
    M = oracle.num_blocks(grid, block)
    W = draw_matrix(M, seed=12)
    path = "tc_fused" if M <= 256 else "tc"
    check_full(f"tc_fused/{name}", q, k, v, W, grid, block, "bf16", "relu", 1e-6, path)


@pytest.mark.parametrize("name", sorted(TC_CASES))
def test_single_launch_equals_split_launches_bitwise(name):
    """The persistent single launch runs the same arithmetic as the three
    launches (same operands, same MMA order per item and tile), whatever CTA
    takes which item: the outputs are identical bit for bit, run after run."""
    B, H, d, grid, block = TC_CASES[name]
    N = int(np.prod(grid))
    q, k, v = draw_qkv(B, N, H, d, seed=37, dtype="bf16")
    W = draw_matrix(oracle.num_blocks(grid, block), seed=38)
    single = "tc_fused" if oracle.num_blocks(grid, block) <= 256 else "tc"
    a = run(q, k, v, W, grid, block, path=single).cpu()
    b = run(q, k, v, W, grid, block, path=single).cpu()
    c = run(q, k, v, W, grid, block, path="tc").cpu()
    assert torch.equal(a, b)
    assert torch.equal(a, c)


@pytest.mark.parametrize("B", [1, 7])
def test_single_launch_batches_straddling_mixing_tiles(B):
    """Mixing tiles of 128 summary columns that straddle two batches (H (d + 1) d
    is not a multiple of 128) wait for both batches' summaries and count for
    both batches' readout."""
    H, d, grid, block = 5, 32, (16, 32), (8, 16)
    q, k, v = draw_qkv(B, 512, H, d, seed=39, dtype="bf16")
    W = draw_matrix(oracle.num_blocks(grid, block), seed=40)
    check_full(f"tc_straddle/B{B}", q, k, v, W, grid, block, "bf16", "relu", 1e-6, "tc_fused")


@pytest.mark.parametrize("name", sorted(TC_CASES))
def test_simt_path_bf16_small(name):
    B, H, d, grid, block = TC_CASES[name]
    N = int(np.prod(grid))
    q, k, v = draw_qkv(B, N, H, d, seed=13, dtype="bf16")
    W = mhla.init_mixing(grid, block, "exp")
    check_full(f"simt/{name}", q, k, v, W, grid, block, "bf16", "relu", 1e-6, "simt")


SIMT_CASES = {
    "d48_block3x5": (2, 2, 48, (9, 10), (3, 5)),
    "d7_3d": (1, 3, 7, (2, 6, 4), (1, 3, 2)),
    "d128_w4": (1, 1, 128, (8, 8), (2, 2)),
    "deit_like": (4, 3, 64, (14, 14), (2, 2)),
    "d1": (1, 2, 1, (4, 4), (2, 2)),
}


@pytest.mark.parametrize("name", sorted(SIMT_CASES))
@pytest.mark.parametrize("phi", ["relu", "relu_eps"])
def test_simt_path_fp32_small(name, phi):
    B, H, d, grid, block = SIMT_CASES[name]
    N = int(np.prod(grid))
    q, k, v = draw_qkv(B, N, H, d, seed=17, dtype="f32")
    M = oracle.num_blocks(grid, block)
    W = draw_matrix(M, seed=18)
    check_full(f"simt_f32/{name}/{phi}", q, k, v, W, grid, block, "f32", phi, 1e-6, "simt")


# Fused short-sequence path: N <= 256 tokens, M <= 96 blocks.  Cases cover one
# and two query tiles, a ragged last key chunk (N not a multiple of 32), a single
# token, one block, one block per token, the 96-block limit, 3-D grids and both d.
FUSED_CASES = {
    "deit_like_d64": (3, 3, 64, (14, 14), (2, 2)),
    "n1_d64": (2, 1, 64, (1, 1), (1, 1)),
    "n37_d64_w1": (2, 2, 64, (1, 37), (1, 1)),
    "n100_d32": (2, 3, 32, (10, 10), (2, 5)),
    "n128_d32": (2, 2, 32, (8, 16), (4, 4)),
    "n129_d64": (1, 2, 64, (3, 43), (3, 1)),
    "n250_d32": (1, 2, 32, (10, 25), (5, 5)),
    "n256_d64_m1": (1, 2, 64, (16, 16), (16, 16)),
    "m96_d64": (1, 1, 64, (12, 16), (2, 1)),
    "3d_d64": (2, 2, 64, (4, 6, 8), (2, 3, 2)),
    "3d_d32": (1, 3, 32, (3, 8, 8), (1, 4, 4)),
}


@pytest.mark.parametrize("name", sorted(FUSED_CASES))
@pytest.mark.parametrize("phi", ["relu", "relu_eps"])
def test_fused_path_small(name, phi):
    B, H, d, grid, block = FUSED_CASES[name]
    N = int(np.prod(grid))
    q, k, v = draw_qkv(B, N, H, d, seed=31, dtype="bf16")
    M = oracle.num_blocks(grid, block)
    W = draw_matrix(M, seed=32)                  # asymmetric: a transposed W would show
    check_full(f"fused/{name}/{phi}", q, k, v, W, grid, block, "bf16", phi, 1e-6, "fused")


def test_fused_path_takes_slices_of_one_projection_and_is_deterministic():
    B, N, H, d, grid, block = 2, 196, 3, 64, (14, 14), (2, 2)
    qkv = draw_qkv(B, N, 3 * H, d, seed=33)[0].view(B, N, 3, H, d)
    W = mhla.init_mixing(grid, block, "linear")
    qd, Wd = qkv.to(DEV), torch.from_numpy(W).to(DEV)
    outs = [mhla.forward(qd[:, :, 0], qd[:, :, 1], qd[:, :, 2], Wd, grid, block, path="fused") for _ in range(2)]
    torch.cuda.synchronize()
    assert mhla.device_status() == 0
    assert torch.equal(outs[0], outs[1])
    ref = oracle.forward(as_f64(qkv[:, :, 0]), as_f64(qkv[:, :, 1]), as_f64(qkv[:, :, 2]), W, grid, block)
    assert normwise(as_f64(outs[0].cpu()), ref) <= TOL["bf16"]


def test_fused_path_agrees_with_the_three_launch_path():
    B, H, d, grid, block = 2, 3, 64, (16, 16), (16, 8)
    q, k, v = draw_qkv(B, 256, H, d, seed=34)
    W = mhla.init_mixing(grid, block, "cos")
    a = run(q, k, v, W, grid, block, path="fused").cpu()
    b = run(q, k, v, W, grid, block, path="tc").cpu()
    assert normwise(as_f64(a), as_f64(b)) <= TOL["bf16"]


# The tensor-core forward on contiguous 64-token blocks (1-D sequences, rows of
# 64): summaries and mixing as usual, the readout per 128-token tile of two blocks.
TILE_CASES = {
    "seq_d64": (2, 3, 64, (1, 1024), (1, 64)),
    "seq_d32": (1, 2, 32, (1, 512), (1, 64)),
    "rows_d64": (2, 2, 64, (16, 64), (1, 64)),
    "m512_d64": (1, 1, 64, (1, 32768), (1, 64)),
}


@pytest.mark.parametrize("name", sorted(TILE_CASES))
@pytest.mark.parametrize("phi", ["relu", "relu_eps"])
def test_tensor_core_tile_readout(name, phi):
    B, H, d, grid, block = TILE_CASES[name]
    N = int(np.prod(grid))
    q, k, v = draw_qkv(B, N, H, d, seed=35, dtype="bf16")
    W = draw_matrix(oracle.num_blocks(grid, block), seed=36)
    check_full(f"tile/{name}/{phi}", q, k, v, W, grid, block, "bf16", phi, 1e-6, "tc")


def test_tiny_fp32_workload():
    wl = WORKLOADS["tiny_16x16_fp32"]
    q, k, v = draw_workload(wl)
    W = mhla.init_mixing(wl.grid, wl.block, wl.transform, wl.local_thres, wl.exp_sigma)
    check_full("workload/tiny", q, k, v, W, wl.grid, wl.block, "f32", wl.phi, wl.eps)


def test_tiny_fp32_relu_eps_mode():
    wl = WORKLOADS["tiny_16x16_fp32"]
    q, k, v = draw_workload(wl)
    W = mhla.init_mixing(wl.grid, wl.block, wl.transform)
    check_full("workload/tiny/relu_eps", q, k, v, W, wl.grid, wl.block, "f32", "relu_eps", 1e-6)


# ------------------------------------------------------------------ full-size workloads

def sample_bh(B, H, n):
    pairs = [(0, 0), (B - 1, H - 1), (B // 2, H // 2), (0, H - 1), (B - 1, 0)]
    out = []
    for p in pairs:
        if p not in out:
            out.append(p)
    return out[:n]


_CACHE = {}


def workload_inputs(name):
    if name not in _CACHE:
        _CACHE.clear()
        wl = WORKLOADS[name]
        _CACHE[name] = (wl, *draw_workload(wl))
    return _CACHE[name]


@pytest.mark.parametrize("name,samples", [
    ("deit_t_14x14", None), ("dit_s2_4096px", 3), ("sana_4096px", 3), ("video_20x32x32", 3),
    ("sweep_64x64", None), ("sweep_128x128", 4), ("sweep_256x256", 2), ("sweep_512x512", 2),
    ("lm_causal_4096", 3),
])
def test_workload_parity(name, samples):
    wl, q, k, v = workload_inputs(name)
    W = mhla.init_mixing(wl.grid, wl.block, wl.transform, wl.local_thres, wl.exp_sigma)
    out = as_f64(run(q, k, v, W, wl.grid, wl.block, wl.phi, wl.eps).cpu())
    pairs = [(b, h) for b in range(wl.B) for h in range(wl.H)] if samples is None else sample_bh(wl.B, wl.H, samples)
    worst = {"normwise": 0.0, "frobenius": 0.0, "p999": 0.0}
    for b, h in pairs:
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1), slice(None))
        ref = oracle.forward(as_f64(q[sl]), as_f64(k[sl]), as_f64(v[sl]), W, wl.grid, wl.block,
                             PHI[wl.phi], wl.eps)
        rep = error_report(out[sl], ref)
        worst = {key: max(worst[key], rep[key]) for key in worst}
        err = rep["normwise"]
        assert err <= TOL[wl.dtype], f"{name} (b={b}, h={h}): normwise error {err:.3e}"
    log(f"workload/{name}", err=worst["normwise"], pairs=len(pairs), **worst)
    assert np.isfinite(out).all()


@pytest.mark.parametrize("name", ["dit_s2_4096px", "sana_4096px", "video_20x32x32"])
def test_workload_single_launch_equals_split_launches(name):
    """At full size, in the launch configuration the benchmark times: the single
    persistent launch and the three launches agree bit for bit."""
    wl, q, k, v = workload_inputs(name)
    W = mhla.init_mixing(wl.grid, wl.block, wl.transform, wl.local_thres, wl.exp_sigma)
    a = run(q, k, v, W, wl.grid, wl.block, wl.phi, wl.eps, path="tc_fused")
    b = run(q, k, v, W, wl.grid, wl.block, wl.phi, wl.eps, path="tc")
    assert torch.equal(a, b)


def test_workload_w_matches_oracle_bitwise_at_large_m():
    for name in ("dit_s2_4096px", "sweep_512x512"):
        wl = WORKLOADS[name]
        W = mhla.init_mixing(wl.grid, wl.block, wl.transform, wl.local_thres, wl.exp_sigma)
        ref = oracle.mixing_matrix(wl.grid, wl.block, wl.transform, wl.local_thres, wl.exp_sigma)
        assert np.array_equal(W.view(np.uint32), ref.view(np.uint32))


# ------------------------------------------------------------------ edge cases

@pytest.mark.parametrize("path", ["tc", "simt", "fused"])
def test_zero_query_rows_give_zero(path):
    B, H, d, grid, block = 1, 2, 64, (16, 16), (16, 8)
    q, k, v = draw_qkv(B, 256, H, d, seed=21)
    q[0, 5, 1, :] = -torch.abs(q[0, 5, 1, :]) - 0.25     # phi(q) = 0 exactly
    q[0, 200, 0, :] = 0.0
    W = mhla.init_mixing(grid, block, "linear")
    out = run(q, k, v, W, grid, block, path=path).cpu()
    assert torch.all(out[0, 5, 1] == 0) and torch.all(out[0, 200, 0] == 0)


@pytest.mark.parametrize("path", ["tc", "simt", "fused"])
def test_constant_values_give_weighted_mean(path):
    B, H, d, grid, block = 1, 2, 64, (16, 16), (16, 8)
    q, k, _ = draw_qkv(B, 256, H, d, seed=22)
    v = torch.full_like(q, 0.75)
    W = mhla.init_mixing(grid, block, "exp")
    out = as_f64(run(q, k, v, W, grid, block, eps=0.0, path=path).cpu())
    # every phi(q_t) is non-zero here, so each output is a weighted mean of 0.75
    assert (np.maximum(as_f64(q), 0).max(axis=-1) > 0).all()
    assert np.abs(out - 0.75).max() <= 0.75 * 2 ** -7


@pytest.mark.parametrize("path", ["tc", "simt"])
def test_strided_slices_of_one_projection(path):
    B, N, H, d, grid, block = 2, 512, 3, 64, (16, 32), (16, 8)
    qkv = draw_qkv(B, N, 3 * H, d, seed=23)[0].view(B, N, 3, H, d)
    q, k, v = qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2]
    W = draw_matrix(oracle.num_blocks(grid, block), seed=24)
    qd = qkv.to(DEV)
    out = mhla.forward(qd[:, :, 0], qd[:, :, 1], qd[:, :, 2], torch.from_numpy(W).to(DEV), grid, block, path=path)
    torch.cuda.synchronize()
    ref = oracle.forward(as_f64(q), as_f64(k), as_f64(v), W, grid, block)
    assert normwise(as_f64(out.cpu()), ref) <= TOL["bf16"]


def test_paths_agree_and_tensor_core_path_is_deterministic():
    B, H, d, grid, block = 2, 3, 64, (32, 32), (16, 8)
    q, k, v = draw_qkv(B, 1024, H, d, seed=25)
    W = mhla.init_mixing(grid, block, "cos")
    a = run(q, k, v, W, grid, block, path="tc").cpu()
    b = run(q, k, v, W, grid, block, path="tc").cpu()
    assert torch.equal(a, b)
    c = run(q, k, v, W, grid, block, path="simt").cpu()
    assert normwise(as_f64(a), as_f64(c)) <= TOL["bf16"]


def test_explicit_workspace_and_errors():
    B, H, d, grid, block = 1, 2, 64, (16, 16), (16, 8)
    q, k, v = draw_qkv(B, 256, H, d, seed=26)
    W = mhla.init_mixing(grid, block, "linear")
    qd = q.to(DEV)
    need = mhla.workspace_size(qd, grid, block, "tc")
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    a = run(q, k, v, W, grid, block, path="tc", workspace=ws).cpu()
    b = run(q, k, v, W, grid, block, path="tc").cpu()
    assert torch.equal(a, b)
    with pytest.raises(mhla.MhlaError) as e:
        run(q, k, v, W, grid, block, path="tc", workspace=ws[: need - 256])
    assert e.value.status == 6


def test_empty_batch():
    q = torch.empty(0, 256, 2, 64, dtype=torch.bfloat16, device=DEV)
    W = torch.ones(4, 4, device=DEV)
    out = mhla.forward(q, q, q, W, (16, 16), (8, 8))
    assert out.shape == q.shape


def test_profile_reports_every_kernel():
    B, H, d, grid, block = 1, 2, 64, (16, 16), (16, 8)
    q, k, v = draw_qkv(B, 256, H, d, seed=27)
    W = mhla.init_mixing(grid, block, "linear")
    mhla.profile_begin()
    run(q, k, v, W, grid, block, path="tc")
    run(q, k, v, W, grid, block, path="tc_fused")
    run(q, k, v, W, grid, block, path="simt")
    run(q, k, v, W, grid, block, path="fused")
    prof = mhla.profile_end()
    for name in ("tc_fused", "tc_summary", "tc_mix", "tc_output", "simt_summary", "simt_mix", "simt_output",
                 "tc_small"):
        assert prof[name][0] == 1 and prof[name][1] > 0.0, name
