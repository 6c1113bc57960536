"""GPU parity of the module around the core (LayerNorm, 5 x 5 positional term,
the whole module with its projections) against the float64 module oracle.

bf16 storage between the steps bounds the agreement: every stored value is
rounded once to bf16 (relative 2^-9), so element checks take 2^-7 of the value
plus a small absolute floor, and the module output is held to the 2e-2
normwise bound of bf16 inputs with float32 accumulation,
max |y - y_ref| / max |y_ref|, the bar every parity test here uses (the
relative Frobenius error is logged beside it with MHLA_PARITY_LOG set).
"""

import json
import os

import numpy as np
import pytest
import torch

import oracle
import token_level_head_block_gb300 as mhla
from token_level_head_block_gb300.synth import as_f64, draw_module_params, draw_tokens

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _bf16_close(got, ref, rel=2.0 ** -7, abs_=1e-3):
    err = np.abs(got - ref)
    bad = err > rel * np.abs(ref) + abs_
    assert not bad.any(), f"{bad.sum()} of {bad.size} elements off, worst {err.max():.3g}"


def _normwise(got, ref):
    """The parity bar: the largest elementwise error against the largest |ref|."""
    return float(np.abs(got - ref).max() / np.abs(ref).max())


def _frobenius(got, ref):
    return float(np.linalg.norm((got - ref).ravel()) / np.linalg.norm(ref.ravel()))


def _log(case, **kw):
    path = os.environ.get("MHLA_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": case, **kw}) + "\n")


@pytest.mark.parametrize("rows,C", [(1, 64), (37, 384), (1000, 256), (129, 1024), (64, 2048), (5, 520)])
def test_layer_norm(rows, C):
    x = draw_tokens(1, rows, C, seed=11 + C)[0]
    rng = np.random.default_rng(C)
    w = torch.from_numpy((1 + 0.1 * rng.standard_normal(C)).astype(np.float32))
    b = torch.from_numpy((0.1 * rng.standard_normal(C)).astype(np.float32))
    y = mhla.layer_norm(x.to(DEV), w.to(DEV), b.to(DEV), eps=1e-5)
    torch.cuda.synchronize()
    ref = oracle.layer_norm(as_f64(x), as_f64(w), as_f64(b), 1e-5)
    _bf16_close(as_f64(y.cpu()), ref, abs_=2e-3)


def test_layer_norm_in_place_and_constant_rows():
    C = 128
    x = draw_tokens(1, 16, C, seed=3)[0]
    x[3] = 2.5                              # a constant row normalises to the bias
    w, b = torch.ones(C), torch.full((C,), 0.25)
    xd = x.to(DEV)
    mhla.layer_norm(xd, w.to(DEV), b.to(DEV), out=xd)
    torch.cuda.synchronize()
    ref = oracle.layer_norm(as_f64(x), as_f64(w), as_f64(b))
    got = as_f64(xd.cpu())
    _bf16_close(got, ref, abs_=2e-3)
    assert np.all(got[3] == 0.25)


LINEAR_CASES = [
    # (rows, k, n_out, bias): one tile and a ragged one on every axis (rows past
    # a 128-row tile, n_out past a column tile and not a multiple of 64, k past a
    # 64-wide chunk), the module's DiT-S/2 shapes, the largest C; k <= 384 keeps
    # a slice of w resident per CTA, larger k streams both operands
    (1, 8, 8, True),
    (300, 72, 136, True),
    (512, 384, 1152, True),
    (1000, 384, 384, False),
    (257, 2048, 264, True),
    (700, 512, 200, True),
    (4096, 64, 256, False),
]


@pytest.mark.parametrize("rows,k,n_out,bias", LINEAR_CASES)
def test_linear_layer(rows, k, n_out, bias):
    """The projections' tensor-core GEMM against the float64 nn.Linear of the
    module oracle: float32 accumulation leaves only the final bf16 rounding."""
    x = draw_tokens(1, rows, k, seed=31 + k)[0]
    rng = np.random.default_rng(n_out)
    w = torch.from_numpy((rng.standard_normal((n_out, k)) / np.sqrt(k)).astype(np.float32)).to(torch.bfloat16)
    b = torch.from_numpy((0.1 * rng.standard_normal(n_out)).astype(np.float32)).to(torch.bfloat16) if bias else None
    y = mhla.linear(x.to(DEV), w.to(DEV), None if b is None else b.to(DEV))
    torch.cuda.synchronize()
    assert mhla.device_status() == 0
    ref = oracle.linear(as_f64(x), as_f64(w), None if b is None else as_f64(b))
    got = as_f64(y.cpu())
    _bf16_close(got, ref, abs_=2e-3)
    assert _normwise(got, ref) <= 2e-2


def test_linear_refuses_bad_shapes_and_empty_rows():
    x = torch.zeros(4, 12, dtype=torch.bfloat16, device=DEV)            # k % 8 != 0
    w = torch.zeros(16, 12, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(mhla.MhlaError) as e:
        mhla.linear(x, w)
    assert e.value.status == 3
    x0 = torch.zeros(0, 16, dtype=torch.bfloat16, device=DEV)
    w0 = torch.zeros(8, 16, dtype=torch.bfloat16, device=DEV)
    assert mhla.linear(x0, w0).shape == (0, 8)


LEPE_CASES = [
    # (B, grid, H, d)
    (2, (13, 21), 2, 32),         # ragged tiles on both axes, C = 64
    (1, (64, 64), 6, 64),         # DiT-like channels, C = 384
    (1, (8, 40), 3, 32),          # C = 96: a partial 64-channel chunk
    (2, (3, 9, 17), 2, 64),       # 3-D grid: every frame on its own
    (1, (1, 5), 1, 8),            # a single row narrower than the kernel
]


@pytest.mark.parametrize("B,grid,H,d", LEPE_CASES)
def test_lepe_add_strided_v(B, grid, H, d):
    N = int(np.prod(grid))
    C = H * d
    rng = np.random.default_rng(N + C)
    # v as the third C-slice of a [B, N, 3C] projection (the module's layout)
    qkv = draw_tokens(B, N, 3 * C, seed=17)
    v_full = qkv.to(DEV)
    v = v_full[:, :, 2 * C:].view(B, N, H, d)
    o = draw_tokens(B, N, C, seed=19)
    o_dev = o.to(DEV).view(B, N, H, d).contiguous()
    w = torch.from_numpy((0.2 * rng.standard_normal((C, 5, 5))).astype(np.float32))
    bias = torch.from_numpy((0.1 * rng.standard_normal(C)).astype(np.float32))
    mhla.lepe_add(v, o_dev, grid, w.to(DEV), bias.to(DEV))
    torch.cuda.synchronize()
    v_ref = as_f64(qkv)[:, :, 2 * C:]
    ref = as_f64(o) + oracle.lepe(v_ref, grid, as_f64(w), as_f64(bias))
    _bf16_close(as_f64(o_dev.cpu()).reshape(B, N, C), ref, abs_=2e-3)


MODULE_CASES = [
    # (name, B, grid, block, heads, d, lepe, biases, transform)
    ("tiny_simt_core", 2, (16, 16), (4, 4), 2, 32, True, True, "linear"),
    ("dit_like_tc_core", 1, (64, 64), (16, 16), 6, 64, True, True, "exp"),
    ("video_like_3d", 1, (4, 16, 16), (2, 8, 8), 2, 64, True, False, "linear"),
    ("no_lepe_no_bias", 2, (32, 32), (8, 8), 4, 32, False, False, "cos"),
]


@pytest.mark.parametrize("name,B,grid,block,heads,d,lepe,biases,transform", MODULE_CASES,
                         ids=[c[0] for c in MODULE_CASES])
def test_module_forward(name, B, grid, block, heads, d, lepe, biases, transform):
    N, C = int(np.prod(grid)), heads * d
    x = draw_tokens(B, N, C, seed=101)
    p = draw_module_params(C, seed=202, lepe=lepe, biases=biases)
    W = mhla.init_mixing(grid, block, transform)
    pd = {k: t.to(DEV) for k, t in p.items()}
    y = mhla.module_forward(x.to(DEV), pd, torch.from_numpy(W).to(DEV), grid, block, heads, phi="relu_eps",
                            eps=1e-6)
    torch.cuda.synchronize()
    assert mhla.device_status() == 0
    ref = oracle.module_forward(as_f64(x), {k: as_f64(t) for k, t in p.items()}, W.astype(np.float64), grid,
                                block, heads, oracle.PHI_RELU_EPS, 1e-6)
    got = as_f64(y.cpu())
    err = _normwise(got, ref)
    _log(f"module_{name}", err=err, frobenius=_frobenius(got, ref))
    assert err <= 2e-2, f"{name}: normwise error {err:.3e}"


def test_module_with_workspace_and_in_place():
    B, grid, block, heads, d = 1, (32, 32), (16, 16), 2, 64
    N, C = 1024, 128
    x = draw_tokens(B, N, C, seed=5)
    p = {k: t.to(DEV) for k, t in draw_module_params(C, seed=6).items()}
    W = torch.from_numpy(mhla.init_mixing(grid, block)).to(DEV)
    ws = torch.empty(mhla.module_workspace_size(B, N, C, heads, grid, block), dtype=torch.uint8, device=DEV)
    a = mhla.module_forward(x.to(DEV), p, W, grid, block, heads, workspace=ws)
    xd = x.to(DEV)
    mhla.module_forward(xd, p, W, grid, block, heads, out=xd, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a, xd)


def test_module_rejects_bad_shapes():
    x = torch.zeros(1, 64, 60, dtype=torch.bfloat16, device=DEV)     # C % 8 != 0
    p = {k: t.to(DEV) for k, t in draw_module_params(64, seed=1).items()}
    W = torch.ones(1, 1, device=DEV)
    with pytest.raises(mhla.MhlaError):
        mhla.module_forward(x, p, W, (8, 8), (8, 8), 2)


def test_module_refuses_before_any_launch():
    """A request the core refuses (here W inside the buffer the core writes)
    is turned down before the LayerNorm or the projection runs: the workspace
    comes back untouched."""
    B, grid, block, heads, d = 1, (16, 16), (4, 4), 2, 32
    N, C = 256, 64
    x = draw_tokens(B, N, C, seed=8).to(DEV)
    p = {k: t.to(DEV) for k, t in draw_module_params(C, seed=9).items()}
    ws = torch.full((mhla.module_workspace_size(B, N, C, heads, grid, block),), 0x5A, dtype=torch.uint8, device=DEV)
    M = mhla.num_blocks(grid, block)
    W_inside = ws[:M * M * 4].view(torch.float32)       # overlaps the normalised input / core output buffer
    with pytest.raises(mhla.MhlaError) as e:
        mhla.module_forward(x, p, W_inside, grid, block, heads, workspace=ws)
    assert e.value.status == 1
    torch.cuda.synchronize()
    assert bool((ws == 0x5A).all())


def test_lepe_add_many_frames():
    """More (frame, channel chunk) tiles than a 16-bit grid axis holds: the
    persistent kernel walks them with a 64-bit tile index."""
    B, grid, H, d = 22000, (2, 3), 3, 64          # 22000 frames x 3 channel chunks = 66000 tiles
    N, C = 6, 192
    rng = np.random.default_rng(23)
    v = draw_tokens(B, N, C, seed=24)
    o = draw_tokens(B, N, C, seed=25)
    o_dev = o.to(DEV).view(B, N, H, d)
    w = torch.from_numpy((0.2 * rng.standard_normal((C, 5, 5))).astype(np.float32))
    bias = torch.from_numpy((0.1 * rng.standard_normal(C)).astype(np.float32))
    mhla.lepe_add(v.to(DEV).view(B, N, H, d), o_dev, grid, w.to(DEV), bias.to(DEV))
    torch.cuda.synchronize()
    got = as_f64(o_dev.cpu()).reshape(B, N, C)
    for b in (0, 1, 4097, 12345, B - 1):          # frames are independent: a sample against the oracle
        ref = as_f64(o[b:b + 1]) + oracle.lepe(as_f64(v[b:b + 1]), grid, as_f64(w), as_f64(bias))
        _bf16_close(got[b:b + 1], ref, abs_=2e-3)
