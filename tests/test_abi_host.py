"""Host-side checks of the C ABI: no GPU needed, no kernel is launched.

The library must load and export every function include/mhla.h declares; the
host W builder must reproduce the oracle's W bit for bit; every malformed request
must be rejected with its documented status before any GPU work is queued.
"""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import token_level_head_block_gb300 as mhla
from tests.golden.write_golden import CASES, case_name, load
from token_level_head_block_gb300.workloads import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mhla.h")

OK, INVALID, SHAPE, UNSUPPORTED, CUDA, TIMEOUT, WORKSPACE = range(7)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mhla_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    return mhla.lib()


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert {"mhla_forward", "mhla_init_mixing", "mhla_workspace_size"} <= set(names)
    for name in names:
        assert hasattr(L, name), name


def test_version_and_status_strings(L):
    assert b"sm_103a" in L.mhla_version()
    for code in range(7):
        assert L.mhla_status_string(code).decode() == mhla.STATUS[code]
    assert L.mhla_status_string(99) == b"unknown status"


@pytest.mark.parametrize("case", CASES, ids=[case_name(*c) for c in CASES])
def test_init_mixing_matches_stored_fixture_bitwise(case):
    W = mhla.init_mixing(case[0], case[1], case[2], local_thres=case[3], exp_sigma=case[4])
    assert np.array_equal(W.view(np.uint32), load()[case_name(*case)].view(np.uint32))


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_init_mixing_matches_oracle_bitwise_on_workloads(name):
    wl = WORKLOADS[name]
    if wl.M > 300:
        pytest.skip("python-loop oracle W is slow at this M; covered on the GPU box")
    W = mhla.init_mixing(wl.grid, wl.block, wl.transform, wl.local_thres, wl.exp_sigma)
    ref = oracle.mixing_matrix(wl.grid, wl.block, wl.transform, wl.local_thres, wl.exp_sigma)
    assert np.array_equal(W.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("transform", list(mhla.TRANSFORMS))
def test_init_mixing_rectangular_and_single_block(transform):
    W = mhla.init_mixing((12, 20), (4, 4), transform, 1.5, 2.5)
    ref = oracle.mixing_matrix((12, 20), (4, 4), transform, 1.5, 2.5)
    assert np.array_equal(W.view(np.uint32), ref.view(np.uint32))
    assert mhla.init_mixing((8, 8), (8, 8), transform).tolist() == [[1.0]]


def test_num_blocks_and_bad_shapes(L):
    assert mhla.num_blocks((256, 256), (16, 16)) == 256
    assert mhla.num_blocks((20, 32, 32), (4, 8, 8)) == 80
    for g, b in [((14, 14), (4, 4)), ((16, 16), (4, 4, 1)), ((0, 4), (1, 1))]:
        with pytest.raises(mhla.MhlaError) as e:
            mhla.num_blocks(g, b)
        assert e.value.status == SHAPE


def test_init_mixing_rejects_bad_arguments(L):
    g, b = mhla.shape3((8, 8)), mhla.shape3((4, 4))
    buf = (ctypes.c_float * 16)()      # M = 4 blocks -> 16 entries
    call = lambda t, lt, s, cap, p=buf: L.mhla_init_mixing(ctypes.byref(g), ctypes.byref(b), t, lt, s, p, cap)
    assert call(0, 1.5, 3.0, 16) == OK
    assert call(5, 1.5, 3.0, 16) == INVALID         # unknown transform
    assert call(2, 1.5, 0.0, 16) == INVALID         # exp with sigma 0
    assert call(4, -1.0, 3.0, 16) == INVALID        # local with negative threshold
    assert call(0, 1.5, 3.0, 15) == INVALID         # W too small
    assert call(0, 1.5, 3.0, 16, None) == INVALID   # null W


# ------------------------------------------------------------ forward validation

FAKE = 1 << 40          # a 256-byte aligned address that is never dereferenced here


def contig(B, N, H, d, dtype="bf16", base=FAKE):
    return mhla.tensor_desc(base, dtype, (B, N, H, d), (N * H * d, H * d, d))


def call_forward(L, q, k, v, o, grid, block, W=FAKE + (1 << 36), phi=(0, 1e-6), ws=None, ws_bytes=0, path=0):
    return L.mhla_forward(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), ctypes.c_void_p(W),
                          ctypes.byref(mhla.shape3(grid)), ctypes.byref(mhla.shape3(block)),
                          ctypes.byref(mhla.Phi(*phi)), ctypes.byref(o),
                          ctypes.c_void_p(ws) if ws else None, ws_bytes, None, path)


def four(B, N, H, d, dtype="bf16"):
    span = B * N * H * d * 4 + 4096
    return [contig(B, N, H, d, dtype, FAKE + i * span) for i in range(4)]


def test_forward_rejects_malformed_requests_before_any_launch(L):
    q, k, v, o = four(2, 256, 3, 64)
    grid, block = (16, 16), (4, 4)
    assert call_forward(L, q, k, v, o, (16, 15), block) == SHAPE           # grid product != N
    assert call_forward(L, q, k, v, o, grid, (5, 4)) == SHAPE              # block does not tile
    assert call_forward(L, q, k, v, o, grid, (4, 4, 4)) == SHAPE           # ndim mismatch
    k2 = contig(2, 256, 3, 32, base=k.data)
    assert call_forward(L, q, k2, v, o, grid, block) == SHAPE              # d differs
    v2 = contig(2, 256, 3, 64, "f32", base=v.data)
    assert call_forward(L, q, k, v2, o, grid, block) == SHAPE              # dtype differs
    assert call_forward(L, q, k, v, q, grid, block) == INVALID             # out aliases q
    assert call_forward(L, q, k, v, o, grid, block, W=0) == INVALID        # null W
    assert call_forward(L, q, k, v, o, grid, block, W=o.data + 64) == INVALID   # W inside out
    assert call_forward(L, q, k, v, o, grid, block, phi=(7, 1e-6)) == INVALID   # unknown phi
    assert call_forward(L, q, k, v, o, grid, block, phi=(0, -1.0)) == INVALID   # negative eps
    assert call_forward(L, q, k, v, o, grid, block, phi=(0, float("inf"))) == INVALID
    bad = contig(2, 256, 3, 200, base=q.data)
    assert call_forward(L, bad, bad, bad, contig(2, 256, 3, 200, base=o.data), grid, block) == INVALID
    o_overlap = mhla.tensor_desc(o.data, "bf16", (2, 256, 3, 64), (256 * 3 * 64, 3 * 64, 32))
    assert call_forward(L, q, k, v, o_overlap, grid, block) == INVALID    # heads overlap in out
    for path in (0, 1, 3):   # auto (the fused path here, which needs no workspace), CUDA cores, fused
        assert call_forward(L, q, k, v, o, grid, block, ws=FAKE + 7, ws_bytes=1 << 30, path=path) == WORKSPACE
        assert call_forward(L, q, k, v, o, grid, block, ws=None, ws_bytes=16, path=path) == WORKSPACE
    assert call_forward(L, q, k, v, o, grid, block, ws=FAKE, ws_bytes=16, path=1) == WORKSPACE  # too small
    assert call_forward(L, q, k, v, o, grid, block, path=9) == INVALID                          # unknown path


def test_forward_explicit_tensor_core_path_refuses_ineligible_problems(L):
    q, k, v, o = four(1, 196, 3, 64)                                # 2x2 blocks: 4 tokens per block
    assert call_forward(L, q, k, v, o, (14, 14), (2, 2), path=2) == UNSUPPORTED
    q, k, v, o = four(1, 256, 1, 32, "f32")                         # fp32 runs on CUDA cores only
    assert call_forward(L, q, k, v, o, (16, 16), (16, 16), path=2) == UNSUPPORTED


def test_forward_explicit_fused_path_refuses_ineligible_problems(L):
    q, k, v, o = four(1, 1024, 2, 64)                               # more than 256 tokens
    assert call_forward(L, q, k, v, o, (32, 32), (16, 8), path=3) == UNSUPPORTED
    q, k, v, o = four(1, 256, 2, 64)                                # M = 128 > 96 blocks
    assert call_forward(L, q, k, v, o, (16, 16), (1, 2), path=3) == UNSUPPORTED
    q, k, v, o = four(1, 196, 3, 48)                                # d = 48
    assert call_forward(L, q, k, v, o, (14, 14), (2, 2), path=3) == UNSUPPORTED
    q, k, v, o = four(1, 196, 3, 64, "f32")                         # float32
    assert call_forward(L, q, k, v, o, (14, 14), (2, 2), path=3) == UNSUPPORTED
    ts = [mhla.tensor_desc(t.data, "bf16", (1, 196, 3, 64), (196 * 3 * 68, 3 * 68, 68)) for t in four(1, 196, 3, 64)]
    assert call_forward(L, *ts, (14, 14), (2, 2), path=3) == UNSUPPORTED   # strides break the 16-byte rule


def test_empty_batch_is_a_no_op(L):
    q, k, v, o = four(0, 256, 3, 64)
    assert call_forward(L, q, k, v, o, (16, 16), (4, 4)) == OK
    q, k, v, o = four(2, 256, 0, 64)
    assert call_forward(L, q, k, v, o, (16, 16), (4, 4)) == OK


def select(L, q, grid, block, strides=None):
    ts = four(q[0], q[1], q[2], q[3], q[4] if len(q) > 4 else "bf16")
    if strides:
        ts = [mhla.tensor_desc(t.data, t.dtype, (t.B, t.N, t.H, t.d), strides) for t in ts]
    return L.mhla_select_path(*(ctypes.byref(t) for t in ts), ctypes.byref(mhla.shape3(grid)),
                              ctypes.byref(mhla.shape3(block)))


def test_path_selection(L):
    SIMT, TC, FUSED = 1, 2, 3
    for name in ("dit_s2_4096px", "sana_4096px", "video_20x32x32", "sweep_64x64", "sweep_512x512"):
        wl = WORKLOADS[name]
        assert select(L, (wl.B, wl.N, wl.H, wl.d), wl.grid, wl.block) == TC, name
    wl = WORKLOADS["lm_causal_4096"]                 # contiguous 64-token blocks: the tile readout
    assert select(L, (wl.B, wl.N, wl.H, wl.d), wl.grid, wl.block) == TC
    wl = WORKLOADS["deit_t_14x14"]                   # 196 tokens, 49 blocks: one fused launch
    assert select(L, (wl.B, wl.N, wl.H, wl.d), wl.grid, wl.block) == FUSED
    wl = WORKLOADS["tiny_16x16_fp32"]
    assert select(L, (wl.B, wl.N, wl.H, wl.d, "f32"), wl.grid, wl.block) == SIMT
    # short sequences take the fused kernel even where the three-launch path applies
    assert select(L, (1, 256, 2, 64), (16, 16), (16, 16)) == FUSED
    assert select(L, (2, 37, 1, 32), (1, 37), (1, 1)) == FUSED
    # d = 48 has no tensor-core kernel; 64-token blocks cannot fill a 128-row tile;
    # 128 blocks of 2 tokens exceed the fused kernel's 96 blocks.
    assert select(L, (1, 256, 2, 48), (16, 16), (16, 16)) == SIMT
    assert select(L, (1, 1024, 2, 64), (32, 32), (8, 8)) == SIMT
    assert select(L, (1, 256, 2, 64), (16, 16), (1, 2)) == SIMT
    # strides that break TMA's 16-byte rule fall back to CUDA cores
    assert select(L, (1, 256, 2, 64), (16, 16), (16, 16), strides=(256 * 2 * 68, 2 * 68, 68)) == SIMT
    # q, k, v taken as slices of one [B, N, 3, H, d] projection still qualify
    st = (512 * 3 * 2 * 64, 3 * 2 * 64, 64)
    q, k, v = (mhla.tensor_desc(FAKE + 2 * i * 2 * 64, "bf16", (2, 512, 2, 64), st) for i in range(3))
    o = contig(2, 512, 2, 64, base=FAKE + (1 << 30))
    assert L.mhla_select_path(*(ctypes.byref(t) for t in (q, k, v, o)), ctypes.byref(mhla.shape3((16, 32))),
                              ctypes.byref(mhla.shape3((16, 8)))) == TC
    st = (196 * 3 * 3 * 64, 3 * 3 * 64, 64)
    q, k, v = (mhla.tensor_desc(FAKE + 2 * i * 3 * 64, "bf16", (2, 196, 3, 64), st) for i in range(3))
    o = contig(2, 196, 3, 64, base=FAKE + (1 << 30))
    assert L.mhla_select_path(*(ctypes.byref(t) for t in (q, k, v, o)), ctypes.byref(mhla.shape3((14, 14))),
                              ctypes.byref(mhla.shape3((2, 2)))) == FUSED


def test_workspace_sizes(L):
    wl = WORKLOADS["dit_s2_4096px"]
    q = contig(wl.B, wl.N, wl.H, wl.d)
    M, BH, d = wl.M, wl.B * wl.H, wl.d
    n = ctypes.c_size_t()
    assert L.mhla_workspace_size(ctypes.byref(q), ctypes.byref(mhla.shape3(wl.grid)),
                                 ctypes.byref(mhla.shape3(wl.block)), 2, ctypes.byref(n)) == OK
    expect = M * M * 2 + M * BH * (d + 1) * d * 2 + BH * M * d * d * 2 + BH * M * d * 4
    assert expect <= n.value < expect + 4 * 256 and n.value % 256 == 0
    assert L.mhla_workspace_size(ctypes.byref(q), ctypes.byref(mhla.shape3(wl.grid)),
                                 ctypes.byref(mhla.shape3(wl.block)), 1, ctypes.byref(n)) == OK
    assert n.value >= 2 * BH * M * d * (d + 1) * 4
    wl = WORKLOADS["deit_t_14x14"]                     # the fused path needs no workspace
    q = contig(wl.B, wl.N, wl.H, wl.d)
    for path in (0, 3):
        assert L.mhla_workspace_size(ctypes.byref(q), ctypes.byref(mhla.shape3(wl.grid)),
                                     ctypes.byref(mhla.shape3(wl.block)), path, ctypes.byref(n)) == OK
        assert n.value == 0


# ------------------------------------------------------------ backward validation

def call_backward(L, q, k, v, g, dq, dk, dv, grid, block, W=FAKE + (1 << 36), dW=FAKE + (1 << 37),
                  phi=(0, 1e-6), ws=None, ws_bytes=0, path=0):
    return L.mhla_backward(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), ctypes.c_void_p(W),
                           ctypes.byref(mhla.shape3(grid)), ctypes.byref(mhla.shape3(block)),
                           ctypes.byref(mhla.Phi(*phi)), ctypes.byref(g), ctypes.byref(dq), ctypes.byref(dk),
                           ctypes.byref(dv), ctypes.c_void_p(dW) if dW else None,
                           ctypes.c_void_p(ws) if ws else None, ws_bytes, None, path)


def seven(B, N, H, d, dtype="bf16"):
    span = B * N * H * d * 4 + 4096
    return [contig(B, N, H, d, dtype, FAKE + i * span) for i in range(7)]


def test_backward_rejects_malformed_requests_before_any_launch(L):
    q, k, v, g, dq, dk, dv = seven(2, 1024, 3, 64)
    grid, block = (32, 32), (16, 8)
    assert call_backward(L, q, k, v, g, dq, dk, dv, (32, 31), block) == SHAPE
    assert call_backward(L, q, k, v, g, dq, dk, dv, grid, (5, 8)) == SHAPE
    dk2 = contig(2, 1024, 3, 32, base=dk.data)
    assert call_backward(L, q, k, v, g, dq, dk2, dv, grid, block) == SHAPE          # d differs
    g2 = contig(2, 1024, 3, 64, "f32", base=g.data)
    assert call_backward(L, q, k, v, g2, dq, dk, dv, grid, block) == SHAPE          # dtype differs
    assert call_backward(L, q, k, v, g, dq, dq, dv, grid, block) == INVALID         # dq and dk alias
    assert call_backward(L, q, k, v, g, q, dk, dv, grid, block) == INVALID          # dq aliases q
    assert call_backward(L, q, k, v, g, dq, dk, g, grid, block) == INVALID          # dv aliases dout
    assert call_backward(L, q, k, v, g, dq, dk, dv, grid, block, W=0) == INVALID    # null W
    assert call_backward(L, q, k, v, g, dq, dk, dv, grid, block, dW=0) == INVALID   # null dW
    assert call_backward(L, q, k, v, g, dq, dk, dv, grid, block, dW=FAKE + (1 << 36) + 64) == INVALID  # dW in W
    assert call_backward(L, q, k, v, g, dq, dk, dv, grid, block, dW=dq.data + 128) == INVALID          # dW in dq
    assert call_backward(L, q, k, v, g, dq, dk, dv, grid, block, W=dk.data) == INVALID                 # W in dk
    assert call_backward(L, q, k, v, g, dq, dk, dv, grid, block, phi=(3, 1e-6)) == INVALID
    over = mhla.tensor_desc(dv.data, "bf16", (2, 1024, 3, 64), (1024 * 3 * 64, 3 * 64, 32))
    assert call_backward(L, q, k, v, g, dq, dk, over, grid, block) == INVALID       # heads overlap in dv
    assert call_backward(L, q, k, v, g, dq, dk, dv, grid, block, ws=FAKE + 7, ws_bytes=1 << 40) == WORKSPACE
    assert call_backward(L, q, k, v, g, dq, dk, dv, grid, block, ws=FAKE, ws_bytes=16) == WORKSPACE
    assert call_backward(L, q, k, v, g, dq, dk, dv, grid, block, ws=None, ws_bytes=16) == WORKSPACE
    assert call_backward(L, q, k, v, g, dq, dk, dv, grid, (4, 4), path=2) == UNSUPPORTED   # 16-token blocks
    st68 = (1024 * 3 * 68, 3 * 68, 68)
    dv68 = mhla.tensor_desc(dv.data, "bf16", (2, 1024, 3, 64), st68)
    assert call_backward(L, q, k, v, g, dq, dk, dv68, grid, block, path=2) == UNSUPPORTED   # TMA-unfit dv
    assert call_backward(L, q, k, v, g, dq, dk, dv, grid, block, path=3) == UNSUPPORTED
    assert call_backward(L, q, k, v, g, dq, dk, dv, grid, block, path=9) == INVALID


def test_backward_workspace_size(L):
    wl = WORKLOADS["dit_s2_4096px"]
    q = contig(wl.B, wl.N, wl.H, wl.d)
    M, BH, d = wl.M, wl.B * wl.H, wl.d
    sizes = {}
    for path in (0, 1, 2):
        n = ctypes.c_size_t()
        assert L.mhla_backward_workspace_size(ctypes.byref(q), ctypes.byref(mhla.shape3(wl.grid)),
                                              ctypes.byref(mhla.shape3(wl.block)), path, ctypes.byref(n)) == OK
        assert n.value % 256 == 0
        sizes[path] = n.value
    simt = 3 * BH * M * d * (d + 1) * 4 + BH * M * M * 4
    assert simt <= sizes[1] < simt + 4 * 256
    groups = (BH * (d + 1) * d + 127) // 128
    tc = 2 * M * M * 2 + 2 * M * groups * 128 * 2 + BH * M * d * d * 2 + BH * M * d * 4
    # + the dW partial products: one 256 x 256 tile of dW (M = 256) split over up to 100 CTAs
    tiles = ((M + 255) // 256) ** 2
    nsplit = min(groups, -(-100 // tiles))
    assert tc < sizes[2] <= tc + nsplit * M * M * 4 + 8 * 256
    assert sizes[0] == max(sizes[1], sizes[2])                         # AUTO: enough for either path
    assert L.mhla_backward_workspace_size(ctypes.byref(q), ctypes.byref(mhla.shape3(wl.grid)),
                                          ctypes.byref(mhla.shape3(wl.block)), 3, ctypes.byref(n)) == UNSUPPORTED


# ------------------------------------------------------------ causal validation

def call_causal(L, q, k, v, o, grid, block, W=FAKE + (1 << 36), phi=(0, 1e-6), ws=None, ws_bytes=0, path=0):
    return L.mhla_forward_causal(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), ctypes.c_void_p(W),
                                 ctypes.byref(mhla.shape3(grid)), ctypes.byref(mhla.shape3(block)),
                                 ctypes.byref(mhla.Phi(*phi)), ctypes.byref(o),
                                 ctypes.c_void_p(ws) if ws else None, ws_bytes, None, path)


def test_causal_rejects_malformed_requests_before_any_launch(L):
    q, k, v, o = four(2, 1024, 3, 64)
    assert call_causal(L, q, k, v, o, (32, 32), (4, 4)) == SHAPE               # blocks not contiguous
    assert call_causal(L, q, k, v, o, (32, 32), (2, 2)) == SHAPE
    assert call_causal(L, q, k, v, o, (1, 1000), (1, 8)) == SHAPE              # grid product != N
    assert call_causal(L, q, k, v, o, (1, 1024), (1, 64), W=0) == INVALID
    assert call_causal(L, q, k, v, q, (1, 1024), (1, 64)) == INVALID           # out aliases q
    assert call_causal(L, q, k, v, o, (1, 1024), (1, 32), path=2) == UNSUPPORTED   # 32-token blocks
    q2, k2, v2, o2 = four(2, 1000, 3, 64)
    assert call_causal(L, q2, k2, v2, o2, (1, 1000), (1, 125), path=2) == UNSUPPORTED   # N not a multiple of 128
    assert call_causal(L, q, k, v, o, (1, 1024), (1, 64), path=3) == UNSUPPORTED
    assert call_causal(L, q, k, v, o, (1, 1024), (1, 64), ws=FAKE + 8, ws_bytes=1 << 30) == WORKSPACE
    assert call_causal(L, q, k, v, o, (1, 1024), (1, 64), ws=FAKE, ws_bytes=16) == WORKSPACE
    assert call_causal(L, q, k, v, o, (1, 1024), (1, 64), ws=None, ws_bytes=16) == WORKSPACE
    n = ctypes.c_size_t()
    assert L.mhla_causal_workspace_size(ctypes.byref(q), ctypes.byref(mhla.shape3((32, 32))),
                                        ctypes.byref(mhla.shape3((8, 32))), 1, ctypes.byref(n)) == OK
    simt = n.value
    assert simt == 2 * ((2 * 3 * 4 * 64 * 65 * 4 + 255) // 256 * 256)       # two float32 summary buffers
    assert L.mhla_causal_workspace_size(ctypes.byref(q), ctypes.byref(mhla.shape3((32, 32))),
                                        ctypes.byref(mhla.shape3((8, 32))), 2, ctypes.byref(n)) == OK
    tc = n.value                                                             # 8 units of 128 tokens
    units, groups = 8, (2 * 3 * 65 * 64 + 127) // 128
    assert tc >= units * 8 * 2 + units * groups * 128 * 2 + 2 * 3 * units * 64 * 64 * 2 + 2 * 3 * units * 64 * 4
    assert L.mhla_causal_workspace_size(ctypes.byref(q), ctypes.byref(mhla.shape3((32, 32))),
                                        ctypes.byref(mhla.shape3((8, 32))), 0, ctypes.byref(n)) == OK
    assert n.value == max(tc, simt)
    assert L.mhla_causal_workspace_size(ctypes.byref(q), ctypes.byref(mhla.shape3((32, 32))),
                                        ctypes.byref(mhla.shape3((8, 8))), 0, ctypes.byref(n)) == SHAPE
    e = four(0, 1024, 3, 64)
    assert call_causal(L, *e, (32, 32), (8, 32)) == OK                         # empty batch: nothing queued


def call_backward_causal(L, q, k, v, g, dq, dk, dv, grid, block, W=FAKE + (1 << 36), dW=FAKE + (1 << 37),
                         phi=(0, 1e-6), ws=None, ws_bytes=0, path=0):
    return L.mhla_backward_causal(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), ctypes.c_void_p(W),
                                  ctypes.byref(mhla.shape3(grid)), ctypes.byref(mhla.shape3(block)),
                                  ctypes.byref(mhla.Phi(*phi)), ctypes.byref(g), ctypes.byref(dq),
                                  ctypes.byref(dk), ctypes.byref(dv), ctypes.c_void_p(dW) if dW else None,
                                  ctypes.c_void_p(ws) if ws else None, ws_bytes, None, path)


def test_causal_backward_rejects_malformed_requests_before_any_launch(L):
    q, k, v, g, dq, dk, dv = seven(2, 1024, 3, 64)
    grid, block = (1, 1024), (1, 64)
    assert call_backward_causal(L, q, k, v, g, dq, dk, dv, (32, 32), (4, 4)) == SHAPE   # blocks not contiguous
    assert call_backward_causal(L, q, k, v, g, dq, dk, dv, (1, 1000), (1, 8)) == SHAPE
    dk2 = contig(2, 1024, 3, 32, base=dk.data)
    assert call_backward_causal(L, q, k, v, g, dq, dk2, dv, grid, block) == SHAPE
    assert call_backward_causal(L, q, k, v, g, dq, dq, dv, grid, block) == INVALID     # dq and dk alias
    assert call_backward_causal(L, q, k, v, g, dq, dk, g, grid, block) == INVALID      # dv aliases dout
    assert call_backward_causal(L, q, k, v, g, dq, dk, dv, grid, block, W=0) == INVALID
    assert call_backward_causal(L, q, k, v, g, dq, dk, dv, grid, block, dW=0) == INVALID
    assert call_backward_causal(L, q, k, v, g, dq, dk, dv, grid, block, dW=FAKE + (1 << 36) + 64) == INVALID
    assert call_backward_causal(L, q, k, v, g, dq, dk, dv, grid, block, phi=(3, 1e-6)) == INVALID
    assert call_backward_causal(L, q, k, v, g, dq, dk, dv, grid, block, ws=FAKE + 7, ws_bytes=1 << 40) == WORKSPACE
    assert call_backward_causal(L, q, k, v, g, dq, dk, dv, grid, block, ws=FAKE, ws_bytes=16) == WORKSPACE
    for path in (3, 4):
        assert call_backward_causal(L, q, k, v, g, dq, dk, dv, grid, block, path=path) == UNSUPPORTED
    # TC (tensor-core summaries and mixing) takes bf16, d = 64, 64-token blocks; it
    # gets as far as the workspace check here
    assert call_backward_causal(L, q, k, v, g, dq, dk, dv, grid, block, ws=FAKE, ws_bytes=16, path=2) == WORKSPACE
    f32 = seven(2, 1024, 3, 64, "f32")
    assert call_backward_causal(L, *f32, grid, block, path=2) == UNSUPPORTED          # float32 inputs
    assert call_backward_causal(L, q, k, v, g, dq, dk, dv, (1, 1024), (1, 256), path=2) == UNSUPPORTED  # w = 256
    assert call_backward_causal(L, q, k, v, g, dq, dk, dv, grid, block, path=9) == INVALID
    n = ctypes.c_size_t()
    BH, M, N, d = 6, 16, 1024, 64
    KS = 16  # the dW partial products split d (d + 1) = 4160 entries in 16 runs (6 tiles are too few CTAs)
    need = 3 * BH * M * d * (d + 1) * 4 + BH * KS * M * M * 4 + BH * M * 4 + BH * N * (d + 4) * 4
    groups = (BH * (d + 1) * d + 127) // 128
    nsplit = min(groups, 152)   # the tensor-core dW product's splits (a small tile: one per SM)
    tc = M * M * 2 + M * groups * 128 * 2 + BH * M * d * d * 2 + BH * M * d * 4 + nsplit * M * M * 4
    for path, extra in ((0, tc), (1, 0), (2, tc)):
        assert L.mhla_backward_causal_workspace_size(ctypes.byref(q), ctypes.byref(mhla.shape3(grid)),
                                                     ctypes.byref(mhla.shape3(block)), path,
                                                     ctypes.byref(n)) == OK
        assert n.value % 256 == 0 and need + extra <= n.value < need + extra + 11 * 256, path
    assert L.mhla_backward_causal_workspace_size(ctypes.byref(q), ctypes.byref(mhla.shape3((32, 32))),
                                                 ctypes.byref(mhla.shape3((4, 4))), 0, ctypes.byref(n)) == SHAPE
    assert L.mhla_backward_causal_workspace_size(ctypes.byref(f32[0]), ctypes.byref(mhla.shape3(grid)),
                                                 ctypes.byref(mhla.shape3(block)), 2,
                                                 ctypes.byref(n)) == UNSUPPORTED


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    """With the library absent the binding raises on first use; it has no other
    path to fall back on (the package never imports the oracle)."""
    monkeypatch.setattr(mhla, "_lib", None)
    monkeypatch.setattr(mhla, "_LIB_PATH", str(tmp_path / "libmhla.so"))
    with pytest.raises(mhla.MhlaError, match="missing"):
        mhla.lib()
    with pytest.raises(mhla.MhlaError):
        mhla.init_mixing((16, 16), (4, 4))


def test_package_sources_never_import_the_oracle():
    pkg = os.path.join(ROOT, "token_level_head_block_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith(".py"):
                text = open(os.path.join(dirpath, fn)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, flags=re.M), fn


def test_noalloc_refuses_oversized_problems_before_touching_the_device(L):
    """A problem whose scratch exceeds the library's fixed array comes back as
    MHLA_ERR_WORKSPACE from the host checks alone (were the device consulted
    first, a machine without one would answer MHLA_ERR_CUDA instead)."""
    fn = L.mhla_forward_noalloc
    P = ctypes.POINTER
    fn.argtypes = [P(mhla.Tensor), P(mhla.Tensor), P(mhla.Tensor), ctypes.c_void_p, P(mhla.Shape3),
                   P(mhla.Shape3), P(mhla.Phi), P(mhla.Tensor), ctypes.c_void_p, ctypes.c_int32]
    fn.restype = ctypes.c_int
    q, k, v, o = four(64, 196, 3, 64)                 # float32 summaries on the CUDA cores: ~313 MB
    grid, block = mhla.shape3((14, 14)), mhla.shape3((2, 2))
    need = ctypes.c_size_t(0)
    assert L.mhla_workspace_size(ctypes.byref(q), ctypes.byref(grid), ctypes.byref(block), 1,
                                 ctypes.byref(need)) == OK
    m = re.search(r"#define MHLA_NOALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", open(HEADER).read())
    assert need.value > int(m.group(1)) << int(m.group(2))
    st = fn(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), ctypes.c_void_p(FAKE + (1 << 36)), ctypes.byref(grid),
            ctypes.byref(block), ctypes.byref(mhla.Phi(0, 1e-6)), ctypes.byref(o), None, 1)
    assert st == WORKSPACE



def test_stall_hook_refuses_bad_arguments_on_the_host(L):
    """The timeout-path diagnostic hook validates before touching the device."""
    L.mhla_debug_stall_waits.argtypes = [ctypes.c_int32, ctypes.c_uint64]
    L.mhla_debug_stall_waits.restype = ctypes.c_int
    assert L.mhla_debug_stall_waits(-2, 0) == 1          # warp outside -1 .. 31
    assert L.mhla_debug_stall_waits(32, 1000000) == 1
    assert L.mhla_debug_stall_waits(1, 999) == 1         # limit below 1 us
    assert L.mhla_debug_stall_waits(1, 2000000000) == 1  # limit above 1 s
