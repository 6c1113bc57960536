"""Host-side checks of the module entry points: validation and workspace sizing,
no GPU needed and no kernel launched (every request here is rejected, or only
sized, before any GPU work)."""

import ctypes

import pytest

import token_level_head_block_gb300 as mhla

OK, INVALID, SHAPE, UNSUPPORTED, CUDA, TIMEOUT, WORKSPACE = range(7)


def _ws(B, N, C, heads, grid, block):
    n = ctypes.c_size_t(0)
    st = mhla.lib().mhla_module_workspace_size(B, N, C, heads, ctypes.byref(mhla.shape3(grid)),
                                               ctypes.byref(mhla.shape3(block)), ctypes.byref(n))
    return st, n.value


def test_workspace_holds_the_buffers_of_the_dit_shape():
    B, N, C = 4, 65536, 384
    st, n = _ws(B, N, C, 6, (256, 256), (16, 16))
    assert st == OK
    R = B * N
    assert n >= R * C * 2 + R * 3 * C * 2 + (32 << 20)
    assert n % 256 == 0


@pytest.mark.parametrize("B,N,C,heads,grid,block,status", [
    (1, 64, 60, 2, (8, 8), (8, 8), UNSUPPORTED),      # C % 8
    (1, 64, 64, 3, (8, 8), (8, 8), INVALID),          # heads do not divide C
    (1, 64, 4096, 16, (8, 8), (8, 8), UNSUPPORTED),   # C > 2048
    (1, 64, 40, 2, (8, 8), (8, 8), UNSUPPORTED),      # d = 20 is not a multiple of 8
    (1, 64, 64, 2, (8, 9), (8, 8), SHAPE),            # grid does not hold N tokens
    (1, 64, 64, 2, (8, 8), (3, 8), SHAPE),            # block does not tile the grid
    (-1, 64, 64, 2, (8, 8), (8, 8), INVALID),
    (1, 1 << 34, 64, 2, (1 << 17, 1 << 17), (1 << 9, 1 << 9), UNSUPPORTED),   # LayerNorm grid past 2^31 CTAs
])
def test_workspace_size_rejects(B, N, C, heads, grid, block, status):
    assert _ws(B, N, C, heads, grid, block)[0] == status


def test_empty_batch_needs_nothing():
    assert _ws(0, 64, 64, 2, (8, 8), (8, 8)) == (OK, 0)


def test_layer_norm_rejects_before_launch():
    L = mhla.lib()
    p = ctypes.c_void_p(1 << 20)
    assert L.mhla_layer_norm(p, p, 4, 12, p, p, 1e-5, None) == UNSUPPORTED        # C % 8
    assert L.mhla_layer_norm(p, p, 4, 4096, p, p, 1e-5, None) == UNSUPPORTED      # C > 2048
    assert L.mhla_layer_norm(p, p, 4, 64, p, p, -1.0, None) == INVALID            # eps < 0
    assert L.mhla_layer_norm(None, p, 4, 64, p, p, 1e-5, None) == INVALID         # null input
    assert L.mhla_layer_norm(ctypes.c_void_p((1 << 20) + 8), p, 4, 64, p, p, 1e-5, None) == INVALID  # alignment
    assert L.mhla_layer_norm(p, ctypes.c_void_p((1 << 20) + 64), 4, 64, p, p, 1e-5, None) == INVALID  # overlap
    assert L.mhla_layer_norm(p, p, 0, 64, p, p, 1e-5, None) == OK                 # nothing to do


def _view(addr, B, N, H, d, sb, sn, sh):
    return mhla.tensor_desc(addr, 0, (B, N, H, d), (sb, sn, sh))


def test_lepe_add_rejects_before_launch():
    L = mhla.lib()
    w = ctypes.c_void_p(1 << 24)
    good_v = _view(1 << 20, 1, 64, 2, 32, 64 * 192, 192, 32)
    good_o = _view(1 << 22, 1, 64, 2, 32, 64 * 64, 64, 32)
    g = mhla.shape3((8, 8))
    bad_d = _view(1 << 20, 1, 64, 2, 12, 64 * 24, 24, 12)
    bad_d_o = _view(1 << 22, 1, 64, 2, 12, 64 * 24, 24, 12)
    assert L.mhla_lepe_add(ctypes.byref(bad_d), ctypes.byref(bad_d_o), ctypes.byref(g), w, w, None) == UNSUPPORTED
    assert L.mhla_lepe_add(ctypes.byref(good_v), ctypes.byref(good_o), ctypes.byref(mhla.shape3((8, 9))), w, w,
                           None) == SHAPE
    assert L.mhla_lepe_add(ctypes.byref(good_v), ctypes.byref(good_o), ctypes.byref(g), None, w, None) == INVALID
    overlap = _view((1 << 20) + 64, 1, 64, 2, 32, 64 * 64, 64, 32)
    assert L.mhla_lepe_add(ctypes.byref(good_v), ctypes.byref(overlap), ctypes.byref(g), w, w, None) == INVALID
    misaligned = _view((1 << 22) + 8, 1, 64, 2, 32, 64 * 64, 64, 32)
    assert L.mhla_lepe_add(ctypes.byref(good_v), ctypes.byref(misaligned), ctypes.byref(g), w, w,
                           None) == UNSUPPORTED
