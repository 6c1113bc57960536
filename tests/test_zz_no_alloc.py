"""The allocation-free forward entry point, mhla_forward_noalloc, through the C ABI.

It exists for callers that may not allocate device memory where they run the
forward (an inference engine's plugin inside the engine's enqueue step, a serving
loop that fixes its memory at start-up): it takes its scratch from a 64 MiB array
compiled into the library instead of a caller workspace or cudaMallocAsync.
Its output must match the regular entry point's within the parity tolerance, on
two calls in a row with different inputs (the shared scratch carries nothing from
one call to the next), and a problem needing more scratch than the array holds
must be refused before any GPU work.  This file is collected last and needs
nothing from the other tests.
"""

import ctypes

import numpy as np
import pytest
import torch

import token_level_head_block_gb300 as mhla
from token_level_head_block_gb300.synth import as_f64, draw_matrix, draw_qkv

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: 2e-2, torch.float32: 1e-4}
DEV = torch.device("cuda:0")
P = ctypes.POINTER


def noalloc_fn():
    fn = mhla.lib().mhla_forward_noalloc
    fn.argtypes = [P(mhla.Tensor), P(mhla.Tensor), P(mhla.Tensor), ctypes.c_void_p, P(mhla.Shape3),
                   P(mhla.Shape3), P(mhla.Phi), P(mhla.Tensor), ctypes.c_void_p, ctypes.c_int32]
    fn.restype = ctypes.c_int
    return fn


def desc(t):
    dt = "bf16" if t.dtype == torch.bfloat16 else "f32"
    return mhla.tensor_desc(t.data_ptr(), dt, tuple(t.shape), (t.stride(0), t.stride(1), t.stride(2)))


def call_noalloc(q, k, v, W, grid, block, out, path="auto"):
    stream = torch.cuda.current_stream(DEV).cuda_stream
    return noalloc_fn()(ctypes.byref(desc(q)), ctypes.byref(desc(k)), ctypes.byref(desc(v)),
                        ctypes.c_void_p(W.data_ptr()), ctypes.byref(mhla.shape3(grid)),
                        ctypes.byref(mhla.shape3(block)), ctypes.byref(mhla.Phi(0, 1e-6)),
                        ctypes.byref(desc(out)), ctypes.c_void_p(stream) if stream else None,
                        mhla.PATHS[path])


def normwise(a, b):
    a, b = as_f64(a.cpu()), as_f64(b.cpu())
    return float(np.abs(a - b).max() / np.abs(b).max())


@pytest.mark.parametrize("case", [
    # (B, H, d, grid, block, dtype): tensor-core path, then the CUDA-core path
    (2, 3, 64, (32, 48), (16, 8), "bf16"),
    (1, 2, 32, (16, 16), (4, 4), "f32"),
])
def test_noalloc_matches_regular_entry_point_twice_in_a_row(case):
    B, H, d, grid, block, dtype = case
    N = int(np.prod(grid))
    M = mhla.num_blocks(grid, block)
    W = torch.from_numpy(draw_matrix(M, seed=31)).to(DEV)
    for seed in (41, 42):                               # two calls in a row, different inputs
        q, k, v = (t.to(DEV) for t in draw_qkv(B, N, H, d, seed=seed, dtype=dtype))
        out = torch.full_like(q, float("nan"))
        assert call_noalloc(q, k, v, W, grid, block, out) == 0
        ref = mhla.forward(q, k, v, W, grid, block)
        torch.cuda.synchronize()
        assert mhla.device_status() == 0
        err = normwise(out, ref)
        assert err <= TOL[q.dtype], f"seed {seed}: normwise difference {err:.3e}"


def test_noalloc_refuses_problems_beyond_its_scratch():
    # 64 x 3 heads of a 14 x 14 grid with 2 x 2 blocks on the CUDA-core path
    # keep float32 summaries: about 313 MB of scratch, far above the 64 MiB array.
    B, H, d, grid, block = 64, 3, 64, (14, 14), (2, 2)
    q = torch.randn(B, 196, H, d, device=DEV).to(torch.bfloat16)
    need = mhla.workspace_size(q, grid, block, "simt")
    assert need > (64 << 20)
    out = torch.full_like(q, 7.0)
    W = torch.ones(49, 49, device=DEV)
    assert call_noalloc(q, q, q, W, grid, block, out, path="simt") == 6   # MHLA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)                                      # nothing ran
