"""The allocation-free forward entry point, mhla_forward_noalloc, through the C ABI.

It exists for callers that may not allocate device memory where they run the
forward (an inference engine's plugin inside the engine's enqueue step, a serving
loop that fixes its memory at start-up): it takes its scratch from a 64 MiB array
compiled into the library instead of a caller workspace or cudaMallocAsync.

The first call in a context is its set-up (it loads the array there); a call
with an empty batch does exactly that and nothing else, and is made first, as a
caller would at start-up.  The output must then match the float64 oracle at the
parity bar and the regular entry point within the same bar, on two calls in a
row with different inputs (the shared scratch carries nothing from one call to
the next).  The CUDA-core cases run before the tensor-core case, so the
tensor-core call reads over scratch bytes another layout left behind.  A problem
needing more scratch than the array holds must be refused before any GPU work.
This file is collected last and needs nothing from the other tests.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
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


def normwise(got, ref):
    return float(np.abs(got - ref).max() / np.abs(ref).max())


def test_noalloc_set_up_call_with_an_empty_batch():
    """The start-up call a caller makes: B = 0 sets the array up and queues nothing."""
    grid, block, H, d = (16, 16), (4, 4), 2, 32
    q = torch.empty(0, 256, H, d, dtype=torch.float32, device=DEV)
    W = torch.ones(16, 16, device=DEV)
    assert call_noalloc(q, q, q, W, grid, block, torch.empty_like(q)) == 0
    torch.cuda.synchronize()
    assert mhla.device_status() == 0


@pytest.mark.parametrize("case", [
    # (B, H, d, grid, block, dtype, path): the CUDA cores first, so the
    # tensor-core call runs over scratch left behind by another layout
    (1, 2, 32, (16, 16), (4, 4), "f32", "simt"),
    (2, 4, 64, (32, 64), (8, 16), "bf16", "simt"),
    (2, 3, 64, (32, 48), (16, 8), "bf16", "tc"),
], ids=["simt_f32", "simt_bf16_larger_scratch", "tc_bf16"])
def test_noalloc_matches_oracle_and_regular_entry_point_twice_in_a_row(case):
    B, H, d, grid, block, dtype, path = case
    N = int(np.prod(grid))
    M = mhla.num_blocks(grid, block)
    W_host = draw_matrix(M, seed=31)
    W = torch.from_numpy(W_host).to(DEV)
    for seed in (41, 42):                               # two calls in a row, different inputs
        qh, kh, vh = draw_qkv(B, N, H, d, seed=seed, dtype=dtype)
        q, k, v = qh.to(DEV), kh.to(DEV), vh.to(DEV)
        out = torch.full_like(q, float("nan"))
        assert call_noalloc(q, k, v, W, grid, block, out, path=path) == 0
        regular = mhla.forward(q, k, v, W, grid, block, path=path)
        torch.cuda.synchronize()
        assert mhla.device_status() == 0
        got = as_f64(out.cpu())
        ref = oracle.forward(as_f64(qh), as_f64(kh), as_f64(vh), W_host.astype(np.float64), grid, block)
        err = normwise(got, ref)
        assert err <= TOL[q.dtype], f"seed {seed}: normwise error against the oracle {err:.3e}"
        diff = normwise(got, as_f64(regular.cpu()))
        assert diff <= TOL[q.dtype], f"seed {seed}: normwise difference from mhla_forward {diff:.3e}"


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
