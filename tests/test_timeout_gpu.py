"""The timeout path of the device-side waits, exercised on the GPU without a
fault, trap or hang.

Every kernel waits on its pipeline barriers with a bound (time and polls); a
wait that gives up raises its CTA's abort flag and the device error word, the
other roles stop, copies in flight drain and tensor memory is released.  That
exit is taken only when a completion is lost, so it is forced here with the
library's diagnostic hook (mhla_debug_stall_waits): the waits of one warp
index of every kernel that find their barrier not yet complete behave as if it
never completed and give up after 1 ms.  The warp is one whose waits do poll:
the MMA issuer (warp 1) of the pipelined kernels, the control warp (warp 8)
of the short-sequence kernel, whose workers' barriers are often complete at
the first poll.  Each call must then report MHLA_ERR_TIMEOUT with bit 0 (a wait gave up)
and without bit 1 (a drain of copies in flight failed), and the same call made
again after the hook is off must give the oracle's result on the same context.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import token_level_head_block_gb300 as mhla
from token_level_head_block_gb300.synth import as_f64, draw_matrix, draw_module_params, draw_qkv, draw_tokens

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
TIMEOUT = 5


def raw_status():
    """(status, flags) of mhla_device_status without raising."""
    flags = ctypes.c_uint32(0)
    st = mhla.lib().mhla_device_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream) or None,
                                       ctypes.byref(flags))
    return int(st), int(flags.value)


def normwise(got, ref):
    return float(np.abs(got - ref).max() / np.abs(ref).max())


def forward_case(path, B=1, H=2, d=64, grid=(32, 32), block=(16, 16)):
    N = int(np.prod(grid))
    q, k, v = draw_qkv(B, N, H, d, seed=61, dtype="bf16")
    W = draw_matrix(oracle.num_blocks(grid, block), seed=62)
    Wd = torch.from_numpy(W).to(DEV)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)

    def call():
        return mhla.forward(qd, kd, vd, Wd, grid, block, path=path)

    def check(out):
        ref = oracle.forward(as_f64(q), as_f64(k), as_f64(v), W, grid, block)
        return normwise(as_f64(out.cpu()), ref)
    return call, check


def backward_case():
    B, H, d, grid, block = 1, 2, 64, (32, 32), (16, 8)
    q, k, v = draw_qkv(B, 1024, H, d, seed=63, dtype="bf16")
    g = draw_qkv(B, 1024, H, d, seed=64, dtype="bf16")[0]
    W = mhla.init_mixing(grid, block, "exp")
    dev = [t.to(DEV) for t in (q, k, v, g)]
    Wd = torch.from_numpy(W).to(DEV)

    def call():
        return mhla.backward(dev[0], dev[1], dev[2], Wd, dev[3], grid, block, path="tc")[0]

    def check(dq):
        ref = oracle.backward(as_f64(q), as_f64(k), as_f64(v), W, as_f64(g), grid, block)[0]
        return normwise(as_f64(dq.cpu()), ref)
    return call, check


def causal_case():
    B, H, d, grid, block = 1, 2, 64, (1, 1024), (1, 64)
    q, k, v = draw_qkv(B, 1024, H, d, seed=65, dtype="bf16")
    W = mhla.init_mixing(grid, block, "linear")
    dev = [t.to(DEV) for t in (q, k, v)]
    Wd = torch.from_numpy(W).to(DEV)

    def call():
        return mhla.forward_causal(dev[0], dev[1], dev[2], Wd, grid, block, path="tc")

    def check(out):
        ref = oracle.forward_causal(as_f64(q), as_f64(k), as_f64(v), W, grid, block)
        return normwise(as_f64(out.cpu()), ref)
    return call, check


def module_case():
    B, grid, block, heads = 1, (32, 32), (16, 16), 2
    N, C = 1024, 128
    x = draw_tokens(B, N, C, seed=66)
    p = draw_module_params(C, seed=67)
    W = mhla.init_mixing(grid, block)
    xd, pd, Wd = x.to(DEV), {k: t.to(DEV) for k, t in p.items()}, torch.from_numpy(W).to(DEV)

    def call():
        return mhla.module_forward(xd, pd, Wd, grid, block, heads)

    def check(y):
        ref = oracle.module_forward(as_f64(x), {k: as_f64(t) for k, t in p.items()}, W.astype(np.float64), grid,
                                    block, heads, oracle.PHI_RELU_EPS, 1e-6)
        return normwise(as_f64(y.cpu()), ref)
    return call, check


CASES = {
    # name: (case, warp whose waits stall)
    "forward_three_launches": (lambda: forward_case("tc"), 1),
    "forward_single_launch": (lambda: forward_case("tc_fused"), 1),
    "forward_short_sequence": (lambda: forward_case("fused", B=2, H=3, grid=(14, 14), block=(2, 2)), 8),
    "backward": (backward_case, 1),
    "causal": (causal_case, 1),
    "module": (module_case, 1),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_bounded_wait_runs_out_then_the_context_recovers(name):
    make, warp = CASES[name]
    call, check = make()
    assert raw_status() == (0, 0)
    mhla.debug_stall_waits(warp, 1_000_000)         # that warp of every kernel: waits give up after 1 ms
    try:
        call()
        torch.cuda.synchronize()
        status, flags = raw_status()
    finally:
        mhla.debug_stall_waits(-1)
    assert status == TIMEOUT, (status, flags)
    assert flags & 1, f"no wait gave up: flags {flags:#x}"
    assert not flags & 2, f"copies in flight did not drain: flags {flags:#x}"
    assert raw_status() == (0, 0)                   # the word was cleared by the read
    out = call()                                    # the same context, hook off
    torch.cuda.synchronize()
    assert raw_status() == (0, 0)
    assert check(out) <= 2e-2
