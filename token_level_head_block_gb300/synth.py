"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

Draws only: q, k, v ~ N(0, 1) as float32 from ``numpy.random.default_rng(seed)``
in the order q, k, v, each a full ``[B, N, H, d]`` array, then (for bf16
workloads) a round-to-nearest-even cast.  Nothing here computes any part of the
attention; the oracle and the CUDA path both read these same buffers.
"""

from __future__ import annotations

import numpy as np
import torch


def draw_qkv(B, N, H, d, seed, dtype="bf16"):
    """Return CPU torch tensors q, k, v of shape [B, N, H, d] in ``dtype``."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(3):
        a = rng.standard_normal((B, N, H, d), dtype=np.float32)
        t = torch.from_numpy(a)
        if dtype == "bf16":
            t = t.to(torch.bfloat16)
        elif dtype != "f32":
            raise ValueError(f"unsupported dtype {dtype}")
        out.append(t)
    return tuple(out)


def draw_workload(wl, seed=None):
    """Inputs of a named workload (see ``workloads.WORKLOADS``)."""
    return draw_qkv(wl.B, wl.N, wl.H, wl.d, wl.seed if seed is None else seed, wl.dtype)


def draw_matrix(M, seed, low=0.0, high=1.0):
    """A random M x M float32 matrix with entries uniform in [low, high)."""
    rng = np.random.default_rng(seed)
    return rng.uniform(low, high, size=(M, M)).astype(np.float32)


def as_f64(t):
    """Exact float64 copy of a CPU tensor (bf16 and fp32 decode exactly)."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def draw_tokens(B, N, C, seed):
    """x ~ N(0, 1), [B, N, C], bf16 (round to nearest even from float32)."""
    rng = np.random.default_rng(seed)
    return torch.from_numpy(rng.standard_normal((B, N, C), dtype=np.float32)).to(torch.bfloat16)


def draw_module_params(C, seed, lepe=True, biases=True):
    """Seeded parameters of the module around the core, as CPU torch tensors:
    LayerNorm weight 1 + 0.1 N(0, 1) and bias 0.1 N(0, 1) (float32); projection
    weights N(0, 1 / C) and biases 0.1 N(0, 1) (bf16); 5 x 5 positional kernels
    0.2 N(0, 1) and bias 0.1 N(0, 1) (float32).  Drawn in that order."""
    rng = np.random.default_rng(seed)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    bf16 = lambda a: f32(a).to(torch.bfloat16)
    p = {"ln_weight": f32(1 + 0.1 * rng.standard_normal(C)), "ln_bias": f32(0.1 * rng.standard_normal(C)),
         "qkv_weight": bf16(rng.standard_normal((3 * C, C)) / np.sqrt(C)),
         "out_weight": bf16(rng.standard_normal((C, C)) / np.sqrt(C))}
    qkv_b, out_b = 0.1 * rng.standard_normal(3 * C), 0.1 * rng.standard_normal(C)
    if biases:
        p["qkv_bias"], p["out_bias"] = bf16(qkv_b), bf16(out_b)
    lw, lb = 0.2 * rng.standard_normal((C, 5, 5)), 0.1 * rng.standard_normal(C)
    if lepe:
        p["lepe_weight"], p["lepe_bias"] = f32(lw), f32(lb)
    return p
