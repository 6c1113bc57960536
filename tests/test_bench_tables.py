"""The benchmark's per-kernel tables and CPU legs, checked on the host.

Every kernel name the library times (its `KernelTimer` names, including the
projections' names passed to the linear-layer helper) must have an algorithmic
work entry, so the roofline of whichever kernel dominates a pass is never
reported against zero work; and the module pass's CPU leg must run the module
oracle end to end.
"""

import os
import re

import numpy as np
import pytest

import bench
from token_level_head_block_gb300.workloads import WORKLOADS

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "token_level_head_block_gb300",
                    "csrc")


def timed_kernel_names():
    names = set()
    for fn in os.listdir(CSRC):
        if not fn.endswith(".cu"):
            continue
        text = open(os.path.join(CSRC, fn)).read()
        for call in re.findall(r"KernelTimer timer\(([^;]*)\);", text):
            names.update(re.findall(r'"([a-z_0-9]+)"', call))
        names.update(re.findall(r'launch_gemm\("([a-z_0-9]+)"', text))
    # mhla_gemm labels the stand-alone linear-layer entry point, which no
    # benchmark pass launches (the module's projections carry their own names)
    names.discard("mhla_gemm")
    return names


def test_every_timed_kernel_has_work():
    names = timed_kernel_names()
    assert {"tc_summary", "tc_mix", "tc_output", "tc_tile_output", "mhla_lepe_add", "mhla_gemm_qkv"} <= names
    wl = WORKLOADS["dit_s2_4096px"]
    for name in sorted(names):
        bound, work = bench.kernel_work(wl, name)
        assert bound in ("hbm", "tensor", "alu"), name
        assert work > 0, name


def test_module_projection_flops():
    wl = WORKLOADS["dit_s2_4096px"]
    C = wl.H * wl.d
    assert bench.kernel_work(wl, "mhla_gemm_qkv") == ("tensor", 2 * wl.B * wl.N * C * 3 * C)
    assert bench.kernel_work(wl, "mhla_gemm_out") == ("tensor", 2 * wl.B * wl.N * C * C)


def test_module_cpu_leg_runs_the_oracle():
    wl = WORKLOADS["tiny_16x16_fp32"]
    x, params = bench.module_inputs(wl, 7)
    assert tuple(x.shape) == (wl.B, wl.N, wl.H * wl.d)
    import oracle
    W = oracle.mixing_matrix(wl.grid, wl.block, wl.transform, wl.local_thres, wl.exp_sigma)
    rate, n, el = bench.oracle_module_rate(wl, x, params, W, 0.0, max_items=1)
    assert n == 1 and el > 0 and rate == pytest.approx(wl.N / el)
    assert np.isfinite(rate)
