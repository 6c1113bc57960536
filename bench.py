#!/usr/bin/env python3
"""Throughput of the MHLA forward pass on GB300 (tokens/s and HBM roofline).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                  [--pass forward|backward|causal|causal_backward|module]

One step = one MHLA forward (summaries, mixing GEMM, outputs) over
one synthetic batch of the workload, inputs resident in HBM; with
``--pass backward`` one step is one backward pass (dq, dk, dv, dW for a seeded
dout); with ``--pass causal`` one causal (chunkwise) MHLA forward and with
``--pass causal_backward`` its backward pass; with ``--pass
module`` one forward of the whole module around the core (LayerNorm, qkv
projection, MHLA, 5 x 5 positional term, output projection) on x [B, N, H * d].  Rank 0 prints one
JSON line.  With N > 1 (torchrun) every rank runs an independent batch on its own
GPU (replicas, weak scaling); ranks meet only for the timing barrier and the
max-over-ranks reduction.  ``--impl reference`` times the float64 CPU oracle on
the host cores instead (rank 0 only), on bounded samples of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import itertools
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from token_level_head_block_gb300.workloads import HEADLINE, WORKLOADS  # noqa: E402

METRIC = "MHLA forward tokens/sec at 1 GB300; achieved HBM GB/s as fraction of peak"
METRIC_BWD = "MHLA backward (dq, dk, dv, dW) tokens/sec at 1 GB300; achieved HBM GB/s as fraction of peak"
METRIC_CAUSAL = "causal MHLA forward tokens/sec at 1 GB300; achieved HBM GB/s as fraction of peak"
METRIC_CAUSAL_BWD = ("causal MHLA backward (dq, dk, dv, dW) tokens/sec at 1 GB300; achieved HBM GB/s as fraction "
                     "of peak")
METRIC_MODULE = ("MHLA module forward (LayerNorm, qkv projection, MHLA, 5x5 positional term, output projection) "
                 "tokens/sec at 1 GB300")
METRICS = {"forward": METRIC, "backward": METRIC_BWD, "causal": METRIC_CAUSAL, "causal_backward": METRIC_CAUSAL_BWD,
           "module": METRIC_MODULE}
ORACLE_WHAT = {"forward": "oracle (blocked form)", "backward": "backward oracle", "causal": "causal oracle",
               "causal_backward": "causal backward oracle"}
UNIT = "tokens/s"
L2_BYTES = 129 * 1024 * 1024
ROTATE_CAP = 256   # copies at most (the tiny workload stays inside L2 even so)


def rotation(tensors, l2_bytes):
    """Copies of a step's tensors (inputs and outputs) to cycle through, one set per
    step: a set is touched again only after more than 1.5x the L2 size of other
    traffic, so every step reads its inputs from HBM.  One set when a step alone
    moves that much."""
    step_bytes = sum(t.numel() * t.element_size() for t in tensors)
    n = 1 if step_bytes >= 1.5 * l2_bytes else min(ROTATE_CAP, -(-int(1.5 * l2_bytes) // step_bytes) + 1)
    return [tuple(tensors)] + [tuple(t.clone() for t in tensors) for _ in range(n - 1)], step_bytes
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------- distributed harness

def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def dist_init(backend):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(x, device=None):
    """Maximum of a float over all ranks (x itself without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_throughput(units_per_rank, world, steps, max_elapsed_s):
    """Units processed by all ranks divided by the slowest rank's time."""
    return units_per_rank * world * steps / max_elapsed_s


# ----------------------------------------------------------------- clocks

CLOCK_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi sampling every 200 ms of the benchmark's GPU."""

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="mhla_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu=timestamp,{CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        rows = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
            os.unlink(self.path)
        return summarize_clocks(rows)


def summarize_clocks(rows):
    def num(x):
        try:
            return float(x)
        except ValueError:
            return None
    sm = [num(r[1]) for r in rows if num(r[1]) is not None]
    smax = [num(r[2]) for r in rows if num(r[2]) is not None]
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
            "reasons": reasons, "samples": len(rows),
            "power_w_max": max((num(r[3]) or 0.0) for r in rows) if rows else None}


# ----------------------------------------------------------------- roofline inputs

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# Source files a kernel's code lives in (with the shared inline-PTX header).
KERNEL_SOURCES = {"tc_summary": ("tc_summary.cu", "tc_fwd_bodies.cuh"), "tc_mix": ("tc_mix.cu", "tc_fwd_bodies.cuh"),
                  "tc_output": ("tc_output.cu", "tc_fwd_bodies.cuh"), "tc_fused": ("tc_fused.cu", "tc_fwd_bodies.cuh"),
                  "tc_small": "small_kernels.cu", "simt_summary": "simt_kernels.cu",
                  "simt_mix": "simt_kernels.cu", "simt_output": "simt_kernels.cu",
                  "tc_bwd_query": "bwd_tc_kernels.cu", "tc_bwd_key": "bwd_tc_kernels.cu",
                  "tc_dw": "bwd_tc_kernels.cu", "simt_bwd_query": "simt_kernels.cu",
                  "simt_bwd_key": "simt_kernels.cu", "simt_dw": "simt_kernels.cu",
                  "simt_causal_output": "simt_kernels.cu", "tc_causal_tile": "causal_tc_kernels.cu",
                  "simt_causal_bwd_query": "simt_kernels.cu", "simt_causal_bwd_key": "simt_kernels.cu",
                  "simt_ds_to_summary": "simt_kernels.cu",
                  "simt_dw_causal_and_wt": "simt_kernels.cu",
                  "tc_tile_output": "causal_tc_kernels.cu", "mhla_lepe_add": "module_kernels.cu",
                  "mhla_ln_rows": "module_kernels.cu", "mhla_gemm_qkv": "gemm_kernels.cu",
                  "mhla_gemm_out": "gemm_kernels.cu"}


def kernel_source_digest(kernel):
    """Hash of the source files of one kernel: a profile summary taken on other
    code than the current one does not count."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "token_level_head_block_gb300", "csrc")
    own = KERNEL_SOURCES.get(kernel, ())
    for name in ((own,) if isinstance(own, str) else tuple(own)) + ("ptx.cuh", "tc_common.cuh"):
        p = os.path.join(csrc, name)
        if name and os.path.exists(p):
            with open(p, "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    d = re.search(r"kernel_source_digest:\s*([0-9a-f]+)", text)
    if not m or not d or d.group(1) != kernel_source_digest(kernel):
        return None
    return int(m.group(1))


def kernel_work(wl, name):
    """(bound, algorithmic bytes or flops per launch) of each kernel of the path."""
    io = wl.B * wl.N * wl.H * wl.d * wl.elem_bytes
    BH, M, d = wl.B * wl.H, wl.M, wl.d
    table = {
        "tc_summary": ("hbm", 2 * io), "simt_summary": ("hbm", 2 * io),
        "tc_output": ("hbm", 2 * io), "simt_output": ("hbm", 2 * io),
        "tc_mix": ("tensor", 2 * M * M * BH * d * (d + 1)), "simt_mix": ("alu", 2 * M * M * BH * d * (d + 1)),
        "tc_small": ("hbm", 4 * io),
        # the whole forward in one persistent launch: read q, k, v, write o
        "tc_fused": ("hbm", 4 * io),
        # backward: read q, dout, write dq; read k, v, write dk, dv; dW = dS~ . S^T
        "tc_bwd_query": ("hbm", 3 * io), "simt_bwd_query": ("hbm", 3 * io),
        "tc_bwd_key": ("hbm", 4 * io), "simt_bwd_key": ("hbm", 4 * io),
        "tc_dw": ("tensor", 2 * M * M * BH * d * (d + 1)), "simt_dw": ("alu", 2 * M * M * BH * d * (d + 1)),
        # causal: read q, k, v, write o
        "simt_causal_output": ("hbm", 4 * io), "tc_causal_tile": ("hbm", 4 * io),
        # causal backward: read q, k, v, dout, write dq and the float32 dnum, dden
        # rows; read q, k, v and those rows, write dk, dv
        "simt_causal_bwd_query": ("hbm", 5 * io + BH * wl.N * (d + 1) * 4),
        "simt_causal_bwd_key": ("hbm", 5 * io + BH * wl.N * (d + 1) * 4),
        # causal backward, path TC: dS< to the bf16 summary layout; dW made causal and
        # W's strict lower triangle transposed
        "simt_ds_to_summary": ("hbm", BH * M * d * (d + 1) * (4 + 2)),
        "simt_dw_causal_and_wt": ("hbm", M * M * (4 + 2) + 2 * M * M * 4 + BH * M * 4),
        # readout of contiguous 64-token blocks: read q, write o
        "tc_tile_output": ("hbm", 2 * io),
        # module: x -> LayerNorm; qkv = xn W^T; o += lepe(v) (read v, o; write o); y = o W^T
        "mhla_ln_rows": ("hbm", 2 * io), "mhla_lepe_add": ("hbm", 3 * io),
        "mhla_gemm_qkv": ("tensor", 2 * wl.tokens * (wl.H * d) * 3 * (wl.H * d)),
        "mhla_gemm_out": ("tensor", 2 * wl.tokens * (wl.H * d) * (wl.H * d)),
    }
    return table.get(name, ("hbm", 0))


# ----------------------------------------------------------------- CPU oracle baseline

def blas_threads():
    import ctypes
    try:
        with open("/proc/self/maps") as f:
            libs = sorted({line.split()[-1] for line in f if "openblas" in line.lower() and ".so" in line})
    except OSError:
        libs = []
    for lib in libs:
        try:
            L = ctypes.CDLL(lib)
        except OSError:
            continue
        for sym in ("openblas_get_num_threads", "openblas_get_num_threads64_",
                    "scipy_openblas_get_num_threads64_", "scipy_openblas_get_num_threads"):
            fn = getattr(L, sym, None)
            if fn is not None:
                fn.restype = ctypes.c_int
                return int(fn())
    return os.cpu_count() or 1


def runs_of(n, total, what):
    """How many oracle runs a timed sample made over `total` units named `what`
    (the sampler cycles through them, so n may exceed total)."""
    if n <= total:
        return f"{n} of the {total} {what}"
    return f"{n} runs cycling over the {total} {what}"


def oracle_sample_rate(wl, q, k, v, W, budget_s, max_slices=None, g=None, causal=False):
    """Times the oracle (the backward oracle when dout g is given; the causal
    ones with ``causal``) on (b, h)
    slices until budget_s elapses (at least one slice).  Returns (tokens/s,
    slices, seconds); a slice of one head counts N / H tokens."""
    import oracle
    from token_level_head_block_gb300.synth import as_f64
    phi = oracle.PHI_RELU if wl.phi == "relu" else oracle.PHI_RELU_EPS
    pairs = [(b, h) for b in range(wl.B) for h in range(wl.H)]
    done, t0 = 0, time.perf_counter()
    while True:
        b, h = pairs[done % len(pairs)]
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1), slice(None))
        if causal and g is not None:
            oracle.backward_causal(as_f64(q[sl]), as_f64(k[sl]), as_f64(v[sl]), W, as_f64(g[sl]), wl.grid, wl.block,
                                   phi, wl.eps)
        elif causal:
            oracle.forward_causal(as_f64(q[sl]), as_f64(k[sl]), as_f64(v[sl]), W, wl.grid, wl.block, phi, wl.eps)
        elif g is None:
            oracle.forward(as_f64(q[sl]), as_f64(k[sl]), as_f64(v[sl]), W, wl.grid, wl.block, phi, wl.eps)
        else:
            oracle.backward(as_f64(q[sl]), as_f64(k[sl]), as_f64(v[sl]), W, as_f64(g[sl]), wl.grid, wl.block, phi,
                            wl.eps)
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_slices and done >= max_slices):
            break
    return done * wl.N / wl.H / el, done, el


def module_inputs(wl, seed):
    """Seeded x [B, N, H * d] and module parameters for the module pass."""
    from token_level_head_block_gb300.synth import draw_module_params, draw_tokens
    C = wl.H * wl.d
    return draw_tokens(wl.B, wl.N, C, seed), draw_module_params(C, seed + 1)


def oracle_module_rate(wl, x, params, W, budget_s, max_items=None):
    """Times the module oracle on whole batch elements (the projections mix the
    heads, so a batch element is the smallest unit) until budget_s elapses.
    Returns (tokens/s, batch elements, seconds)."""
    import oracle
    from token_level_head_block_gb300.synth import as_f64
    phi = oracle.PHI_RELU if wl.phi == "relu" else oracle.PHI_RELU_EPS
    p64 = {k: as_f64(t) for k, t in params.items()}
    done, t0 = 0, time.perf_counter()
    while True:
        b = done % wl.B
        oracle.module_forward(as_f64(x[b:b + 1]), p64, W, wl.grid, wl.block, wl.H, phi, wl.eps)
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_items and done >= max_items):
            break
    return done * wl.N / el, done, el


def draw_dout(wl, seed=None):
    """Seeded dL/d(out) for the backward pass, N(0, 1) in the workload's dtype."""
    from token_level_head_block_gb300.synth import draw_qkv
    return draw_qkv(wl.B, wl.N, wl.H, wl.d, wl.seed + 100 if seed is None else seed, wl.dtype)[0]


# ----------------------------------------------------------------- arms

def run_reference(args, wl):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import numpy as np  # noqa: F401
    import oracle
    from token_level_head_block_gb300.synth import draw_workload
    W = oracle.mixing_matrix(wl.grid, wl.block, wl.transform, wl.local_thres, wl.exp_sigma)
    if args.pass_ == "module":
        x, params = module_inputs(wl, wl.seed + 300)
        for _ in range(args.warmup):
            oracle_module_rate(wl, x, params, W, 0.0, max_items=1)
        times = []
        for _ in range(args.steps):
            times.append(oracle_module_rate(wl, x, params, W, 1e9, max_items=1)[2])
        total = sum(times)
        value = args.steps * wl.N / total
        sample = f"each step: one of the {wl.B} batch elements of {wl.name}, float64 numpy module oracle"
        print(json.dumps({
            "impl": "reference", "metric": METRICS[args.pass_], "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {**wl.describe(), "pass": "module",
                                            "parallelism": "host cores (BLAS threads)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }))
        return
    q, k, v = draw_workload(wl)
    g = draw_dout(wl) if args.pass_ in ("backward", "causal_backward") else None
    causal = args.pass_ in ("causal", "causal_backward")
    per_step = max(1, args.ref_slices)
    for _ in range(args.warmup):
        oracle_sample_rate(wl, q, k, v, W, 0.0, max_slices=1, g=g, causal=causal)
    times = []
    for _ in range(args.steps):
        _, n, el = oracle_sample_rate(wl, q, k, v, W, 1e9, max_slices=per_step, g=g, causal=causal)
        times.append(el)
    total = sum(times)
    value = args.steps * per_step * wl.N / wl.H / total
    cores = blas_threads()
    what = ORACLE_WHAT[args.pass_]
    sample = (f"each step: {per_step} of the {wl.B * wl.H} (batch, head) slices of {wl.name}, "
              f"float64 numpy {what}; a slice counts N/H tokens")
    print(json.dumps({
        "impl": "reference", "metric": METRICS[args.pass_], "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {**wl.describe(), "parallelism": "host cores (BLAS threads)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def run_ours(args, wl):
    import torch
    import token_level_head_block_gb300 as mhla
    from token_level_head_block_gb300.synth import draw_workload

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist_init("nccl")
    mhla.lib()

    bwd = args.pass_ in ("backward", "causal_backward")
    module = args.pass_ == "module"
    q_h, k_h, v_h = draw_workload(wl, seed=wl.seed + rank)      # each replica its own batch
    g_h = draw_dout(wl, seed=wl.seed + 100 + rank) if bwd else None
    W_h = mhla.init_mixing(wl.grid, wl.block, wl.transform, wl.local_thres, wl.exp_sigma)
    q, k, v = (t.to(dev) for t in (q_h, k_h, v_h))
    W = torch.from_numpy(W_h).to(dev)
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)
    l2_bytes = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", L2_BYTES)
    turn = itertools.count()   # step counter: which input set the next step takes
    if module:
        x_h, params_h = module_inputs(wl, wl.seed + 300 + rank)
        x = x_h.to(dev)
        params = {name: t.to(dev) for name, t in params_h.items()}
        y = torch.empty_like(x)
        ws = torch.empty(mhla.module_workspace_size(wl.B, wl.N, wl.H * wl.d, wl.H, wl.grid, wl.block),
                         dtype=torch.uint8, device=dev)
        sets, set_bytes = rotation([x, y], l2_bytes)

        def step():
            xx, yy = sets[next(turn) % len(sets)]
            mhla.module_forward(xx, params, W, wl.grid, wl.block, wl.H, phi=wl.phi, eps=wl.eps, out=yy,
                                workspace=ws, stream=stream)
    elif args.pass_ == "causal":
        ws = torch.empty(mhla.causal_workspace_size(q, wl.grid, wl.block), dtype=torch.uint8, device=dev)
        sets, set_bytes = rotation([q, k, v, out], l2_bytes)

        def step():
            qq, kk, vv, oo = sets[next(turn) % len(sets)]
            mhla.forward_causal(qq, kk, vv, W, wl.grid, wl.block, phi=wl.phi, eps=wl.eps, out=oo, workspace=ws,
                                stream=stream)
    elif bwd:
        g = g_h.to(dev)
        dq, dk, dv, dW = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(W)
        causal_bwd = args.pass_ == "causal_backward"
        ws_size = mhla.backward_causal_workspace_size if causal_bwd else mhla.backward_workspace_size
        bwd_call = mhla.backward_causal if causal_bwd else mhla.backward
        ws = torch.empty(ws_size(q, wl.grid, wl.block), dtype=torch.uint8, device=dev)
        sets, set_bytes = rotation([q, k, v, g, dq, dk, dv], l2_bytes)

        def step():
            qq, kk, vv, gg, dqq, dkk, dvv = sets[next(turn) % len(sets)]
            bwd_call(qq, kk, vv, W, gg, wl.grid, wl.block, phi=wl.phi, eps=wl.eps, dq=dqq, dk=dkk, dv=dvv, dW=dW,
                     workspace=ws, stream=stream)
    else:
        ws = torch.empty(mhla.workspace_size(q, wl.grid, wl.block, args.path), dtype=torch.uint8, device=dev)
        sets, set_bytes = rotation([q, k, v, out], l2_bytes)

        def step():
            qq, kk, vv, oo = sets[next(turn) % len(sets)]
            mhla.forward(qq, kk, vv, W, wl.grid, wl.block, phi=wl.phi, eps=wl.eps, out=oo, workspace=ws,
                         stream=stream, path=args.path)
    path = mhla.select_path(q, k, v, out, wl.grid, wl.block) if args.path == "auto" else args.path

    def timed(n, body):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(dev)
        torch.cuda.synchronize(dev)
        start.record(stream)
        for _ in range(n):
            body()
        end.record(stream)
        torch.cuda.synchronize(dev)
        barrier(dev)
        return start.elapsed_time(end) / 1e3

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if mhla.device_status() != 0:
        raise SystemExit("device wait flag set during warm-up")

    gpu_uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    sampler = ClockSampler(gpu_uuid)
    sampler.start()
    t_end = time.time() + args.sustain
    while time.time() < t_end:             # sustained load so the clock samples mean something
        for _ in range(50):
            step()
        torch.cuda.synchronize(dev)
    el_main = timed(args.steps, step)                       # pass A: the headline number
    mhla.profile_begin()
    el_prof = timed(args.steps, step)                       # pass B: per-kernel attribution
    prof = mhla.profile_end()
    clocks = sampler.stop()
    if mhla.device_status() != 0:
        raise SystemExit("device wait flag set during the timed region")

    max_el = max_over_ranks(el_main, dev)
    value = whole_job_throughput(wl.tokens, world, args.steps, max_el)
    ms_per_step = 1e3 * max_el / args.steps

    # e2e: host buffers in pinned memory, copies inside the timed region.  The
    # batch elements of a forward (plain, causal or module) are independent, so
    # the step is cut into batch chunks on three streams: the H2D copy of chunk
    # c + 1, the library call on chunk c and the D2H copy of chunk c - 1 overlap.
    # The backward's dW sums over the batch, so its copies stay serial.
    e2e = None
    if not args.no_e2e:
        hq, hk, hv = (t.pin_memory() for t in (q_h, k_h, v_h))
        n_chunks = min(wl.B, 8)
        bounds = [(c * wl.B // n_chunks, (c + 1) * wl.B // n_chunks) for c in range(n_chunks)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        if module:
            hx, hy = x_h.pin_memory(), torch.empty_like(x_h).pin_memory()
            ins, outs = [(x, hx)], [(hy, y)]

            def call(b0, b1):
                mhla.module_forward(x[b0:b1], params, W, wl.grid, wl.block, wl.H, phi=wl.phi, eps=wl.eps,
                                    out=y[b0:b1], workspace=ws, stream=stream)
        elif bwd:
            hg = g_h.pin_memory()
            hdq, hdk, hdv = (torch.empty_like(q_h).pin_memory() for _ in range(3))
            hdW = torch.empty(dW.shape, dtype=dW.dtype).pin_memory()
        else:
            ho = torch.empty_like(q_h).pin_memory()
            ins, outs = [(q, hq), (k, hk), (v, hv)], [(ho, out)]
            causal = args.pass_ == "causal"

            def call(b0, b1):
                fn = mhla.forward_causal if causal else mhla.forward
                kw = {} if causal else {"path": args.path}
                fn(q[b0:b1], k[b0:b1], v[b0:b1], W, wl.grid, wl.block, phi=wl.phi, eps=wl.eps, out=out[b0:b1],
                   workspace=ws, stream=stream, **kw)

        if bwd:
            def e2e_step():
                for dst, src in ((q, hq), (k, hk), (v, hv), (g, hg)):
                    dst.copy_(src, non_blocking=True)
                step()
                for dst, src in ((hdq, dq), (hdk, dk), (hdv, dv), (hdW, dW)):
                    dst.copy_(src, non_blocking=True)
        else:
            def e2e_step():
                s_in.wait_stream(stream)             # the previous step has fully finished
                for b0, b1 in bounds:
                    with torch.cuda.stream(s_in):
                        for dst, src in ins:
                            dst[b0:b1].copy_(src[b0:b1], non_blocking=True)
                    stream.wait_stream(s_in)
                    call(b0, b1)
                    s_out.wait_stream(stream)
                    with torch.cuda.stream(s_out):
                        for dst, src in outs:
                            dst[b0:b1].copy_(src[b0:b1], non_blocking=True)
                stream.wait_stream(s_out)            # the step ends when its last copy has landed

        for _ in range(2):
            e2e_step()
        n_e2e = max(3, min(args.steps, 50))
        el_e2e = max_over_ranks(timed(n_e2e, e2e_step), dev)
        io = wl.B * wl.N * wl.H * wl.d * wl.elem_bytes
        e2e = {"value": whole_job_throughput(wl.tokens, world, n_e2e, el_e2e), "unit": UNIT,
               "h2d_bytes_per_step": io if module else (4 if bwd else 3) * io,
               "d2h_bytes_per_step": 3 * io + wl.M * wl.M * 4 if bwd else io, "steps": n_e2e,
               "ms_per_step": 1e3 * el_e2e / n_e2e,
               "copies": "serial on the compute stream (dW sums over the batch)" if bwd else
                         f"{n_chunks} batch chunks; H2D, library call and D2H on three streams, overlapped"}

    # roofline of the dominant kernel, from the per-kernel events of pass B
    peaks, peak_src = load_peaks()
    kern = {name: {"launches": n, "avg_us": 1e3 * ms / n, "share": 0.0} for name, (n, ms) in prof.items()}
    total_ms = sum(ms for _, ms in prof.values()) or 1.0
    for name, (_, ms) in prof.items():
        kern[name]["share"] = ms / total_ms
    dominant = max(prof, key=lambda n: prof[n][1])
    bound, work = kernel_work(wl, dominant)
    avg_s = prof[dominant][1] / 1e3 / prof[dominant][0]
    if bound == "hbm":
        achieved, peak, unit = work / avg_s / 1e9, float(peaks["hbm_gbs"]), "GB/s"
    else:
        achieved = work / avg_s / 1e12
        peak, unit = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])), "TFLOP/s"
    traffic = profiled_traffic(dominant, wl.name)
    roofline = {"kernel": dominant, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "traffic": traffic, "algorithmic_per_launch": work,
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback"}
    # read q, k, v (+ dout) and write o (dq, dk, dv)
    pass_bytes = wl.algorithmic_bytes * 7 // 4 if bwd else wl.algorithmic_bytes
    fwd_gbs = pass_bytes / (max_el / args.steps) / 1e9
    forward_roofline = {"bound": "hbm", "achieved": fwd_gbs, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                        "frac": fwd_gbs / float(peaks["hbm_gbs"]), "bytes_per_step": pass_bytes}
    if module:
        # the two projections carry the step's flops: 8 tokens C^2
        C = wl.H * wl.d
        flops = 8 * wl.tokens * C * C
        tf = flops / (max_el / args.steps) / 1e12
        tpeak = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
        forward_roofline = {"bound": "tensor", "achieved": tf, "peak": tpeak, "unit": "TFLOP/s", "frac": tf / tpeak,
                            "flops_per_step": flops, "note": "projection flops over the whole step"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and module:
        rate, n, el = oracle_module_rate(wl, x_h, params_h, W_h.astype("float64"), args.cpu_seconds)
        cpu = {"value": rate, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
               "sample": f"{runs_of(n, wl.B, 'batch elements')} of {wl.name} in {el:.1f} s, float64 numpy "
                         "module oracle"}
    elif rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, n, el = oracle_sample_rate(wl, q_h, k_h, v_h, W_h, args.cpu_seconds, g=g_h,
                                         causal=args.pass_ in ("causal", "causal_backward"))
        what = ORACLE_WHAT[args.pass_]
        cpu = {"value": rate, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
               "sample": f"{runs_of(n, wl.B * wl.H, '(batch, head) slices')} of {wl.name} in {el:.1f} s, "
                         f"float64 numpy {what}; a slice counts N/H tokens"}

    launches = sum(n for n, _ in prof.values())
    if len(sets) == 1:
        l2_note = f"inputs and outputs {set_bytes / 1e6:.0f} MB per step > L2 {l2_bytes / 2**20:.0f} MiB (no flush)"
    else:
        l2_note = (f"{len(sets)} copies of the step's inputs and outputs ({set_bytes / 1e6:.1f} MB each) taken in "
                   f"turn: {len(sets) * set_bytes / 1e6:.0f} MB against L2 {l2_bytes / 2**20:.0f} MiB"
                   + (", every step reads its inputs from HBM" if (len(sets) - 1) * set_bytes > l2_bytes
                      else ", still inside L2 (a launch-bound case)"))
    if rank == 0:
        line = {
            "impl": "ours", "metric": METRICS[args.pass_], "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if wl.dtype == "bf16" else "f32",
            "data": "synthetic",
            "config": {**wl.describe(), "pass": args.pass_,
                       "path": ("tc (summaries, mixings, dW) + warp-level mma (per-token steps)" if "tc_summary" in prof
                                else "simt")
                               if args.pass_ == "causal_backward" else
                               ("tc" if "tc_bwd_query" in prof else "simt") if bwd else
                               ("module (core: " + path + ")") if module else
                               (("tc" if "tc_causal_tile" in prof else "simt") if args.pass_ == "causal" else path),
                       "global_batch": wl.B * world, "seq_len": wl.N,
                       "parallelism": f"replicas x{world} (independent batches, no collective)",
                       "l2": l2_note,
                       "clock_window": f"{args.sustain:.1f} s sustained run of the same step, then both timed passes"},
            "clocks": clocks, "e2e": e2e, "gpu_launches": launches,
            "roofline": roofline, f"{args.pass_}_roofline": forward_roofline,
            "kernels": kern, "profiled_pass_ms_per_step": 1e3 * el_prof / args.steps,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--sustain", type=float, default=2.0, help="seconds of load before timing (clock samples)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="budget of the CPU oracle baseline")
    ap.add_argument("--ref-slices", type=int, default=1, help="(batch, head) slices per reference step")
    ap.add_argument("--pass", dest="pass_", choices=sorted(METRICS), default="forward")
    ap.add_argument("--path", default="auto", choices=["auto", "tc", "tc_fused", "simt", "fused"],
                    help="forward kernels (auto: what the library picks; tc_fused: the single persistent launch)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)      # at least three untimed warm-up steps
    wl = WORKLOADS[args.workload]
    _, world, _ = dist_env()
    if world != args.gpus and world > 1:
        print(f"warning: WORLD_SIZE={world} but --gpus {args.gpus}", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
