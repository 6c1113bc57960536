"""The benchmark's multi-rank harness on CPU (gloo, world size 2).

Replica ranks exchange nothing but the timing barrier and one max-reduction of
their elapsed times; the whole-job throughput divides every rank's units by the
slowest rank's time.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r, w = bench.dist_init("gloo")
    bench.barrier()
    elapsed = 1.0 + rank            # rank 1 is the slow one
    m = bench.max_over_ranks(elapsed)
    out[rank] = (r, w, m, bench.whole_job_throughput(1000, w, 10, m))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_max_reduction_and_throughput():
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
    assert out[0] == (0, 2, 2.0, 1000 * 2 * 10 / 2.0)
    assert out[1] == (1, 2, 2.0, 1000 * 2 * 10 / 2.0)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_throughput(262144, 1, 200, 0.04) == pytest.approx(262144 * 200 / 0.04)


def test_clock_summary_flags_throttling():
    rows = [["t", "1800", "2070", "900", "0x0", "Not Active", "Not Active", "Not Active", "Active"],
            ["t", "1900", "2070", "950", "0x0", "Not Active", "Active", "Not Active", "Not Active"],
            ["t", "2000", "2070", "1000", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"]]
    s = bench.summarize_clocks(rows)
    assert s["sm_mhz"] == 1900 and s["sm_max_mhz"] == 2070 and s["samples"] == 3
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


@pytest.mark.parametrize("pass_", ["forward", "backward", "causal", "module"])
def test_reference_arm_prints_one_contract_line(pass_):
    """`--impl reference` times the oracle on the host alone and prints one JSON
    line with the keys the benchmark contract names."""
    import json
    import subprocess
    import sys
    wl = "lm_causal_4096" if pass_ == "causal" else "tiny_16x16_fp32"
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--pass", pass_,
                        "--workload", wl, "--steps", "2", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 3
    assert line["value"] > 0 and line["unit"] == "tokens/s" and line["config"]["workload"] == wl
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_rotation_keeps_small_steps_out_of_l2():
    import torch

    l2 = 1000
    # a step that alone moves more than 1.5x L2: one set, the tensors themselves
    big = [torch.zeros(2000, dtype=torch.uint8)]
    sets, nbytes = bench.rotation(big, l2)
    assert len(sets) == 1 and sets[0][0] is big[0] and nbytes == 2000
    # a small step: enough copies that a set is touched again only after > 1.5x L2
    q, o = torch.arange(50, dtype=torch.int32), torch.zeros(50, dtype=torch.int32)   # 400 bytes a step
    sets, nbytes = bench.rotation([q, o], l2)
    assert nbytes == 400
    assert (len(sets) - 1) * nbytes > 1.5 * l2
    assert sets[0][0] is q
    for s in sets[1:]:
        assert torch.equal(s[0], q) and s[0].data_ptr() != q.data_ptr() and s[1].data_ptr() != o.data_ptr()
    # never more than the cap
    sets, _ = bench.rotation([torch.zeros(1, dtype=torch.uint8)], l2)
    assert len(sets) == bench.ROTATE_CAP
