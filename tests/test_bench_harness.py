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
