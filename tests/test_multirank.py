"""The multi-GPU host path of the benchmark, on CPU with two gloo ranks.

Every rank runs an independent replica of the workload (no data exchange); the
job's rate is the units all ranks processed over the slowest rank's time, and
only rank 0 prints.  These tests run the rank arithmetic and the launch under
torchrun with the gloo backend on 127.0.0.1.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    units = 100.0 * (rank + 1)   # rank r processed 100 (r+1) tokens
    ms = 10.0 * (rank + 1)       # in 10 (r+1) ms
    res = {
        "max": bench.max_over_ranks(ms, world),
        "sum": bench.sum_over_ranks(units, world),
        "rate": bench.job_throughput(units, ms, world),
    }
    bench.barrier(world)
    out[rank] = res
    dist.destroy_process_group()


def test_rank_reductions_over_two_gloo_ranks():
    world, port = 2, free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        assert res[r]["max"] == 20.0
        assert res[r]["sum"] == 300.0
        # 300 tokens over the slowest rank's 20 ms
        assert abs(res[r]["rate"] - 15000.0) < 1e-9


def test_single_rank_reductions_are_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.sum_over_ranks(7.0, 1) == 7.0
    assert bench.job_throughput(50.0, 10.0, 1) == 5000.0


def test_reference_arm_under_torchrun_prints_once():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "1", "--cpu-seconds", "0.25"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle"


@pytest.mark.parametrize("workload", ["decode", "shared", "lmhead"])
def test_reference_arm_json_line_keeps_the_contract(workload):
    """One rank, the oracle arm: one JSON line with the contract's keys, the workload's
    name and routing, a bounded oracle sample and a zero-copy e2e record."""
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--workload", workload, "--steps", "1",
           "--warmup", "1", "--cpu-seconds", "0.25"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in rec, key
    assert rec["impl"] == "reference" and rec["unit"] == "tokens/s" and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] >= 1
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["e2e"]["value"] == rec["value"]
    cfg = rec["config"]
    if workload == "shared":
        assert cfg["workload"] == "moe_layer_shared_decode_batch1" and cfg["top_k"] == 6 and cfg["n_shared"] == 1
    elif workload == "lmhead":
        assert cfg["workload"] == "lmhead_V131072_T1" and cfg["V"] == 131072
    else:
        assert cfg["workload"] == "moe_layer_decode_batch1" and cfg["top_k"] == 8 and cfg["n_shared"] == 0


def test_clock_summary_counts_only_samples_under_load():
    """The clocks record: median SM clock over samples drawing well above idle power,
    and every throttle reason seen in any sample."""
    sys.path.insert(0, ROOT)
    import bench
    cs = bench.ClockSampler(0)
    idle = "0, 1100, 2032, 200.0, 0x0, Not Active, Not Active, Not Active, Not Active"
    busy = "0, {}, 2032, 900.0, 0x0, Not Active, Not Active, Not Active, {}"
    cs.lines = [idle, busy.format(2032, "Not Active"), busy.format(1990, "Active"), busy.format(2032, "Not Active"),
                idle, "garbage"]
    s = cs.summary()
    assert s["sm_mhz"] == 2032 and s["sm_max_mhz"] == 2032 and s["samples"] == 5
    assert s["samples_under_load"] == 3 and s["reasons"] == ["sw_power_cap"]


def test_timing_record_reports_the_median_region():
    sys.path.insert(0, ROOT)
    import bench
    rec = bench.timing_record([3.0, 1.0, 2.0, 2.5, 100.0], 20, "x")
    assert rec["regions"] == 5 and rec["steps_per_region"] == 20
    assert rec["region_ms"] == {"min": 1.0, "median": 2.5, "max": 100.0}
    assert bench.n_region_graphs(20, 64) == 4 and bench.n_region_graphs(2000, 64) == 1
    assert bench.n_region_graphs(1, 64) == 16
