"""Host logic of bench.py's N-replica path on CPU: two gloo ranks (127.0.0.1), the max over
ranks of the timed region and the job-wide time per step; the reference arm runs on rank 0 only."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, ms_by_rank, steps, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        res = bench.job_timing(ms_by_rank[rank], steps, world, dist, "cpu")
        dist.barrier()
        out[rank] = res
    finally:
        dist.destroy_process_group()


def test_job_timing_two_gloo_ranks():
    world, steps = 2, 4
    ms_by_rank = [10.0, 14.0]
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), ms_by_rank, steps, out), nprocs=world,
                           join=True, start_method="spawn")
        res = dict(out)
    # every rank sees the slowest rank's time; 2 replicas finish 2 * 4 steps in 14 ms
    assert res[0] == res[1] == (14.0, 3.5, 1.75)


def test_job_timing_single_rank():
    assert bench.job_timing(12.0, 4, 1) == (12.0, 3.0, 3.0)


def test_reference_arm_other_ranks_do_no_work(capsys):
    class A:
        steps, warmup = 1, 0

    bench.run_reference(A(), rank=1)
    assert capsys.readouterr().out == ""


def test_reference_arm_json_contract():
    # the oracle arm prints one JSON line with the step metric, its own cpu_baseline and an e2e
    # entry without host copies (a bounded sample: 2 of 32 layers, scaled)
    import json
    import subprocess

    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "ms/step"
    assert d["higher_is_better"] is False and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "ms/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == bench.WORKLOAD
