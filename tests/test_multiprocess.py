"""The multi-rank path of bench.py on the CPU (gloo, world size 2).

The path shards only as independent replicas: every rank runs its own step on
its own GPU with no collective on the data path.  What crosses ranks is the
timing: a barrier before the timed region and the max of the per-rank step times
after it, from which the whole-job (weak-scaling) throughput is computed.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        bench.barrier()
        local_step_s = 0.010 * (rank + 1)            # rank 1 is the slower replica
        slowest = bench.max_over_ranks(local_step_s)
        value = bench.job_throughput(1000.0, world, slowest)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"slowest": slowest, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_replica_timing_aggregates_over_gloo_ranks(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r in res:
        assert r["slowest"] == pytest.approx(0.020)           # max over ranks, on every rank
        assert r["value"] == pytest.approx(2 * 1000.0 / 0.020)  # all units / slowest time


def test_single_process_helpers_are_identities():
    sys.path.insert(0, ROOT)
    import bench
    bench.barrier()
    assert bench.max_over_ranks(0.25) == 0.25
    assert bench.job_throughput(10.0, 1, 2.0) == 5.0


def test_reference_arm_prints_on_rank0_only():
    """Under a 2-rank launch only rank 0 runs the reference arm and prints one line."""
    outs = []
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()), OMP_NUM_THREADS="2")
        procs.append(subprocess.Popen(
            [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
             "--steps", "1", "--warmup", "3", "--config", "tiny_decode"],
            cwd=ROOT, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    for p in procs:
        out, err = p.communicate(timeout=600)
        assert p.returncode == 0, err
        outs.append([l for l in out.splitlines() if l.strip()])
    assert outs[1] == []
    assert len(outs[0]) == 1
    line = json.loads(outs[0][0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle"
