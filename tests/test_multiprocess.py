"""The multi-rank host path of bench.py on the CPU (gloo, world size 2): each rank runs
its own replica (independent problems, different seeds), the job time is the slowest
rank's, the throughput counts every rank's work, and under torchrun the reference arm
runs on rank 0 only and prints one line. No GPU: the data path has no collective, so the
only multi-rank logic is this host logic."""
from __future__ import annotations

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


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    import seeded_inputs as si
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = bench.replica(si.WORKLOADS["tiny"], rank)
    # each rank "measured" a different time; the job takes the slowest one's
    t = bench.max_over_ranks(1.0 + rank * 0.5)
    res = {"rank": rank, "seed": w.seed, "max_time": t, "q_head": [int(v) for v in si.make_inputs(w)["q"].ravel()[:16]],
           "value": bench.whole_job_tflops(1e12, 10, dist.get_world_size(), t)}
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(res, f)
    dist.barrier()
    dist.destroy_process_group()


def test_gloo_two_ranks_replicas_and_max_time(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    r = [json.load(open(tmp_path / f"rank{i}.json")) for i in range(world)]
    assert r[0]["seed"] != r[1]["seed"], "replicas must be independent problems"
    assert r[0]["q_head"] != r[1]["q_head"], "the replicas' inputs must differ"
    assert r[0]["max_time"] == r[1]["max_time"] == 1.5  # the slowest rank's time on every rank
    # every rank's work over the slowest time: 2 ranks x 10 steps x 1 TFLOP / 1.5 s
    assert abs(r[0]["value"] - 2 * 10 / 1.5) < 1e-9 and r[0]["value"] == r[1]["value"]


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.whole_job_tflops(2e12, 5, 1, 2.0) == 5.0


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    """`torchrun --nproc-per-node 2 bench.py --impl reference`: rank 0 runs the oracle on
    its bounded sample and prints the line; rank 1 exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--workload", "tiny"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=240, cwd=ROOT,
                       env=dict(os.environ, OMP_NUM_THREADS="1"))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


if __name__ == "__main__":
    pytest.main([__file__, "-q"])
