"""bench.py's multi-rank host logic on the CPU (gloo, world size 2).

Each rank of a multi-GPU bench run is an independent replica of the MSM; the
job's time is the slowest rank's, the units are all ranks' together, and only
rank 0 prints.  These tests run that logic as two gloo processes.
"""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, values, out_dir):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        if ROOT not in sys.path:
            sys.path.insert(0, ROOT)
        import bench
        got = bench.max_over_ranks(values[rank], world)
        with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as f:
            json.dump(got, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_single_process_is_identity():
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    values = [1.5, 7.25]  # rank 1 is the slow one
    mp.start_processes(_rank_main, args=(2, _free_port(), values, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for rank in range(2):
        with open(tmp_path / ("rank%d.json" % rank)) as f:
            assert json.load(f) == max(values)


def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    lines = [line for line in r.stdout.splitlines() if line.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["value"] == d["value"] and d["cpu_baseline"]["kind"] == "oracle"
