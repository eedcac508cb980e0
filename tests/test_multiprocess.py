"""The multi-rank path of bench.py on CPU (gloo, world size 2).

On the GPU machine every rank runs an independent replica of the workload: the
only cross-rank steps are the barriers and the max over ranks of the timed
region, and rank 0 alone prints the line.  These tests run those steps with
two CPU processes, and the reference arm under torchrun, where rank 0 alone
works and prints.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        own = [0.25, 0.75][rank]   # seconds this rank's timed region took
        total = bench.max_over_ranks(own, world, torch.device("cpu"))
        out[rank] = (total, bench.whole_job_tflops(world, 2.0e12, 4, total))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_with_two_gloo_ranks():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
        got = dict(out)
    # both ranks see the slowest rank's time; the value counts both replicas
    assert got[0] == got[1] == (0.75, world * 2.0e12 * 4 / 0.75 / 1e12)


def test_reference_arm_under_torchrun_prints_once_from_rank_zero():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1", "--workload", "small_full_s256_d64"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
