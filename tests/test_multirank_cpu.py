"""The multi-rank path of bench.py on CPU (gloo, world size 2): each rank runs
an independent replica, the ranks meet at barriers around the timed region,
and rank 0 reports the maximum over ranks.  Also the reference arm under
torchrun: rank 0 alone runs the oracle and prints the line."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update({"WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, _ = bench._dist()
    assert (r, w) == (rank, world)
    assert dist.get_backend() == "gloo"
    bench._barrier(w)
    out[rank] = bench._max_over_ranks(1.5 + rank, w)
    bench._barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_over_ranks():
    world, port = 2, _free_port()
    out = mp.get_context("spawn").Manager().dict()   # no fork of a threaded test process
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_reference_arm_prints_one_line_from_rank_0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--workload", "tiny_b2_q1_h16kv1_2k3k", "--steps", "1", "--warmup", "0",
           "--gpus", "2"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
