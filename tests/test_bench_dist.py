"""The multi-rank path of bench.py on CPU: two gloo ranks (one process each)
rendezvous, pass the barrier, take the maximum over ranks of a per-rank time,
and only rank 0 of the reference arm does any work or prints."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import json, os, sys
sys.path.insert(0, os.environ["QMM_TEST_ROOT"])
import bench
world, rank, local = bench.setup_dist(2)
t = bench.max_over_ranks(world, 1.5 + rank, "cpu")
bench.barrier(world)

class A:
    steps, warmup, gpus = 1, 3, 2
if rank != 0:
    bench.run_reference(A(), world, rank)      # ranks other than 0 return at once, printing nothing
import torch.distributed as dist
dist.destroy_process_group()
print(json.dumps({"rank": rank, "world": world, "local": local, "max": t}))
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_barrier_and_max_over_ranks():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2",
                   LOCAL_RANK=str(rank), QMM_BENCH_BACKEND="gloo", QMM_TEST_ROOT=ROOT)
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER], env=env, cwd=ROOT, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=180)
        assert p.returncode == 0, err[-2000:]
        lines = [ln for ln in out.strip().splitlines() if ln.startswith("{")]
        assert len(lines) == 1, out
        outs.append(json.loads(lines[0]))
    outs.sort(key=lambda d: d["rank"])
    assert [d["rank"] for d in outs] == [0, 1]
    assert all(d["world"] == 2 and d["max"] == 2.5 for d in outs)
    assert [d["local"] for d in outs] == [0, 1]
