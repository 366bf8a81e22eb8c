"""The bench's multi-rank plumbing on CPU: two gloo ranks as separate processes.

Replicas share no data path: the only cross-rank steps are the barriers around the timed
region and the max over ranks of the elapsed time.  These run here through the bench's own
helpers, as torchrun would launch them (RANK / WORLD_SIZE / MASTER_* in the environment,
rendezvous on 127.0.0.1)."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import json, os, sys
sys.path.insert(0, os.environ["REPO_ROOT"])
import torch.distributed as dist
import bench
rank = int(os.environ["RANK"])
dist.init_process_group("gloo")
bench._barrier(dist)
# rank r "took" 1.5 * (r + 1) ms: every rank must see the slowest one
t = bench._max_over_ranks(dist, 1.5 * (rank + 1), "cpu")
class A:
    steps, warmup, ref_step_seconds = 1, 0, 0.1
# the reference arm runs on rank 0 only; other ranks return at once without work
ref = bench.run_reference(A, 2, rank) if rank != 0 else "skipped"
bench._barrier(dist)
dist.destroy_process_group()
print(json.dumps({"rank": rank, "max_ms": t, "ref": ref}))
"""


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_two_gloo_ranks_barrier_and_max_over_ranks():
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), REPO_ROOT=ROOT, CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            o, e = p.communicate(timeout=120)
        except subprocess.TimeoutExpired:
            p.kill()
            o, e = p.communicate()
        assert p.returncode == 0, e[-2000:]
        outs.append(json.loads(o.strip().splitlines()[-1]))
    assert sorted(o["rank"] for o in outs) == [0, 1]
    for o in outs:
        assert o["max_ms"] == 3.0
    assert [o["ref"] for o in outs if o["rank"] == 1] == [None]
