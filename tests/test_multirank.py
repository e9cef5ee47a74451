"""World-size-2 runs of the bench's host-side rank logic on CPU (gloo):
barrier, max-over-ranks timing, summed work, and the reference arm printing
on rank 0 only.  The workload shards as independent replicas, so there is no
data-path collective to test."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import bench
args = bench.parse()
world, rank, local = bench.dist_setup(args)
bench.barrier(world)
mx = bench.max_over_ranks(world, 10.0 * (rank + 1))
sm = bench.sum_over_ranks(world, 3.0 + rank)
print(json.dumps({{"rank": rank, "world": world, "max": mx, "sum": sm}}), flush=True)
import torch.distributed as dist
dist.destroy_process_group()
"""


def launch(code, extra_env=None, args=()):
    port = free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        env.update(extra_env or {})
        procs.append(subprocess.Popen([sys.executable, "-c", code, *args], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                      text=True, cwd=ROOT))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=300)
        assert p.returncode == 0, err
        outs.append(out)
    return outs


def test_rank_reductions_world2():
    outs = launch(WORKER.format(root=ROOT))
    rows = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    for r in rows:
        assert r["world"] == 2 and r["max"] == 20.0 and r["sum"] == 7.0


def test_reference_arm_prints_on_rank0_only():
    code = f"import sys; sys.path.insert(0, {ROOT!r}); sys.argv=['bench.py']+sys.argv[1:]; import bench; bench.main()"
    outs = launch(code, args=("--impl", "reference", "--steps", "1", "--warmup", "0"))
    lines0 = [l for l in outs[0].splitlines() if l.startswith("{")]
    lines1 = [l for l in outs[1].splitlines() if l.startswith("{")]
    assert len(lines0) == 1 and lines1 == []
    rec = json.loads(lines0[0])
    assert rec["impl"] == "reference" and rec["value"] > 0 and rec["n_gpus"] == 2
