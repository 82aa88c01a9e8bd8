"""The N>1 path of bench.py on CPU: independent replicas, barrier, max-over-ranks
timing and rank-0-only output, with gloo ranks on 127.0.0.1 (world size 2)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


WORKER = r"""
import os, sys, json
sys.path.insert(0, os.environ["ROOT"])
import bench
world, rank, local = bench.dist_setup()
t = 1.5 if rank == 0 else 4.25          # each replica's own step time
m = bench.allreduce_max(t, world)
bench.barrier(world)
print(json.dumps({"rank": rank, "world": world, "max": m}), flush=True)
import torch.distributed as dist
dist.destroy_process_group()
"""


def _run_ranks(code, world=2, extra_env=None):
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, ROOT=ROOT, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(world),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        env.update(extra_env or {})
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        o, e = p.communicate(timeout=240)
        assert p.returncode == 0, e
        outs.append(o)
    return outs


def test_replicas_take_the_max_over_ranks():
    outs = _run_ranks(WORKER)
    res = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    assert sorted(r["rank"] for r in res) == [0, 1]
    assert all(r["world"] == 2 and r["max"] == 4.25 for r in res)


def test_reference_arm_prints_on_rank0_only():
    code = ("import os,sys; sys.path.insert(0, os.environ['ROOT']); sys.argv=['bench.py','--impl','reference',"
            "'--workload','tiny_t37_h512_e32','--steps','2','--warmup','3','--ref-tokens','2']; import bench; bench.main()")
    outs = _run_ranks(code)
    lines0 = [l for l in outs[0].splitlines() if l.startswith("{")]
    lines1 = [l for l in outs[1].splitlines() if l.startswith("{")]
    assert len(lines0) == 1 and not lines1
    d = json.loads(lines0[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["value"] > 0
