"""Expert parallelism on the CPU: gloo ranks (world size 2) split the experts in two contiguous
ranges, move every (token, slot) pair's activation row to its expert's owner and the outputs back
with the library's orchestration (mxfp4_mixture_experts_top_gb300.ep.ep_forward, two all-to-alls),
and each rank's layer output equals the single-rank oracle's for its tokens. The expert arithmetic is
the oracle's (test backend); the product's CUDA steps are checked on a GPU in test_gpu_ep.py."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import os, sys, json
sys.path.insert(0, os.environ["ROOT"]); sys.path.insert(0, os.path.join(os.environ["ROOT"], "tests"))
import numpy as np, torch, torch.distributed as dist
import oracle
from mxfp4_mixture_experts_top_gb300 import ep, synth
from ep_oracle_backend import OracleEPBackend
dist.init_process_group("gloo")
rank, G = dist.get_rank(), dist.get_world_size()
cfg = json.loads(os.environ["CFG"])
L = synth.make_layer(T=cfg["T"], H=cfg["H"], E=cfg["E"], k=cfg["k"], I=cfg["I"], seed=cfg["seed"])
logits = L["logits"].copy()
if cfg.get("only_first_half"):           # every token routed to the first rank's experts
    logits[:, cfg["E"] // 2:] -= 1000.0
Tr = cfg["T"] // G
tok = np.arange(rank * Tr, (rank + 1) * Tr, dtype=np.int32)
x = torch.from_numpy(L["x_bits"][tok].view(np.int16).copy()).view(torch.bfloat16)
lg = torch.from_numpy(np.ascontiguousarray(logits[tok]))
y = ep.ep_forward(x, lg, cfg["k"], OracleEPBackend(L, rank, G), group=dist.group.WORLD).numpy()
ids, w, _ = oracle.route(logits, cfg["k"])
ref = oracle.forward(L, ids, w, tokens=tok)
print(json.dumps({"rank": rank, "equal": bool(np.array_equal(y, ref)),
                  "max_abs": float(np.abs(y - ref).max()), "n": int(len(tok))}), flush=True)
dist.destroy_process_group()
"""


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _run(cfg, world=2):
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, ROOT=ROOT, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(world),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="", CFG=json.dumps(cfg))
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        o, e = p.communicate(timeout=300)
        assert p.returncode == 0, e
        outs.append(json.loads(o.strip().splitlines()[-1]))
    return outs


@pytest.mark.parametrize("cfg", [
    dict(T=24, H=256, I=128, E=8, k=3, seed=5),                         # uniform routing
    dict(T=18, H=128, I=256, E=16, k=6, seed=9),                        # every token on both ranks
    dict(T=20, H=128, I=128, E=8, k=2, seed=3, only_first_half=True),   # the second rank receives no rows
])
def test_expert_parallel_layer_equals_the_single_rank_oracle(cfg):
    res = _run(cfg)
    assert sorted(r["rank"] for r in res) == [0, 1]
    for r in res:
        assert r["equal"], r


def test_send_counts_are_the_owners_runs():
    from mxfp4_mixture_experts_top_gb300 import ep
    offsets = [0, 3, 3, 7, 12, 12, 20, 21, 25]          # E = 8
    assert ep.send_counts(offsets, 8, 2) == [12, 13]
    assert ep.send_counts(offsets, 8, 4) == [3, 9, 8, 5]
    assert ep.send_counts(offsets, 8, 1) == [25]
    with pytest.raises(ValueError):
        ep.send_counts(offsets, 8, 3)
