"""Expert parallelism of the MXFP4 MoE layer over the ranks of a torch.distributed group.

Host orchestration: experts are split in contiguous ranges, rank g owning experts
[g*EPR, (g+1)*EPR) with EPR = E / G. Each rank

1. routes and permutes its own tokens over all E experts,
2. packs the activation row of every (token, slot) pair in (expert, token) order,
   so the rows for rank g form one contiguous run (``moe_ep_dispatch_pack``),
3. sends the runs to their owners and receives the rows routed to its own experts
   (one all-to-all), runs the grouped expert GEMMs on them with k = 1 and weight 1
   (the per-pair expert outputs), and sends the outputs back in the order received
   (one all-to-all),
4. combines its pairs' outputs in slot order (``moe_ep_combine``), which is the
   single-GPU combine.

The layer is the one of "DeepSeek V4 Flash 单卡 MI300X" (txtmix.com) §一 and §三;
the pages run it on one GPU and do not shard it.

The arithmetic of every step runs in a backend: ``CudaEPBackend`` calls the CUDA
library only (routing, permutation, pack, GEMMs and combine are its kernels); the
host code here moves the counts and runs the two all-to-alls. A group of one rank
skips the collectives.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import moe


def send_counts(offsets, E: int, G: int):
    """Rows this rank sends to each rank: the (expert, token)-ordered pairs of rank g's experts are the
    run offsets[g*EPR] .. offsets[(g+1)*EPR]."""
    if E % G:
        raise ValueError(f"{E} experts do not split evenly over {G} ranks")
    epr = E // G
    return [int(offsets[(g + 1) * epr]) - int(offsets[g * epr]) for g in range(G)]


def _all_to_all(out: torch.Tensor, inp: torch.Tensor, out_splits, in_splits, group):
    """all_to_all_single along dim 0; bf16 rows travel as int32 pairs (gloo moves neither bf16 nor int16)."""
    import torch.distributed as dist
    if inp.dtype == torch.bfloat16:
        out, inp = out.view(torch.int32), inp.view(torch.int32)
    dist.all_to_all_single(out, inp, output_split_sizes=list(out_splits), input_split_sizes=list(in_splits),
                           group=group)


def ep_forward(x: torch.Tensor, logits: torch.Tensor, k: int, backend, group=None) -> torch.Tensor:
    """The layer output of this rank's tokens with the experts spread over the group's ranks.

    x: [T, H] bf16, logits: [T, E] fp32 (this rank's tokens), on the backend's device. Returns y
    [T, H] fp32. With `group` None (or of size 1) every expert is local and nothing is exchanged."""
    import torch.distributed as dist
    G = 1 if group is None else dist.get_world_size(group)
    T, H = x.shape
    E = logits.shape[1]
    ids, w, perm = backend.route_permute(logits, k)
    send = send_counts(backend.offsets_on_host(perm), E, G)
    send_x, send_ids = backend.pack(x, perm, k, E // G)
    if G == 1:
        recv_x, recv_ids, recv = send_x, send_ids, send
    else:
        dev = backend.collective_device
        sc = torch.tensor(send, dtype=torch.int64, device=dev)
        rc = torch.empty(G, dtype=torch.int64, device=dev)
        dist.all_to_all_single(rc, sc, group=group)
        recv = [int(v) for v in rc.tolist()]
        recv_x = torch.empty((sum(recv), H), dtype=send_x.dtype, device=send_x.device)
        recv_ids = torch.empty(max(sum(recv), 1), dtype=torch.int32, device=send_x.device)
        _all_to_all(recv_x, send_x[:sum(send)], recv, send, group)
        _all_to_all(recv_ids[:sum(recv)], send_ids[:sum(send)], recv, send, group)
    out = backend.local_forward(recv_x[:sum(recv)], recv_ids[:sum(recv)])
    if G == 1:
        returned = out
    else:
        returned = torch.empty((T * k, H), dtype=out.dtype, device=out.device)
        _all_to_all(returned, out, send, recv, group)
    return backend.combine(returned, ids, w, perm)


@dataclass
class CudaEPBackend:
    """The rank's share of one layer on its GPU: prepacked weights of its EPR experts. Every step
    calls the CUDA library (no arithmetic on the host)."""

    H: int
    I: int
    E: int
    epr: int
    packed_local: torch.Tensor
    block_m: int = 16
    collective_device: str = "cuda"

    @classmethod
    def create(cls, rank: int, G: int, H: int, I: int, E: int, w13_q, w13_s, w2_q, w2_s, block_m: int = 16,
               collective_device: str = "cuda"):
        """w13_q ... w2_s: the canonical MXFP4 weights of all E experts (device tensors); the rank
        prepacks its own range [rank*E/G, (rank+1)*E/G)."""
        epr = E // G
        lo, hi = rank * epr, (rank + 1) * epr
        desc = moe.make_desc(1, H, I, epr, 1, block_m)
        packed = moe.prepack(desc, w13_q[lo:hi].contiguous(), w13_s[lo:hi].contiguous(), w2_q[lo:hi].contiguous(),
                             w2_s[lo:hi].contiguous())
        return cls(H, I, E, epr, packed, block_m, collective_device)

    def route_permute(self, logits, k):
        ids, w, _, perm = moe.route_permute(logits, k, self.block_m)
        return ids, w, perm

    @staticmethod
    def offsets_on_host(perm):
        return perm["offsets"].cpu().tolist()

    @staticmethod
    def pack(x, perm, k, epr):
        return moe.ep_dispatch_pack(x, perm, k, epr)

    def local_forward(self, recv_x, recv_ids):
        """Expert outputs of the received rows: the layer with k = 1 and weight 1 over the local experts."""
        n = recv_x.shape[0]
        if n == 0:
            return torch.empty((0, self.H), dtype=torch.float32, device=recv_x.device)
        ids = recv_ids.view(n, 1)
        perm = moe.permute(ids, self.epr, self.block_m)
        desc = moe.make_desc(n, self.H, self.I, self.epr, 1, self.block_m)
        ws = torch.empty(moe.workspace_bytes(desc), dtype=torch.uint8, device=recv_x.device)
        ones = torch.ones((n, 1), dtype=torch.float32, device=recv_x.device)
        return moe.forward(desc, recv_x.contiguous(), self.packed_local, ones, perm, ws)

    @staticmethod
    def combine(returned, ids, w, perm):
        return moe.ep_combine(returned.contiguous(), ids, w, perm)
