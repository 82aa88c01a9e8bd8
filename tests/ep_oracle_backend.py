"""Test backend for the expert-parallel orchestration: the same steps as the CUDA backend, each
computed by the float64 oracle or written out with numpy from its definition. Test infrastructure
only (it imports the oracle); the product backend is mxfp4_mixture_experts_top_gb300.ep.CudaEPBackend."""
import numpy as np
import torch

import oracle


class OracleEPBackend:
    collective_device = "cpu"

    def __init__(self, L, rank, G, block_m=16):
        self.L, self.block_m = L, block_m
        self.E = L["E"]
        self.epr = self.E // G
        self.lo = rank * self.epr

    def route_permute(self, logits, k):
        ids, w, _ = oracle.route(logits.numpy(), k)
        perm = oracle.permute(ids, self.E, self.block_m)
        return torch.from_numpy(ids), torch.from_numpy(w), perm

    @staticmethod
    def offsets_on_host(perm):
        return perm["offsets"].tolist()

    def pack(self, x, perm, k, epr):
        """Pairs in (expert, token) order: the real rows of each expert's segment of the permutation."""
        c, pad, r2p = perm["counts"], perm["padded_offsets"], perm["row_to_pair"]
        order = np.concatenate([r2p[pad[e]:pad[e] + c[e]] for e in range(self.E)]).astype(np.int64)
        experts = np.repeat(np.arange(self.E), c)
        send_x = x[torch.from_numpy(order // k)]
        return send_x, torch.from_numpy((experts % epr).astype(np.int32))

    def local_forward(self, recv_x, recv_ids):
        """Per-row expert outputs: the oracle's layer with k = 1 and weight 1 over this rank's experts."""
        L, lo, n = self.L, self.lo, recv_x.shape[0]
        sl = slice(lo, lo + self.epr)
        layer = dict(T=n, H=L["H"], I=L["I"], E=self.epr, k=1,
                     x_bits=recv_x.view(torch.int16).numpy().view(np.uint16),
                     w13_q=np.ascontiguousarray(L["w13_q"][sl]), w13_s=np.ascontiguousarray(L["w13_s"][sl]),
                     w2_q=np.ascontiguousarray(L["w2_q"][sl]), w2_s=np.ascontiguousarray(L["w2_s"][sl]))
        if n == 0:
            return torch.zeros((0, L["H"]), dtype=torch.float64)
        y = oracle.forward(layer, recv_ids.numpy().reshape(n, 1), np.ones((n, 1)))
        return torch.from_numpy(y)

    def combine(self, returned, ids, w, perm):
        """y[t] = sum_j w[t, j] * returned[send position of pair (t, j)], slots ascending, float64."""
        ret = returned.numpy()
        ids, w = ids.numpy(), w.numpy()
        T, k = ids.shape
        off, pad, p2r = perm["offsets"], perm["padded_offsets"], perm["pair_to_row"]
        y = np.zeros((T, ret.shape[1]))
        for t in range(T):
            acc = np.zeros(ret.shape[1])
            for j in range(k):
                p = t * k + j
                e = ids[t, j]
                acc = acc + w[t, j] * ret[off[e] + p2r[p] - pad[e]]
            y[t] = acc
        return torch.from_numpy(y)
