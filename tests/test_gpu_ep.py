"""Expert parallelism on the GPU: the dispatch pack and the combine kernels against their
definitions, and the whole expert-parallel layer (routing, pack, the rank's expert GEMMs, combine)
against the oracle: with one rank, and with two ranks emulated in one process on one GPU (the
all-to-alls replaced by slicing the same buffers, nothing waits on another kernel)."""
import numpy as np
import pytest
import torch

import oracle
from mxfp4_mixture_experts_top_gb300 import ep, synth

pytestmark = pytest.mark.gpu

TOL = 2e-2


def _close(name, y, ref):
    rms = np.sqrt(np.mean(ref ** 2))
    err = np.abs(y.astype(np.float64) - ref).max()
    print(f"[{name}] max|gpu-oracle|/rms = {err / rms:.3e}")
    assert err <= TOL * rms


def _layer(T=40, H=256, I=128, E=8, k=3, seed=21):
    return synth.make_layer(T=T, H=H, E=E, k=k, I=I, seed=seed)


def _dev(L):
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    x = up(L["x_bits"].view(np.int16)).view(torch.bfloat16)
    return x, up(L["logits"]), [up(L[n]) for n in ("w13_q", "w13_s", "w2_q", "w2_s")]


def test_pack_and_combine_match_their_definitions(gpu_lib):
    moe = gpu_lib
    L = _layer()
    x, logits, _ = _dev(L)
    T, H, E, k, epr = L["T"], L["H"], L["E"], L["k"], 4
    ids, w, _, perm = moe.route_permute(logits, k, 16)
    send_x, send_ids = moe.ep_dispatch_pack(x, perm, k, epr)
    torch.cuda.synchronize()
    ids_np = ids.cpu().numpy()
    c, pad, r2p = (perm[n].cpu().numpy() for n in ("counts", "padded_offsets", "row_to_pair"))
    order = np.concatenate([r2p[pad[e]:pad[e] + c[e]] for e in range(E)])
    assert np.array_equal(send_x.view(torch.int16).cpu().numpy(), L["x_bits"].view(np.int16)[order // k])
    assert np.array_equal(send_ids.cpu().numpy()[:T * k], (np.repeat(np.arange(E), c) % epr).astype(np.int32))
    # combine of an arbitrary returned buffer: the slot-ordered weighted sum of each pair's row
    ret = torch.randn(T * k, H, device="cuda")
    y = moe.ep_combine(ret, ids, w, perm)
    torch.cuda.synchronize()
    off, p2r = perm["offsets"].cpu().numpy(), perm["pair_to_row"].cpu().numpy()
    r, wn = ret.cpu().numpy().astype(np.float64), w.cpu().numpy().astype(np.float64)
    pos = off[ids_np.ravel()] + p2r - pad[ids_np.ravel()]
    want = np.einsum("tj,tjh->th", wn, r[pos].reshape(T, k, H))
    assert np.abs(y.cpu().numpy() - want).max() <= 1e-5 * np.abs(want).max()


def test_expert_parallel_layer_one_rank(gpu_lib):
    L = _layer()
    x, logits, wts = _dev(L)
    be = ep.CudaEPBackend.create(0, 1, L["H"], L["I"], L["E"], *wts)
    y = ep.ep_forward(x, logits, L["k"], be).cpu().numpy()
    ids, w, _ = oracle.route(L["logits"], L["k"])
    _close("ep one rank", y, oracle.forward(L, ids, w))


@pytest.mark.parametrize("T,H,I,E,k", [(40, 256, 128, 8, 3), (300, 512, 256, 32, 6)])
def test_expert_parallel_layer_two_ranks_in_one_process(gpu_lib, T, H, I, E, k):
    moe = gpu_lib
    L = _layer(T=T, H=H, I=I, E=E, k=k, seed=T + E)
    x, logits, wts = _dev(L)
    G, epr, half = 2, E // 2, T // 2
    be = [ep.CudaEPBackend.create(r, G, H, I, E, *wts) for r in range(G)]
    toks = [slice(0, half), slice(half, T)]
    st = []                                  # per sender: ids, w, perm, send buffers, runs
    for r in range(G):
        ids, w, perm = be[r].route_permute(logits[toks[r]].contiguous(), k)
        sx, sids = be[r].pack(x[toks[r]].contiguous(), perm, k, epr)
        runs = ep.send_counts(perm["offsets"].cpu().tolist(), E, G)
        st.append((ids, w, perm, sx, sids, np.concatenate([[0], np.cumsum(runs)])))
    outs = []
    for g in range(G):                       # receiver g: the runs for its experts, in sender order
        rx = torch.cat([s[3][s[5][g]:s[5][g + 1]] for s in st])
        rids = torch.cat([s[4][s[5][g]:s[5][g + 1]] for s in st])
        outs.append(be[g].local_forward(rx, rids))
    ys = []
    for r in range(G):                       # sender r gets its pairs' outputs back in send order
        parts, cut = [], 0
        for g in range(G):
            before = sum(int(st[q][5][g + 1] - st[q][5][g]) for q in range(r))
            n = int(st[r][5][g + 1] - st[r][5][g])
            parts.append(outs[g][before:before + n])
        ret = torch.cat(parts)
        ys.append(be[r].combine(ret, st[r][0], st[r][1], st[r][2]))
    y = torch.cat(ys).cpu().numpy()
    ids, w, _ = oracle.route(L["logits"], k)
    _close(f"ep two ranks T{T} E{E}", y, oracle.forward(L, ids, w))
