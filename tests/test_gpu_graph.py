"""A whole layer step captured in one CUDA graph.

The step is route+permute, then the forward's gather, W13, W2 and combine.
Inside the graph the kernels stay chained by programmatic dependent launch.
Replaying the graph on inputs written into the captured buffers after capture
must give bit-identical results to the eager calls on the same inputs (the
layer is deterministic), and no device error.
"""
import numpy as np
import pytest
import torch

from mxfp4_mixture_experts_top_gb300 import synth

pytestmark = pytest.mark.gpu


def _layer(moe, gpu_layers, L, flags=0):
    T, H, I, E, k = L["T"], L["H"], L["I"], L["E"], L["k"]
    desc = moe.make_desc(T, H, I, E, k, 16, 0.0, flags)
    ws = torch.empty(max(moe.workspace_bytes(desc), 1024), dtype=torch.uint8, device="cuda")
    cap = moe.rows_capacity(T, E, k, 16)
    dev = torch.device("cuda")
    bufs = dict(ids=torch.empty((T, k), dtype=torch.int32, device=dev),
                w=torch.empty((T, k), dtype=torch.float32, device=dev),
                bm=torch.empty((T, (E + 31) // 32), dtype=torch.int32, device=dev),
                perm=dict(counts=torch.empty(E, dtype=torch.int32, device=dev),
                          offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                          padded_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                          row_to_pair=torch.empty(max(cap, 1), dtype=torch.int32, device=dev),
                          pair_to_row=torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)),
                perm_err=torch.zeros(4, dtype=torch.int32, device=dev),
                y=torch.empty((T, H), dtype=torch.float32, device=dev))
    return moe.MoELayer(desc, gpu_layers.packed(L), ws, bufs)


@pytest.mark.parametrize("name,flags", [
    ("tiny_t37_h512_e32", 0),
    ("decode_t8_h4096_e256", 0),         # the fused decode GEMMs
    ("decode_t8_h4096_e256", 1),         # the same with the atomic combine (y zeroed by the gather)
    ("stacked_t300", 0),                 # two-pass gather, stacked token tiles (28 rows per expert)
])
def test_graph_replay_matches_eager(gpu_lib, gpu_layers, name, flags):
    moe = gpu_lib
    L = (synth.make_layer(T=300, H=256, E=64, k=6, I=128, seed=300) if name == "stacked_t300"
         else synth.make_config(name))
    layer = _layer(moe, gpu_layers, L, flags)
    x0, lg0 = gpu_layers.inputs(L)
    x, logits = x0.clone(), lg0.clone()
    graph, y_graph = layer.capture_graph(x, logits)

    # other inputs of the same shapes, written into the captured buffers after capture
    rng = np.random.default_rng(7)
    perm_rows = torch.from_numpy(rng.permutation(L["T"])).to("cuda")
    for xin, lgin in ((x0, lg0), (x0[perm_rows].contiguous(), lg0[perm_rows].flip(1).contiguous())):
        x.copy_(xin)
        logits.copy_(lgin)
        graph.replay()
        torch.cuda.synchronize()
        got = y_graph.clone()
        ids_graph = layer.bufs["ids"].clone()
        assert layer.forward_error() == 0
        y_eager = layer(xin, lgin).clone()
        torch.cuda.synchronize()
        assert layer.forward_error() == 0
        assert torch.equal(layer.bufs["ids"], ids_graph)
        if flags & moe.FLAG_FAST_COMBINE:    # the atomic combine's add order varies from run to run
            assert (got - y_eager).abs().max().item() <= 1e-5 * y_eager.abs().max().item(), name
        else:
            assert torch.equal(got, y_eager), f"{name}: graph replay differs from the eager step"
