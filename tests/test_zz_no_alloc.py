"""moe_mxfp4_forward_noalloc: the forward for callers that cannot allocate
device memory where they run the layer (allocation-free runtimes, plugins
whose host owns all device memory). It uses the library's static scratch
array instead of a workspace; its output must match moe_mxfp4_forward.

Kept in a file of its own, collected last, so that a run stopping at the first
failure has already run every other test. Passes alone in a fresh process
and after the other tests (the scratch array then holds stale contents from
earlier calls, which the entry point must not depend on).
"""
import ctypes

import numpy as np
import pytest
import torch

from mxfp4_mixture_experts_top_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = 2e-2   # the layer tolerance used by every parity test: max err <= TOL * rms


def _prepare(moe, L, block_m=16):
    dev = torch.device("cuda")
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    T, H, I, E, k = L["T"], L["H"], L["I"], L["E"], L["k"]
    desc = moe.make_desc(T, H, I, E, k, block_m)
    packed = moe.prepack(desc, up(L["w13_q"]), up(L["w13_s"]), up(L["w2_q"]), up(L["w2_s"]))
    x = up(L["x_bits"].view(np.int16)).view(torch.bfloat16)
    ids, w, _ = moe.route(up(L["logits"]), k)
    perm = moe.permute(ids, E, block_m)
    return desc, packed, x, w, perm


def _close(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    rms = np.sqrt(np.mean(b ** 2))
    return np.abs(a - b).max() <= TOL * rms


@pytest.mark.parametrize("T,H,I,E,k", [(37, 512, 256, 32, 6), (8, 4096, 2048, 32, 6)])
def test_noalloc_matches_forward_on_two_calls_in_a_row(gpu_lib, T, H, I, E, k):
    moe = gpu_lib
    L = synth.make_layer(T=T, H=H, E=E, k=k, I=I, seed=3)
    desc, packed, x, w, perm = _prepare(moe, L)
    ws = torch.empty(moe.workspace_bytes(desc), dtype=torch.uint8, device="cuda")
    ref = moe.forward(desc, x, packed, w, perm, ws)

    # first call: through the C ABI, the library supplies the scratch
    y1 = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    moe.forward_noalloc(desc, x, packed, w, perm, y=y1)
    # second call right after, on different activations (same routing): the
    # scratch now holds the first call's intermediates
    x2 = (x.float() * -0.5).to(torch.bfloat16)
    ref2 = moe.forward(desc, x2, packed, w, perm, ws)
    y2 = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    moe.forward_noalloc(desc, x2, packed, w, perm, y=y2)
    torch.cuda.synchronize()
    assert torch.isfinite(y1).all() and torch.isfinite(y2).all()
    assert _close(y1, ref) and _close(y2, ref2)


def test_noalloc_rejects_layers_larger_than_its_scratch(gpu_lib):
    moe = gpu_lib
    desc = moe.make_desc(2048, 4096, 2048, 256, 6, 16)
    assert moe.workspace_bytes(desc) > moe.NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 20)     # never dereferenced: the size check fails first
    rc = moe.load().moe_mxfp4_forward_noalloc(ctypes.byref(desc), fake, fake, fake, fake, fake, fake, fake, None)
    assert rc == 4   # MOE_ERR_WORKSPACE
