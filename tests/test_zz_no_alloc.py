"""moe_mxfp4_forward_noalloc: the forward for callers that cannot allocate
device memory where they run the layer (allocation-free runtimes, plugins
whose host owns all device memory). It uses the library's static scratch
array instead of a workspace, runs the same kernels, and so must return
exactly what moe_mxfp4_forward returns.

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

MOE_ERR_WORKSPACE, MOE_ERR_DEVICE = 4, 6


def _inputs(moe, gpu_layers, L, block_m=16):
    T, H, I, E, k = L["T"], L["H"], L["I"], L["E"], L["k"]
    desc = moe.make_desc(T, H, I, E, k, block_m)
    x, logits = gpu_layers.inputs(L)
    ids, w, _ = moe.route(logits, k)
    perm = moe.permute(ids, E, block_m)
    return desc, gpu_layers.packed(L), x, w, perm


def _reference(moe, desc, x, packed, w, perm):
    ws = torch.empty(moe.workspace_bytes(desc), dtype=torch.uint8, device="cuda")
    y = moe.forward(desc, x, packed, w, perm, ws)
    torch.cuda.synchronize()
    assert moe.read_device_error(ws[:4].view(torch.int32)) == 0
    return y


def _noalloc(moe, desc, x, packed, w, perm):
    y = torch.full((desc.T, desc.H), float("nan"), dtype=torch.float32, device="cuda")
    moe.forward_noalloc(desc, x, packed, w, perm, y=y)
    torch.cuda.synchronize()
    assert moe.noalloc_read_device_error() == 0
    return y


@pytest.mark.parametrize("T,H,I,E,k", [(37, 512, 256, 32, 6), (8, 4096, 2048, 32, 6)])
def test_noalloc_matches_forward_on_two_calls_in_a_row(gpu_lib, gpu_layers, T, H, I, E, k):
    moe = gpu_lib
    L = synth.make_layer(T=T, H=H, E=E, k=k, I=I, seed=3)
    desc, packed, x, w, perm = _inputs(moe, gpu_layers, L)
    ref = _reference(moe, desc, x, packed, w, perm)
    y1 = _noalloc(moe, desc, x, packed, w, perm)
    # second call right after, on different activations (same routing): the scratch now holds
    # the first call's intermediates
    x2 = (x.float() * -0.5).to(torch.bfloat16)
    ref2 = _reference(moe, desc, x2, packed, w, perm)
    y2 = _noalloc(moe, desc, x2, packed, w, perm)
    assert torch.isfinite(y1).all() and torch.isfinite(y2).all()
    assert torch.equal(y1, ref) and torch.equal(y2, ref2)


def _largest_T(moe, H, I, E, k, block_m=16):
    T = 1
    while moe.workspace_bytes(moe.make_desc(T + 1, H, I, E, k, block_m)) <= moe.NOALLOC_SCRATCH_BYTES:
        T += 1
    return T


def test_noalloc_at_its_size_limit_after_larger_and_smaller_calls(gpu_lib, gpu_layers):
    """The 256-expert layer at the largest token count the array holds (25 tokens, as the header
    documents), then a smaller call with another routing, then the largest again on new activations:
    every call bit-exact against moe_mxfp4_forward, so nothing depends on what an earlier call left in
    the array."""
    moe = gpu_lib
    H, I, E, k = 4096, 2048, 256, 6
    Tmax = _largest_T(moe, H, I, E, k)
    assert Tmax == 25
    big = synth.make_layer(T=Tmax, H=H, E=E, k=k, I=I, seed=0)
    small = synth.make_config("decode_t8_h4096_e256")            # same weights (seed 0), other tokens
    seq = [(big, 1.0), (small, 1.0), (big, -0.75)]
    for L, scale in seq:
        desc, packed, x, w, perm = _inputs(moe, gpu_layers, L)
        x = (x.float() * scale).to(torch.bfloat16)
        ref = _reference(moe, desc, x, packed, w, perm)
        y = _noalloc(moe, desc, x, packed, w, perm)
        assert torch.isfinite(y).all()
        assert torch.equal(y, ref), f"T={L['T']} differs from moe_mxfp4_forward"


def test_noalloc_rejects_layers_larger_than_its_scratch(gpu_lib):
    moe = gpu_lib
    lib = moe.load()
    fake = ctypes.c_void_p(1 << 20)     # never dereferenced: the size check fails first
    for T in (26, 2048):                # one token past the documented limit, and a prefill chunk
        desc = moe.make_desc(T, 4096, 2048, 256, 6, 16)
        assert moe.workspace_bytes(desc) > moe.NOALLOC_SCRATCH_BYTES
        rc = lib.moe_mxfp4_forward_noalloc(ctypes.byref(desc), fake, fake, fake, fake, fake, fake, fake, None)
        assert rc == MOE_ERR_WORKSPACE


def test_noalloc_reports_a_corrupt_permutation_entry(gpu_lib, gpu_layers):
    """A row_to_pair entry outside [0, T*k) is skipped and recorded in the array's error word,
    which moe_mxfp4_noalloc_read_device_error reads and clears; tokens that do not use it match."""
    moe = gpu_lib
    L = synth.make_config("tiny_t37_h512_e32")
    desc, packed, x, w, perm = _inputs(moe, gpu_layers, L)
    T, k = L["T"], L["k"]
    clean = _noalloc(moe, desc, x, packed, w, perm)
    bad = {n: v.clone() for n, v in perm.items()}
    r2p = bad["row_to_pair"].cpu().numpy()
    real = np.flatnonzero(r2p >= 0)
    row = int(real[len(real) // 3])
    pair = int(r2p[row])
    bad["row_to_pair"][row] = T * k + 9
    y = torch.empty((T, L["H"]), dtype=torch.float32, device="cuda")
    moe.forward_noalloc(desc, x, packed, w, bad, y=y)
    torch.cuda.synchronize()
    assert moe.noalloc_read_device_error() == MOE_ERR_DEVICE
    assert moe.noalloc_read_device_error() == 0                      # read-and-clear
    keep = torch.ones(T, dtype=torch.bool, device="cuda")
    keep[pair // k] = False
    assert torch.equal(y[keep], clean[keep])
