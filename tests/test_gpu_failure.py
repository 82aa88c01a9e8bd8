"""Failure detection on the GPU without a fault.

- A bounded pipeline wait that nothing completes gives up, by its time limit
  or by the CTA's abort flag, and records MOE_ERR_TIMEOUT. The device stays
  usable: the layer computes bit-identical results before and after.
- A permutation entry outside [0, T*k) reaching the forward is skipped and
  reported (MOE_ERR_DEVICE); every token that does not use it is unaffected.
"""
import numpy as np
import pytest
import torch

from mxfp4_mixture_experts_top_gb300 import synth

pytestmark = pytest.mark.gpu

MOE_ERR_DEVICE, MOE_ERR_TIMEOUT = 6, 7


def _tiny_forward(moe, gpu_layers, L, perm=None):
    x, logits = gpu_layers.inputs(L)
    T, H, I, E, k = L["T"], L["H"], L["I"], L["E"], L["k"]
    d = moe.make_desc(T, H, I, E, k, 16)
    ids, w, _ = moe.route(logits, k)
    if perm is None:
        perm = moe.permute(ids, E, 16, error=torch.zeros(4, dtype=torch.int32, device="cuda"))
    ws = torch.empty(moe.workspace_bytes(d), dtype=torch.uint8, device="cuda")
    y = moe.forward(d, x, gpu_layers.packed(L), w, perm, ws)
    torch.cuda.synchronize()
    return y, moe.read_device_error(ws[:4].view(torch.int32)), perm


def test_bounded_wait_times_out_and_reports(gpu_lib):
    moe = gpu_lib
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(1, dtype=torch.int64, device="cuda")
    moe.selftest_bounded_wait(5_000_000, 0, err, elapsed)         # 5 ms limit, nobody arrives
    torch.cuda.synchronize()
    ns = int(elapsed.item())
    assert moe.read_device_error(err) == MOE_ERR_TIMEOUT
    assert 5_000_000 <= ns < 500_000_000, ns
    print(f"[bounded wait] gave up after {ns / 1e6:.2f} ms (limit 5 ms)")


def test_abort_flag_ends_a_wait_early(gpu_lib):
    moe = gpu_lib
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(1, dtype=torch.int64, device="cuda")
    moe.selftest_bounded_wait(500_000_000, 2_000_000, err, elapsed)   # limit 500 ms, abort after 2 ms
    torch.cuda.synchronize()
    ns = int(elapsed.item())
    assert moe.read_device_error(err) == MOE_ERR_TIMEOUT
    assert 2_000_000 <= ns < 100_000_000, ns
    print(f"[bounded wait] aborted after {ns / 1e6:.2f} ms (abort at 2 ms, limit 500 ms)")


def test_device_usable_after_timeouts(gpu_lib, gpu_layers):
    moe = gpu_lib
    L = synth.make_config("tiny_t37_h512_e32")
    before, e0, _ = _tiny_forward(moe, gpu_layers, L)
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(1, dtype=torch.int64, device="cuda")
    for _ in range(3):
        moe.selftest_bounded_wait(2_000_000, 0, err, elapsed)
    torch.cuda.synchronize()
    assert moe.read_device_error(err) == MOE_ERR_TIMEOUT
    after, e1, _ = _tiny_forward(moe, gpu_layers, L)
    assert e0 == 0 and e1 == 0
    assert torch.equal(before, after)


def test_forward_skips_and_reports_a_corrupt_permutation_entry(gpu_lib, gpu_layers):
    moe = gpu_lib
    L = synth.make_config("tiny_t37_h512_e32")
    T, k = L["T"], L["k"]
    y_clean, err_clean, perm = _tiny_forward(moe, gpu_layers, L)
    assert err_clean == 0
    bad = {n: v.clone() for n, v in perm.items()}
    r2p = bad["row_to_pair"].cpu().numpy()
    real_rows = np.flatnonzero(r2p >= 0)
    row = int(real_rows[len(real_rows) // 2])
    pair = int(r2p[row])
    bad["row_to_pair"][row] = T * k + 5                            # outside [0, T*k)
    y_bad, err_bad, _ = _tiny_forward(moe, gpu_layers, L, perm=bad)
    assert err_bad == MOE_ERR_DEVICE
    keep = np.ones(T, dtype=bool)
    keep[pair // k] = False                                       # the token whose pair lost its row
    assert torch.equal(y_bad[torch.from_numpy(keep).cuda()], y_clean[torch.from_numpy(keep).cuda()])
