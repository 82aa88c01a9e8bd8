"""GPU parity of routing and permutation: bit-exact with the oracle.

Covers every workload, fuzzed shapes with ties and signed zeros, padding-lane
canaries (rows past T and pairs past T*k must never be read or counted: the
mask fixed in "DeepSeek V4 Flash 单卡 MI300X" (txtmix.com) §三), guard words
after every output, device-side rejection of out-of-range ids, and
determinism.
"""
import numpy as np
import pytest
import torch

import oracle
from mxfp4_mixture_experts_top_gb300 import synth

pytestmark = pytest.mark.gpu

CONFIGS = synth.CONFIG_ORDER


def _route_gpu(moe, logits_np, k):
    lg = torch.from_numpy(logits_np).cuda()
    ids, w, bm = moe.route(lg, k)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy(), bm.cpu().numpy().view(np.uint32)


def _check_route(moe, logits_np, k):
    ids, w, bm = _route_gpu(moe, logits_np, k)
    ids_r, w_r, bm_r = oracle.route(logits_np, k)
    np.testing.assert_array_equal(ids, ids_r)
    np.testing.assert_array_equal(bm, bm_r)
    assert np.abs(w.astype(np.float64) - w_r).max(initial=0) <= 1e-6
    if len(w):
        assert np.abs(w.astype(np.float64).sum(1) - 1).max() <= 1e-6
    return ids


def _check_permute(moe, ids_np, E, block_m):
    ids = torch.from_numpy(ids_np).cuda()
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = moe.permute(ids, E, block_m, error=err)
    torch.cuda.synchronize()
    ref = oracle.permute(ids_np, E, block_m)
    T, k = ids_np.shape
    cap = oracle.rows_capacity(T, E, k, block_m)
    for name in ("counts", "offsets", "padded_offsets"):
        np.testing.assert_array_equal(out[name].cpu().numpy(), ref[name], err_msg=name)
    np.testing.assert_array_equal(out["row_to_pair"].cpu().numpy()[:cap], ref["row_to_pair"])
    np.testing.assert_array_equal(out["pair_to_row"].cpu().numpy()[:T * k], ref["pair_to_row"])
    assert moe.read_device_error(err) == 0


@pytest.mark.parametrize("name", CONFIGS)
def test_route_and_permute_workloads_bit_exact(gpu_lib, name):
    L = synth.make_config(name)
    ids = _check_route(gpu_lib, L["logits"], L["k"])
    for block_m in (16, 128):
        _check_permute(gpu_lib, ids, L["E"], block_m)


@pytest.mark.parametrize("T", [1, 31, 32, 33, 37, 127, 128, 129, 1000])
@pytest.mark.parametrize("E,k", [(8, 1), (8, 8), (32, 6), (40, 6), (256, 6), (256, 8), (1024, 32)])
def test_route_permute_fuzz_with_ties(gpu_lib, T, E, k):
    rng = np.random.default_rng(T * 7919 + E * 31 + k)
    if (T + E) % 2:
        pool = np.array([-2.0, -0.0, 0.0, 0.5, 0.5, 1.0, 3.25], dtype=np.float32)   # heavy ties, both zeros
        logits = pool[rng.integers(0, len(pool), size=(T, E))]
    else:
        logits = rng.standard_normal((T, E)).astype(np.float32)
    ids = _check_route(gpu_lib, logits, k)
    for block_m in (16, 64):
        _check_permute(gpu_lib, ids, E, block_m)


def test_padding_lane_canaries(gpu_lib):
    """Rows past T hold +1e30 / NaN logits and extra valid-looking ids; outputs
    carry guard words. Nothing past the logical sizes may be read or written."""
    moe = gpu_lib
    T, E, k, block_m = 37, 32, 6, 16
    L = synth.make_config("tiny_t37_h512_e32")
    slack = np.full((T + 5, E), 1e30, dtype=np.float32)
    slack[T + 2:] = np.nan
    slack[:T] = L["logits"]
    lg = torch.from_numpy(slack).cuda()
    GUARD = -123456789
    ids_buf = torch.full((T * k + 64,), GUARD, dtype=torch.int32, device="cuda")
    w_buf = torch.full((T * k + 64,), 7.0, dtype=torch.float32, device="cuda")
    bm_buf = torch.full((T + 8,), GUARD, dtype=torch.int32, device="cuda")
    moe.route(lg[:T], k, out=(ids_buf[:T * k].view(T, k), w_buf[:T * k].view(T, k), bm_buf[:T].view(T, 1)))
    torch.cuda.synchronize()
    ids_r, _, bm_r = oracle.route(L["logits"], k)
    np.testing.assert_array_equal(ids_buf[:T * k].cpu().numpy().reshape(T, k), ids_r)
    np.testing.assert_array_equal(bm_buf[:T].cpu().numpy().view(np.uint32).reshape(T, 1), bm_r)
    assert (ids_buf[T * k:].cpu().numpy() == GUARD).all()
    assert (w_buf[T * k:].cpu().numpy() == 7.0).all()
    assert (bm_buf[T:].cpu().numpy() == GUARD).all()

    # ids: T*k real pairs followed by extra ids that a global-bound-only mask would count
    extra = np.concatenate([ids_r.ravel(), np.zeros(200, np.int32)]).astype(np.int32)
    ids_dev = torch.from_numpy(extra).cuda()
    cap = oracle.rows_capacity(T, E, k, block_m)
    out = dict(counts=torch.full((E + 16,), GUARD, dtype=torch.int32, device="cuda"),
               offsets=torch.full((E + 17,), GUARD, dtype=torch.int32, device="cuda"),
               padded_offsets=torch.full((E + 17,), GUARD, dtype=torch.int32, device="cuda"),
               row_to_pair=torch.full((cap + 64,), GUARD, dtype=torch.int32, device="cuda"),
               pair_to_row=torch.full((T * k + 64,), GUARD, dtype=torch.int32, device="cuda"))
    moe.permute(ids_dev[:T * k].view(T, k), E, block_m, out=out)
    torch.cuda.synchronize()
    ref = oracle.permute(ids_r, E, block_m)
    np.testing.assert_array_equal(out["counts"][:E].cpu().numpy(), ref["counts"])
    np.testing.assert_array_equal(out["padded_offsets"][:E + 1].cpu().numpy(), ref["padded_offsets"])
    np.testing.assert_array_equal(out["row_to_pair"][:cap].cpu().numpy(), ref["row_to_pair"])
    np.testing.assert_array_equal(out["pair_to_row"][:T * k].cpu().numpy(), ref["pair_to_row"])
    for name, n in (("counts", E), ("offsets", E + 1), ("padded_offsets", E + 1), ("row_to_pair", cap),
                    ("pair_to_row", T * k)):
        assert (out[name][n:].cpu().numpy() == GUARD).all(), name


def test_out_of_range_ids_are_reported_not_faulted(gpu_lib):
    moe = gpu_lib
    ids = np.array([[0, 1], [2, 9], [-1, 3]], dtype=np.int32)      # E = 4: 9 and -1 are invalid
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = moe.permute(torch.from_numpy(ids).cuda(), 4, 16, error=err)
    torch.cuda.synchronize()
    assert moe.read_device_error(err) == 6
    assert moe.read_device_error(err) == 0                           # cleared by the read
    p2r = out["pair_to_row"].cpu().numpy()
    assert p2r[3] == -1 and p2r[4] == -1
    assert out["counts"].cpu().numpy().tolist() == [1, 1, 1, 1]


def test_route_permute_deterministic(gpu_lib):
    L = synth.make_config("prefill_t8191_zipf_h4096_e256")
    lg = torch.from_numpy(L["logits"]).cuda()
    a = gpu_lib.route(lg, 6)
    b = gpu_lib.route(lg, 6)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    pa = gpu_lib.permute(a[0], 256, 16)
    pb = gpu_lib.permute(b[0], 256, 16)
    for n in pa:
        assert torch.equal(pa[n], pb[n])


@pytest.mark.parametrize("T", [0, 1, 8, 37, 127, 128, 129, 512, 1501, 8191])
@pytest.mark.parametrize("E,k,block_m", [(256, 6, 16), (32, 6, 128), (1024, 32, 16), (8, 8, 64)])
def test_fused_route_permute_matches_oracle(gpu_lib, T, E, k, block_m):
    """moe_route_permute (one launch up to T = 128; above, routing, then the one-block permutation up
    to 2,048 pairs and the chunked one beyond) gives the oracle's ids, weights, bitmatrix and
    permutation, with heavy ties in half of the cases."""
    rng = np.random.default_rng(T * 131 + E + k)
    if T % 2:
        pool = np.array([-1.0, -0.0, 0.0, 0.25, 0.25, 2.0], dtype=np.float32)
        logits = pool[rng.integers(0, len(pool), size=(T, E))]
    else:
        logits = rng.standard_normal((T, E)).astype(np.float32)
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    ids, w, bm, perm = gpu_lib.route_permute(torch.from_numpy(logits).cuda(), k, block_m, error=err)
    torch.cuda.synchronize()
    ids_r, w_r, bm_r = oracle.route(logits, k)
    ref = oracle.permute(ids_r, E, block_m)
    np.testing.assert_array_equal(ids.cpu().numpy().reshape(T, k), ids_r)
    np.testing.assert_array_equal(bm.cpu().numpy().view(np.uint32).reshape(bm_r.shape), bm_r)
    assert np.abs(w.cpu().numpy().astype(np.float64) - w_r).max(initial=0) <= 1e-6
    for name in ("counts", "offsets", "padded_offsets"):
        np.testing.assert_array_equal(perm[name].cpu().numpy(), ref[name], err_msg=name)
    cap = oracle.rows_capacity(T, E, k, block_m)
    np.testing.assert_array_equal(perm["row_to_pair"].cpu().numpy()[:cap], ref["row_to_pair"])
    np.testing.assert_array_equal(perm["pair_to_row"].cpu().numpy()[:T * k], ref["pair_to_row"])
    assert gpu_lib.read_device_error(err) == 0


@pytest.mark.parametrize("T,E,k,block_m,skew", [
    (342, 256, 6, 16, 0.0),        # 2052 pairs: just past the one-block limit, 8 chunks of 256
    (300, 1024, 8, 16, 1.0),       # 2400 pairs over 1024 experts: 2 chunks of 1024 (the last takes 352 more)
    (683, 256, 6, 16, 0.0),        # 4098 pairs
    (1366, 37, 6, 128, 8.0),       # 8196 pairs: a second chunk of 4 pairs; E not a multiple of 8
    (1024, 8, 8, 64, 0.0),         # 8192 pairs: exactly one chunk
    (8191, 256, 6, 16, 30.0),      # one expert takes nearly every token
    (3000, 1024, 32, 16, 2.0),     # 96,000 pairs over 1024 experts (128 blocks)
    (20000, 5, 5, 32, 0.0),        # every token picks every expert
])
def test_multi_block_permute_guards_and_skew(gpu_lib, T, E, k, block_m, skew):
    """The many-block permutation (more than 2048 pairs) is bit-exact and writes nothing past
    its outputs: every output carries guard words after its logical end."""
    moe = gpu_lib
    rng = np.random.default_rng(T + E)
    if k == E:
        ids = np.stack([rng.permutation(E) for _ in range(T)]).astype(np.int32)
    else:
        p = np.exp(skew * rng.random(E))
        ids = np.stack([rng.choice(E, size=k, replace=False, p=p / p.sum()) for _ in range(T)]).astype(np.int32)
    GUARD = -987654321
    cap = oracle.rows_capacity(T, E, k, block_m)
    out = dict(counts=torch.full((E + 16,), GUARD, dtype=torch.int32, device="cuda"),
               offsets=torch.full((E + 17,), GUARD, dtype=torch.int32, device="cuda"),
               padded_offsets=torch.full((E + 17,), GUARD, dtype=torch.int32, device="cuda"),
               row_to_pair=torch.full((cap + 64,), GUARD, dtype=torch.int32, device="cuda"),
               pair_to_row=torch.full((T * k + 64,), GUARD, dtype=torch.int32, device="cuda"))
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    moe.permute(torch.from_numpy(ids).cuda(), E, block_m, out=out, error=err)
    torch.cuda.synchronize()
    ref = oracle.permute(ids, E, block_m)
    np.testing.assert_array_equal(out["counts"][:E].cpu().numpy(), ref["counts"])
    np.testing.assert_array_equal(out["offsets"][:E + 1].cpu().numpy(), ref["offsets"])
    np.testing.assert_array_equal(out["padded_offsets"][:E + 1].cpu().numpy(), ref["padded_offsets"])
    np.testing.assert_array_equal(out["row_to_pair"][:cap].cpu().numpy(), ref["row_to_pair"])
    np.testing.assert_array_equal(out["pair_to_row"][:T * k].cpu().numpy(), ref["pair_to_row"])
    for name, n in (("counts", E), ("offsets", E + 1), ("padded_offsets", E + 1), ("row_to_pair", cap),
                    ("pair_to_row", T * k)):
        assert (out[name][n:].cpu().numpy() == GUARD).all(), name
    assert moe.read_device_error(err) == 0


def test_multi_block_permute_reports_out_of_range_ids(gpu_lib):
    moe = gpu_lib
    T, E, k = 1000, 64, 6
    rng = np.random.default_rng(5)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ids[17, 2] = E + 3
    ids[901, 0] = -2
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = moe.permute(torch.from_numpy(ids).cuda(), E, 16, error=err)
    torch.cuda.synchronize()
    assert moe.read_device_error(err) == 6
    p2r = out["pair_to_row"].cpu().numpy()
    assert p2r[17 * k + 2] == -1 and p2r[901 * k] == -1
    good = ids.ravel()[(ids.ravel() >= 0) & (ids.ravel() < E)]
    np.testing.assert_array_equal(out["counts"].cpu().numpy(), np.bincount(good, minlength=E))
    r2p = out["row_to_pair"].cpu().numpy()
    real = r2p[r2p >= 0]
    assert len(real) == T * k - 2 and (p2r[real] >= 0).all()
