"""Pins for the CPU oracle: each check compares it with something other than itself.

Pins used: the OCP MX format tables (tests/golden), torch's float8_e8m0fnu
conversion, brute-force sorting for top-k, torch.topk, scipy's softmax,
closed forms of the renormalised softmax, numpy's bincount / cumsum /
stable argsort for the permutation, a dense torch float64 SwiGLU MLP for the
one-expert case, a dense per-expert-mask formulation of the whole layer, and
a hand-computed one-hot layer.
"""
import math
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from mxfp4_mixture_experts_top_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                a, b = line.split()
                rows.append((int(a), float(b)))
    return rows


E2M1_TABLE = np.array([v for _, v in _golden("e2m1_ocp_mx.txt")])


def _decode_table(q, s):
    """Dense float64 weights from nibbles/scales via the OCP table (not the oracle's decoder)."""
    lo = E2M1_TABLE[q & 0xF]
    hi = E2M1_TABLE[q >> 4]
    vals = np.stack([lo, hi], axis=-1).reshape(*q.shape[:-1], q.shape[-1] * 2)
    scale = np.ldexp(1.0, s.astype(np.int64) - 127)
    return vals * np.repeat(scale, 32, axis=-1)


# ---------------------------------------------------------------- formats

def test_e2m1_all_codes_match_ocp_table():
    for code, val in _golden("e2m1_ocp_mx.txt"):
        got = oracle.e2m1_value(code)
        assert got == val and math.copysign(1, got) == math.copysign(1, val), code


def test_e8m0_golden_and_torch():
    for s, val in _golden("e8m0_ocp_mx.txt"):
        got = oracle.e8m0_value(s)
        assert (math.isnan(got) and math.isnan(val)) or got == val, s
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64)
    for s in range(255):
        assert oracle.e8m0_value(s) == ref[s].item(), s
    assert math.isnan(oracle.e8m0_value(255)) and math.isnan(ref[255].item())


# ---------------------------------------------------------------- routing

def _brute_topk(row, k):
    order = sorted(range(len(row)), key=lambda e: (-float(row[e]), e))
    return order[:k]


@pytest.mark.parametrize("E,k", [(1, 1), (2, 1), (5, 3), (8, 2), (10, 6), (10, 10)])
def test_route_brute_force_with_ties(E, k):
    rng = np.random.default_rng(E * 100 + k)
    T = 300
    # few distinct values so ties are common; include both zeros
    pool = np.array([-1.5, -0.0, 0.0, 0.25, 0.25, 2.0], dtype=np.float32)
    logits = pool[rng.integers(0, len(pool), size=(T, E))]
    ids, w, bm = oracle.route(logits, k)
    for t in range(T):
        assert list(ids[t]) == _brute_topk(logits[t], k)
    # weights: softmax over all E (scipy), restricted to the chosen, renormalised
    from scipy.special import softmax
    p = softmax(logits.astype(np.float64), axis=1)
    sel = np.take_along_axis(p, ids.astype(np.int64), 1)
    np.testing.assert_allclose(w, sel / sel.sum(1, keepdims=True), rtol=1e-13, atol=1e-15)


def test_route_matches_torch_topk_without_ties():
    rng = np.random.default_rng(7)
    logits = rng.standard_normal((257, 256)).astype(np.float32)
    assert all(len(np.unique(r)) == 256 for r in logits)
    ids, _, _ = oracle.route(logits, 6)
    ref = torch.topk(torch.from_numpy(logits), 6, dim=1, sorted=True).indices.numpy()
    np.testing.assert_array_equal(ids, ref)


def test_route_signed_zero_ties_go_to_lower_index():
    logits = np.array([[-1.0, 0.0, -2.0, -0.0],
                       [-1.0, -0.0, -2.0, 0.0],
                       [-0.0, -0.0, 0.0, 0.0]], dtype=np.float32)
    ids, w, _ = oracle.route(logits, 2)
    assert ids.tolist() == [[1, 3], [1, 3], [0, 1]]
    np.testing.assert_allclose(w, 0.5, rtol=0, atol=1e-15)


def test_route_weight_closed_forms():
    # equal logits -> 1/k
    ids, w, _ = oracle.route(np.full((3, 32), 1.25, np.float32), 6)
    assert ids.tolist() == [list(range(6))] * 3
    np.testing.assert_allclose(w, 1 / 6, rtol=1e-15)
    # chosen set holds m values a and k-m values b: w_a = e^a / (m e^a + (k-m) e^b)
    a, b, m, k = 2.0, 0.5, 2, 5
    row = np.full(20, -30.0, np.float32)
    row[[3, 11]] = a
    row[[0, 5, 19]] = b
    ids, w, _ = oracle.route(row[None], k)
    assert ids[0].tolist() == [3, 11, 0, 5, 19]
    z = m * math.exp(a) + (k - m) * math.exp(b)
    np.testing.assert_allclose(w[0], [math.exp(a) / z] * 2 + [math.exp(b) / z] * 3, rtol=1e-14)
    # shifting every logit by a constant changes nothing
    ids2, w2, _ = oracle.route(row[None] + np.float32(3.0), k)
    assert ids2.tolist() == ids.tolist()
    np.testing.assert_allclose(w2, w, rtol=1e-14)


def test_route_bitmatrix_and_invariants():
    L = synth.make_config("tiny_t37_h512_e32")
    ids, w, bm = oracle.route(L["logits"], 6)
    T, E = L["logits"].shape
    assert bm.shape == (T, 1)
    for t in range(T):
        assert len(set(ids[t].tolist())) == 6                      # k distinct experts
        bits = [e for e in range(E) if (int(bm[t, e // 32]) >> (e % 32)) & 1]
        assert bits == sorted(ids[t].tolist())                     # popcount k, same set
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-13)  # combine weights sum to 1
    assert (w > 0).all()
    # E not a multiple of 32: the last word keeps only real experts
    logits = np.random.default_rng(1).standard_normal((5, 40)).astype(np.float32)
    ids, _, bm = oracle.route(logits, 4)
    assert bm.shape == (5, 2) and (bm[:, 1] >> 8 == 0).all()


# ---------------------------------------------------------------- permutation

@pytest.mark.parametrize("T,E,k,block_m", [(0, 4, 2, 16), (1, 1, 1, 1), (37, 32, 6, 128),
                                           (37, 32, 6, 16), (200, 8, 3, 64), (129, 256, 6, 16)])
def test_permute_matches_numpy(T, E, k, block_m):
    rng = np.random.default_rng(T + E)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32) if T else np.zeros((0, k), np.int32)
    got = oracle.permute(ids, E, block_m)
    flat = ids.ravel()
    counts = np.bincount(flat, minlength=E)
    np.testing.assert_array_equal(got["counts"], counts)
    np.testing.assert_array_equal(got["offsets"], np.concatenate([[0], np.cumsum(counts)]))
    padded = np.concatenate([[0], np.cumsum(-(-counts // block_m) * block_m)])
    np.testing.assert_array_equal(got["padded_offsets"], padded)
    order = np.argsort(flat, kind="stable")          # pairs sorted by expert, then pair index
    r2p = got["row_to_pair"]
    assert len(r2p) == oracle.rows_capacity(T, E, k, block_m)
    real = r2p[r2p >= 0]
    np.testing.assert_array_equal(real, order)        # rows in expert-major, token-ascending order
    for e in range(E):
        seg = r2p[padded[e]:padded[e + 1]]
        assert (seg[:counts[e]] >= 0).all() and (seg[counts[e]:] == -1).all()
    assert (r2p[padded[E]:] == -1).all()
    p2r = got["pair_to_row"]
    np.testing.assert_array_equal(r2p[p2r], np.arange(T * k))   # bijection pair <-> real row
    assert counts.sum() == T * k


def _padded_total(ids, E, block_m):
    """Rows the padded permutation uses, from numpy's bincount (independent of the oracle)."""
    c = np.bincount(ids.ravel(), minlength=E)
    return int((-(-c // block_m) * block_m).sum())


@pytest.mark.parametrize("T,E,k,block_m", [(1, 8, 3, 16), (5, 32, 6, 16), (8, 256, 6, 16), (21, 128, 6, 128),
                                           (37, 256, 6, 64)])
def test_rows_capacity_attained_when_every_pair_has_its_own_expert(T, E, k, block_m):
    """T*k <= E pairs on T*k distinct experts: every pair opens a segment padded by block_m - 1
    rows, so the padded permutation fills the capacity exactly (no smaller bound is valid)."""
    assert T * k <= E
    ids = np.random.default_rng(T).permutation(E)[:T * k].reshape(T, k).astype(np.int32)
    cap = oracle.rows_capacity(T, E, k, block_m)
    assert _padded_total(ids, E, block_m) == cap == T * k * block_m
    got = oracle.permute(ids, E, block_m)
    assert got["padded_offsets"][E] == cap


def test_rows_capacity_attained_with_more_pairs_than_experts():
    """P = 20 pairs on E = 8 experts, block_m = 4, counts (5, 5, 5, 1, 1, 1, 1, 1): every count
    is 1 mod 4, so all 8 segments carry 3 padding rows: 20 + 8 * 3 = 44 rows, the capacity."""
    E, k, bm = 8, 2, 4
    flat = [0] * 5 + [1] * 5 + [2] * 5 + [3, 4, 5, 6, 7]
    ids = np.array([[flat[t], flat[t + 10]] for t in range(10)], np.int32)
    assert all(len(set(r)) == k for r in ids.tolist())
    cap = oracle.rows_capacity(10, E, k, bm)
    assert _padded_total(ids, E, bm) == cap == 44
    assert oracle.permute(ids, E, bm)["padded_offsets"][E] == cap


@pytest.mark.parametrize("seed", range(6))
def test_rows_capacity_bounds_random_and_skewed_routings(seed):
    """No routing needs more rows than the capacity (uniform and heavily skewed draws)."""
    rng = np.random.default_rng(seed)
    for _ in range(20):
        E = int(rng.integers(1, 300))
        k = int(rng.integers(1, min(E, 8) + 1))
        T = int(rng.integers(0, 400))
        bm = int(rng.choice([1, 16, 32, 64, 128]))
        p = rng.random(E) ** (1 + 6 * rng.random())
        ids = np.stack([rng.choice(E, size=k, replace=False, p=p / p.sum()) for _ in range(T)]).astype(np.int32) \
            if T else np.zeros((0, k), np.int32)
        assert _padded_total(ids, E, bm) <= oracle.rows_capacity(T, E, k, bm)


def test_permute_rejects_out_of_range_ids():
    with pytest.raises(oracle.OracleError):
        oracle.permute(np.array([[0, 4]], np.int32), 4, 16)
    with pytest.raises(oracle.OracleError):
        oracle.permute(np.array([[-1, 1]], np.int32), 4, 16)


# ---------------------------------------------------------------- forward

def _tiny_layer(T, H, E, k, I, seed):
    return synth.make_layer(T=T, H=H, E=E, k=k, I=I, seed=seed)


def _dense_reference(L, ids, w, limit=0.0):
    """Dense per-expert-mask formulation in torch float64 (independent of the oracle's loops)."""
    x = torch.from_numpy(synth.bf16_bits_to_f64(L["x_bits"]))
    W13 = torch.from_numpy(_decode_table(L["w13_q"], L["w13_s"]))   # [E, 2I, H]
    W2 = torch.from_numpy(_decode_table(L["w2_q"], L["w2_s"]))      # [E, H, I]
    I = L["I"]
    gu = torch.einsum("th,enh->ten", x, W13)
    g, u = gu[..., :I], gu[..., I:]
    if limit > 0:
        g = torch.clamp(g, max=limit)
        u = torch.clamp(u, -limit, limit)
    a = torch.nn.functional.silu(g) * u
    o = torch.einsum("tei,eci->tec", a, W2)                          # every expert for every token
    mask = torch.zeros(L["T"], L["E"], dtype=torch.float64)
    mask.scatter_(1, torch.from_numpy(ids).long(), torch.from_numpy(w))
    return torch.einsum("te,tec->tc", mask, o).numpy()


def test_forward_single_expert_is_dense_swiglu_mlp():
    L = _tiny_layer(T=7, H=64, E=1, k=1, I=32, seed=3)
    ids = np.zeros((7, 1), np.int32)
    w = np.ones((7, 1))
    y = oracle.forward(L, ids, w)
    x = torch.from_numpy(synth.bf16_bits_to_f64(L["x_bits"]))
    W13 = torch.from_numpy(_decode_table(L["w13_q"], L["w13_s"]))[0]
    W2 = torch.from_numpy(_decode_table(L["w2_q"], L["w2_s"]))[0]
    ref = (torch.nn.functional.silu(x @ W13[:32].T) * (x @ W13[32:].T)) @ W2.T
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-9)


@pytest.mark.parametrize("limit", [0.0, 10.0])
def test_forward_matches_dense_mask_formulation(limit):
    L = _tiny_layer(T=11, H=64, E=6, k=2, I=32, seed=5)
    ids, w, _ = oracle.route(L["logits"], 2)
    y = oracle.forward(L, ids, w, swiglu_limit=limit)
    ref = _dense_reference(L, ids, w, limit)
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.abs(y - ref).max() <= 1e-12 * rms


def test_forward_clamp_changes_large_activations():
    L = _tiny_layer(T=4, H=512, E=2, k=1, I=64, seed=9)
    ids, w, _ = oracle.route(L["logits"], 1)
    y0 = oracle.forward(L, ids, w)
    y1 = oracle.forward(L, ids, w, swiglu_limit=10.0)
    assert np.abs(y0 - y1).max() > 0.1 * np.sqrt(np.mean(y0 ** 2))


def test_forward_one_hot_hand_computed():
    # x = 1 everywhere; gate weights all 1.0, up weights all 0.5 (scale 2^0):
    # g = 32, u = 16, a = SiLU(32) * 16 for every n. W2 has a single nonzero,
    # element (c=3, n=5) = 6.0 * 2^1, so y[3] = 12 * a and every other y is 0.
    H = I = 32
    one = synth.bf16_bits_from_f64(np.ones((1, H)))
    w13_q = np.zeros((1, 2 * I, H // 2), np.uint8)
    w13_q[0, :I] = 0x22          # codes 2, 2 -> 1.0
    w13_q[0, I:] = 0x11          # codes 1, 1 -> 0.5
    w13_s = np.full((1, 2 * I, 1), 127, np.uint8)
    w2_q = np.zeros((1, H, I // 2), np.uint8)
    w2_q[0, 3, 2] = 0x70         # byte 2 high nibble = element n=5, code 7 -> 6.0
    w2_s = np.full((1, H, 1), 128, np.uint8)
    L = dict(T=1, H=H, I=I, E=1, k=1, x_bits=one, w13_q=w13_q, w13_s=w13_s, w2_q=w2_q, w2_s=w2_s)
    y = oracle.forward(L, np.zeros((1, 1), np.int32), np.ones((1, 1)))
    a = 32.0 / (1.0 + math.exp(-32.0)) * 16.0
    expect = np.zeros(H)
    expect[3] = 12.0 * a
    np.testing.assert_allclose(y[0], expect, rtol=1e-15, atol=0)


def test_grouped_form_equals_plain_definition_and_padding_is_inert():
    L = synth.make_config("tiny_t37_h512_e32")
    ids, w, _ = oracle.route(L["logits"], 6)
    y = oracle.forward(L, ids, w)
    for block_m in (1, 16, 128):
        perm = oracle.permute(ids, 32, block_m)
        yg = oracle.forward_grouped(L, w, perm)
        rms = np.sqrt(np.mean(y ** 2))
        assert np.abs(yg - y).max() <= 1e-12 * rms


def test_forward_token_subset_matches_full():
    L = _tiny_layer(T=9, H=64, E=4, k=2, I=32, seed=2)
    ids, w, _ = oracle.route(L["logits"], 2)
    full = oracle.forward(L, ids, w)
    sub = oracle.forward(L, ids, w, tokens=[8, 0, 4])
    np.testing.assert_array_equal(sub, full[[8, 0, 4]])


def test_oracle_is_thread_count_invariant():
    code = ("import numpy as np, oracle; from mxfp4_mixture_experts_top_gb300 import synth;"
            "L=synth.make_config('tiny_t37_h512_e32'); ids,w,_=oracle.route(L['logits'],6);"
            "y=oracle.forward(L,ids,w); import sys; sys.stdout.buffer.write(y.tobytes())")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    outs = []
    for n in ("1", "4"):
        env = dict(os.environ, OMP_NUM_THREADS=n, PYTHONPATH=root)
        outs.append(subprocess.run([sys.executable, "-c", code], env=env, cwd=root,
                                   capture_output=True, check=True).stdout)
    assert outs[0] == outs[1] and len(outs[0]) == 37 * 512 * 8
