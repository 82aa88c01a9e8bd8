"""GPU parity of the MXFP4 layer: decoder bit-exact, layer output within
2e-2 * rms of the float64 oracle on every workload.

Small workloads compare every output. The 4096-wide workloads compare every
output of a stratified token set chosen from the oracle's routing so that the
GEMMs are checked on every expert the batch touches: the last token of each
touched expert (it sits in that expert's last, partly filled, padded block),
one token in each 64-row block of the three most loaded experts (every token
block of the prefill tiles), and the first and last token of the batch. They
run in the same launch configuration as the benchmark (block_m 16, persistent
grid of one CTA per SM). Measured error ratios and expert coverage are
printed.
"""
import numpy as np
import pytest
import torch

import oracle
from mxfp4_mixture_experts_top_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = 2e-2   # max |gpu - oracle| <= TOL * rms(oracle)


def _oracle_decode_bf16_bits(q, s):
    """Expected bf16 bits of every weight: the oracle's E2M1 x E8M0 product (exact in bf16)."""
    e2m1 = np.array([oracle.e2m1_value(c) for c in range(16)])
    e8m0 = np.array([oracle.e8m0_value(v) for v in range(256)])
    vals = np.stack([e2m1[q & 0xF], e2m1[q >> 4]], -1).reshape(*q.shape[:-1], q.shape[-1] * 2)
    vals = vals * np.repeat(e8m0[s], 32, axis=-1)
    return (vals.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_decoder_bit_exact_on_workload_weights(gpu_lib, gpu_layers):
    moe = gpu_lib
    L = synth.make_config("tiny_t37_h512_e32")
    packed = gpu_layers.packed(L)
    d = moe.make_desc(L["T"], L["H"], L["I"], L["E"], L["k"], 16)
    for e in (0, 7, L["E"] - 1):
        w13 = moe.dequant_bf16(d, packed, 0, e).view(torch.int16).cpu().numpy().view(np.uint16)
        np.testing.assert_array_equal(w13, _oracle_decode_bf16_bits(L["w13_q"][e], L["w13_s"][e]))
        w2 = moe.dequant_bf16(d, packed, 1, e).view(torch.int16).cpu().numpy().view(np.uint16)
        np.testing.assert_array_equal(w2, _oracle_decode_bf16_bits(L["w2_q"][e], L["w2_s"][e]))


def test_decoder_bit_exact_all_codes_all_scales(gpu_lib):
    """Every E2M1 code under every finite E8M0 scale (0..254), incl. subnormal results."""
    moe = gpu_lib
    H, I, E = 256, 128, 1
    rng = np.random.default_rng(11)
    w13_q = rng.integers(0, 256, size=(E, 2 * I, H // 2), dtype=np.uint8)
    w13_q[0, :16, :8] = (np.arange(16, dtype=np.uint8)[:, None] * 17)          # both nibbles = code c
    w13_s = (np.arange(E * 2 * I * H // 32) % 255).astype(np.uint8).reshape(E, 2 * I, H // 32)
    w2_q = rng.integers(0, 256, size=(E, H, I // 2), dtype=np.uint8)
    w2_s = ((np.arange(E * H * I // 32) * 7) % 255).astype(np.uint8).reshape(E, H, I // 32)
    dv = lambda a: torch.from_numpy(a).cuda()
    d = moe.make_desc(1, H, I, E, 1, 16)
    packed = moe.prepack(d, dv(w13_q), dv(w13_s), dv(w2_q), dv(w2_s))
    got13 = moe.dequant_bf16(d, packed, 0, 0).view(torch.int16).cpu().numpy().view(np.uint16)
    got2 = moe.dequant_bf16(d, packed, 1, 0).view(torch.int16).cpu().numpy().view(np.uint16)
    np.testing.assert_array_equal(got13, _oracle_decode_bf16_bits(w13_q[0], w13_s[0]))
    np.testing.assert_array_equal(got2, _oracle_decode_bf16_bits(w2_q[0], w2_s[0]))
    assert set(np.unique(w13_s).tolist()) == set(range(255))


def _run_layer(moe, gpu_layers, L, block_m=16, swiglu_limit=0.0, flags=0):
    x, logits = gpu_layers.inputs(L)
    packed = gpu_layers.packed(L)
    T, H, I, E, k = L["T"], L["H"], L["I"], L["E"], L["k"]
    d = moe.make_desc(T, H, I, E, k, block_m, swiglu_limit, flags)
    ids, w, _ = moe.route(logits, k)
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    perm = moe.permute(ids, E, block_m, error=err)
    ws = torch.empty(moe.workspace_bytes(d), dtype=torch.uint8, device="cuda")
    y = moe.forward(d, x, packed, w, perm, ws)
    torch.cuda.synchronize()
    assert moe.read_device_error(err) == 0
    assert moe.read_device_error(ws[:4].view(torch.int32)) == 0
    return dict(y=y, ids=ids, w=w, perm=perm, ws=ws, desc=d, x=x)


def stratified_tokens(ids, block=64, seed=0):
    """Tokens whose outputs, compared in full, reach every token block of every touched expert.

    Rows of an expert are its tokens in ascending order (the permutation is
    stable), so cell (e, b) is rows [b*block, (b+1)*block) of expert e. Every
    cell gets a checked token: first the last token of each touched expert
    (its last, partly filled, padded block), then, for the cells still
    uncovered, a token at a seeded position inside the cell; each chosen token
    covers its cell in all k of its experts. With block = 64 every token block
    of the 16- to 96-row tiles holds a checked token. Tokens 0 and T-1 are
    added. Returns (tokens, covered experts, touched experts, cells)."""
    T, k = ids.shape
    rng = np.random.default_rng(seed)
    E = int(ids.max()) + 1
    rank = np.empty_like(ids)                    # row of pair (t, j) inside its expert's segment
    for e in range(E):
        m = ids == e
        rank[m] = np.arange(int(m.sum()))        # boolean indexing walks (t, j) in row-major order
    cells = set(zip(ids.ravel().tolist(), (rank.ravel() // block).tolist()))
    chosen, covered_cells = set(), set()

    def take(t):
        chosen.add(int(t))
        covered_cells.update(zip(ids[t].tolist(), (rank[t] // block).tolist()))

    for t in (0, T - 1):
        take(t)
    counts = np.bincount(ids.ravel(), minlength=E)
    touched = np.flatnonzero(counts)
    for e in touched:
        take(np.flatnonzero((ids == e).any(1))[-1])
    for e in np.argsort(-counts, kind="stable"):
        if counts[e] == 0:
            break
        rows = np.flatnonzero((ids == e).any(1))
        for b in range(-(-len(rows) // block)):
            if (int(e), b) not in covered_cells:
                seg = rows[b * block:(b + 1) * block]
                take(seg[rng.integers(0, len(seg))])
    assert covered_cells == cells
    tok = np.array(sorted(chosen), dtype=np.int32)
    return tok, len(np.unique(ids[tok].ravel())), len(touched), len(cells)


def _compare(name, y_gpu, y_ref):
    y_gpu = y_gpu.astype(np.float64)
    rms = np.sqrt(np.mean(y_ref ** 2))
    err = np.abs(y_gpu - y_ref)
    ratio = err.max() / rms
    print(f"[{name}] max|gpu-oracle|/rms = {ratio:.3e}, rms err/rms = {np.sqrt(np.mean(err ** 2)) / rms:.3e}")
    assert np.isfinite(y_gpu).all()
    assert ratio <= TOL, f"{name}: max err {err.max():.4g} > {TOL} * rms {rms:.4g}"
    return ratio


@pytest.mark.parametrize("block_m", [16, 128])
def test_forward_tiny_all_outputs(gpu_lib, gpu_layers, block_m):
    L = synth.make_config("tiny_t37_h512_e32")
    r = _run_layer(gpu_lib, gpu_layers, L, block_m)
    ids_r, w_r, _ = oracle.route(L["logits"], L["k"])
    assert np.array_equal(r["ids"].cpu().numpy(), ids_r)
    _compare(f"tiny bm{block_m}", r["y"].cpu().numpy(), oracle.forward(L, ids_r, w_r))


def _e4m3_values():
    """All 256 E4M3 codes (OCP FP8: bias 7, 3 mantissa bits, subnormals; S.1111.111 is NaN)."""
    c = np.arange(256)
    s, e, m = c >> 7, (c >> 3) & 15, c & 7
    v = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1 + m / 8.0, e - 7))
    v = np.where(s == 1, -v, v)
    v[(c & 0x7F) == 0x7F] = np.nan
    return v


def _terms(ws, off_q, off_s, nt, R, K):
    """Sum of the MXFP8 terms stored at (off_q, off_s): value[row, k]. Terms are E4M3 bytes
    [K/128][nt][R][128] (slab-major); scales are 32-bit words [K/128][nt][RS] (RS = R rounded
    up to 4) whose byte b holds the E8M0 scale of 32-element block 4 * slab + b."""
    RS = (R + 3) // 4 * 4
    q = ws[off_q:off_q + nt * R * K].cpu().numpy().reshape(K // 128, nt, R, 128).transpose(1, 2, 0, 3).reshape(nt, R, K)
    sw = ws[off_s:off_s + (K // 128) * nt * RS * 4].cpu().numpy().reshape(K // 128, nt, RS, 4)
    sc = sw.transpose(1, 2, 0, 3).reshape(nt, RS, K // 32)[:, :R].astype(int)
    v = _e4m3_values()[q] * np.ldexp(1.0, np.repeat(sc, 32, axis=2) - 127)
    return v.sum(0)


def test_forward_tiny_intermediates(gpu_lib, gpu_layers):
    """Diagnostic: the activation terms of both GEMMs against float64. The x
    terms reproduce every bf16 input (2 terms: 4 + 4 significant bits); the h
    terms keep SiLU(gate)*up to about 4 bits per term (the term count is read
    off the workspace layout)."""
    moe = gpu_lib
    L = synth.make_config("tiny_t37_h512_e32")
    r = _run_layer(moe, gpu_layers, L, 16)
    lay = moe.workspace_layout(r["desc"])
    R = moe.rows_capacity(L["T"], L["E"], L["k"], 16)
    Rv = int(r["perm"]["padded_offsets"][-1].item())
    I, H, k = L["I"], L["H"], L["k"]
    ws = r["ws"]
    x = synth.bf16_bits_to_f64(L["x_bits"])
    r2p = r["perm"]["row_to_pair"].cpu().numpy()[:Rv]
    real = r2p >= 0                  # padding rows are not written (their outputs are never stored)
    xg = _terms(ws, lay["xq"], lay["xs"], 2, R, H)[:Rv][real]
    want = x[r2p[real] // k]
    # exact unless a 32-element block spans more than E4M3's range (then the smallest values keep
    # fewer bits): measured on these inputs about 2 in 10^4 elements, each off by < 1e-6 * max|x|
    assert np.mean(xg == want) > 0.999 and np.abs(xg - want).max() <= 1e-6 * np.abs(x).max()
    nt_h = (lay["hs"] - lay["hq"]) // (R * I)
    h_gpu = _terms(ws, lay["hq"], lay["hs"], nt_h, R, I)[:Rv]
    ids = r["ids"].cpu().numpy()
    e2m1 = np.array([oracle.e2m1_value(c) for c in range(16)])
    worst = 0.0
    for row in range(Rv):
        p = r2p[row]
        if p < 0:
            continue
        t, e = p // k, ids[p // k, p % k]
        q, s = L["w13_q"][e], L["w13_s"][e]
        W = np.stack([e2m1[q & 0xF], e2m1[q >> 4]], -1).reshape(2 * I, H) * np.repeat(np.ldexp(1.0, s.astype(int) - 127), 32, 1)
        gu = W @ x[t]
        h = gu[:I] / (1 + np.exp(-gu[:I])) * gu[I:]
        worst = max(worst, np.abs(h_gpu[row] - h).max() / np.sqrt(np.mean(h ** 2)))
    print(f"[tiny h] {nt_h} terms: max|h_terms-h|/rms(h) = {worst:.3e}")
    # the residual after t terms is at most half an E4M3 ulp of term t, 2^(4 - 4t) of the block's
    # largest value (<= 448 * 2^e1), and a block's largest |h| is a few rms(h) of its row
    assert worst < {2: 3e-2, 3: 3e-3}[nt_h]


@pytest.mark.parametrize("T,H,I,E,k,block_m", [(300, 256, 128, 64, 6, 64),     # 28 rows per expert
                                                 (700, 256, 256, 8, 2, 128)])   # 175: token-major tiles
def test_gather_two_pass_terms(gpu_lib, gpu_layers, T, H, I, E, k, block_m):
    """Above 16 rows per expert on average the gather converts each token once and stores its terms
    to all k of its rows (through an inverse of row_to_pair). Every real row against the token's
    bf16 values (padding rows are not written)."""
    moe = gpu_lib
    L = synth.make_layer(T=T, H=H, E=E, k=k, I=I, seed=T * 3 + E)
    r = _run_layer(moe, gpu_layers, L, block_m)
    lay = moe.workspace_layout(r["desc"])
    R = moe.rows_capacity(T, E, k, block_m)
    Rv = int(r["perm"]["padded_offsets"][-1].item())
    x = synth.bf16_bits_to_f64(L["x_bits"])
    r2p = r["perm"]["row_to_pair"].cpu().numpy()[:Rv]
    assert (r2p < 0).any(), "the case should hold padding rows"
    real = r2p >= 0
    xg = _terms(r["ws"], lay["xq"], lay["xs"], 2, R, H)[:Rv][real]
    want = x[r2p[real] // k]
    assert np.mean(xg == want) > 0.999 and np.abs(xg - want).max() <= 1e-6 * np.abs(x).max()


def test_forward_decode_t8_all_outputs(gpu_lib, gpu_layers):
    L = synth.make_config("decode_t8_h4096_e256")
    r = _run_layer(gpu_lib, gpu_layers, L)
    ids_r, w_r, _ = oracle.route(L["logits"], L["k"])
    assert np.array_equal(r["ids"].cpu().numpy(), ids_r)
    _compare("decode t8", r["y"].cpu().numpy(), oracle.forward(L, ids_r, w_r))


LARGE = ["decode_t512_h4096_e256", "prefill_t2048_h4096_e256", "prefill_t8191_zipf_h4096_e256"]


def _compared_tokens(L, ids_r):
    """All tokens for the small workloads; the stratified set for the 4096-wide batches."""
    if L["T"] <= 64:
        return np.arange(L["T"], dtype=np.int32), None
    tok, covered, touched, cells = stratified_tokens(ids_r)
    assert covered == touched, f"stratified set reaches {covered} of {touched} touched experts"
    return tok, f"{len(tok)} tokens, experts covered {covered}/{touched}, 64-row blocks covered {cells}/{cells}"


@pytest.mark.parametrize("name", LARGE)
def test_forward_large_stratified_tokens(gpu_lib, gpu_layers, name):
    L = synth.make_config(name)
    r = _run_layer(gpu_lib, gpu_layers, L)
    ids_r, w_r, _ = oracle.route(L["logits"], L["k"])
    assert np.array_equal(r["ids"].cpu().numpy(), ids_r)
    tok, what = _compared_tokens(L, ids_r)
    y = r["y"].cpu().numpy()
    assert np.isfinite(y).all()
    _compare(f"{name}: {what}", y[tok], oracle.forward(L, ids_r, w_r, tokens=tok))


@pytest.mark.parametrize("name", synth.CONFIG_ORDER)
def test_forward_swiglu_clamp_variant(gpu_lib, gpu_layers, name):
    """The SwiGLU clamp (limit 10) on every workload, hence on every tile configuration."""
    L = synth.make_config(name)
    r = _run_layer(gpu_lib, gpu_layers, L, swiglu_limit=10.0)
    ids_r, w_r, _ = oracle.route(L["logits"], L["k"])
    tok, what = _compared_tokens(L, ids_r)
    _compare(f"{name} clamp10: {what or 'all tokens'}", r["y"].cpu().numpy()[tok],
             oracle.forward(L, ids_r, w_r, tokens=tok, swiglu_limit=10.0))


@pytest.mark.parametrize("T,H,I,E,k", [(1, 256, 128, 8, 2), (17, 128, 256, 16, 4), (200, 256, 128, 5, 3),
                                       (300, 128, 128, 64, 6),
                                       (40, 256, 128, 1024, 6),     # > 512 experts: the wide-E decode W2 tiles
                                       (11000, 128, 128, 1024, 6),  # > 64 rows per expert, H % 256 != 0, > 512 experts: wide-E 96-row tiles
                                       (700, 256, 256, 8, 2),       # token-major tiles, all outputs
                                       (600, 384, 128, 8, 2),       # H % 256 != 0: 96-row tiles, an odd number of W2 output tiles
                                       (600, 384, 256, 32, 6)])     # 112 rows per expert, H % 256 != 0: 96-row tiles, <= 512 experts
def test_forward_fuzz_shapes(gpu_lib, gpu_layers, T, H, I, E, k):
    L = synth.make_layer(T=T, H=H, E=E, k=k, I=I, seed=T + E)
    r = _run_layer(gpu_lib, gpu_layers, L)
    ids_r, w_r, _ = oracle.route(L["logits"], k)
    _compare(f"fuzz {T}x{H}x{I} E{E} k{k}", r["y"].cpu().numpy(), oracle.forward(L, ids_r, w_r))


@pytest.mark.parametrize("T,H,I,E,k,flags", [
    (8, 512, 512, 64, 6, 0),           # decode, 8-row fused GEMMs: gather, GEMMs, combine
    (8, 512, 512, 64, 6, 1),           # the same with the atomic combine: no combine kernel
    (40, 256, 128, 1024, 6, 0),        # more than 512 experts: decode tiles in two GEMM launches
    (300, 256, 128, 64, 6, 0),         # 28 rows per expert: two-pass gather, stacked token tiles
    (700, 256, 256, 8, 2, 0),          # 175 rows per expert: token-major tiles
])
def test_forward_launches_what_its_plan_says(gpu_lib, gpu_layers, T, H, I, E, k, flags):
    """The kernels the GPU ran for one forward, counted by the CUDA profiler, are the number
    moe_mxfp4_forward_plan reports, and every one of them is this library's."""
    moe = gpu_lib
    L = synth.make_layer(T=T, H=H, E=E, k=k, I=I, seed=T + E)
    x, logits = gpu_layers.inputs(L)
    packed = gpu_layers.packed(L)
    ids, w, _ = moe.route(logits, k)
    perm = moe.permute(ids, E, 16)
    d = moe.make_desc(T, H, I, E, k, 16, 0.0, flags)
    ws = torch.empty(moe.workspace_bytes(d), dtype=torch.uint8, device="cuda")
    moe.forward(d, x, packed, w, perm, ws)            # warm-up: attributes, tensor maps
    torch.cuda.synchronize()
    from torch.profiler import ProfilerActivity, profile
    with profile(activities=[ProfilerActivity.CUDA]):     # the process's first session may start late
        moe.forward(d, x, packed, w, perm, ws)
        torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        moe.forward(d, x, packed, w, perm, ws)
        torch.cuda.synchronize()
    kernels = [e.name for e in prof.events() if e.device_type.name == "CUDA" and "memcpy" not in e.name.lower()
               and "memset" not in e.name.lower()]
    if not kernels:
        pytest.skip("the CUDA profiler recorded no kernels on this host")
    plan = moe.forward_plan(d)
    assert all("moe" in n for n in kernels), kernels
    assert len(kernels) == plan["launches"], (kernels, plan)


@pytest.mark.parametrize("block_m", [16, 64, 128])
@pytest.mark.parametrize("T,H,I,E,k,limit,zipf", [
    (1200, 512, 256, 64, 2, 0.0, False),      # 37.5 rows per expert
    (500, 256, 384, 16, 2, 10.0, False),      # 62.5 rows per expert (some above 64: two token blocks), clamp,
                                              # three 256-row W13 blocks
    (40, 256, 256, 1, 1, 0.0, False),         # one expert, k = 1
    (2000, 256, 128, 1024, 16, 0.0, False),   # 1,024 experts, 31 rows each
    (1500, 512, 256, 128, 4, 0.0, True),      # skewed routing: hot experts hold several token blocks
    (600, 768, 256, 64, 4, 0.0, False),       # 37.5 rows per expert, three 256-row W2 blocks (H = 768)
    (1200, 256, 128, 40, 1, 10.0, False),     # k = 1, clamp
])
def test_forward_stacked_token_tiles(gpu_lib, gpu_layers, T, H, I, E, k, limit, zipf, block_m):
    """17 to 64 rows per expert with H a multiple of 256 selects the token-major tiles of 64 token rows
    whose two activation terms are stacked as the MMA's 128 A rows (paired epilogue warps add the
    halves): every output against the oracle, with partial token blocks, rows of the next expert inside
    a block, the clamp, one expert and more than 512 experts."""
    moe = gpu_lib
    assert 16 < T * k / E <= 64 or zipf
    L = synth.make_layer(T=T, H=H, E=E, k=k, I=I, zipf_bias=zipf, seed=T + 7 * H)
    r = _run_layer(moe, gpu_layers, L, block_m=block_m, swiglu_limit=limit)
    assert moe.forward_plan(r["desc"])["regime"] == "mid"
    ids_r, w_r, _ = oracle.route(L["logits"], k)
    assert np.array_equal(r["ids"].cpu().numpy(), ids_r)
    _compare(f"stacked {T}x{H}x{I} E{E} k{k} L{limit} bm{block_m}{' zipf' if zipf else ''}", r["y"].cpu().numpy(),
             oracle.forward(L, ids_r, w_r, swiglu_limit=limit))


@pytest.mark.parametrize("block_m", [16, 128])
@pytest.mark.parametrize("T,H,I,E,k,limit", [(1200, 512, 256, 16, 4, 0.0),   # 300 rows per expert: 3 token blocks
                                             (1000, 256, 384, 5, 3, 10.0),   # 600 rows per expert, clamp, I/128 odd
                                             (520, 768, 128, 2, 1, 0.0),     # 260 rows per expert, three W2 blocks
                                             (300, 256, 128, 1, 1, 0.0),     # one expert, k = 1
                                             (11000, 256, 128, 1024, 6, 0.0)])  # 1,024 experts, 64.5 rows each
def test_forward_token_major_tiles(gpu_lib, gpu_layers, T, H, I, E, k, limit, block_m):
    """More than 64 rows per expert on average selects the token-major tiles (128 token rows x 256
    weight rows, terms summed by the tensor core): every output against the oracle, with small and
    large row padding, partial last token blocks and rows of the next expert inside a tile."""
    L = synth.make_layer(T=T, H=H, E=E, k=k, I=I, seed=T + H)
    r = _run_layer(gpu_lib, gpu_layers, L, block_m=block_m, swiglu_limit=limit)
    ids_r, w_r, _ = oracle.route(L["logits"], k)
    y = r["y"].cpu().numpy()
    assert np.isfinite(y).all()
    _compare(f"token-major {T}x{H}x{I} E{E} k{k} bm{block_m} L{limit}", y,
             oracle.forward(L, ids_r, w_r, swiglu_limit=limit))


FAST_CASES = [("decode_t8_h4096_e256", None), ("tiny_t37_h512_e32", None),
              ("prefill_t2048_h4096_e256", None), ("prefill_t8191_zipf_h4096_e256", None),
              (None, (600, 384, 256, 32, 6)), (None, (1000, 256, 384, 5, 3))]


@pytest.mark.parametrize("name,shape", FAST_CASES)
def test_fast_combine_matches_oracle_and_default(gpu_lib, gpu_layers, name, shape):
    """MOE_FLAG_FAST_COMBINE on every tile family: the decode shapes (up to 16 rows per expert) take
    the atomic combine (W2 adds w * o into a zeroed y), the larger ones keep the slot-ordered
    combine. Either way within the parity tolerance of the oracle and equal to the default path up
    to fp32 rounding order (|diff| <= 1e-5 * max|y|). y starts as NaN, so every output must be
    written."""
    moe = gpu_lib
    if name:
        L = synth.make_config(name)
    else:
        T, H, I, E, k = shape
        L = synth.make_layer(T=T, H=H, E=E, k=k, I=I, seed=T + H + 1)
    det = _run_layer(moe, gpu_layers, L)["y"].clone()
    x, logits = gpu_layers.inputs(L)
    d = moe.make_desc(L["T"], L["H"], L["I"], L["E"], L["k"], 16, 0.0, moe.FLAG_FAST_COMBINE)
    ids, w, _ = moe.route(logits, L["k"])
    perm = moe.permute(ids, L["E"], 16)
    ws = torch.empty(moe.workspace_bytes(d), dtype=torch.uint8, device="cuda")
    y = torch.full((L["T"], L["H"]), float("nan"), dtype=torch.float32, device="cuda")
    moe.forward(d, x, gpu_layers.packed(L), w, perm, ws, y)
    torch.cuda.synchronize()
    assert moe.read_device_error(ws[:4].view(torch.int32)) == 0
    assert torch.isfinite(y).all()
    diff = (y - det).abs().max().item()
    assert diff <= 1e-5 * det.abs().max().item(), diff
    ids_r, w_r, _ = oracle.route(L["logits"], L["k"])
    tok, what = _compared_tokens(L, ids_r)
    _compare(f"fast combine {name or shape}: {what or 'all tokens'}", y.cpu().numpy()[tok],
             oracle.forward(L, ids_r, w_r, tokens=tok))


@pytest.mark.parametrize("name", ["decode_t8_h4096_e256", "tiny_t37_h512_e32", "prefill_t8191_zipf_h4096_e256"])
def test_bf16_output_is_the_rounded_fp32_output(gpu_lib, gpu_layers, name):
    """out_dtype MOE_OUT_BF16: y is the fp32 result of the same slot-ordered combine rounded to
    nearest even, bit for bit (also with MOE_FLAG_FAST_COMBINE, which bf16 output does not take)."""
    moe = gpu_lib
    L = synth.make_config(name)
    ref = _run_layer(moe, gpu_layers, L)["y"]
    x, logits = gpu_layers.inputs(L)
    ids, w, _ = moe.route(logits, L["k"])
    perm = moe.permute(ids, L["E"], 16)
    for flags in (0, moe.FLAG_FAST_COMBINE):
        d = moe.make_desc(L["T"], L["H"], L["I"], L["E"], L["k"], 16, 0.0, flags, moe.OUT_BF16)
        ws = torch.empty(moe.workspace_bytes(d), dtype=torch.uint8, device="cuda")
        y = moe.forward(d, x, gpu_layers.packed(L), w, perm, ws)
        torch.cuda.synchronize()
        assert y.dtype == torch.bfloat16 and moe.read_device_error(ws[:4].view(torch.int32)) == 0
        assert torch.equal(y, ref.to(torch.bfloat16)), f"flags {flags}"


@pytest.mark.parametrize("name", ["tiny_t37_h512_e32", "prefill_t2048_h4096_e256", "prefill_t8191_zipf_h4096_e256"])
def test_forward_reports_bad_rows_and_clears_the_word_on_the_next_call(gpu_lib, gpu_layers, name):
    """A row_to_pair entry >= T*k is recorded in the workspace's error word (by the W2 GEMM) on both
    gather paths; the next forward clears the word first thing, so a clean call after a bad one
    reads 0 without an explicit clear in between."""
    moe = gpu_lib
    L = synth.make_config(name)
    x, logits = gpu_layers.inputs(L)
    T, k = L["T"], L["k"]
    d = moe.make_desc(T, L["H"], L["I"], L["E"], k, 16)
    ids, w, _ = moe.route(logits, k)
    perm = moe.permute(ids, L["E"], 16)
    ws = torch.empty(moe.workspace_bytes(d), dtype=torch.uint8, device="cuda")
    bad = {n: v.clone() for n, v in perm.items()}
    r2p = bad["row_to_pair"].cpu().numpy()
    row = int(np.flatnonzero(r2p >= 0)[len(np.flatnonzero(r2p >= 0)) // 2])
    bad["row_to_pair"][row] = T * k + 5
    moe.forward(d, x, gpu_layers.packed(L), w, bad, ws)
    torch.cuda.synchronize()
    word = ws[:4].view(torch.int32)
    assert int(word.item()) == 6                                      # MOE_ERR_DEVICE, not yet cleared
    moe.forward(d, x, gpu_layers.packed(L), w, perm, ws)
    torch.cuda.synchronize()
    assert moe.read_device_error(word) == 0


@pytest.mark.parametrize("T,H,I,E,k,limit", [(8, 512, 512, 64, 6, 0.0), (16, 1024, 512, 48, 4, 0.0),
                                             (3, 4096, 2048, 256, 6, 10.0), (1, 512, 1024, 8, 1, 0.0),
                                             (170, 768, 512, 512, 6, 0.0)])
def test_fused_decode_gemms_match_two_launches_and_oracle(gpu_lib, gpu_layers, T, H, I, E, k, limit):
    """At most 2 rows per expert, W13 and W2 run as one persistent launch in which an expert's W2
    tiles wait for its W13 tiles through counters in the workspace. Its output equals the two-launch
    path (which the forward takes when events are recorded between kernels) bit for bit, and the
    oracle within tolerance; the same with the atomic combine and with bf16 output."""
    moe = gpu_lib
    L = synth.make_layer(T=T, H=H, E=E, k=k, I=I, seed=T * 13 + E)
    x, logits = gpu_layers.inputs(L)
    packed = gpu_layers.packed(L)
    ids, w, _ = moe.route(logits, k)
    perm = moe.permute(ids, E, 16)
    d = moe.make_desc(T, H, I, E, k, 16, limit)
    ws = torch.empty(moe.workspace_bytes(d), dtype=torch.uint8, device="cuda")
    fused = moe.forward(d, x, packed, w, perm, ws).clone()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    for e in evs:
        e.record()
    two = torch.empty_like(fused)
    moe.forward_timed(d, x, packed, w, perm, ws, two, evs)
    torch.cuda.synchronize()
    assert moe.read_device_error(ws[:4].view(torch.int32)) == 0
    assert torch.equal(fused, two)
    ids_r, w_r, _ = oracle.route(L["logits"], k)
    _compare(f"fused decode {T}x{H}x{I} E{E} k{k} L{limit}", fused.cpu().numpy(),
             oracle.forward(L, ids_r, w_r, swiglu_limit=limit))
    df = moe.make_desc(T, H, I, E, k, 16, limit, moe.FLAG_FAST_COMBINE)
    fast = moe.forward(df, x, packed, w, perm, ws)
    db = moe.make_desc(T, H, I, E, k, 16, limit, 0, moe.OUT_BF16)
    yb = moe.forward(db, x, packed, w, perm, ws)
    torch.cuda.synchronize()
    assert moe.read_device_error(ws[:4].view(torch.int32)) == 0
    assert (fast - fused).abs().max().item() <= 1e-5 * fused.abs().max().item()
    assert torch.equal(yb, fused.to(torch.bfloat16))


def test_forward_deterministic(gpu_lib, gpu_layers):
    L = synth.make_config("decode_t512_h4096_e256")
    a = _run_layer(gpu_lib, gpu_layers, L)["y"].clone()
    b = _run_layer(gpu_lib, gpu_layers, L)["y"]
    assert torch.equal(a, b)
