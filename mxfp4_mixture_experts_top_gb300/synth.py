"""Seeded synthetic inputs for the MXFP4 mixture-of-experts layer.

This module only draws numbers. It holds none of the layer's arithmetic: no
MXFP4 decode, no routing, no GEMM. Both the CUDA path (through the tests and
the benchmark) and the CPU oracle take their inputs from here.

Generator (one counter-based stream per tensor):
  * ``splitmix64`` (Steele, Lea, Flood, "Fast splittable pseudorandom number
    generators", OOPSLA 2014): value ``i`` of stream ``s`` under seed ``seed``
    is ``mix(key(seed, s) + (i + 1) * 0x9E3779B97F4A7C15)``, where ``mix`` is
    the published splitmix64 output function.
  * Normal draws: Box-Muller in float64 on two 53-bit uniforms, then rounded
    to bfloat16 with round-to-nearest-even.
  * MXFP4 element bytes: raw generator bytes (so both nibbles are uniform over
    all 16 E2M1 codes). E8M0 scale bytes: ``127 + u`` with ``u`` uniform over
    the integers ``-6 .. -2`` (i.e. block scales ``2**u``).
  * Router logits: ``x @ Wr`` with ``Wr ~ N(0, 1/H)`` in bfloat16, accumulated
    in float64 and rounded once to float32. The router GEMM is outside the
    layer; its fp32 result is the layer's input.
  * Skewed prefill: a per-expert bias ``3 * ln(p_rank)`` with Zipf(s=1.2) rank
    probabilities over the E experts, ranks assigned to experts by a seeded
    Fisher-Yates permutation, added to the float64 logits before the single
    rounding to float32.

The five workloads are those of a DeepSeek-V4-Flash-shaped MoE layer (256
experts, top-6; "DeepSeek V4 Flash 单卡 MI300X" (txtmix.com), §一): a tiny
layer that is not a multiple of the 128-row tile, one decode step with 7
draft tokens, 64 decode streams of 8 tokens, a 2,048-token prefill chunk and
a Zipf-skewed 8,191-token prefill.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from functools import lru_cache

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_STREAM_MUL = np.uint64(0xD1B54A32D192ED03)

STREAM_X = 1
STREAM_WR = 2
STREAM_W13_Q = 3
STREAM_W13_S = 4
STREAM_W2_Q = 5
STREAM_W2_S = 6
STREAM_BIAS_PERM = 7

# Workloads, named by what they are. H, I: hidden and expert-intermediate width.
CONFIGS = {
    "tiny_t37_h512_e32": dict(T=37, H=512, E=32, k=6, I=256, zipf_bias=False),
    "decode_t8_h4096_e256": dict(T=8, H=4096, E=256, k=6, I=2048, zipf_bias=False),
    "decode_t512_h4096_e256": dict(T=512, H=4096, E=256, k=6, I=2048, zipf_bias=False),
    "prefill_t2048_h4096_e256": dict(T=2048, H=4096, E=256, k=6, I=2048, zipf_bias=False),
    "prefill_t8191_zipf_h4096_e256": dict(T=8191, H=4096, E=256, k=6, I=2048, zipf_bias=True),
}
CONFIG_ORDER = list(CONFIGS)

_CHUNK = 1 << 22  # uint64 draws per work item


def _mix(z: np.ndarray) -> np.ndarray:
    """splitmix64 output function on a uint64 array (wrapping arithmetic)."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    a = np.array([seed & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    b = np.array([stream], dtype=np.uint64) * _STREAM_MUL
    return _mix(a ^ b)[0]


def _draw_chunk(key: np.uint64, start: int, n: int) -> np.ndarray:
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    return _mix(idx * GOLDEN + key)


def u64_stream(seed: int, stream: int, n: int, start: int = 0, threads: int = 8) -> np.ndarray:
    """Values ``start .. start+n-1`` of one counter-based splitmix64 stream."""
    key = _key(seed, stream)
    if n <= _CHUNK:
        return _draw_chunk(key, start, n)
    out = np.empty(n, dtype=np.uint64)
    spans = [(s, min(_CHUNK, n - s)) for s in range(0, n, _CHUNK)]

    def work(span):
        s, m = span
        out[s:s + m] = _draw_chunk(key, start + s, m)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(work, spans))
    return out


def random_bytes(seed: int, stream: int, n: int) -> np.ndarray:
    """``n`` generator bytes (little-endian bytes of consecutive draws)."""
    words = u64_stream(seed, stream, (n + 7) // 8)
    return words.view(np.uint8)[:n].copy() if n % 8 else words.view(np.uint8)


def normals(seed: int, stream: int, n: int) -> np.ndarray:
    """``n`` standard normal float64 values (Box-Muller on paired draws)."""
    u = u64_stream(seed, stream, 2 * n).reshape(n, 2)
    scale = 2.0 ** -53
    u1 = ((u[:, 0] >> np.uint64(11)).astype(np.float64) + 1.0) * scale  # (0, 1]
    u2 = (u[:, 1] >> np.uint64(11)).astype(np.float64) * scale          # [0, 1)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def bf16_bits_from_f64(a: np.ndarray) -> np.ndarray:
    """Round float64 values (normal range) to bfloat16, nearest-even; uint16 bits."""
    a = np.asarray(a, dtype=np.float64)
    m, e = np.frexp(a)
    r = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)  # 8 significant bits, ties to even
    return (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def e8m0_scales(seed: int, stream: int, n: int, lo: int = -6, hi: int = -2) -> np.ndarray:
    """E8M0 bytes ``127 + u``, ``u`` uniform over the integers ``lo .. hi``."""
    d = u64_stream(seed, stream, n)
    span = np.uint64(hi - lo + 1)
    u = ((d >> np.uint64(32)) * span) >> np.uint64(32)  # Lemire multiply-shift, 0 .. span-1
    return (u.astype(np.int64) + (127 + lo)).astype(np.uint8)


def zipf_bias(seed: int, E: int, s: float = 1.2, amp: float = 3.0) -> np.ndarray:
    """Per-expert bias ``amp * ln(p_rank(e))`` with Zipf(s) rank probabilities.

    Ranks 1..E are assigned to experts by a Fisher-Yates shuffle driven by its
    own stream, so the hot experts are not simply the low indices.
    """
    perm = np.arange(E)
    d = u64_stream(seed, STREAM_BIAS_PERM, E)
    for i in range(E - 1, 0, -1):
        j = int((int(d[i]) >> 32) * (i + 1) >> 32)
        perm[i], perm[j] = perm[j], perm[i]
    ranks = np.arange(1, E + 1, dtype=np.float64)
    p = ranks ** -s
    p /= p.sum()
    bias = np.empty(E, dtype=np.float64)
    bias[perm] = amp * np.log(p)  # expert perm[r-1] gets rank r
    return bias


@lru_cache(maxsize=1)
def mxfp4_weights(seed: int, E: int, H: int, I: int):
    """Canonical MXFP4 expert weights, shared by every workload with these sizes.

    Returns ``(w13_q, w13_s, w2_q, w2_s)``:
      * ``w13_q`` uint8 [E, 2I, H/2]: rows [0, I) gate, [I, 2I) up; byte j of a
        row holds element 2j in its low nibble and 2j+1 in its high nibble.
      * ``w13_s`` uint8 [E, 2I, H/32]: one E8M0 scale per 32 consecutive K.
      * ``w2_q`` uint8 [E, H, I/2], ``w2_s`` uint8 [E, H, I/32]: same encoding.
    """
    assert H % 32 == 0 and I % 32 == 0
    w13_q = random_bytes(seed, STREAM_W13_Q, E * 2 * I * H // 2).reshape(E, 2 * I, H // 2)
    w13_s = e8m0_scales(seed, STREAM_W13_S, E * 2 * I * H // 32).reshape(E, 2 * I, H // 32)
    w2_q = random_bytes(seed, STREAM_W2_Q, E * H * I // 2).reshape(E, H, I // 2)
    w2_s = e8m0_scales(seed, STREAM_W2_S, E * H * I // 32).reshape(E, H, I // 32)
    return w13_q, w13_s, w2_q, w2_s


def activations(seed: int, T: int, H: int) -> np.ndarray:
    """x: bfloat16 bits [T, H], entries N(0, 1)."""
    return bf16_bits_from_f64(normals(seed, STREAM_X, T * H)).reshape(T, H)


def router_logits(seed: int, x_bits: np.ndarray, E: int, zipf: bool) -> np.ndarray:
    """fp32 [T, E] router logits for bf16 activations (router GEMM outside the layer)."""
    T, H = x_bits.shape
    wr = bf16_bits_to_f64(bf16_bits_from_f64(normals(seed, STREAM_WR, H * E) / math.sqrt(H)))
    logits = bf16_bits_to_f64(x_bits) @ wr.reshape(H, E)
    if zipf:
        logits = logits + zipf_bias(seed, E)[None, :]
    return logits.astype(np.float32)


def make_layer(T: int, H: int, E: int, k: int, I: int, zipf_bias: bool = False, seed: int = 0):
    """All inputs of one layer call as host numpy arrays."""
    x = activations(seed, T, H)
    logits = router_logits(seed, x, E, zipf_bias)
    w13_q, w13_s, w2_q, w2_s = mxfp4_weights(seed, E, H, I)
    return dict(T=T, H=H, E=E, k=k, I=I, seed=seed, x_bits=x, logits=logits,
                w13_q=w13_q, w13_s=w13_s, w2_q=w2_q, w2_s=w2_s)


def make_config(name: str, seed: int = 0):
    return make_layer(seed=seed, **CONFIGS[name])
