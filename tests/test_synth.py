"""The seeded input generator: deterministic, correctly distributed, shared weights."""
import numpy as np

from mxfp4_mixture_experts_top_gb300 import synth


def test_streams_are_deterministic_and_distinct():
    a = synth.u64_stream(0, 1, 1000)
    assert np.array_equal(a, synth.u64_stream(0, 1, 1000))
    assert np.array_equal(a[500:], synth.u64_stream(0, 1, 500, start=500))   # counter-based
    assert not np.array_equal(a, synth.u64_stream(0, 2, 1000))
    assert not np.array_equal(a, synth.u64_stream(1, 1, 1000))


def test_chunked_generation_equals_single_chunk():
    n = synth._CHUNK + 1234
    big = synth.u64_stream(3, 5, n)
    assert np.array_equal(big[:1000], synth.u64_stream(3, 5, 1000))
    assert np.array_equal(big[-7:], synth.u64_stream(3, 5, 7, start=n - 7))


def test_distributions():
    z = synth.normals(0, 9, 200_000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    s = synth.e8m0_scales(0, 4, 100_000)
    assert set(np.unique(s).tolist()) == {121, 122, 123, 124, 125}
    b = synth.random_bytes(0, 3, 160_000)
    lo, hi = np.bincount(b & 0xF, minlength=16), np.bincount(b >> 4, minlength=16)
    assert lo.min() > 9000 and hi.min() > 9000      # nibbles uniform over 16 codes


def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -9])
    bits = synth.bf16_bits_from_f64(vals)
    back = synth.bf16_bits_to_f64(bits)
    assert back.tolist() == [1.0, 1.0, 1.0 + 2 ** -6, -2.5, 1.0]


def test_configs_share_weights_and_shapes():
    L = synth.make_config("tiny_t37_h512_e32")
    assert L["x_bits"].shape == (37, 512) and L["logits"].shape == (37, 32)
    assert L["w13_q"].shape == (32, 512, 256) and L["w13_s"].shape == (32, 512, 16)
    assert L["w2_q"].shape == (32, 512, 128) and L["w2_s"].shape == (32, 512, 8)
    assert L["logits"].dtype == np.float32


def test_zipf_bias_skews_routing():
    bias = synth.zipf_bias(0, 256)
    assert np.isclose(np.exp(bias / 3).sum(), 1.0)
    assert len(np.unique(bias)) == 256 and np.argmax(bias) != 0 or bias[0] != bias.max()
