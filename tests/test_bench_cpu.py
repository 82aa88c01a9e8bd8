"""bench.py's work accounting, on the CPU: the algorithmic bytes and flops
behind every roofline fraction it prints."""
import numpy as np

import bench
from mxfp4_mixture_experts_top_gb300 import moe


def test_per_expert_bytes_match_the_format_and_the_library():
    # MXFP4: 4 bits per weight plus one E8M0 byte per 32 weights
    w13, w2 = bench.per_expert_bytes(4096, 2048)
    assert (w13, w2) == (2 * 2048 * 4096 // 2 + 2 * 2048 * 4096 // 32, 4096 * 2048 // 2 + 4096 * 2048 // 32)
    assert (w13, w2) == (8_912_896, 4_456_448)
    lib = moe.load()
    for E, H, I in ((256, 4096, 2048), (32, 512, 256), (5, 256, 128)):
        d = moe.make_desc(8, H, I, E, 2, 16)
        a, b = bench.per_expert_bytes(H, I)
        assert lib.moe_mxfp4_packed_bytes(d) == E * (a + b)


def test_algorithmic_counts_touched_experts_and_routed_pairs():
    T, H, I, E, k = 8, 4096, 2048, 256, 6
    L = dict(T=T, H=H, I=I, E=E, k=k)
    ids = np.arange(T * k).reshape(T, k) % 45          # 45 distinct experts, 48 pairs
    a = bench.algorithmic(L, ids)
    P = T * k
    assert a["touched"] == 45
    assert a["w13_kernel_bytes"] == 45 * 8_912_896 + 2 * P * (H + H // 32) + 2 * P * (I + I // 32)
    assert a["w13_kernel_bytes"] == 401_688_576        # the decode figure quoted with the W13 roofline
    assert a["w2_kernel_bytes"] == 45 * 4_456_448 + 2 * P * (I + I // 32) + 4 * P * H
    assert a["gemms_kernel_bytes"] == a["w13_kernel_bytes"] + a["w2_kernel_bytes"] == 603_217_920
    assert a["layer_bytes"] == 45 * (8_912_896 + 4_456_448) + T * H * 2 + T * E * 4 + T * H * 4
    assert a["flops"] == 6.0 * P * H * I == a["gemms_flops"]
    # executed: W13 (2I rows) against 2 x terms, W2 (H rows) against 2 h terms
    assert a["mma_flops"] == 2.0 * P * H * I * (2 * 2 + 2) == a["gemms_mma_flops"]
    # the library's own term counts (as bench.py reads them off the workspace layout at run time)
    assert bench.term_counts(moe, moe.make_desc(T, H, I, E, k, 16)) == (bench.NT_X, bench.NT_H)


class _Ev:
    """A stand-in for a recorded CUDA event at a fixed time (ms)."""
    def __init__(self, t):
        self.t = t

    def elapsed_time(self, other):
        return other.t - self.t


def test_event_pass_times_the_fused_launch_as_one_interval():
    """Events 0..6: start, after route+permute, before the gather, after it, after W13, after W2, after
    the combine. With both GEMMs in one launch no event sits between them: "gemms" is 3 -> 5."""
    ev = [_Ev(t) for t in (0.0, 0.010, 0.010, 0.018, 0.5, 0.130, 0.138)]   # event 4 never recorded
    pk, total, _ = bench.summarize([ev], fused=True)
    assert set(pk) == {"route_permute", "gather", "gemms", "combine"}
    assert abs(pk["gemms"] - 0.112) < 1e-12 and abs(pk["combine"] - 0.008) < 1e-12
    ev = [_Ev(t) for t in (0.0, 0.010, 0.010, 0.018, 0.100, 0.140, 0.148)]
    pk, _, _ = bench.summarize([ev])
    assert abs(pk["w13"] - 0.082) < 1e-12 and abs(pk["w2"] - 0.040) < 1e-12 and "gemms" not in pk


def test_kernel_labels_follow_the_forward_plan():
    for T, H, want in ((8, 4096, "moe_gemm_decode_kernel"), (512, 4096, "moe_gemm_kernel<W13*>"),
                       (2048, 4096, "W13Rows64"), (2048, 640, "moe_gemm_kernel<W13*>"),
                       (8191, 4096, "moe_gemm_rows_kernel<W13Rows>")):
        plan = moe.forward_plan(moe.make_desc(T, H, 2048, 256, 6, 16))
        names = bench.kernel_names(plan, H)
        label = names["gemms"] if plan["fused_gemms"] else names["w13"]
        assert want in label, (T, H, plan, label)


def test_roofline_bound_follows_the_executed_work():
    """Decode W13 (45 experts, 48 pairs) is HBM-bound; the skewed prefill W13 (17 experts, 49,146
    pairs, two x terms) is tensor-bound. achieved counts the useful work only."""
    peaks = (6800.0, 1900.0, 1700.0, "test")
    T, H, I, E, k = 8, 4096, 2048, 256, 6
    dec = bench.algorithmic(dict(T=T, H=H, I=I, E=E, k=k), np.arange(T * k).reshape(T, k) % 45)
    r = bench.kernel_roofline("decode", "w13", dec, 0.1, peaks)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - dec["w13_kernel_bytes"] / 1e-4 / 1e9) < 1e-6 * r["achieved"]
    T = 8191
    ids = np.array([[(t + j) % 17 for j in range(k)] for t in range(T)])
    pre = bench.algorithmic(dict(T=T, H=H, I=I, E=E, k=k), ids)
    r = bench.kernel_roofline("prefill", "w13", pre, 1.4, peaks)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] == 2 * 1900.0
    assert abs(r["achieved"] - 4.0 * T * k * H * I / 1.4e-3 / 1e12) < 1e-9 * r["achieved"]
    assert abs(r["executed_frac"] - 2 * r["frac"]) < 1e-12
    assert abs(r["frac_of_bf16_peak"] - 2 * r["frac"]) < 1e-12        # useful flops against the bf16 rate
    assert abs(r["frac_of_mxfp4_peak"] - r["frac"] / 3) < 1e-12       # against 6 x bf16


def test_both_arms_report_the_same_config():
    L = dict(T=8191, H=4096, I=2048, E=256, k=6)
    a = bench.workload_config("prefill_t8191_zipf_h4096_e256", L, 17)
    assert a == bench.workload_config("prefill_t8191_zipf_h4096_e256", dict(L), 17)
    assert a["workload"] == bench.DEFAULT_WORKLOAD and a["touched_experts"] == 17
