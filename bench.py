#!/usr/bin/env python
"""Benchmark of the MXFP4 MoE layer hot path on GB300.

One step = one pass of the whole layer over one batch of synthetic input:
moe_route -> moe_permute -> moe_mxfp4_forward (gather, W13 GEMM + SiLU*up,
W2 GEMM, combine). Default (headline) workload: the largest one, a Zipf-skewed
8,191-token prefill (H=4096, E=256, top-6, I=2048). The other 4096-wide
workloads (decode T=8 with 7 draft tokens, 64 decode streams T=512, a
2,048-token prefill chunk) are timed with shorter runs in the same process
and reported under `per_config`, each with its own roofline.

Timing: W untimed warm-up steps, then exactly K steps between a barrier and
a device synchronise on both sides. The L2 cache is flushed (a write of twice
its size) before every step, outside the per-step CUDA events; `value` is
tokens over the summed per-step device time. `e2e` repeats the step through
the public API with pinned host buffers: one host->device copy of x and the
logits (kept in one pinned buffer), the calls, device->host copy of y, all
inside the timed region.
`graph` times the same step replayed from one CUDA graph (route+permute and
the forward captured once), as a serving stack runs a decode step; `step_ms`
gives the p10/p50/p90 of the timed steps.

Under torchrun each rank runs an independent replica (weak scaling, no
collective on the data path); rank 0 prints the JSON line with the maximum
per-rank time.

--impl reference times the float64 CPU oracle on a bounded token sample of
the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s and % of HBM / MXFP4-tensor roofline; route µs/layer"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "prefill_t8191_zipf_h4096_e256"
PER_CONFIG = ["decode_t8_h4096_e256", "decode_t512_h4096_e256", "prefill_t2048_h4096_e256"]
L2_NOTE = "flushed before every timed GPU step by a write of twice the L2 size (n/a on the CPU arm)"


def per_expert_bytes(H, I):
    """Prepacked MXFP4 bytes (nibbles + E8M0 scales) of one expert's W13 and W2."""
    w13 = 2 * I * H // 2 + 2 * I * H // 32
    w2 = H * I // 2 + H * I // 32
    return w13, w2


NT_X, NT_H = 2, 2   # MXFP8 terms of the activations, x (bf16) and h = SiLU(gate)*up (the library's; run-time
                    # figures use the counts read off its workspace layout, term_counts())


def algorithmic(L, ids, nt_x=NT_X, nt_h=NT_H):
    """Algorithmic bytes and flops of one step.

    W13 kernel: touched experts' MXFP4 W13 bytes (nibbles + E8M0 scales), the P gathered
    activation rows as nt_x E4M3 terms with one scale byte per 32 elements, and the P rows of
    h written as nt_h terms with their scales. W2 kernel: touched experts' W2 bytes, the h terms
    read back, and the fp32 per-pair outputs written. Layer: touched experts' W13 + W2 bytes,
    x (bf16), logits (fp32), y (fp32). Useful flops: 6 P H I (4 P H I for W13, 2 P I H for W2);
    executed tensor flops: nt_x (W13) and nt_h (W2) times the useful ones."""
    T, H, I, E, k = L["T"], L["H"], L["I"], L["E"], L["k"]
    touched = int(len(np.unique(ids)))
    P = T * k
    w13, w2 = per_expert_bytes(H, I)
    w13_kernel = touched * w13 + nt_x * P * (H + H // 32) + nt_h * P * (I + I // 32)
    w2_kernel = touched * w2 + nt_h * P * (I + I // 32) + 4 * P * H
    layer = touched * (w13 + w2) + T * H * 2 + T * E * 4 + T * H * 4
    flops = 6.0 * P * H * I
    mma_flops = 2.0 * P * H * I * (2 * nt_x + nt_h)
    d = dict(touched=touched, w13_kernel_bytes=w13_kernel, w2_kernel_bytes=w2_kernel, layer_bytes=layer,
             flops=flops, w13_flops=4.0 * P * H * I, w2_flops=2.0 * P * H * I,
             w13_mma_flops=4.0 * P * H * I * nt_x, w2_mma_flops=2.0 * P * H * I * nt_h, mma_flops=mma_flops)
    # both GEMMs in one launch (the smallest batches): the sum of the two
    for key in ("kernel_bytes", "flops", "mma_flops"):
        d[f"gemms_{key}"] = d[f"w13_{key}"] + d[f"w2_{key}"]
    return d


def term_counts(moe, desc):
    """(x terms, h terms) the library uses for this layer, read off its workspace layout."""
    lay = moe.workspace_layout(desc)
    R = moe.rows_capacity(desc.T, desc.E, desc.k, desc.block_m)
    return (lay["xs"] - lay["xq"]) // (R * desc.H), (lay["hs"] - lay["hq"]) // (R * desc.I)


KERNEL_NAMES = {"w13": "moe_gemm_kernel<W13*> (grouped W13 GEMM + SiLU*up + h terms)",
                "w2": "moe_gemm_kernel<W2*> (grouped W2 GEMM)",
                "gemms": "moe_gemm_decode_kernel (W13 GEMM + SiLU*up + h terms, then W2: one persistent launch)"}
ROWS_KERNEL_NAMES = {"w13": "moe_gemm_rows_kernel<W13Rows> (token-major grouped W13 GEMM + SiLU*up + h terms)",
                     "w2": "moe_gemm_rows_kernel<W2Rows> (token-major grouped W2 GEMM)"}
ROWS64_KERNEL_NAMES = {"w13": "moe_gemm_rows_kernel<W13Rows64> (token-major, 64 token rows x 2 stacked terms; grouped "
                              "W13 GEMM + SiLU*up + h terms)",
                       "w2": "moe_gemm_rows_kernel<W2Rows64> (token-major, 64 token rows x 2 stacked terms; grouped "
                             "W2 GEMM)"}


def kernel_names(plan, H):
    """Names of the GEMM kernels the library launches for a layer, from its forward plan: token-major
    tiles in the "huge" regime, stacked token-major tiles in the "mid" regime when H is a multiple of 256,
    weight-major tiles otherwise (one fused launch where the plan says so)."""
    if plan["regime"] == "huge":
        return ROWS_KERNEL_NAMES
    if plan["regime"] == "mid" and H % 256 == 0:
        return ROWS64_KERNEL_NAMES
    return KERNEL_NAMES


def kernel_roofline(name, key, alg, ms, peaks, names=KERNEL_NAMES):
    """Roofline of one GEMM launch (key "w13", "w2", or "gemms" for both in one launch): bound by HBM or by the tensor pipe,
    whichever needs more time for the work it executes (all activation terms) at the measured
    peaks; `achieved` counts the algorithmic (useful) bytes or flops."""
    hbm, bf16, bf16_sus, kind = peaks
    mxf8 = MXF8_OVER_BF16 * bf16
    kernel = names[key]
    nbytes, flops, mma = alg[f"{key}_kernel_bytes"], alg[f"{key}_flops"], alg[f"{key}_mma_flops"]
    traffic, source = traffic_per_launch(name, key, nbytes)
    if mma / (mxf8 * 1e12) > nbytes / (hbm * 1e9):
        ach = flops / (ms / 1e3) / 1e12
        r = {"kernel": kernel, "bound": "tensor", "achieved": ach, "peak": mxf8, "unit": "TFLOP/s",
             "frac": ach / mxf8, "executed_frac": mma / (ms / 1e3) / 1e12 / mxf8,
             "frac_of_sustained": ach / (MXF8_OVER_BF16 * bf16_sus),
             "frac_of_bf16_peak": ach / bf16,
             "frac_of_mxfp4_peak": ach / (FP4_OVER_BF16 * bf16),
             "peak_source": f"{kind} bf16_tflops (burst) x {MXF8_OVER_BF16:g}: kind::mxf8f6f4 is nominally twice "
                            "the dense bf16 rate; achieved counts useful flops, executed_frac all activation terms; "
                            f"frac_of_bf16_peak: useful flops against the measured dense bf16 rate (a bf16-activation "
                            f"path's ceiling); frac_of_mxfp4_peak: against {FP4_OVER_BF16:g} x that, the nominal dense "
                            "FP4 (kind::mxf4) rate, which needs FP4 activations that the parity bar rules out",
             "flops_per_launch": flops}
    else:
        ach = nbytes / (ms / 1e3) / 1e9
        r = {"kernel": kernel, "bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
             "peak_source": f"{kind} hbm_gbs"}
    r.update({"traffic": traffic, "traffic_source": source, "bytes_per_launch": nbytes, "avg_launch_ms": ms})
    return r


def traffic_per_launch(workload: str, kernel: str, alg_bytes: float):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu table
    (profiles/traffic.json): measured on that workload itself, or on a smaller case and scaled by
    the algorithmic bytes. None when the kernel sources changed since the capture or no capture
    exists."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None, None
    with open(path) as f:
        d = json.load(f)
    h = hashlib.sha256()
    for rel in d["kernel_sources"]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    if h.hexdigest() != d["kernel_sources_sha256"]:
        return None, "kernel sources changed since the ncu capture"
    for ent in d["entries"]:
        if ent["workload"] == workload and ent["kernel"] == kernel:
            if "dram_bytes_per_launch" in ent:
                return ent["dram_bytes_per_launch"], ent["capture"]
            return ent["traffic_over_algorithmic"] * alg_bytes, ent["capture"]
    return None, "no ncu capture of this kernel on this workload"


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("hbm_gbs"), d.get("bf16_tflops"), d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# The GEMMs run tcgen05 kind::mxf8f6f4 (8-bit operand path: E2M1 weights, E4M3 activation terms),
# nominally twice the dense bf16 rate (4.5 vs 2.25 PFLOP/s); its peak is the measured bf16 figure
# times that ratio. The dense FP4 rate (kind::mxf4, both operands E2M1) is nominally six times the
# bf16 rate (13.5 PFLOP/s); it is reported for context only, since FP4 activations miss the
# 2e-2 parity bar by far.
MXF8_OVER_BF16 = 2.0
FP4_OVER_BF16 = 6.0


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.index), "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def oracle_sample(L, n_tokens: int, min_seconds: float, max_reps: int = 50):
    """Time route + forward of the float64 oracle on the first n_tokens tokens."""
    import oracle
    tok = np.arange(min(n_tokens, L["T"]), dtype=np.int32)
    reps, t0 = 0, time.perf_counter()
    while True:
        ids, w, _ = oracle.route(L["logits"], L["k"])
        oracle.forward(L, ids, w, tokens=tok)
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or reps >= max_reps:
            break
    return len(tok) * reps / el, el, reps, len(tok)


def load_workload(name: str):
    """A named workload, or custom:T,H,I,E,k (uniform routing) / customz:T,H,I,E,k (routing logits
    with the Zipf expert bias of the skewed prefill), seed 0, for small profiling cases."""
    from mxfp4_mixture_experts_top_gb300 import synth
    for prefix, zipf in (("custom:", False), ("customz:", True)):
        if name.startswith(prefix):
            T, H, I, E, k = (int(v) for v in name[len(prefix):].split(","))
            return synth.make_layer(T=T, H=H, E=E, k=k, I=I, seed=0, zipf_bias=zipf)
    return synth.make_config(name)


def workload_config(name, L, touched):
    """The `config` object of both arms' JSON lines (identical for the same workload)."""
    return {"workload": name, "T": L["T"], "H": L["H"], "I": L["I"], "E": L["E"], "k": L["k"], "block_m": 16,
            "touched_experts": int(touched), "l2": L2_NOTE}


def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    L = load_workload(args.workload)
    touched = len(np.unique(oracle.route(L["logits"], L["k"])[0]))
    n_tok = args.ref_tokens
    for _ in range(args.warmup):
        oracle_sample(L, n_tok, 0.0, 1)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_sample(L, n_tok, 0.0, 1)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = n_tok / (ms / 1e3)
    cores = oracle.max_threads()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded splitmix64; sizes of the workload)",
        "config": workload_config(args.workload, L, touched),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"route of all {L['T']} tokens + float64 forward of {n_tok} tokens per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def time_workload(moe, L, steps, warmup, flush_buf, events_per_step=True):
    """Time K device steps of one workload; returns per-kernel and per-step times (ms)."""
    import torch
    dev = torch.device("cuda")
    T, H, I, E, k = L["T"], L["H"], L["I"], L["E"], L["k"]
    x = torch.from_numpy(L["x_bits"].view(np.int16)).to(dev).view(torch.bfloat16)
    logits = torch.from_numpy(L["logits"]).to(dev)
    w = tuple(torch.from_numpy(np.ascontiguousarray(L[n])).to(dev) for n in ("w13_q", "w13_s", "w2_q", "w2_s"))
    layer = moe.MoELayer.create(T, H, I, E, k, *w, block_m=16, device=dev)
    del w
    b = layer.bufs
    fused = moe.forward_plan(layer.desc)["fused_gemms"]

    def step(evs):
        """One layer step with an event between kernels: each kernel timed alone (no overlap). Where the
        library runs both GEMMs as one launch, no event goes between them, so that launch is timed."""
        evs[0].record()
        moe.route_permute(logits, k, 16, out=(b["ids"], b["w"], b["bm"]), perm_out=b["perm"], error=b["perm_err"])
        evs[1].record()
        lib_ev = [evs[2], evs[3], None, evs[5], evs[6]] if fused else evs[2:7]
        moe.forward_timed(layer.desc, x, layer.packed, b["w"], b["perm"], layer.workspace, b["y"], lib_ev)

    def step_fast():
        """One layer step as a user runs it: consecutive kernels overlap their start with the previous end."""
        moe.route_permute(logits, k, 16, out=(b["ids"], b["w"], b["bm"]), perm_out=b["perm"], error=b["perm_err"])
        moe.forward(layer.desc, x, layer.packed, b["w"], b["perm"], layer.workspace, b["y"])

    def mk():
        # events are created (first record) here so the library can re-record their handles
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(7)]
        for e in evs:
            e.record()
        return evs
    for _ in range(warmup):
        flush_buf.zero_()
        step(mk())
        flush_buf.zero_()
        step_fast()
    torch.cuda.synchronize()
    assert layer.forward_error() == 0, "device error during warm-up"
    return layer, x, logits, step, mk, step_fast


def route_us_graph(moe, layer, logits, flush_buf, reps=20, rounds=5):
    """Device time (µs) of one moe_route_permute call: `reps` calls captured in one CUDA graph and
    replayed between two events after an L2 flush, so no host launch latency enters the interval.
    The first call reads the logits from HBM, the others find them in L2 (as a layer does when the
    router GEMM has just written them). Median over `rounds` replays."""
    import torch
    b, d = layer.bufs, layer.desc

    def call():
        moe.route_permute(logits, d.k, d.block_m, out=(b["ids"], b["w"], b["bm"]), perm_out=b["perm"],
                          error=b["perm_err"])
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(reps):
            call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(rounds)]
    graph.replay()
    for a, e in ev:
        flush_buf.zero_()
        a.record()
        graph.replay()
        e.record()
    torch.cuda.synchronize()
    del graph
    return 1e3 * float(np.median([a.elapsed_time(e) for a, e in ev])) / reps


def time_fast(step_fast, flush_buf, steps):
    """Device time (ms) of each of `steps` layer steps, L2 flushed before each, events only around the step."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush_buf.zero_()
        ev[i][0].record()
        step_fast()
        ev[i][1].record()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def time_fast_combine(moe, layer, x, logits, flush_buf, steps):
    """Device time (ms) of each of `steps` steps with MOE_FLAG_FAST_COMBINE (up to 16 rows per expert
    W2 adds w * o into y with reduction atomics: no per-pair rows, no combine kernel), L2 flushed
    before each. Not bit-reproducible where taken, so not the headline; reported beside it."""
    import copy
    import torch
    d = copy.copy(layer.desc)
    d.flags = moe.FLAG_FAST_COMBINE
    b = layer.bufs
    k = d.k

    def step():
        moe.route_permute(logits, k, d.block_m, out=(b["ids"], b["w"], b["bm"]), perm_out=b["perm"],
                          error=b["perm_err"])
        moe.forward(d, x, layer.packed, b["w"], b["perm"], layer.workspace, b["y"])
    for _ in range(3):
        flush_buf.zero_()
        step()
    st = time_fast(step, flush_buf, steps)
    torch.cuda.synchronize()
    assert layer.forward_error() == 0, "device error in the fast-combine steps"
    return st


def summarize(evsets, fused=False):
    # events: 0 start, 1 after route+permute, 2 before gather, 3 after gather, 4 after W13, 5 after W2, 6 after combine
    # (with both GEMMs in one launch, event 4 is not recorded and "gemms" is the launch from 3 to 5)
    keys = ["route_permute", "gather"] + (["gemms"] if fused else ["w13", "w2"]) + ["combine"]
    out = {k: [] for k in keys}
    total = []
    for ev in evsets:
        t = [ev[0].elapsed_time(e) for e in ev]
        out["route_permute"].append(t[2] - t[0])
        out["gather"].append(t[3] - t[2])
        if fused:
            out["gemms"].append(t[5] - t[3])
        else:
            out["w13"].append(t[4] - t[3])
            out["w2"].append(t[5] - t[4])
        out["combine"].append(t[6] - t[5])
        total.append(t[6])
    return {k: float(np.mean(v)) for k, v in out.items()}, float(np.sum(total)), [float(v) for v in total]


def load_logits(layer, L):
    import torch
    return torch.from_numpy(L["logits"]).to(layer.packed.device)


def measure_config(moe, name, L, steps, warmup, flush_buf, peaks):
    """Short run of one workload for `per_config`: step times (L2 flushed before each), the per-kernel
    event pass, and the rooflines of the layer and of both GEMMs."""
    import torch
    hbm, bf16, bf16_sus, _ = peaks
    lay, x, logits, step, mk, fast = time_workload(moe, L, steps, warmup, flush_buf)
    st = time_fast(fast, flush_buf, steps)
    ms = float(np.mean(st))
    fc_ms = float(np.mean(time_fast_combine(moe, lay, x, logits, flush_buf, steps)))
    evs = [mk() for _ in range(steps)]
    for ev in evs:
        flush_buf.zero_()
        step(ev)
    torch.cuda.synchronize()
    assert lay.forward_error() == 0, f"device error in {name}"
    plan = moe.forward_plan(lay.desc)
    pk, _, _ = summarize(evs, plan["fused_gemms"])
    route_us = route_us_graph(moe, lay, load_logits(lay, L), flush_buf)
    nt_x, nt_h = term_counts(moe, lay.desc)
    a = algorithmic(L, lay.bufs["ids"].cpu().numpy(), nt_x, nt_h)
    mxf8 = MXF8_OVER_BF16 * bf16
    out = {
        "tokens_per_s": L["T"] / (ms / 1e3), "ms_per_step": ms, "touched_experts": a["touched"],
        "fast_combine": {"tokens_per_s": L["T"] / (fc_ms / 1e3), "ms_per_step": fc_ms},
        "activation_terms": {"x": nt_x, "h": nt_h},
        "step_ms": {"p10": float(np.percentile(st, 10)), "p50": float(np.percentile(st, 50)),
                    "p90": float(np.percentile(st, 90))},
        "route_us": route_us, "route_us_event_pass": 1e3 * pk["route_permute"], "kernel_ms": pk,
        "layer_roofline": {"bytes": a["layer_bytes"], "hbm_frac": a["layer_bytes"] / (ms / 1e3) / 1e9 / hbm,
                           "flops": a["flops"],
                           "mxf8_frac_useful": a["flops"] / (ms / 1e3) / 1e12 / mxf8,
                           "mxf8_frac_executed": a["mma_flops"] / (ms / 1e3) / 1e12 / mxf8},
        "forward_plan": plan,
    }
    if plan["fused_gemms"]:
        out["gemms_roofline"] = kernel_roofline(name, "gemms", a, pk["gemms"], peaks, kernel_names(plan, L["H"]))
    else:
        out["w13_roofline"] = kernel_roofline(name, "w13", a, pk["w13"], peaks, kernel_names(plan, L["H"]))
        out["w2_roofline"] = kernel_roofline(name, "w2", a, pk["w2"], peaks, kernel_names(plan, L["H"]))
    return out, lay, a


def run_ours(args, world, rank, local):
    import torch
    from mxfp4_mixture_experts_top_gb300 import moe
    moe.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 128 * 1024 * 1024)
    flush_buf = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
    peaks = measured_peaks()
    hbm_peak, bf16_peak, bf16_sus, peak_kind = peaks
    mxf8 = MXF8_OVER_BF16 * bf16_peak

    L = load_workload(args.workload)
    layer, x, logits, step, mk, step_fast = time_workload(moe, L, args.steps, args.warmup, flush_buf)
    T, H, I, E, k = L["T"], L["H"], L["I"], L["E"], L["k"]

    visible = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    smi_index = visible.split(",")[local] if visible else str(local)
    sampler = ClockSampler(smi_index)
    sampler.start()
    time.sleep(0.3)
    for _ in range(max(args.warmup, 3)):       # keep the GPU busy while the sampler starts
        flush_buf.zero_()
        step_fast()
    torch.cuda.synchronize()

    n0 = moe.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    step_ms = time_fast(step_fast, flush_buf, args.steps)
    wall = time.perf_counter() - wall0
    barrier(world)
    launches = moe.launch_count() - n0
    clocks = sampler.stop()
    assert layer.forward_error() == 0, "device error in the timed region"
    total_ms = allreduce_max(float(np.sum(step_ms)), world)

    # per-kernel times: a separate pass with an event between kernels (each kernel alone, no overlap)
    evsets = [mk() for _ in range(min(args.steps, 50))]
    for ev in evsets:
        flush_buf.zero_()
        step(ev)
    torch.cuda.synchronize()
    plan = moe.forward_plan(layer.desc)
    per_kernel, _, _ = summarize(evsets, plan["fused_gemms"])
    route_us = route_us_graph(moe, layer, logits, flush_buf)
    ms_per_step = total_ms / args.steps
    value = world * T / (ms_per_step / 1e3)

    ids = layer.bufs["ids"].cpu().numpy()
    nt_x, nt_h = term_counts(moe, layer.desc)
    alg = algorithmic(L, ids, nt_x, nt_h)
    if plan["fused_gemms"]:
        roofline = kernel_roofline(args.workload, "gemms", alg, per_kernel["gemms"], peaks, kernel_names(plan, L["H"]))
        other = None
    else:
        dominant = "w13" if per_kernel["w13"] >= per_kernel["w2"] else "w2"
        roofline = kernel_roofline(args.workload, dominant, alg, per_kernel[dominant], peaks, kernel_names(plan, L["H"]))
        other = kernel_roofline(args.workload, "w2" if dominant == "w13" else "w13", alg,
                                per_kernel["w2" if dominant == "w13" else "w13"], peaks, kernel_names(plan, L["H"]))
    layer_gbs = alg["layer_bytes"] / (ms_per_step / 1e3) / 1e9
    layer_tflops = alg["flops"] / (ms_per_step / 1e3) / 1e12

    # ---- end to end through the public API with pinned host buffers, as a serving loop runs it: every
    # step copies its inputs (x, then the logits, 16-byte aligned since H is a multiple of 128, in one
    # pinned buffer, one copy) to the device, runs the layer and reads y back into pinned memory. The
    # copies run on their own streams, double-buffered, so step i's read-back and step i+1's upload
    # overlap the layer's kernels; every copy of every step is inside the timed region.
    in_bytes = T * H * 2 + T * E * 4
    in_host = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    in_host[:T * H * 2].copy_(torch.from_numpy(L["x_bits"].view(np.uint8).reshape(-1)))
    in_host[T * H * 2:].copy_(torch.from_numpy(np.ascontiguousarray(L["logits"]).view(np.uint8).reshape(-1)))
    in_dev = [torch.empty(in_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    x_dev = [b_[:T * H * 2].view(torch.bfloat16).view(T, H) for b_ in in_dev]
    lg_dev = [b_[T * H * 2:].view(torch.float32).view(T, E) for b_ in in_dev]
    y_dev = [torch.empty((T, H), dtype=torch.float32, device=dev) for _ in range(2)]
    y_host = [torch.empty((T, H), dtype=torch.float32).pin_memory() for _ in range(2)]
    comp = torch.cuda.current_stream()
    up_s, down_s = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    bl = layer.bufs

    def e2e_steps(n):
        for i in range(n):
            j = i % 2
            with torch.cuda.stream(up_s):
                if i >= 2:
                    up_s.wait_event(ev_comp[j])            # step i-2 has read this input buffer
                in_dev[j].copy_(in_host, non_blocking=True)
                ev_in[j].record(up_s)
            comp.wait_event(ev_in[j])
            if i >= 2:
                comp.wait_event(ev_out[j])                 # step i-2's y has been read back
            moe.route_permute(lg_dev[j], k, 16, out=(bl["ids"], bl["w"], bl["bm"]), perm_out=bl["perm"],
                              error=bl["perm_err"])
            moe.forward(layer.desc, x_dev[j], layer.packed, bl["w"], bl["perm"], layer.workspace, y_dev[j])
            ev_comp[j].record(comp)
            with torch.cuda.stream(down_s):
                down_s.wait_event(ev_comp[j])
                y_host[j].copy_(y_dev[j], non_blocking=True)
                ev_out[j].record(down_s)

    e2e_steps(max(args.warmup, 2))
    torch.cuda.synchronize()
    assert torch.equal(x_dev[0], x) and torch.equal(lg_dev[1], logits)
    assert torch.equal(y_host[0], y_host[1]) and torch.equal(y_dev[0].cpu(), y_host[0])
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    e2e_steps(args.steps)
    torch.cuda.synchronize()
    e2e_ms = allreduce_max(1e3 * (time.perf_counter() - t0), world) / args.steps
    assert layer.forward_error() == 0, "device error in the end-to-end steps"
    # ---- the same step replayed from one CUDA graph (how a serving stack runs a decode step)
    graph, _ = layer.capture_graph(x, logits)
    g_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for _ in range(args.warmup):
        flush_buf.zero_()
        graph.replay()
    for a, b in g_ev:
        flush_buf.zero_()
        a.record()
        graph.replay()
        b.record()
    torch.cuda.synchronize()
    assert layer.forward_error() == 0, "device error in the graph replays"
    g_ms = allreduce_max(float(np.sum([a.elapsed_time(b) for a, b in g_ev])), world) / args.steps
    del graph
    graph_line = {"value": world * T / (g_ms / 1e3), "unit": UNIT, "ms_per_step": g_ms,
                  "how": "route+permute+forward captured in one CUDA graph, replayed; L2 flushed before each replay"}
    fc = time_fast_combine(moe, layer, x, logits, flush_buf, args.steps)
    fc_ms = float(np.mean(fc))
    fast_line = {"value": world * T / (fc_ms / 1e3), "unit": UNIT, "ms_per_step": fc_ms,
                 "how": "the same step with MOE_FLAG_FAST_COMBINE, which lets the library add w * o into y "
                        "with fp32 reduction atomics from W2 (no per-pair rows, no combine kernel) where that is "
                        "faster, up to 16 rows per expert; larger batches keep the slot-ordered combine. Not "
                        "bit-reproducible where taken, so not the headline"}
    e2e = {"value": world * T / (e2e_ms / 1e3), "unit": UNIT, "ms_per_step": e2e_ms,
           "h2d_bytes_per_step": T * H * 2 + T * E * 4, "d2h_bytes_per_step": T * H * 4,
           "how": "public API (moe_route_permute + moe_mxfp4_forward) with pinned host buffers: per step one "
                  "host-to-device copy of x and the logits and one device-to-host copy of y, on their own "
                  "streams, double-buffered so they overlap the neighbouring steps' kernels; wall time of "
                  "the K steps from a synchronised start to the last copy's end; no L2 flush (each step's "
                  "inputs plus the touched expert weights exceed L2)"}
    del layer, x, logits, in_dev, x_dev, lg_dev, y_dev
    torch.cuda.empty_cache()

    # ---- the other 4096-wide workloads: shorter runs, each with its own roofline
    per_config = {}
    if rank == 0 and not args.no_per_config:
        for name in PER_CONFIG:
            if name == args.workload:
                continue
            n = max(3, min(args.steps, 20))
            per_config[name], lay_c, _ = measure_config(moe, name, load_workload(name), n, max(3, min(args.warmup, 5)),
                                                        flush_buf, peaks)
            del lay_c
            torch.cuda.empty_cache()

    # ---- CPU baseline: the oracle on the host cores, bounded sample
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        v, el, reps, ntok = oracle_sample(L, args.ref_tokens, args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
               "sample": f"{reps} x (route of all {T} tokens + float64 forward of {ntok} tokens), {el:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None,
            "dtype": f"mxf8f6f4 (MXFP4 weights E2M1 x E8M0 on tcgen05 block-scaled MMAs; activations as MXFP8 "
                     f"terms: x {nt_x}, h {nt_h}; fp32 accumulate)",
            "data": "synthetic (seeded splitmix64 inputs of the workload's shapes and distributions)",
            "config": workload_config(args.workload, L, alg["touched"]),
            "route_us_per_layer": route_us,
            "route_us_how": "moe_route_permute device time: 20 calls in one CUDA graph, replayed after an L2 flush "
                            "(median of 5 replays / 20); kernel_ms.route_permute is the event-pass interval, which "
                            "also holds the host's launch latency",
            "kernel_ms": per_kernel,
            "kernel_ms_pass": "separate pass, an event between kernels (each kernel alone); the timed steps "
                              "overlap each kernel's start with the previous kernel's end",
            "layer_roofline": {"bytes": alg["layer_bytes"], "achieved_gbs": layer_gbs, "hbm_frac": layer_gbs / hbm_peak,
                               "flops": alg["flops"], "achieved_tflops": layer_tflops,
                               "mxf8_peak_tflops": mxf8,
                               "mxf8_frac_useful": layer_tflops / mxf8,
                               "mxf8_frac_executed": layer_tflops * alg["mma_flops"] / alg["flops"] / mxf8,
                               "mxf8_frac_useful_of_sustained": layer_tflops / (MXF8_OVER_BF16 * bf16_sus)},
            "roofline": roofline,
            "other_gemm_roofline": other,
            "forward_plan": plan,
            "e2e": e2e,
            "gpu_launches": launches,
            "wall_s_timed": wall,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "step_ms": {"p10": float(np.percentile(step_ms, 10)), "p50": float(np.percentile(step_ms, 50)),
                        "p90": float(np.percentile(step_ms, 90))},
            "graph": graph_line,
            "fast_combine": fast_line,
        }
        if per_config:
            line["per_config"] = per_config
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    help="a named workload, or custom:T,H,I,E,k / customz:T,H,I,E,k (Zipf-biased routing), seed 0, "
                         "for small profiling cases")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the shorter runs of the other 4096-wide workloads (profiling runs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-tokens", type=int, default=4)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
