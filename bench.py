"""MoE-layer tokens/s on one GB300 (or N independent replicas), with roofline and CPU-oracle baseline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl {ours,reference}]

One step = one pass of the whole layer (router GEMM, top-k, dispatch, gate/up and down grouped
GEMMs, combine) over one batch of synthetic tokens, through the C ABI (moe_forward). The default
workload is the DeepSeek-V3-shaped prefill layer (16384 tokens, h 7168, 256 routed experts top-8 +
1 shared, intermediate 2048); its 22.6 GB of expert weights are read every step, far more than L2.

Prints ONE JSON line on rank 0. The headline fields are the default workload's; on one GPU the line
also carries ``sustained`` (the same step back to back for about 3 s, with its own clock samples) and
``per_config``: the same measurements for every other configuration of the layer (tiny, Mixtral-shaped,
DeepSeek-V3-shaped decode, FP8 and decode with NVFP4 expert weights), each with its tokens/s, layer
roofline fraction, expert-GEMM roofline, CUDA-graph and end-to-end rates, clocks and CPU-oracle rate.
Configurations whose weights and activations fit in L2 (tiny) are timed with L2 flushed between steps.
``--impl reference`` times the CPU oracle instead (on the host cores, bounded samples of the same
workload, nothing on the GPU).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/sec on 1 GB300; % of roofline (HBM or tensor-pipe)"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def weight_bytes(wl):
    """bytes per expert-weight element: bf16 2; e4m3 1 (+ 4 / 128^2 of fp32 scales); NVFP4 1/2 + 1/16
    (an e4m3 scale per 16 elements)"""
    return {"bf16": 2.0, "fp8": 1.0 + 4.0 / 16384, "nvfp4": 0.5 + 1.0 / 16}[wl.dtype]


def gemm_bytes(wl, active_experts):
    """Algorithmic bytes of the expert-GEMM pair of one step: the weights of the experts with rows (and
    the shared expert's) read once, the expert-major rows read, the SwiGLU product written and read
    back, the route-weighted rows written."""
    R_tot = wl.T * wl.k + (wl.T if wl.has_shared else 0)
    act = 1.0 if wl.dtype == "fp8" else 2.0
    w = (active_experts * 3.0 * wl.h * wl.I + 3.0 * wl.h * wl.I_shared) * weight_bytes(wl)
    return w + R_tot * (wl.h * act + 2.0 * wl.I * act + 2.0 * wl.h)


def layer_counts(wl, active_experts):
    """Algorithmic FLOPs and bytes of one layer step (inputs, outputs and the weights that must be
    read; the permute buffers are overhead, not algorithmic)."""
    T, h, E, k, I, Is = wl.T, wl.h, wl.E, wl.k, wl.I, wl.I_shared
    wbytes = weight_bytes(wl)
    gemm_flops = 6.0 * T * k * h * I + 6.0 * T * h * Is
    flops = 2.0 * T * h * E + gemm_flops
    bytes_ = (2.0 * T * h * 2  # x in, y out (bf16)
              + 4.0 * E * h + (4.0 * E if wl.bias_range is not None else 0.0)  # router weight, bias
              + active_experts * 3.0 * h * I * wbytes + 3.0 * h * Is * wbytes)
    return flops, gemm_flops, bytes_


# the sources each grouped-GEMM kernel is compiled from (a DRAM capture is valid while they are unchanged)
GEMM_KERNEL_SOURCES = {
    "grouped_gemm_bf16_kernel": ("gemm.cu", "gemm_common.cuh", "common.cuh"),
    "grouped_gemm_bf16_pair_kernel": ("gemm_pair.cu", "gemm_common.cuh", "common.cuh"),
    "grouped_gemm_fp8_kernel": ("gemm_fp8.cu", "gemm_common.cuh", "common.cuh"),
    "grouped_gemm_nvfp4_kernel": ("gemm_fp4.cu", "gemm_common.cuh", "common.cuh"),
}


def gemm_source_sha(kernel):
    """sha256 over the sources one grouped-GEMM kernel is compiled from."""
    h = hashlib.sha256()
    for f in GEMM_KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(ROOT, "routing_dispatch_expert_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def gemm_split_bytes(wl, active_experts):
    """Algorithmic bytes of the gate/up and of the down launch of moe_expert_ffn (the shared expert, if
    any, as one more group): the weights of the experts with rows (and the shared expert's) read once,
    the expert-major rows read, the SwiGLU product written (gate/up) and read back (down), the expert
    outputs written (down)."""
    R_tot = wl.T * wl.k + (wl.T if wl.has_shared else 0)
    act = 1.0 if wl.dtype == "fp8" else 2.0
    wb = weight_bytes(wl)
    groups = active_experts + (1 if wl.has_shared else 0)
    gate_up = groups * 2.0 * wl.I * wl.h * wb + R_tot * wl.h * act + R_tot * wl.I * act
    down = groups * 1.0 * wl.h * wl.I * wb + R_tot * wl.I * act + R_tot * wl.h * 2.0
    return gate_up, down


def gemm_traffic_from_profile(wl, active_experts):
    """DRAM bytes per expert-GEMM launch (mean of the gate/up and down launches) of this workload, from
    the committed ncu summary: the two launches were captured on a small case of the same kernel (a few
    GB on the device), and their measured bytes are scaled to the full workload by the ratio of the full
    to the small case's algorithmic bytes (the traffic grows with the weights of the active experts and
    the rows, which is what the algorithmic bytes count). None if the capture was not taken on the
    current sources of its kernel or has no entry for this workload."""
    p = os.path.join(ROOT, "profiles", "grouped_gemm_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    entry = d.get("workloads", {}).get(wl.name)
    if not entry or entry.get("kernel_source_sha256") != gemm_source_sha(entry["kernel"]):
        return None
    ratio = sum(entry["measured_bytes"]) / sum(entry["small_case_algorithmic_bytes"])
    return ratio * sum(gemm_split_bytes(wl, active_experts)) / 2.0


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled in the background during a timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"moe_bench_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.gpu)], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        rows = [l.split(", ") for l in open(self.path).read().strip().splitlines() if l.count(",") >= 8]
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip().lower() == "active"})
        # samples under load: the top half of the observed power draw
        load = sm
        if power and len(power) == len(sm):
            thr = float(np.median(power))
            load = [s for s, p in zip(sm, power) if p >= thr] or sm
        return {"sm_mhz": float(np.median(load)) if load else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


class HostExpertWeights:
    """bf16 weights of a workload's experts from the seeded host generator, generated on first use
    and kept (the oracle's inputs; their generation is not part of the timed oracle)."""

    def __init__(self, wl):
        import synth

        self.wl, self.synth, self.cache = wl, synth, {}

    def __call__(self, e):
        if e not in self.cache:
            self.cache[e] = self.synth.expert_weights(self.wl, e)
        return self.cache[e]


def time_cpu_oracle(wl, budget_s, weights=None):
    """The oracle as it stands, on a bounded sample of the workload's tokens, on the host cores.

    Sample: S consecutive tokens of the workload's seeded input go through the oracle's router GEMM,
    top-k, permutation and dispatch copy, the expert FFN of every routed row with its own expert's
    weights (the real expert mix of those tokens; FP8 layers quantise each expert's weights and the
    rows as the oracle does), the shared expert's rows, and the combine. Only the oracle's calls are
    timed; the experts' bf16 weights come from the seeded host generator (`weights`, cached, untimed).
    S is sized from a small first run so that the timed oracle work takes about `budget_s`. Returns
    (tokens/s, S, timed seconds, experts used)."""
    import oracle
    import synth

    kw = dict(k=wl.k, n_group=wl.n_group, topk_group=wl.topk_group,
              score=oracle.SOFTMAX if wl.score == "softmax" else oracle.SIGMOID, renorm=wl.renorm,
              routed_scale=wl.routed_scale)
    w_r = synth.router_weight(wl)
    bias = synth.bias(wl)
    mu = synth.skew_shift(wl, w_r)
    weights = weights if weights is not None else HostExpertWeights(wl)

    def ffn(xd_rows, e):
        gu, d = weights(e)
        t0 = time.perf_counter()
        if wl.dtype == "fp8":
            xq, xs = oracle.quant_1x128(oracle.bf16_to_double(xd_rows))
            (gq, gs), (dq, ds) = oracle.quant_weight_128x128(gu), oracle.quant_weight_128x128(d)
            o = oracle.expert_ffn_fp8(xq, xs, gq, gs, dq, ds)
        elif wl.dtype == "nvfp4":
            o = oracle.expert_ffn_nvfp4(xd_rows, oracle.quant_weight_nvfp4(gu), oracle.quant_weight_nvfp4(d))
        else:
            o = oracle.expert_ffn_bf16(xd_rows, gu, d)
        return o, time.perf_counter() - t0

    def run(S):
        x = synth.activations(wl, mu, 0, S)
        t0 = time.perf_counter()
        logits = oracle.router_logits(x, w_r)
        idx, w = oracle.route(logits, bias, **kw)
        counts, offsets, inv_pos, row_token = oracle.permute(idx, wl.E)
        xd = oracle.gather_rows(x, row_token)
        dt = time.perf_counter() - t0
        o_rows = np.empty((S * wl.k, wl.h), np.float64)
        used = 0
        for e in np.nonzero(counts)[0]:
            a, b = int(offsets[e]), int(offsets[e + 1])
            o_rows[a:b], t = ffn(xd[a:b], int(e))
            dt += t
            used += 1
        shared = None
        if wl.has_shared:
            shared, t = ffn(x, "shared")
            dt += t
        t0 = time.perf_counter()
        oracle.combine(o_rows[inv_pos.reshape(-1)].reshape(S, wl.k, wl.h), w, shared)
        return dt + time.perf_counter() - t0, used

    S = 8
    dt, _ = run(S)
    S = int(max(1, min(wl.T, S * budget_s / max(dt, 1e-6))))
    dt, used = run(S)
    return S / dt, S, dt, used


def max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise max of per-rank timings (the job is as slow as its slowest replica)."""
    if dist is None:
        return list(values)
    import torch

    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_tokens_per_s(world, tokens_per_replica, ms_per_step):
    """Whole-job throughput of `world` independent replicas: all tokens over the slowest step time."""
    return world * tokens_per_replica / (ms_per_step * 1e-3)


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def omp_threads():
    v = os.environ.get("OMP_NUM_THREADS")
    return int(v) if v and v.isdigit() else host_cores()


def reference_arm(args, wl, rank, world):
    if rank != 0:
        return
    import oracle

    oracle.build()
    budget = max(0.5, min(4.0, 150.0 / max(1, args.steps + args.warmup)))
    weights = HostExpertWeights(wl)
    for _ in range(args.warmup):
        time_cpu_oracle(wl, budget, weights)
    vals, samples, secs, used = [], [], [], []
    for _ in range(args.steps):
        v, S, dt, u = time_cpu_oracle(wl, budget, weights)
        vals.append(v)
        samples.append(S)
        secs.append(dt)
        used.append(u)
    value = float(np.median(vals))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": float(np.median(secs)) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(wl, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": omp_threads(), "cpu_model": cpu_model(),
                         "kind": "oracle",
                         "sample": f"per step {int(np.median(samples))} of the workload's tokens through the whole "
                                   f"oracle layer, every routed row with its own expert's weights "
                                   f"({int(np.median(used))} experts); oracle calls timed, weight generation not"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


L2_FLUSHED = "flushed between steps (a buffer of 4 x L2 overwritten outside the timed events)"
L2_LARGER = "inputs larger than L2: every step reads all active expert weights (GBs) once"


def config_of(wl, world):
    return {"workload": wl.name, "T": wl.T, "h": wl.h, "E": wl.E, "k": wl.k, "I": wl.I, "I_shared": wl.I_shared,
            "n_group": wl.n_group, "topk_group": wl.topk_group, "score": wl.score, "expert_dtype": wl.dtype,
            "zipf_s": wl.zipf_s, "parallelism": f"replicas x{world}",
            "l2": L2_FLUSHED if fits_in_l2(wl) else L2_LARGER}


def measure_fp8_peak(n=8192, sustain_s=4.0):
    """Dense e4m3 GEMM rate of the vendor library on this GPU, the way the bf16 peak is measured:
    best of 10 n^3 products (burst) and back to back for a few seconds (sustained), 2 n^3 FLOPs each,
    tensor-wise fp32 scales, bf16 out. Context for the FP8 roofline, which uses the measured bf16
    peak times the nominal FP8/bf16 ratio of 2."""
    import torch

    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(0)
    a = (torch.randn(n, n, device=dev, generator=g) * 0.5).to(torch.float8_e4m3fn)
    b = (torch.randn(n, n, device=dev, generator=g) * 0.5).to(torch.float8_e4m3fn)
    one = torch.ones((), device=dev, dtype=torch.float32)
    f = lambda: torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
    for _ in range(3):
        f()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(10):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        f()
        e.record()
        torch.cuda.synchronize()
        best = min(best, s.elapsed_time(e))
    flops = 2.0 * n ** 3
    reps = max(10, int(sustain_s * 1e3 / best))
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(reps):
        f()
    e.record()
    torch.cuda.synchronize()
    sus = s.elapsed_time(e) / reps
    print(json.dumps({"fp8_e4m3_tflops": flops / best / 1e9, "fp8_e4m3_tflops_sustained": flops / sus / 1e9,
                      "n": n, "how": "torch._scaled_mm e4m3 x e4m3 -> bf16, tensor-wise scales; best of 10 "
                                     f"(burst) and {reps} back to back (sustained)"}), flush=True)


PER_CONFIG = ("tiny", "mixtral", "dsv3_decode", "dsv3_fp8", "dsv3_decode_fp4")


def cpu_model():
    """The host CPU's model name (lscpu on Arm, /proc/cpuinfo elsewhere)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform

    return platform.machine()


def make_layer(wl, dev, rde, synth, torch):
    """Config, device weights (FP8 / NVFP4 quantised by the library), workspace and x/y buffers."""
    cfg = rde.make_config(T=wl.T, h=wl.h, E=wl.E, k=wl.k, I=wl.I, I_shared=wl.I_shared, n_group=wl.n_group,
                          topk_group=wl.topk_group, score=wl.score, renorm=wl.renorm, routed_scale=wl.routed_scale,
                          dtype=wl.dtype)
    inp = synth.device_inputs(wl, torch, device=dev)
    wts = dict(w_gu=inp["w_gu"], w_d=inp["w_d"], w_gu_shared=inp["w_gu_shared"], w_d_shared=inp["w_d_shared"])
    if wl.dtype == "fp8":
        wts["w_gu"], wts["s_gu"] = rde.quantize_weights_fp8(inp["w_gu"])
        wts["w_d"], wts["s_d"] = rde.quantize_weights_fp8(inp["w_d"])
        if wl.has_shared:
            wts["w_gu_shared"], wts["s_gu_shared"] = rde.quantize_weights_fp8(inp["w_gu_shared"])
            wts["w_d_shared"], wts["s_d_shared"] = rde.quantize_weights_fp8(inp["w_d_shared"])
        del inp["w_gu"], inp["w_d"]
    elif wl.dtype == "nvfp4":
        for n in ("gu", "d") + (("gu_shared", "d_shared") if wl.has_shared else ()):
            wts["w_" + n], wts["s_" + n], wts["g_" + n] = rde.quantize_weights_nvfp4(inp["w_" + n])
        del inp["w_gu"], inp["w_d"]
    weights = rde.Weights(w_router=inp["w_router"], bias=inp["bias"], **wts)
    ws = rde.alloc_workspace(cfg, dev)
    rde.device_status(cfg, ws)
    return cfg, weights, ws, inp["x"]


def fits_in_l2(wl, props=None):
    """True when a step's weights and activations could stay in L2 between steps (then L2 is flushed)."""
    w = 3.0 * wl.h * wl.I * (wl.E + (1 if wl.has_shared else 0)) * weight_bytes(wl)
    return w + 4.0 * wl.T * wl.h < 2 * getattr(props, "L2_cache_size", 129 << 20)


class Timer:
    """Mean milliseconds of `steps` calls of fn on `stream`, CUDA events on that stream. Without a
    flush buffer the calls run back to back between one pair of events; with one, every call has its
    own pair of events and the buffer (larger than L2) is overwritten between calls, outside them."""

    def __init__(self, torch, stream, flush=None):
        self.torch, self.stream, self.flush = torch, stream, flush

    def __call__(self, fn, steps):
        torch, stream = self.torch, self.stream
        if self.flush is None:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(steps):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b) / steps
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in evs:
            with torch.cuda.stream(stream):
                self.flush.fill_(1)
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b) for a, b in evs]))


def measure(wl, args, dev, dist, rde, synth, torch, steps, gpu_index, sustain_s=0.0):
    """One workload: K timed moe_forward steps (the metric), the same steps through the step entry
    points with the expert-GEMM pair bracketed by events (its roofline), one CUDA graph per step, the
    end-to-end rate from pinned host buffers, and the roofline of the layer. Returns a dict."""
    props = torch.cuda.get_device_properties(dev)
    cfg, weights, ws, x = make_layer(wl, dev, rde, synth, torch)
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream(dev)
    flush = None
    if fits_in_l2(wl, props):
        flush = torch.empty(4 * getattr(props, "L2_cache_size", 129 << 20), dtype=torch.uint8, device=dev)
    timer = Timer(torch, stream, flush)

    for _ in range(args.warmup):
        rde.forward(cfg, x, weights, y, ws)
    torch.cuda.synchronize(dev)
    status = rde.device_status(cfg, ws)
    if status != 0:
        raise SystemExit(f"{wl.name}: device status {status} after warm-up")
    bal = rde.balance(cfg, ws)
    active = bal["active"]

    R = wl.T * wl.k
    R_tot = R + (wl.T if wl.has_shared else 0)
    v = lambda name, dt, shape: rde.ws_view(ws, cfg, name, dt, shape)  # noqa: E731
    xd_dt = torch.uint8 if wl.dtype == "fp8" else torch.bfloat16
    it = dict(logits=v("logits", torch.float32, (wl.T, wl.E)), idx=v("topk_idx", torch.int32, (wl.T, wl.k)),
              w=v("topk_w", torch.float32, (wl.T, wl.k)), counts=v("counts", torch.int32, (wl.E,)),
              offsets=v("offsets", torch.int32, (wl.E + 1,)), inv_pos=v("inv_pos", torch.int32, (wl.T, wl.k)),
              row_token=v("row_token", torch.int32, (R,)), row_weight=v("row_weight", torch.float32, (R,)),
              xd=v("xd", xd_dt, (R_tot, wl.h)), yd=v("yd", torch.bfloat16, (R_tot, wl.h)))
    xs = v("xd_scales", torch.float32, (R_tot, wl.h // 128)) if wl.dtype == "fp8" else None

    # timed region (the metric): K steps of moe_forward, the public fused entry point
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(gpu_index) as clk:
        n0 = rde.launch_count()
        ms_step = timer(lambda: rde.forward(cfg, x, weights, y, ws), steps)
        n1 = rde.launch_count()
        if dist is not None:
            dist.barrier()
    clocks = clk.summary()

    # the same steps through the step entry points, with the expert-GEMM pair (moe_expert_ffn)
    # bracketed by its own events on the same stream: the roofline's timing
    gemm_times = []

    def step_split():
        rde.route(cfg, x, weights, it["idx"], it["w"], logits=it["logits"], ws=ws)
        rde.dispatch(cfg, x, it["idx"], it["w"], it["counts"], it["offsets"], it["inv_pos"], it["row_token"],
                     it["row_weight"], it["xd"], xs, ws)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        rde.expert_ffn(cfg, weights, it["xd"], xs, it["offsets"], it["row_weight"], it["yd"], ws)
        b.record(stream)
        gemm_times.append((a, b))
        rde.combine(cfg, it["yd"], it["inv_pos"], y)

    for _ in range(2):
        step_split()
    torch.cuda.synchronize(dev)
    gemm_times.clear()
    ms_split = timer(step_split, steps)
    gemm_ms = float(np.mean([a.elapsed_time(b) for a, b in gemm_times]))

    # the same layer as one CUDA graph per step (moe_graph_*): launch cost removed
    gstream = torch.cuda.Stream(dev)
    gstream.wait_stream(stream)
    with torch.cuda.stream(gstream):
        graph = rde.Graph(cfg, x, weights, y, ws, gstream)
        for _ in range(2):
            graph.launch()
        gstream.synchronize()
        ms_graph = Timer(torch, gstream, flush)(graph.launch, steps)
    gstream.synchronize()
    del graph

    # end to end through the public API with host buffers: every step copies its x in from pinned host
    # memory and its y out to pinned host memory. With inputs larger than L2 the copies run on their own
    # streams with two device buffers of x and y alternating, so the copy-in of step i+1 and the copy-out
    # of step i-1 overlap the layer of step i (the way a serving loop feeds a layer); when L2 is flushed
    # between steps, each step is the copy-in, the layer and the copy-out in sequence.
    x_host = x.cpu().pin_memory()
    y_host = [torch.empty(y.shape, dtype=y.dtype, pin_memory=True) for _ in range(2)]
    x_dev = [torch.empty_like(x) for _ in range(2)]
    y_dev = [y, torch.empty_like(y)]
    e2e_steps = max(4, steps // 2)
    if flush is not None:
        def e2e_seq():
            x_dev[0].copy_(x_host, non_blocking=True)
            rde.forward(cfg, x_dev[0], weights, y_dev[0], ws)
            y_host[0].copy_(y_dev[0], non_blocking=True)

        e2e_seq()
        torch.cuda.synchronize(dev)
        ms_e2e = timer(e2e_seq, e2e_steps)
    else:
        h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_used = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def e2e_step(i):
            b = i & 1
            if i >= 2:
                h2d.wait_event(ev_used[b])
            with torch.cuda.stream(h2d):
                x_dev[b].copy_(x_host, non_blocking=True)
            ev_in[b].record(h2d)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])
            rde.forward(cfg, x_dev[b], weights, y_dev[b], ws)
            ev_used[b].record(stream)
            d2h.wait_event(ev_used[b])
            with torch.cuda.stream(d2h):
                y_host[b].copy_(y_dev[b], non_blocking=True)
            ev_out[b].record(d2h)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e_s.record(stream)
        h2d.wait_stream(stream)
        d2h.wait_stream(stream)
        for i in range(e2e_steps):
            e2e_step(i)
        stream.wait_event(ev_out[0])
        stream.wait_event(ev_out[1])
        e_e.record(stream)
        torch.cuda.synchronize(dev)
        ms_e2e = e_s.elapsed_time(e_e) / e2e_steps

    # a sustained window: back-to-back moe_forward steps for `sustain_s` seconds, with its own clocks
    sustained = None
    if sustain_s > 0:
        n_sus = max(steps, int(np.ceil(sustain_s * 1e3 / ms_step)))
        torch.cuda.synchronize(dev)
        with ClockSampler(gpu_index) as clk2:
            ms_sus = timer(lambda: rde.forward(cfg, x, weights, y, ws), n_sus)
        sustained = {"steps": n_sus, "seconds": n_sus * ms_sus * 1e-3, "ms_per_step": ms_sus, "clocks": clk2.summary()}

    ms_step, ms_e2e, gemm_ms, ms_graph, ms_split = max_over_ranks([ms_step, ms_e2e, gemm_ms, ms_graph, ms_split], dist,
                                                                  dev)
    status = rde.device_status(cfg, ws)
    if status != 0:
        raise SystemExit(f"{wl.name}: device status {status} after the timed region")

    peaks, peaks_kind = load_peaks()
    n_sms = props.multi_processor_count
    flops, gemm_flops, bytes_ = layer_counts(wl, active)
    p_tc = peaks["bf16_tflops"] * 1e12
    p_hbm = peaks["hbm_gbs"] * 1e9
    # the expert GEMMs run at their own dtype's peak: FP8 = the measured bf16 peak x the nominal
    # dense ratio 4.5 / 2.25 PFLOP/s; the router stays bf16 (fp32-accurate split)
    ratio = 2.0 if wl.dtype == "fp8" else 1.0
    p_gemm = p_tc * ratio
    t_compute = (flops - gemm_flops) / p_tc + gemm_flops / p_gemm
    t_roof = max(t_compute, bytes_ / p_hbm)
    gemm_tflops = gemm_flops / (gemm_ms * 1e-3) / 1e12
    gemm_peak = peaks["bf16_tflops"] * ratio
    gemm_peak_sus = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * ratio
    traffic = gemm_traffic_from_profile(wl, active)
    hbm_bound = t_compute < bytes_ / p_hbm
    if wl.dtype == "fp8":
        gemm_kernel = "grouped_gemm_fp8_kernel"
    elif wl.dtype == "nvfp4":
        gemm_kernel = "grouped_gemm_nvfp4_kernel"
    elif wl.T * wl.k >= 128 * wl.E and (wl.T * wl.k // 256) * (wl.I // 128) > n_sms // 2:
        gemm_kernel = "grouped_gemm_bf16_pair_kernel"
    else:
        gemm_kernel = "grouped_gemm_bf16_kernel"
    if hbm_bound:
        # a weight-streaming step: the expert GEMMs against the measured copy bandwidth
        gb = gemm_bytes(wl, active)
        roof = {"bound": "hbm", "achieved": gb / (gemm_ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": gb / (gemm_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], "traffic": traffic, "algorithmic_bytes": gb,
                "kernel": gemm_kernel + " (gate/up + down launches of one step)",
                "peak_kind": f"HBM copy bandwidth, {peaks_kind}", "tflops": gemm_tflops}
    else:
        roof = {"bound": "tensor", "achieved": gemm_tflops, "peak": gemm_peak, "unit": "TFLOP/s",
                "frac": gemm_tflops / gemm_peak, "traffic": traffic,
                "kernel": gemm_kernel + " (gate/up + down launches of one step)",
                "peak_kind": (f"fp8 = 2 x bf16 burst ({peaks_kind}), nominal ratio" if wl.dtype == "fp8"
                              else f"bf16 burst, {peaks_kind}"),
                "frac_of_sustained": gemm_tflops / gemm_peak_sus,
                "timing": "moe_expert_ffn inside the step-entry-point path, CUDA events on the launching stream"}
    world = 1 if dist is None else dist.get_world_size()
    out = {
        "workload": wl.name, "steps": steps, "ms_per_step": ms_step, "value": job_tokens_per_s(world, wl.T, ms_step),
        "unit": UNIT,
        "l2": L2_FLUSHED if flush is not None else L2_LARGER,
        "roofline": roof,
        "layer_roofline": {"t_roof_ms": t_roof * 1e3, "frac": t_roof / (ms_step * 1e-3), "flops": flops,
                           "bytes": bytes_, "active_experts": active, "bound": "hbm" if hbm_bound else "tensor",
                           "peaks": peaks_kind},
        "balance": {"max_over_mean": bal["max_over_mean"], "active_experts": bal["active"],
                    "dropped_assignments": bal["dropped"]},
        "ms_moe_forward": ms_step, "ms_split_step": ms_split, "ms_expert_ffn": gemm_ms,
        "graph": {"value": job_tokens_per_s(world, wl.T, ms_graph), "unit": UNIT, "ms_per_step": ms_graph,
                  "note": "the same step replayed as one CUDA graph (moe_graph_launch)"},
        "e2e": {"value": job_tokens_per_s(world, wl.T, ms_e2e), "unit": UNIT, "ms_per_step": ms_e2e,
                "h2d_bytes_per_step": int(x.numel() * x.element_size()),
                "d2h_bytes_per_step": int(y.numel() * y.element_size())},
        "gpu_launches": int(n1 - n0), "launches_per_step": (n1 - n0) / steps,
        "clocks": clocks,
    }
    if sustained is not None:
        sustained["value"] = job_tokens_per_s(world, wl.T, sustained["ms_per_step"])
        sustained["unit"] = UNIT
        sustained["layer_roofline_frac"] = t_roof / (sustained["ms_per_step"] * 1e-3)
        out["sustained"] = sustained
    del cfg, weights, ws, x, y, it, xs, flush, x_host, y_host, x_dev, y_dev
    import gc

    gc.collect()
    torch.cuda.empty_cache()
    return out


def cpu_baseline_of(wl, budget_s):
    v_cpu, S, dt, used = time_cpu_oracle(wl, budget_s)
    return {"value": v_cpu, "unit": UNIT, "cores": omp_threads(), "cpu_model": cpu_model(), "kind": "oracle",
            "sample": f"{S} of the workload's tokens through the whole oracle layer in {dt:.1f} s of oracle "
                      f"time, every routed row with its own expert's weights ({used} experts); weight "
                      "generation on the host not timed"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="dsv3_prefill")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="time only the headline workload")
    ap.add_argument("--sustain", type=float, default=3.0, help="seconds of the sustained window (0: none)")
    ap.add_argument("--tokens", type=int, default=None, help="override T (small profiling cases)")
    ap.add_argument("--experts", type=int, default=None, help="override E (small profiling cases)")
    ap.add_argument("--fp8-peak", action="store_true",
                    help="measure the library FP8 GEMM rate (cuBLASLt through torch._scaled_mm) and exit")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.fp8_peak:
        measure_fp8_peak()
        return

    import synth

    wl = synth.WORKLOADS[args.workload]
    small = args.tokens is not None or args.experts is not None
    if small:
        wl = wl.replace(name=f"{wl.name}_T{args.tokens or wl.T}_E{args.experts or wl.E}", T=args.tokens or wl.T,
                        E=args.experts or wl.E)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus)))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        reference_arm(args, wl, rank, world)
        return

    import torch

    import routing_dispatch_expert_gb300 as rde
    from routing_dispatch_expert_gb300 import build as pkg_build

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if rank == 0 or world > 1:
        pkg_build.build()
        synth.build()
    if dist is not None:
        dist.barrier()
    rde.load()
    dev = torch.device("cuda", local_rank)
    gpu_index = os.environ.get("CUDA_VISIBLE_DEVICES", str(local_rank)).split(",")[0] if world == 1 else local_rank

    head = measure(wl, args, dev, dist, rde, synth, torch, args.steps, gpu_index,
                   sustain_s=0.0 if small else args.sustain)
    # every other configuration of the layer, one after another on the same GPU (1-GPU runs only)
    per_config = {}
    if world == 1 and not small and not args.no_per_config:
        for name in PER_CONFIG:
            if name == wl.name:
                continue
            w2 = synth.WORKLOADS[name]
            # sub-millisecond steps: more of them, so the timed region is not a few microseconds
            per_config[name] = measure(w2, args, dev, dist, rde, synth, torch, args.steps, gpu_index)
            if per_config[name]["ms_per_step"] < 1.0:
                per_config[name] = measure(w2, args, dev, dist, rde, synth, torch, args.steps * 25, gpu_index)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_of(wl, 12.0)
        for name, entry in per_config.items():
            entry["cpu_baseline"] = cpu_baseline_of(synth.WORKLOADS[name], 3.0)

    if rank == 0:
        line = {
            "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3" if wl.dtype == "fp8" else "bf16",
            "data": "synthetic", "config": config_of(wl, world),
        }
        for key in ("roofline", "layer_roofline", "balance", "ms_moe_forward", "ms_split_step", "ms_expert_ffn",
                    "graph", "e2e", "gpu_launches", "clocks", "sustained"):
            if key in head:
                line[key] = head[key]
        line["cpu_baseline"] = cpu
        if per_config:
            line["per_config"] = per_config
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
