#!/usr/bin/env python3
"""Benchmark of the GB300 affine-quantised MoE FFN block.

Default workload (one "step" = one decode token through the whole hot path):
a 30-layer stack of independent MoE layers (hidden 2816, inter 704, 128
experts, top-8, 4-bit experts, 8-bit router, group 64; layer l generated with
seed l, all 30 x 128 experts resident in HBM), 256 steps, each step one fresh
N(0,1) hidden state, x_l = rmsnorm_no_scale(h_l), h_{l+1} = h_l + MoE_l(x_l).
The 30 layer calls of a step are captured in one CUDA graph; each call is one
launch of the fused layer kernel, chained with programmatic dependent launch.

Prints one JSON line (see the keys below).  `--impl reference` times the
float64 CPU oracle instead, on a bounded sample of the same workload.

Other workloads for development: --workload layer1 (one layer, T=1),
prefill128 (one layer, T=128, Zipf-skewed routing), batch64 (one layer, 64
independent tokens), prefill30 (30 layers x 128-token chunks, Zipf).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

H, I, E, K = 2816, 704, 128, 8
N_LAYERS = 30
ROUTER_BYTES = E * H + 2 * E * (H // 64) * 2                                   # 382,976
EXPERT_BYTES = 3 * (I * H // 2 + 2 * I * (H // 64) * 2)                          # 3,345,408
MEASURED_PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
CSRC = os.path.join(ROOT, "bit_affine_quantized_gb300", "csrc")
# per-launch DRAM traffic of the fused kernels, from committed ncu summaries:
# (summary file, sources that define the kernel)
TRAFFIC = {
    1: ("decode_layer_kernel_T1.md", ("decode.cu", "common.cuh")),
    128: ("prefill_layer_kernel_T128.md", ("prefill.cu", "fused.cuh", "common.cuh")),
}


# steps of each workload when it is timed as a sub-record of the default line
SUB_STEPS = {"layer1": 64, "batch64": 32, "prefill128": 32, "prefill30": 8}
# the tied 4-bit head (vocabulary 262,144 x hidden 2816, group-64 affine) on one
# decoded token: greedy token only, softcap 30
HEAD_V, HEAD_STEPS, HEAD_SOFTCAP = 262144, 32, 30.0
# the whole-prompt layer: a 4096-row prompt (32 chunks of 128) through the
# 30-layer stack layer-major, each layer one moe_layer_forward_prompt call
PROMPT_ROWS, PROMPT_STEPS = 4096, 4
# expert offload: a 4-layer decode stack (Zipf-skewed routing, the pages'
# premise) with each layer's routed experts in pinned host memory behind 16
# device slots per layer
OFFLOAD_LAYERS, OFFLOAD_SLOTS, OFFLOAD_WARM, OFFLOAD_STEPS = 4, 16, 16, 48


def layer_bytes(n_tokens: int, distinct_routed: int) -> int:
    """Algorithmic bytes of one layer call: router + touched experts + shared
    + bf16 activations in and out."""
    return ROUTER_BYTES + (distinct_routed + 1) * EXPERT_BYTES + 2 * n_tokens * H * 2


WORKLOADS = {
    "decode30": dict(layers=N_LAYERS, tokens=1, zipf=False, rms=False, residual=True,
                     desc="decode, 30-layer MoE stack, 1 token per step, fresh N(0,1) hidden state per step"),
    "layer1": dict(layers=8, tokens=1, zipf=False, rms=True, residual=False,
                   desc="decode, one MoE layer, 1 token per step (8 layer copies rotated: 3.5 GB > L2)"),
    "batch64": dict(layers=8, tokens=64, zipf=False, rms=True, residual=False,
                    desc="batched decode, one MoE layer, 64 independent tokens, uniform routing (8 copies rotated)"),
    "prefill128": dict(layers=8, tokens=128, zipf=True, rms=True, residual=False,
                       desc="prefill chunk, one MoE layer, 128 tokens, Zipf(1.1) logit offsets (8 copies rotated)"),
    "prefill30": dict(layers=N_LAYERS, tokens=128, zipf=True, rms=True, residual=True,
                      desc="prefill, 30-layer MoE stack, 128-token chunks, Zipf(1.1) logit offsets per layer"),
}


# ---------------------------------------------------------------- helpers
def sources_sha256(files) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def traffic_per_launch(T: int):
    """DRAM bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)
    from the committed summary for this token count, or None when there is
    none or the kernel's sources changed since it was taken."""
    if T not in TRAFFIC:
        return None, "no capture for this token count"
    name, files = TRAFFIC[T]
    path = os.path.join(ROOT, "profiles", name)
    try:
        fields = {}
        with open(path) as f:
            for line in f:
                if "=" in line and line.strip().startswith("- "):
                    k, v = line.strip()[2:].split("=", 1)
                    fields[k.strip()] = v.strip().strip("`")
        if fields.get("kernel_sources_sha256") != sources_sha256(files):
            return None, f"profiles/{name}: kernel changed since the capture"
        return int(fields["traffic_bytes_per_launch"]), f"profiles/{name}"
    except Exception as exc:
        return None, f"profiles/{name}: {type(exc).__name__}"


def peaks():
    try:
        with open(MEASURED_PEAKS) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Maximum of a per-rank float over all ranks (identity when world == 1)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- our arm
class Layers:
    """The 30 synthetic layers (seed = layer index), resident in HBM, with the
    Zipf logit offsets of each layer as a separate small tensor: workloads
    with Zipf-skewed routing use the same weights plus that offset."""

    def __init__(self, device, n_layers=N_LAYERS):
        import torch
        import bit_affine_quantized_gb300 as bq
        from synth import gen
        from synth.device import DeviceLayer
        self.layers = [DeviceLayer(l, H, I, E, device=device) for l in range(n_layers)]
        self.bias = [torch.from_numpy(gen.zipf_logit_bias(l, E)).to(device) for l in range(n_layers)]
        dims = bq.make_dims(H, I, E, K)
        self.plain = [bq.layer_weights_from(dims, L.addresses()) for L in self.layers]
        self.zipf = []
        for L, b in zip(self.layers, self.bias):
            addr = dict(L.addresses())
            addr["logit_bias"] = b.data_ptr()
            self.zipf.append(bq.layer_weights_from(dims, addr))

    def weights(self, spec):
        w = self.zipf if spec["zipf"] else self.plain
        return w[:spec["layers"]]


def time_workload(moe, spec, weights, steps, warmup, rank, device, e2e=False, clocks=False):
    """Times `steps` steps of a workload after `warmup` untimed ones.

    A step is one pass of the hot path over one batch of synthetic input:
    for residual workloads every layer of the stack on one chunk (one CUDA
    graph), otherwise one layer call on one chunk, the layer copies rotated
    across steps so that L2 never holds the next step's weights.  Returns
    the step time (CUDA events on the launching stream around the whole
    timed region), the summed duration of the layer calls (events around
    each graph replay), the distinct experts touched, and optionally the
    end-to-end time with host buffers and the clocks sampled meanwhile."""
    import torch
    from synth import gen

    T = spec["tokens"]
    steps_total = warmup + steps
    chunk_seed = 1000 + 7919 * rank
    host_in = np.stack([gen.hidden_states(chunk_seed, s, T, H, rms_normalize=spec["rms"])
                        for s in range(steps_total)])                       # [S, T, H] bf16 bits
    inputs = torch.from_numpy(host_in.view(np.int16)).to(device)
    outputs = torch.empty_like(inputs)
    h = torch.empty((T, H), dtype=torch.int16, device=device)
    y = torch.empty_like(h)
    ws = torch.empty(moe.workspace_bytes(weights[0].dims, T), dtype=torch.uint8, device=device)
    stream = torch.cuda.Stream(device=device)
    ids = torch.empty((len(weights), T, K), dtype=torch.int32, device=device)

    def call(li):
        if spec["residual"]:
            moe.layer_forward_residual(h, T, weights[li], ws, ids_out=ids[li], stream=stream)
        else:
            moe.layer_forward(h, T, weights[li], y, ws, ids_out=ids[li], stream=stream)

    graphs = []
    h.copy_(inputs[0])
    torch.cuda.synchronize(device)
    with torch.cuda.stream(stream):
        if spec["residual"]:
            for li in range(len(weights)):
                call(li)  # warm the code path once outside capture
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for li in range(len(weights)):
                    call(li)
            graphs.append(g)
        else:
            for li in range(len(weights)):
                call(li)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    call(li)
                graphs.append(g)
    torch.cuda.synchronize(device)
    st = moe.get_error()
    if st != 0:
        raise RuntimeError(f"device error status {st} during warm-up")
    out_src = h if spec["residual"] else y

    # launches per layer call, read from the trace slots the kernels stamp
    trace = torch.zeros(4 * 8, dtype=torch.int64, device=device)
    moe.set_trace(trace, 8)
    with torch.cuda.stream(stream):
        call(0)
    torch.cuda.synchronize(device)
    moe.set_trace(None, 0)
    launches_per_call = int((trace.view(8, 4) != 0).any(dim=1).sum())
    calls_per_step = len(weights) if spec["residual"] else 1

    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps_total)]

    def one_step(s):
        h.copy_(inputs[s], non_blocking=True)
        kev[s][0].record(stream)
        graphs[s % len(graphs)].replay()
        kev[s][1].record(stream)
        outputs[s].copy_(out_src, non_blocking=True)

    with torch.cuda.stream(stream):
        for s in range(warmup):
            one_step(s)
    torch.cuda.synchronize(device)
    sampler = None
    if clocks:
        sampler = ClockSampler(torch.device(device).index or 0)
        sampler.start()
        time.sleep(0.3)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for s in range(warmup, steps_total):
            one_step(s)
        ev1.record(stream)
    torch.cuda.synchronize(device)
    res = {"elapsed_ms": ev0.elapsed_time(ev1),
           "kernel_ms": sum(a.elapsed_time(b) for a, b in kev[warmup:steps_total]),
           "launches_per_call": launches_per_call, "calls_per_step": calls_per_step}
    if sampler is not None:
        res["clocks"] = sampler.stop()
    st = moe.get_error()
    if st != 0:
        raise RuntimeError(f"device error status {st} during the timed region")

    # algorithmic bytes: distinct experts actually touched per layer call
    ids_np = ids.cpu().numpy()
    if spec["residual"]:
        distinct = [len(np.unique(ids_np[l])) for l in range(len(weights))]
    else:
        distinct = [len(np.unique(ids_np[(steps_total - 1) % len(graphs)]))]
    res["distinct"] = distinct
    res["bytes_per_call"] = sum(layer_bytes(T, d) for d in distinct) / len(distinct)
    res["bytes_per_step"] = res["bytes_per_call"] * calls_per_step

    if e2e:
        # end to end through the public API with host buffers: pinned H2D of
        # the step's input, the layer calls, D2H of the result, every step
        pin_in = torch.from_numpy(host_in.view(np.int16)).pin_memory()
        pin_out = torch.empty_like(pin_in).pin_memory()
        torch.cuda.synchronize(device)
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for s in range(steps):
                h.copy_(pin_in[s], non_blocking=True)
                graphs[s % len(graphs)].replay()
                pin_out[s].copy_(out_src, non_blocking=True)
                stream.synchronize()
        res["e2e_s"] = time.perf_counter() - t0
    return res


def summary(spec, res, steps, world, hbm):
    """Throughput, per-call time and roofline fraction of one timed workload."""
    T = spec["tokens"]
    call_us = res["kernel_ms"] * 1e3 / (steps * res["calls_per_step"])
    achieved = res["bytes_per_call"] / (call_us / 1e6) / 1e9
    return {"value": world * T * steps / (res["elapsed_ms"] / 1e3), "ms_per_step": res["elapsed_ms"] / steps,
            "call_us": call_us, "achieved": achieved, "frac": achieved / hbm}


def kernel_name(spec, res):
    if res["launches_per_call"] != 1:
        return "router + gate/up + down launches (MOE_*_FUSED=0)"
    return "decode_layer_kernel" if spec["tokens"] == 1 else "prefill_layer_kernel"


def run_ours(args, spec, rank, world, device):
    import bit_affine_quantized_gb300 as bq

    bq.build_library()
    moe = bq.Moe()
    layers = Layers(device)
    hbm, peak_kind = peaks()
    T = spec["tokens"]
    barrier(world)
    res = time_workload(moe, spec, layers.weights(spec), args.steps, args.warmup, rank, device, e2e=True,
                        clocks=True)
    for key in ("elapsed_ms", "kernel_ms", "e2e_s"):
        res[key] = max_over_ranks(res[key], world, device)
    barrier(world)
    sm = summary(spec, res, args.steps, world, hbm)
    fused = res["launches_per_call"] == 1
    traffic, traffic_src = traffic_per_launch(T) if fused else (None, "chained launches")
    line = {
        "metric": args.metric, "value": round(sm["value"], 3), "unit": args.unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sm["ms_per_step"], 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": spec["desc"], "layers": spec["layers"], "tokens_per_step": T, "hidden": H,
                   "inter": I, "experts": E, "top_k": K, "group": 64,
                   "l2": "inputs larger than L2: %.0f MB of touched weights per step (L2 129 MB)%s" % (
                       res["bytes_per_step"] / 1e6, "" if spec["residual"] else "; 8 layer copies rotated"),
                   "cuda_graph": True, "pdl": os.environ.get("MOE_PDL", "1") != "0",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": kernel_name(spec, res),
                     "achieved": round(sm["achieved"], 1), "peak": hbm, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(sm["frac"], 4), "traffic": traffic, "traffic_source": traffic_src,
                     "algorithmic_bytes_per_launch": round(res["bytes_per_call"]),
                     "launch_us": round(sm["call_us"], 3), "launches_timed": args.steps * res["calls_per_step"]},
        "e2e": {"value": round(world * T * args.steps / res["e2e_s"], 3), "unit": args.unit,
                "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * H * 2, "steps": args.steps},
        "gpu_launches": res["launches_per_call"] * res["calls_per_step"] * args.steps,
        "clocks": res["clocks"],
    }
    # the metric's other workloads, each timed on its own region after the main one
    if not args.no_workloads:
        subs = {}
        name = [k for k, v in WORKLOADS.items() if v is spec][0]
        for other, steps in SUB_STEPS.items():
            if other == name:
                continue
            ospec = WORKLOADS[other]
            r = time_workload(moe, ospec, layers.weights(ospec), steps, 3, rank, device)
            for key in ("elapsed_ms", "kernel_ms"):
                r[key] = max_over_ranks(r[key], world, device)
            o = summary(ospec, r, steps, world, hbm)
            otraffic = traffic_per_launch(ospec["tokens"])[0] if r["launches_per_call"] == 1 else None
            subs[other] = {"workload": ospec["desc"], "value": round(o["value"], 3),
                           "unit": "rows/s" if ospec["zipf"] else "tok/s", "steps": steps, "warmup": 3,
                           "ms_per_step": round(o["ms_per_step"], 5), "kernel": kernel_name(ospec, r),
                           "launch_us": round(o["call_us"], 3),
                           "algorithmic_bytes_per_launch": round(r["bytes_per_call"]),
                           "distinct_experts_per_call": round(float(np.mean(r["distinct"])), 2),
                           "achieved_gbs": round(o["achieved"], 1), "frac": round(o["frac"], 4),
                           "traffic": otraffic,
                           "gpu_launches": r["launches_per_call"] * r["calls_per_step"] * steps}
        subs["prompt30"] = time_prompt(moe, layers.weights(WORKLOADS["prefill30"]), device, world)
        subs["head"] = time_head(moe, device, hbm, world)
        subs["offload"] = time_offload(moe, device, world)
        line["workloads"] = subs
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(spec, args.cpu_seconds)
    moe.close()
    return line


def prompt_flops(n_rows: int) -> int:
    """Algorithmic FLOPs of one whole-prompt layer call: the router (2 T E H)
    and the gate, up and down contractions of every routed pair and every
    shared row (2 (T k + T) 3 I H)."""
    return 2 * n_rows * E * H + 2 * n_rows * (K + 1) * 3 * I * H


def time_prompt(moe, weights, device, world):
    """A PROMPT_ROWS-row prompt through the 30-layer stack (Zipf-skewed
    routing), one moe_layer_forward_prompt call per layer, the 30 calls of a
    step in one CUDA graph; CUDA events around each replay (inputs: a fresh
    RMS-normalised prompt per step, 433 MB of weights per layer > L2).  Also
    the per-call duration (events around each of the 30 calls, no graph)
    and, from the launch trace of one call, the two GEMM launches' spans."""
    import torch
    from synth import gen

    T = PROMPT_ROWS
    steps_total = 3 + PROMPT_STEPS
    inputs = torch.from_numpy(np.stack([gen.hidden_states(5000, s, T, H, rms_normalize=True)
                                        for s in range(steps_total)]).view(np.int16)).to(device)
    h = torch.empty((T, H), dtype=torch.int16, device=device)
    ws = torch.empty(moe.prompt_workspace_bytes(weights[0].dims, T), dtype=torch.uint8, device=device)
    st = torch.cuda.Stream(device)

    def step_calls():
        for w in weights:
            moe.layer_forward_prompt(h, T, w, ws, stream=st)

    h.copy_(inputs[0])
    torch.cuda.synchronize(device)
    with torch.cuda.stream(st):
        step_calls()  # warm the code path once outside capture
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            step_calls()
    torch.cuda.synchronize(device)
    assert moe.get_error() == 0, "prompt layer call reported an error"
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps_total)]
    with torch.cuda.stream(st):
        for s in range(steps_total):
            h.copy_(inputs[s], non_blocking=True)
            kev[s][0].record(st)
            g.replay()
            kev[s][1].record(st)
    torch.cuda.synchronize(device)
    assert moe.get_error() == 0, "prompt layer call reported an error"
    step_s = max_over_ranks(statistics.median(a.elapsed_time(b) for a, b in kev[3:]) / 1e3, world, device)
    # per call, events around each call (no graph)
    cev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in weights]
    with torch.cuda.stream(st):
        h.copy_(inputs[0], non_blocking=True)
        for (a, b), w in zip(cev, weights):
            a.record(st)
            moe.layer_forward_prompt(h, T, w, ws, stream=st)
            b.record(st)
    torch.cuda.synchronize(device)
    call_s = statistics.median(a.elapsed_time(b) for a, b in cev) / 1e3
    # per-launch spans of one call from the trace slots (first block past its
    # dependency wait to the last block's exit, device global timer)
    trace = torch.zeros(4 * 8, dtype=torch.int64, device=device)
    moe.set_trace(trace, 8)
    with torch.cuda.stream(st):
        moe.layer_forward_prompt(h, T, weights[0], ws, stream=st)
    torch.cuda.synchronize(device)
    moe.set_trace(None, 0)
    v = [int(q) & 0xFFFFFFFFFFFFFFFF for q in trace.cpu().tolist()]
    m64 = 0xFFFFFFFFFFFFFFFF
    names = ("router", "sort", "gather", "gemm_gate_up", "gemm_down", "combine")
    spans = {n: round(((v[4 * i + 3] - (v[4 * i + 1] ^ m64)) / 1e3), 1) if v[4 * i + 1] and v[4 * i + 3] else None
             for i, n in enumerate(names)}
    launches = sum(1 for i in range(6) if v[4 * i])
    flops = prompt_flops(T)
    gemm_us = (spans["gemm_gate_up"] or 0) + (spans["gemm_down"] or 0)
    peak = tensor_peak()
    del ws, inputs
    return {"workload": "prefill, 30-layer MoE stack, a %d-row prompt per step (32 chunks of 128), Zipf(1.1) logit "
                        "offsets per layer, each layer one whole-prompt call (all chunks' pairs grouped per expert, "
                        "expert tiles of eight in order)" % T,
            "value": round(world * T / step_s, 3), "unit": "rows/s", "steps": PROMPT_STEPS, "warmup": 3,
            "ms_per_step": round(step_s * 1e3, 4), "layer_call_us": round(call_s * 1e6, 2),
            "launches_per_call": launches, "launch_spans_us": spans,
            "roofline": {"bound": "tensor", "unit": "TFLOP/s", "peak": peak[0], "peak_kind": peak[1],
                         "algorithmic_flops_per_call": flops,
                         "achieved_call": round(flops / call_s / 1e12, 1),
                         "frac_call": round(flops / call_s / 1e12 / peak[0], 4),
                         "achieved_gemm": round((flops - 2 * T * E * H) / (gemm_us * 1e-6) / 1e12, 1) if gemm_us else None,
                         "frac_gemm": round((flops - 2 * T * E * H) / (gemm_us * 1e-6) / 1e12 / peak[0], 4)
                         if gemm_us else None},
            "gpu_launches": launches * len(weights) * PROMPT_STEPS}


def tensor_peak():
    """Dense fp16/bf16 tensor peak (TFLOP/s): the measured sustained figure
    (a kernel timed inside a long step), else the fallback."""
    try:
        with open(MEASURED_PEAKS) as f:
            p = json.load(f)
        return float(p["bf16_tflops_sustained"]), "measured sustained bf16 (fp16 runs at the same rate)"
    except Exception:
        return 1700.0, "fallback sustained bf16"


def time_head(moe, device, hbm, world):
    """The tied head, one token per call (greedy token), CUDA events over
    HEAD_STEPS calls on one stream after 3 warm-up calls; its 415 MB of codes,
    scales and biases stream from HBM on every call (larger than L2)."""
    import torch
    import bit_affine_quantized_gb300 as bq
    from synth import gen
    from synth.device import DeviceHead

    head = DeviceHead(11, HEAD_V, H, device=device)
    hw = bq.make_head_weights(head.vocab, head.hidden, *head.addresses())
    x = torch.from_numpy(gen.hidden_states(2026, 0, 1, H, True).view(np.int16)).to(device)
    tok = torch.empty(1, dtype=torch.int32, device=device)
    st = torch.cuda.Stream(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(st):
        for _ in range(3):
            moe.head_forward(x, 1, hw, HEAD_SOFTCAP, tokens=tok, stream=st)
        torch.cuda.synchronize(device)
        e0.record(st)
        for _ in range(HEAD_STEPS):
            moe.head_forward(x, 1, hw, HEAD_SOFTCAP, tokens=tok, stream=st)
        e1.record(st)
    torch.cuda.synchronize(device)
    assert moe.get_error() == 0, "head call reported an error"
    call_s = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, device) / HEAD_STEPS
    nbytes = HEAD_V * H // 2 + HEAD_V * (H // 64) * 4 + H * 2 + 4  # codes, bf16 scales + biases, x, token
    achieved = nbytes / call_s / 1e9
    del head
    return {"workload": "tied 4-bit head, vocabulary %d x hidden %d, one token per call, greedy token, softcap %g"
                        % (HEAD_V, H, HEAD_SOFTCAP),
            "value": round(world / call_s, 3), "unit": "tok/s", "steps": HEAD_STEPS, "warmup": 3,
            "kernel": "head_kernel", "launch_us": round(call_s * 1e6, 3), "algorithmic_bytes_per_launch": nbytes,
            "achieved_gbs": round(achieved, 1), "frac": round(achieved / hbm, 4), "traffic": None,
            "gpu_launches": HEAD_STEPS}


def time_offload(moe, device, world):
    """Decode through OFFLOAD_LAYERS layers with moe_layer_forward_offload:
    the router on the device, the ids to the host, the LFU slot cache, one
    host-to-device copy per missing expert, the block on the slots.  Each call
    waits on the stream (the CPU handoff), so the time is host wall clock over
    OFFLOAD_STEPS steps after OFFLOAD_WARM warm-up steps that fill the caches."""
    import torch
    import bit_affine_quantized_gb300 as bq
    from synth import gen
    from synth.device import DeviceLayer

    dims = bq.make_dims(H, I, E, K)
    layers, hosts, ws_off, slots = [], [], [], []
    for l in range(OFFLOAD_LAYERS):
        L = DeviceLayer(100 + l, H, I, E, device=device, zipf=True)
        n = E * L.stride
        host = torch.empty(n, dtype=torch.uint8, pin_memory=True)
        host.copy_(L.buf[L.experts_off:L.experts_off + n])
        addr = dict(L.addresses())
        addr["experts"] = host.data_ptr()
        layers.append(L)
        hosts.append(host)
        ws_off.append(bq.layer_weights_from(dims, addr))
        slots.append(torch.empty(OFFLOAD_SLOTS * L.stride, dtype=torch.uint8, device=device))
    stride = layers[0].stride
    blob = ws_off[0].layout.down_b + (H * (I // 64) * 2)  # extent of one blob's sub-tensors
    cache = bq.ExpertCache(OFFLOAD_LAYERS, OFFLOAD_SLOTS)
    ws = torch.empty(moe.workspace_bytes(dims, 1), dtype=torch.uint8, device=device)
    h = torch.empty((1, H), dtype=torch.int16, device=device)
    st = torch.cuda.Stream(device)
    inputs = [torch.from_numpy(gen.hidden_states(3000, s, 1, H, False).view(np.int16)).to(device)
              for s in range(OFFLOAD_WARM + OFFLOAD_STEPS)]

    def step(s):
        with torch.cuda.stream(st):
            h.copy_(inputs[s])
            for l in range(OFFLOAD_LAYERS):
                moe.layer_forward_offload(h, cache, l, ws_off[l], slots[l], ws, stream=st)
        torch.cuda.synchronize(device)

    for s in range(OFFLOAD_WARM):
        step(s)
    before = [cache.stats(l) for l in range(OFFLOAD_LAYERS)]
    t0 = time.perf_counter()
    for s in range(OFFLOAD_WARM, OFFLOAD_WARM + OFFLOAD_STEPS):
        step(s)
    elapsed = max_over_ranks(time.perf_counter() - t0, world, device)
    assert moe.get_error() == 0, "offload call reported an error"
    after = [cache.stats(l) for l in range(OFFLOAD_LAYERS)]
    hits = sum(a[0] - b[0] for a, b in zip(after, before))
    misses = sum(a[1] - b[1] for a, b in zip(after, before))
    cache.close()
    per_layer_us = elapsed / (OFFLOAD_STEPS * OFFLOAD_LAYERS) * 1e6
    h2d = misses * blob / OFFLOAD_STEPS
    del layers, hosts, slots
    return {"workload": "decode, %d-layer MoE stack with routed experts in pinned host memory, %d device slots per "
                        "layer, least-frequently-used eviction (recency breaks ties), Zipf(1.1) logit offsets"
                        % (OFFLOAD_LAYERS, OFFLOAD_SLOTS),
            "value": round(world * OFFLOAD_STEPS / elapsed, 3), "unit": "tok/s", "steps": OFFLOAD_STEPS,
            "warmup": OFFLOAD_WARM, "timing": "host wall clock (each call waits on the stream for the ids)",
            "layers": OFFLOAD_LAYERS, "layer_us": round(per_layer_us, 2),
            "hit_rate": round(hits / max(1, hits + misses), 4), "expert_loads_per_step": round(misses / OFFLOAD_STEPS, 2),
            "h2d_bytes_per_step": round(h2d), "gpu_launches": None}


# ---------------------------------------------------------------- oracle arm
def _oracle_sample(spec, seconds: float, chunk: int, layer_cap: int = 30):
    """Times the float64 oracle on a bounded sample of the workload: one
    token-chunk (input `chunk`) through consecutive layers until `seconds` of
    oracle time.  Returns (seconds per (layer, chunk), layers timed)."""
    from oracle import moe_oracle as O
    from synth import gen

    T = spec["tokens"]
    h = gen.hidden_states(1000, chunk, T, H, rms_normalize=spec["rms"])
    spent, timed = 0.0, 0
    for l in range(min(layer_cap, spec["layers"])):
        router = gen.router_weights(l, E, H)
        bias = gen.zipf_logit_bias(l, E) if spec["zipf"] else None
        shared = gen.expert_weights(l, gen.SHARED_ID, H, I)
        x = O.rmsnorm_no_scale(h) if spec["residual"] else h
        ids = O.select_top_k(O.router_logits(x, router, bias), K)          # routing, untimed
        experts = {int(e): gen.expert_weights(l, int(e), H, I) for e in np.unique(ids)}  # inputs, untimed
        t0 = time.perf_counter()
        if spec["residual"]:
            out = O.stack_layer(h, router, experts.__getitem__, shared, K, bias)
            h = out["h_next"]
        else:
            O.moe_block(x, router, experts.__getitem__, shared, K, bias)
        spent += time.perf_counter() - t0
        timed += 1
        if spent >= seconds:
            break
    return spent / timed, timed


def _oracle_steps(spec, steps):
    """Oracle time of layer 0 of the stack on the inputs of the given steps
    (one bounded sample per step of the reference arm)."""
    from oracle import moe_oracle as O
    from synth import gen
    router = gen.router_weights(0, E, H)
    bias = gen.zipf_logit_bias(0, E) if spec["zipf"] else None
    shared = gen.expert_weights(0, gen.SHARED_ID, H, I)
    out = []
    for s in steps:
        h = gen.hidden_states(1000, s, spec["tokens"], H, rms_normalize=spec["rms"])
        x = O.rmsnorm_no_scale(h) if spec["residual"] else h
        ids = O.select_top_k(O.router_logits(x, router, bias), K)
        experts = {int(e): gen.expert_weights(0, int(e), H, I) for e in np.unique(ids)}
        t0 = time.perf_counter()
        if spec["residual"]:
            O.stack_layer(h, router, experts.__getitem__, shared, K, bias)
        else:
            O.moe_block(x, router, experts.__getitem__, shared, K, bias)
        out.append(time.perf_counter() - t0)
    return out


def oracle_cores() -> int:
    """Host cores available to the oracle's worker processes."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def _oracle_pool(name: str, jobs):
    """Runs one child process per job (a list of extra arguments) at once,
    each on one BLAS thread: every host core runs whole layer calls of its
    own, the processes split the work by input chunk or step, and no result
    depends on how many there are.  Returns the children's results in job
    order."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    procs = []
    for extra in jobs:
        cmd = [sys.executable, os.path.abspath(__file__), "--oracle-sample", name, *extra]
        procs.append(subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, env=env))
    out = []
    for p in procs:
        o, e = p.communicate(timeout=1800)
        if p.returncode != 0:
            raise RuntimeError(e[-800:])
        out.append(json.loads(o.strip().splitlines()[-1]))
    return out


def cpu_baseline(spec, seconds: float) -> dict:
    """The float64 oracle on all host cores: one process per core, each
    timing whole layer calls on its own input chunk for about `seconds`."""
    name = [k for k, v in WORKLOADS.items() if v is spec][0]
    cores = oracle_cores()
    try:
        t0 = time.perf_counter()
        res = _oracle_pool(name, [["--cpu-seconds", str(seconds), "--oracle-chunk", str(c)] for c in range(cores)])
        wall = time.perf_counter() - t0
    except Exception as exc:  # reported, never fatal for the GPU number
        return {"value": None, "error": str(exc)[-400:]}
    T = spec["tokens"]
    layers = spec["layers"] if spec["residual"] else 1
    per_core = [T / (per_layer * layers) for per_layer, _ in res]
    calls = sum(n for _, n in res)
    mean_call = float(np.mean([p for p, _ in res]))
    return {"value": round(sum(per_core), 6), "unit": "rows/s" if spec["zipf"] else "tok/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{cores} processes, one per host core, each timing whole layer calls of {T} token(s) on its "
                      f"own input chunk for about {seconds:.0f} s ({calls} calls in all, {mean_call:.2f} s each); "
                      f"per-core throughput = tokens / (seconds per call x {layers} layer(s) per step), summed "
                      f"over the cores; numpy float64, one BLAS thread per process; {wall:.1f} s wall"}


def run_reference(args, spec, rank, world):
    if rank != 0:
        return None
    name = [k for k, v in WORKLOADS.items() if v is spec][0]
    cores = oracle_cores()
    steps = list(range(args.warmup + args.steps))
    per = [p for p in (steps[i::cores] for i in range(cores)) if p]
    t0 = time.perf_counter()
    res = _oracle_pool(name, [["--oracle-steps", ",".join(map(str, p))] for p in per])
    wall = time.perf_counter() - t0
    times = {}
    for p, r in zip(per, res):
        times.update(zip(p, r))
    timed = [times[s] for s in steps[args.warmup:]]
    per_layer = sum(timed) / len(timed)
    layers = spec["layers"] if spec["residual"] else 1
    T = spec["tokens"]
    used = len(per)
    value = used * T / (per_layer * layers)
    unit = "rows/s" if spec["zipf"] else "tok/s"
    return {
        "impl": "reference", "metric": args.metric, "value": round(value, 6), "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_layer * layers * 1e3, 3),
        "ms_per_step_kind": f"extrapolated: layer 0 timed on each step's input ({per_layer * 1e3:.1f} ms), "
                            f"x {layers} layer(s)",
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": spec["desc"], "layers": spec["layers"], "tokens_per_step": T},
        "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": used, "kind": "oracle",
                         "sample": f"each step: layer 0 of the stack for {T} token(s) in the float64 oracle, "
                                   f"scaled to {layers} layer(s); the {len(steps)} steps spread over {used} "
                                   f"processes (one per host core, one BLAS thread each), throughput summed over "
                                   f"them; {wall:.1f} s wall"},
        "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------- main
def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="decode30")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-sample", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-steps", default="", help=argparse.SUPPRESS)
    ap.add_argument("--oracle-chunk", type=int, default=0, help=argparse.SUPPRESS)
    ap.add_argument("--no-workloads", action="store_true",
                    help="time only the selected workload (no sub-records of the other four)")
    args = ap.parse_args(argv)
    if args.oracle_sample:
        spec = WORKLOADS[args.oracle_sample]
        if args.oracle_steps:
            print(json.dumps(_oracle_steps(spec, [int(v) for v in args.oracle_steps.split(",")])))
        else:
            print(json.dumps(_oracle_sample(spec, args.cpu_seconds, args.oracle_chunk)))
        return 0
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    spec = WORKLOADS[args.workload]
    multi = spec["tokens"] > 1
    args.metric = ("MoE-layer prefill rows/s" if multi and spec["zipf"] else
                   "MoE-layer decode tokens/s") + (" (30-layer stack)" if spec["residual"] else " (one layer)")
    args.unit = "rows/s" if multi and spec["zipf"] else "tok/s"
    rank, local_rank, world = dist_env()

    if args.impl == "reference":
        line = run_reference(args, spec, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0

    import torch
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    line = run_ours(args, spec, rank, world, device)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
