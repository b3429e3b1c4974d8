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
    1: ("decode_layer_kernel_T1.md", ("decode.cu", "common.cuh", "kernels.h")),
    128: ("prefill_layer_kernel_T128.md", ("prefill.cu", "fused.cuh", "common.cuh", "kernels.h")),
}


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
def build_layers(spec, device):
    from synth.device import DeviceLayer
    return [DeviceLayer(l, H, I, E, device=device, zipf=spec["zipf"]) for l in range(spec["layers"])]


def run_ours(args, spec, rank, world, device):
    import torch
    import bit_affine_quantized_gb300 as bq
    from synth import gen

    bq.build_library()
    moe = bq.Moe()
    dims = bq.make_dims(H, I, E, K)
    layers = build_layers(spec, device)
    weights = [bq.layer_weights_from(dims, L.addresses()) for L in layers]
    T = spec["tokens"]
    steps_total = args.warmup + args.steps
    # per-step inputs, resident in HBM before the timed region
    chunk_seed = 1000 + 7919 * rank
    host_in = np.stack([gen.hidden_states(chunk_seed, s, T, H, rms_normalize=spec["rms"])
                        for s in range(steps_total)])                       # [S, T, H] bf16 bits
    inputs = torch.from_numpy(host_in.view(np.int16)).to(device)
    outputs = torch.empty_like(inputs)
    h = torch.empty((T, H), dtype=torch.int16, device=device)
    y = torch.empty_like(h)
    ws = torch.empty(moe.workspace_bytes(dims, T), dtype=torch.uint8, device=device)
    stream = torch.cuda.Stream(device=device)
    ids = torch.empty((spec["layers"], T, K), dtype=torch.int32, device=device)

    def step_body():
        # the graph body: all layers of one step on `h`
        for l, w in enumerate(weights):
            li = l % len(weights)
            if spec["residual"]:
                moe.layer_forward_residual(h, T, weights[li], ws, ids_out=ids[li], stream=stream)
            else:
                moe.layer_forward(h, T, weights[li], y, ws, ids_out=ids[li], stream=stream)
            if not spec["residual"]:
                break

    # non-residual workloads rotate layer copies across steps (cold L2)
    graphs = []
    h.copy_(inputs[0])
    torch.cuda.synchronize(device)
    with torch.cuda.stream(stream):
        if spec["residual"]:
            g = torch.cuda.CUDAGraph()
            step_body()  # warm the code path once outside capture
            with torch.cuda.graph(g, stream=stream):
                step_body()
            graphs.append(g)
        else:
            for li, w in enumerate(weights):
                g = torch.cuda.CUDAGraph()
                moe.layer_forward(h, T, w, y, ws, ids_out=ids[li], stream=stream)
                with torch.cuda.graph(g, stream=stream):
                    moe.layer_forward(h, T, w, y, ws, ids_out=ids[li], stream=stream)
                graphs.append(g)
    torch.cuda.synchronize(device)
    st = moe.get_error()
    if st != bq.MOE_OK:
        raise RuntimeError(f"device error status {st} during warm-up")

    out_src = h if spec["residual"] else y

    # launches per layer call, read from the trace slots the kernels stamp
    trace = torch.zeros(4 * 8, dtype=torch.int64, device=device)
    moe.set_trace(trace, 8)
    with torch.cuda.stream(stream):
        if spec["residual"]:
            moe.layer_forward_residual(h, T, weights[0], ws, stream=stream)
        else:
            moe.layer_forward(h, T, weights[0], y, ws, stream=stream)
    torch.cuda.synchronize(device)
    moe.set_trace(None, 0)
    launches_per_call = int((trace.view(8, 4) != 0).any(dim=1).sum())
    calls_per_step = spec["layers"] if spec["residual"] else 1

    # the kernels' own time: events around each graph replay, on its stream
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps_total)]

    def one_step(s):
        h.copy_(inputs[s], non_blocking=True)
        kev[s][0].record(stream)
        graphs[s % len(graphs)].replay()
        kev[s][1].record(stream)
        outputs[s].copy_(out_src, non_blocking=True)

    with torch.cuda.stream(stream):
        for s in range(args.warmup):
            one_step(s)
    torch.cuda.synchronize(device)
    sampler = ClockSampler(torch.cuda.current_device() if device is None else torch.device(device).index or 0)
    barrier(world)
    torch.cuda.synchronize(device)
    sampler.start()
    time.sleep(0.3)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for s in range(args.warmup, steps_total):
            one_step(s)
        ev1.record(stream)
    torch.cuda.synchronize(device)
    elapsed_ms = ev0.elapsed_time(ev1)
    kernel_ms = sum(a.elapsed_time(b) for a, b in kev[args.warmup:steps_total])
    clocks = sampler.stop()
    barrier(world)
    st = moe.get_error()
    if st != bq.MOE_OK:
        raise RuntimeError(f"device error status {st} during the timed region")

    elapsed_ms = max_over_ranks(elapsed_ms, world, device)
    ms_per_step = elapsed_ms / args.steps
    units_per_step = T  # tokens (rows) per step per rank
    value = world * units_per_step * args.steps / (elapsed_ms / 1e3)

    # algorithmic bytes: distinct experts actually touched per layer call
    ids_np = ids.cpu().numpy()
    if spec["residual"]:
        n_calls = spec["layers"]
        distinct = [len(np.unique(ids_np[l])) for l in range(n_calls)]
    else:
        n_calls = 1
        distinct = [len(np.unique(ids_np[(steps_total - 1) % len(graphs)]))]
    bytes_per_step = sum(layer_bytes(T, d) for d in distinct)
    bytes_per_call = bytes_per_step / n_calls
    hbm, peak_kind = peaks()
    # one layer call is one launch of the fused kernel (the dominant and only
    # kernel of the step); its average duration over the timed region
    call_us = max_over_ranks(kernel_ms, world, device) * 1e3 / (args.steps * calls_per_step)
    achieved = bytes_per_call / (call_us / 1e6) / 1e9
    fused = launches_per_call == 1
    traffic, traffic_src = traffic_per_launch(T) if fused else (None, "chained launches")

    # end to end through the public API with host buffers: pinned H2D of the
    # step's input, the layer calls, D2H of the result, every step
    pin_in = torch.from_numpy(host_in.view(np.int16)).pin_memory()
    pin_out = torch.empty_like(pin_in).pin_memory()
    e2e_steps = args.steps
    torch.cuda.synchronize(device)
    barrier(world)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for s in range(e2e_steps):
            h.copy_(pin_in[s], non_blocking=True)
            graphs[s % len(graphs)].replay()
            pin_out[s].copy_(out_src, non_blocking=True)
            stream.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, device)
    e2e_value = world * units_per_step * e2e_steps / e2e_s

    kernel_name = ("decode_layer_kernel" if T == 1 else "prefill_layer_kernel") if fused else \
        "router + gate/up + down launches (MOE_*_FUSED=0)"
    line = {
        "metric": args.metric, "value": round(value, 3), "unit": args.unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": spec["desc"], "layers": spec["layers"], "tokens_per_step": T, "hidden": H,
                   "inter": I, "experts": E, "top_k": K, "group": 64,
                   "l2": "inputs larger than L2: %.0f MB of touched weights per step (L2 129 MB)%s" % (
                       bytes_per_step / 1e6, "" if spec["residual"] else "; 8 layer copies rotated"),
                   "cuda_graph": True, "pdl": os.environ.get("MOE_PDL", "1") != "0",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": kernel_name,
                     "achieved": round(achieved, 1), "peak": hbm, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "traffic": traffic, "traffic_source": traffic_src,
                     "algorithmic_bytes_per_launch": round(bytes_per_call), "launch_us": round(call_us, 3),
                     "launches_timed": args.steps * calls_per_step},
        "e2e": {"value": round(e2e_value, 3), "unit": args.unit, "h2d_bytes_per_step": T * H * 2,
                "d2h_bytes_per_step": T * H * 2, "steps": e2e_steps},
        "gpu_launches": launches_per_call * calls_per_step * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(spec, args.cpu_seconds)
    moe.close()
    return line


# ---------------------------------------------------------------- oracle arm
def _oracle_sample(spec, seconds: float, layer_cap: int = 30):
    """Times the float64 oracle on a bounded sample of the workload: one
    token-chunk through consecutive layers until `seconds` of oracle time.
    Returns (seconds per (layer, chunk), layers timed)."""
    from oracle import moe_oracle as O
    from synth import gen

    T = spec["tokens"]
    h = gen.hidden_states(1000, 0, T, H, rms_normalize=spec["rms"])
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


def _oracle_child(name: str, seconds: float, steps: int = 0):
    """Runs the oracle sample in a child process pinned to one BLAS thread."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-sample", name, "--cpu-seconds", str(seconds),
           "--oracle-steps", str(steps)]
    res = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=1800)
    if res.returncode != 0:
        raise RuntimeError(res.stderr[-800:])
    return json.loads(res.stdout.strip().splitlines()[-1])


def _oracle_steps(spec, steps: int):
    """Per-step oracle time of layer 0 on fresh inputs (reference arm)."""
    from oracle import moe_oracle as O
    from synth import gen
    router = gen.router_weights(0, E, H)
    bias = gen.zipf_logit_bias(0, E) if spec["zipf"] else None
    shared = gen.expert_weights(0, gen.SHARED_ID, H, I)
    out = []
    for s in range(steps):
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


def cpu_baseline(spec, seconds: float) -> dict:
    """Oracle on the host in a child process pinned to one BLAS thread."""
    name = [k for k, v in WORKLOADS.items() if v is spec][0]
    try:
        per_layer, timed = _oracle_child(name, seconds)
    except Exception as exc:  # reported, never fatal for the GPU number
        return {"value": None, "error": str(exc)[-400:]}
    T = spec["tokens"]
    value = T / (per_layer * (spec["layers"] if spec["residual"] else 1))
    return {"value": round(value, 6), "unit": "tok/s", "cores": 1, "kind": "oracle",
            "sample": f"{timed} layer call(s) of {T} token(s) timed ({per_layer:.2f} s each), scaled to "
                      f"{spec['layers'] if spec['residual'] else 1} layer(s) per step; numpy float64, one thread"}


def run_reference(args, spec, rank, world):
    if rank != 0:
        return None
    name = [k for k, v in WORKLOADS.items() if v is spec][0]
    times = _oracle_child(name, 0.0, steps=args.warmup + args.steps)
    timed = times[args.warmup:]
    per_layer = sum(timed) / len(timed)
    layers = spec["layers"] if spec["residual"] else 1
    T = spec["tokens"]
    value = T / (per_layer * layers)
    return {
        "impl": "reference", "metric": args.metric, "value": round(value, 6), "unit": args.unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_layer * layers * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": spec["desc"], "layers": spec["layers"], "tokens_per_step": T},
        "cpu_baseline": {"value": round(value, 6), "unit": args.unit, "cores": 1, "kind": "oracle",
                         "sample": f"each step: layer 0 of the stack for {T} token(s) in the float64 oracle, "
                                   f"scaled to {layers} layer(s)"},
        "e2e": {"value": round(value, 6), "unit": args.unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
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
    ap.add_argument("--oracle-steps", type=int, default=0, help=argparse.SUPPRESS)
    args = ap.parse_args(argv)
    if args.oracle_sample:
        spec = WORKLOADS[args.oracle_sample]
        if args.oracle_steps > 0:
            print(json.dumps(_oracle_steps(spec, args.oracle_steps)))
        else:
            print(json.dumps(_oracle_sample(spec, args.cpu_seconds)))
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
