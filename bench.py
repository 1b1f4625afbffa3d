#!/usr/bin/env python3
"""Throughput benchmark of the MoE FFN layer on GB300.

One step = one moe_forward over one batch of T tokens: route -> group ->
grouped SwiGLU experts -> combine, inputs resident in HBM.  Prints ONE JSON
line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--also NAME,...] [--also-mxfp8 NAME,...]
                  [--also-mxfp8-act NAME,...]
                  [--also-nvfp4 NAME,...] [--also-single NAME,...]

Default workload: the Qwen3-235B-A22B MoE layer on a 64-token decode batch
(d=4096, E=128, top-8, I=1536).  Its 4.8 GB of expert weights exceed the
129 MB L2, so every step streams them from HBM (no flush needed).
--impl reference times the fp64 CPU oracle on the host cores instead.
The "also" entries measure further workloads at N=1: --also with bf16
weights, --also-mxfp8 / --also-nvfp4 with the expert weights quantised to
MXFP8 / NVFP4 once before timing (moe_forward_mxfp8 / moe_forward_nvfp4),
--also-mxfp8-act with MXFP8 weights and MXFP8 tokens (W8A8, act_mxfp8),
--also-single with the whole layer as one kernel launch (single_launch).
A bf16 "also" entry times max(3, K/50) steps (tens of ms, like the burst
bf16 peak: single GEMMs at full clocks); the prefill entry also times,
as a second row, enough steps for about 2 s (like the sustained peak: a
seconds-long GEMM loop under the power cap).  A timed region longer than
1 s is always compared with the sustained peak.
The stdout line stays short (the "also" entries are rows of the fields named
in "also_fields"); the per-kernel breakdown of every entry and the full
roofline records go to stderr, one JSON line each.
Inside the timed region the dominant kernel is bracketed by CUDA events on
every 10th step (for the roofline's achieved rate); the per-kernel breakdown
("kernels") comes from a traced pass of up to 50 steps just before it.
Multi-GPU (torchrun): independent replicas, one per GPU, no collective on
the data path; value = all tokens processed / max time over ranks.
"""

from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

TRACE_EVERY = 10  # timed steps per step whose dominant kernel is bracketed by events
SUSTAINED_S = 2.0  # seconds of the sustained loop of a bf16 "also" entry
METRIC = "MoE-layer tokens/s (prefill, decode) + % of bf16 TC peak / HBM GB/s, 1 GB300"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    from mixture_experts_layer_20_gb300 import workloads as W
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=W.DECODE, choices=sorted(W.WORKLOADS))
    ap.add_argument("--also", default=f"{W.PREFILL},{W.SKEWED},{W.DEEPSEEK},{W.TINY}",
                    help="comma-separated extra workloads measured at N=1 (empty for none)")
    ap.add_argument("--also-single", default=W.DECODE,
                    help="workloads also measured at N=1 as one kernel launch (empty for none)")
    ap.add_argument("--also-mxfp8", default=f"{W.DECODE},{W.PREFILL}",
                    help="workloads also measured at N=1 with MXFP8 expert weights (empty for none)")
    ap.add_argument("--also-nvfp4", default=f"{W.DECODE},{W.PREFILL}",
                    help="workloads also measured at N=1 with NVFP4 expert weights (empty for none)")
    ap.add_argument("--also-mxfp8-act", default=W.DECODE,
                    help="workloads also measured at N=1 with MXFP8 expert weights and MXFP8 "
                         "tokens, W8A8 (decode sizes only; empty for none)")
    ap.add_argument("--weights", choices=["bf16", "mxfp8", "nvfp4", "mxfp8-act"], default="bf16",
                    help="expert weights of the main workload (profiler captures of the "
                         "quantised kernels; e2e is measured for bf16 only)")
    ap.add_argument("--single-launch", action="store_true",
                    help="run the main workload as one kernel launch")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override T (smaller cases for profiler captures)")
    ap.add_argument("--experts", type=int, default=0,
                    help="override E (smaller cases for profiler captures)")
    return ap.parse_args()


def pick_workload(W, args):
    import dataclasses
    w = W.WORKLOADS[args.workload]
    changes = {}
    if args.tokens:
        changes["T"] = args.tokens
    if args.experts:
        changes["E"] = args.experts
    if changes:
        tag = ",".join(f"{k}={v}" for k, v in changes.items())
        w = dataclasses.replace(w, name=f"{w.name}[{tag}]", **changes)
    return w


# ------------------------------------------------------------------ helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(gpu_index)], stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        with open(self.file.name) as f:
            lines = [l.strip() for l in f if l.strip()]
        os.unlink(self.file.name)
        rows = []
        for l in lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 - 0.25 <= r[0] <= t1 + 0.25]
        sample = inside or rows[-3:]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in sample for i, v in enumerate(r[3]) if v == "Active"})
        return {
            "sm_mhz": statistics.median(r[1] for r in sample) if sample else None,
            "sm_max_mhz": max(r[2] for r in sample) if sample else None,
            "reasons": reasons,
            "samples": len(inside),
        }


def source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


GEMM_SOURCES = ["mixture_experts_layer_20_gb300/csrc/moe_gemm.cu",
                "mixture_experts_layer_20_gb300/csrc/moe_expert_gemm.cu",
                "mixture_experts_layer_20_gb300/csrc/moe_expert_gemm.cuh",
                "mixture_experts_layer_20_gb300/csrc/moe_smallm.cu",
                "mixture_experts_layer_20_gb300/csrc/moe_smallm.cuh",
                "mixture_experts_layer_20_gb300/csrc/moe_convert.cuh",
                "mixture_experts_layer_20_gb300/csrc/moe_device.cuh"]


def ncu_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if it still
    describes the current kernel source."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        e = t[kernel][workload]
        if e.get("source_sha") != source_sha(GEMM_SOURCES):
            return None
        return e["dram_bytes_per_launch"]
    except Exception:
        return None


MX_BYTES = 1 + 1 / 32  # MXFP8 weight bytes per parameter: E4M3 code + E8M0 scale per 32
NV_BYTES = 0.5 + 1 / 16  # NVFP4: E2M1 code + E4M3 scale per 16 (tensor scales negligible)


def kernel_work(name, w, counts):
    """Algorithmic (flops, bytes) of one launch of a kernel: each operand and
    result counted once, weights only for experts that received rows."""
    from mixture_experts_layer_20_gb300 import counters as C
    T, d, E, k, I, Is = w.T, w.d, w.E, w.top_k, w.I, w.I_shared
    rows = T * k
    name = name.removesuffix("_smallm")  # the small-M kernels do the same work
    if name == "moe_decode_fused":  # the whole layer in one launch
        return (C.expert_flops(T, k, d, I, Is) + C.router_flops(T, d, E) + 2 * rows * d,
                C.algorithmic_bytes(counts, T, d, E, I, Is))
    touched = sum(1 for c in counts if c > 0)
    if name == "moe_gate_up_swiglu_nvfp4":
        return 4 * rows * d * I, int(touched * 2 * I * d * NV_BYTES) + rows * d * 2 + rows * I * 2
    if name == "moe_down_nvfp4":
        return 2 * rows * d * I, int(touched * d * I * NV_BYTES) + rows * I * 2 + rows * d * 2
    if name == "moe_gate_up_swiglu_mxfp8_a8":  # W8A8: the tokens as MXFP8 codes too
        return (4 * rows * d * I,
                int(touched * 2 * I * d * MX_BYTES + rows * d * MX_BYTES) + rows * I * 2)
    if name == "moe_down_mxfp8_a8":
        return 2 * rows * d * I, int(touched * d * I * MX_BYTES + rows * I * MX_BYTES) + rows * d * 2
    if name == "moe_act_mxfp8":  # two launches a layer (x, then h): their mean
        return 0, int((T * d + rows * I) * (2 + MX_BYTES) / 2)
    if name == "moe_gate_up_swiglu_mxfp8":
        return 4 * rows * d * I, int(touched * 2 * I * d * MX_BYTES) + rows * d * 2 + rows * I * 2
    if name == "moe_down_mxfp8":
        return 2 * rows * d * I, int(touched * d * I * MX_BYTES) + rows * I * 2 + rows * d * 2
    if name == "moe_gate_up_swiglu":
        return 4 * rows * d * I, touched * 2 * I * d * 2 + rows * d * 2 + rows * I * 2
    if name == "moe_down":
        return 2 * rows * d * I, touched * d * I * 2 + rows * I * 2 + rows * d * 2
    if name == "moe_shared_gate_up_swiglu":
        return 4 * T * d * Is, 2 * Is * d * 2 + T * d * 2 + T * Is * 2
    if name == "moe_shared_down":
        return 2 * T * d * Is, d * Is * 2 + T * Is * 2 + T * d * 2
    partial = ((d + 511) // 512) * T * ((E + 15) // 16 * 16) * 4
    if name == "moe_router_logits":
        return C.router_flops(T, d, E), T * d * 2 + E * d * 2 + partial
    if name == "moe_router_topk":
        return 0, partial + rows * 8
    if name == "moe_combine":
        return 2 * rows * d, rows * d * 2 + T * d * 2 + rows * 8 + (T * d * 2 if Is else 0)
    if name == "moe_permute_gather":
        return 0, rows * d * 2 + T * d * 2 + rows * 4
    return 0, rows * 4 * 4


# ------------------------------------------------------------------ output

ALSO_FIELDS = ["workload", "weights", "tokens_per_s", "ms_per_step", "sm_mhz", "clock_reasons",
               "layer_tc_frac", "layer_hbm_frac", "dom_kernel", "dom_bound", "dom_frac", "peak"]
SUSTAINED_FOR = {"qwen3_235b_prefill_T6000"}  # bf16 entries that also get the ~2 s loop


def also_row(name, weights, r, peak_kind):
    """One "also" entry as a row of ALSO_FIELDS (the stdout line stays under
    about 3000 characters, so that a short log tail still holds all of it)."""
    c = r["clocks"] or {}
    roof, layer = r["roofline"], r["layer"]
    return [name, weights, int(round(r["tokens_per_s"])), round(r["ms"], 4), c.get("sm_mhz"),
            ",".join(c.get("reasons", [])), round(layer["tc_peak_frac"], 3),
            round(layer["hbm_frac"], 3),
            roof["kernel"].removeprefix("moe_").replace("_swiglu", ""), roof["bound"],
            round(roof["frac"], 3),
            "sust" if peak_kind == "sustained" else "burst"]


def bench_config(w, world):
    """The workload's config, the same for both arms."""
    return {"workload": w.name, "T": w.T, "d": w.d, "E": w.E, "top_k": w.top_k, "I": w.I,
            "I_shared": w.I_shared, "parallelism": f"replicas x{world}",
            "l2": "inputs > L2 (touched expert weights streamed from HBM each step)"}


def detail_line(label, r):
    """Per-kernel breakdown and full roofline of one entry, for stderr."""
    return json.dumps({"detail": label, "ms_per_step": round(r["ms"], 4), "clocks": r["clocks"],
                       "layer": r["layer"], "roofline": r["roofline"], "kernels": r["kernels"]})


# ------------------------------------------------------------------ ranks
# Replicas: each rank runs the whole layer on its own batch; the job's time is
# the slowest rank's and its throughput all ranks' tokens over that time.

def slowest_rank(dist, ms, device):
    """Max over ranks of a per-rank time (the identity without a process group)."""
    if not dist:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item()


def job_rate(dist, per_rank_rate, world, device):
    """Whole-job rate from per-rank rates: world x the slowest rank's rate."""
    if not dist:
        return per_rank_rate
    import torch
    t = torch.tensor([per_rank_rate], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MIN)
    return t.item() * world


# ------------------------------------------------------------------ our arm

def measure(moe, W, w, params, steps, warmup, rank, world, dist, sampler_index, peaks,
            mxfp8=False, nvfp4=False, single_launch=False, act_mxfp8=False):
    """mxfp8 / nvfp4: the expert weights are quantised once, outside the
    timed region, and every step runs moe_forward_mxfp8 / _nvfp4 on them
    (act_mxfp8: MXFP8 tokens too, W8A8).
    single_launch: every step runs the layer as one kernel launch."""
    import torch
    from mixture_experts_layer_20_gb300 import counters as C
    x = W.make_x(w, device="cuda")
    ws = moe.new_workspace(w.T, w.d, w.E, w.I, w.top_k, w.I_shared, act_mxfp8=act_mxfp8)
    out = torch.empty((w.T, w.d), dtype=torch.bfloat16, device="cuda")
    kw = dict(out=out, ws=ws, router_bias=params["router_bias"],
              w_gate_up_shared=params["w_gate_up_shared"], w_down_shared=params["w_down_shared"])
    fwd_kw = dict(single_launch=True) if single_launch else {}
    if mxfp8:
        mx_gu = moe.moe_mxfp8_quantize(params["w_gate_up"])
        mx_d = moe.moe_mxfp8_quantize(params["w_down"])

        def step():
            moe.moe_forward_mxfp8(x, params["w_router"], mx_gu, mx_d, w.top_k, **kw,
                                  **(dict(act_mxfp8=True) if act_mxfp8 else {}))
    elif nvfp4:
        nv_gu = moe.moe_nvfp4_quantize(params["w_gate_up"])
        nv_d = moe.moe_nvfp4_quantize(params["w_down"])

        def step():
            moe.moe_forward_nvfp4(x, params["w_router"], nv_gu, nv_d, w.top_k, **kw)
    else:
        def step():
            moe.moe_forward(x, params["w_router"], params["w_gate_up"], params["w_down"], w.top_k,
                            **kw, **fwd_kw)

    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize()
    if moe.moe_get_device_status(ws) != moe.MOE_OK:
        raise RuntimeError("device status not OK after warm-up")
    views = moe.workspace_views(ws, w.T, w.d, w.E, w.I, w.top_k, w.I_shared)
    counts = views["expert_counts"].cpu().tolist()

    # Per-kernel breakdown from a traced pass outside the timed region: every
    # traced launch costs two event records, which also delay the next launch.
    moe.moe_profiler_collect()
    moe.moe_profiler_only(None)
    moe.moe_profiler_enable(True)
    n_trace = max(3, min(steps, 50))
    for _ in range(n_trace):
        step()
    torch.cuda.synchronize()
    moe.moe_profiler_enable(False)
    prof = moe.moe_profiler_collect()
    dom = max(prof, key=lambda n: prof[n][1])

    # Timed region: the dominant kernel is bracketed by events on every
    # TRACE_EVERY-th step (its duration gives the roofline's achieved rate);
    # an event pair between two launches also blocks their overlap, so the
    # other steps run without it.
    sampler = ClockSampler(sampler_index) if sampler_index is not None else None
    time.sleep(0.3 if sampler else 0)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    moe.moe_profiler_only(dom)
    l0 = moe.moe_launch_count()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    start.record()
    for i in range(steps):
        traced = i % TRACE_EVERY == 0
        if traced:
            moe.moe_profiler_enable(True)
        step()
        if traced:
            moe.moe_profiler_enable(False)
    stop.record()
    torch.cuda.synchronize()
    t1 = time.time()
    launches = moe.moe_launch_count() - l0
    moe.moe_profiler_only(None)
    dom_n, dom_total = moe.moe_profiler_collect()[dom]
    if dist:
        dist.barrier()
    clocks = sampler.stop(t0, t1) if sampler else None
    ms = slowest_rank(dist, start.elapsed_time(stop) / steps, "cuda")
    if moe.moe_get_device_status(ws) != moe.MOE_OK:
        raise RuntimeError("device status not OK after the timed region")

    # per-kernel breakdown and the dominant kernel's roofline
    kernels = {}
    for name, (n, tot) in prof.items():
        fl, by = kernel_work(name, w, counts)
        avg = tot / n
        kernels[name] = {"launches": n, "avg_ms": round(avg, 5), "share": None,
                         "tflops": round(fl / (avg * 1e-3) / 1e12, 2),
                         "gbs": round(by / (avg * 1e-3) / 1e9, 1), "alg_bytes": int(by)}
    total_k = sum(v[1] for v in prof.values()) or 1.0
    for name, (n, tot) in prof.items():
        kernels[name]["share"] = round(tot / total_k, 4)
    fl, by = kernel_work(dom, w, counts)
    avg_s = dom_total / dom_n * 1e-3
    region_s = ms * steps * 1e-3
    tensor_peak = peaks["bf16_tflops_sustained"] if region_s > 1.0 else peaks["bf16_tflops"]
    t_tensor = fl / (tensor_peak * 1e12)
    t_hbm = by / (peaks["hbm_gbs"] * 1e9)
    if t_tensor >= t_hbm:
        roof = {"bound": "tensor", "achieved": round(fl / avg_s / 1e12, 1), "peak": tensor_peak,
                "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": round(by / avg_s / 1e9, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    tr = ncu_traffic(dom, w.name)
    roof.update({"traffic": tr, "kernel": dom, "algorithmic_bytes": by, "algorithmic_flops": fl,
                 "avg_launch_ms": round(avg_s * 1e3, 5), "launches_averaged": dom_n})

    flops = C.expert_flops(w.T, w.top_k, w.d, w.I, w.I_shared)
    abytes = C.algorithmic_bytes(counts, w.T, w.d, w.E, w.I, w.I_shared)
    if mxfp8 or nvfp4:  # routed expert weights at MX_BYTES / NV_BYTES per parameter, not 2
        tw = C.touched_weight_bytes(counts, w.d, w.I)
        abytes += int(tw * (MX_BYTES if mxfp8 else NV_BYTES) / 2) - tw
    layer = {
        "tflops": round(flops / (ms * 1e-3) / 1e12, 1),
        "tc_peak_frac": round(flops / (ms * 1e-3) / 1e12 / tensor_peak, 4),
        "gbs": round(abytes / (ms * 1e-3) / 1e9, 1),
        "hbm_frac": round(abytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
        "active_experts": sum(1 for c in counts if c > 0),
        "padded_rows_128": C.padded_rows(counts, 128),
    }
    return {"ms": ms, "tokens_per_s": w.T * world / (ms * 1e-3), "launches": launches,
            "clocks": clocks, "roofline": roof, "kernels": kernels, "layer": layer,
            "x": x, "ws": ws, "counts": counts}


def measure_e2e(moe, w, params, ws, x, steps, single_launch=False):
    """Tokens/s end to end through the public API, from pinned host x to pinned
    host out, as a serving loop runs it: two device buffer sets, each with the
    layer captured as a graph (moe_forward_graph over device x / out) and
    replayed with moe_graph_launch; step i's x goes up on a copy stream while
    step i - 1 computes, its out comes back on another while step i + 1
    computes, and the host waits for step i's copy-back and reads the result
    after queueing step i + 1.  Every step moves its own x in and its out back.
    Reported beside it: a graph over the host buffers themselves (H2D, layer,
    D2H on one stream) with a stream synchronisation after every step, and the
    plain moe_forward_host call the same way."""
    import torch
    x_hosts = [x.cpu().pin_memory() for _ in range(2)]
    out_hosts = [torch.empty((w.T, w.d), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    kw = dict(router_bias=params["router_bias"], w_gate_up_shared=params["w_gate_up_shared"],
              w_down_shared=params["w_down_shared"], single_launch=single_launch)
    s = torch.cuda.current_stream()

    def timed(call):
        for _ in range(3):
            call()
            s.synchronize()
        t0 = time.perf_counter()
        for _ in range(steps):
            call()
            s.synchronize()
        return w.T * steps / (time.perf_counter() - t0)

    wts = (params["w_router"], params["w_gate_up"], params["w_down"])
    plain = timed(lambda: moe.moe_forward_host(x_hosts[0], *wts, w.top_k, out_hosts[0], ws, **kw))
    g_host = moe.ForwardGraph(x_hosts[0], *wts, w.top_k, out_hosts[0], ws, **kw)
    synced = timed(lambda: g_host.launch())
    g_host.close()

    x_dev = [torch.empty_like(x) for _ in range(2)]
    out_dev = [torch.empty((w.T, w.d), dtype=torch.bfloat16, device=x.device) for _ in range(2)]
    graphs = [moe.ForwardGraph(x_dev[j], *wts, w.top_k, out_dev[j], ws, **kw) for j in range(2)]
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    seen = []

    def run(n):
        for i in range(n):
            j = i % 2  # buffers of step i - 2: its copy-back was waited for below
            with torch.cuda.stream(up):
                x_dev[j].copy_(x_hosts[j], non_blocking=True)
                ev_in[j].record(up)
            s.wait_event(ev_in[j])
            graphs[j].launch()
            ev_done[j].record(s)
            down.wait_event(ev_done[j])
            with torch.cuda.stream(down):
                out_hosts[j].copy_(out_dev[j], non_blocking=True)
                ev_out[j].record(down)
            if i:
                ev_out[1 - j].synchronize()
                seen.append(out_hosts[1 - j][0, 0].item())  # the host reads step i - 1
        ev_out[(n - 1) % 2].synchronize()
        seen.append(out_hosts[(n - 1) % 2][0, 0].item())

    run(3)
    t0 = time.perf_counter()
    run(steps)
    value = w.T * steps / (time.perf_counter() - t0)
    for g in graphs:
        g.close()
    nbytes = w.T * w.d * 2
    return {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": nbytes,
            "d2h_bytes_per_step": nbytes, "api": "moe_forward_graph+moe_graph_launch, copy streams",
            "synced_value": round(synced, 1), "plain_call_value": round(plain, 1)}


def cpu_baseline(W, w, params, x, target_s=15.0):
    """The oracle, as it stands, on the first S tokens of the same batch."""
    import numpy as np
    import oracle
    xb = W.to_bits(x)
    wr = W.to_bits(params["w_router"])
    bias = None if params["router_bias"] is None else params["router_bias"].cpu().numpy()
    shared = (W.to_bits(params["w_gate_up_shared"]), W.to_bits(params["w_down_shared"])) \
        if params["w_gate_up_shared"] is not None else (None, None)

    class Host:
        def __init__(self, t): self.t, self.c = t, {}
        def __getitem__(self, e):
            e = int(e)
            if e not in self.c:
                self.c[e] = W.to_bits(self.t[e])
            return self.c[e]

    gu, dn = Host(params["w_gate_up"]), Host(params["w_down"])

    def run(S):
        ids, _, _ = oracle.route(xb[:S], wr, w.top_k, bias)
        for e in np.unique(ids):       # host copies of the weights are not timed
            gu[e]; dn[e]
        c0, t0 = time.process_time(), time.perf_counter()
        oracle.forward(xb[:S], wr, gu, dn, w.top_k, router_bias=bias,
                       w_gate_up_shared=shared[0], w_down_shared=shared[1])
        return time.perf_counter() - t0, time.process_time() - c0

    el1, _ = run(1)
    S = int(max(1, min(w.T, target_s / max(el1, 1e-3) * 0.5)))
    el, cpu = run(S)
    return {"value": round(S / el, 3), "unit": "tokens/s", "cores": round(cpu / el, 1),
            "host_cores": os.cpu_count(), "kind": "oracle",
            "sample": f"first {S} of {w.T} tokens of {w.name}, {el:.1f} s wall"}


# ------------------------------------------------------------------ reference arm

def reference_arm(args):
    import numpy as np
    import torch
    import oracle
    from mixture_experts_layer_20_gb300 import workloads as W
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = pick_workload(W, args)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    params = W.make_weights(w, device=dev)
    x = W.make_x(w, device=dev)
    xb = W.to_bits(x)
    wr = W.to_bits(params["w_router"])
    bias = None if params["router_bias"] is None else params["router_bias"].cpu().numpy()
    shared = (W.to_bits(params["w_gate_up_shared"]), W.to_bits(params["w_down_shared"])) \
        if params["w_gate_up_shared"] is not None else (None, None)
    cache_gu, cache_d = {}, {}

    class Host:
        def __init__(self, t, c): self.t, self.c = t, c
        def __getitem__(self, e):
            e = int(e)
            if e not in self.c:
                self.c[e] = W.to_bits(self.t[e])
            return self.c[e]

    gu, dn = Host(params["w_gate_up"], cache_gu), Host(params["w_down"], cache_d)

    def tokens(i, S):
        return [(i * S + j) % w.T for j in range(S)]

    def one(i, S):
        idx = tokens(i, S)
        ids, _, _ = oracle.route(xb[idx], wr, w.top_k, bias)
        for e in np.unique(ids):
            gu[e]; dn[e]
        t0 = time.perf_counter()
        oracle.forward(xb[idx], wr, gu, dn, w.top_k, router_bias=bias,
                       w_gate_up_shared=shared[0], w_down_shared=shared[1])
        return time.perf_counter() - t0

    budget = 150.0 / max(1, args.steps + args.warmup)
    S = max(1, min(w.T, int(budget / max(one(0, 1), 1e-3) * 0.7)))
    for i in range(args.warmup):
        one(i, S)
    c0 = time.process_time()
    times = [one(args.warmup + i, S) for i in range(args.steps)]
    cpu = time.process_time() - c0
    el = sum(times)
    value = S * args.steps / el
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded Gaussian x and weights)",
        "config": bench_config(w, int(os.environ.get("WORLD_SIZE", "1"))),
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "kind": "oracle",
                         "cores": round(cpu / el, 1), "host_cores": os.cpu_count(),
                         "sample": f"{S} tokens of {w.name} per step (rotating through the batch)"},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ main

def main():
    args = parse_args()
    if args.impl == "reference":
        return reference_arm(args)

    import torch
    from mixture_experts_layer_20_gb300 import binding as moe
    from mixture_experts_layer_20_gb300 import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    smi_index = vis.split(",")[local] if vis else local
    peaks, peak_src = load_peaks()

    w = pick_workload(W, args)
    params = W.make_weights(w, device="cuda")
    r = measure(moe, W, w, params, args.steps, args.warmup, rank, world, dist, smi_index, peaks,
                mxfp8=args.weights in ("mxfp8", "mxfp8-act"), nvfp4=args.weights == "nvfp4",
                single_launch=args.single_launch, act_mxfp8=args.weights == "mxfp8-act")
    e2e = None
    if args.weights == "bf16":
        e2e = measure_e2e(moe, w, params, r["ws"], r["x"], max(10, min(args.steps, 100)),
                          single_launch=args.single_launch)
        if dist:
            e2e["value"] = round(job_rate(dist, e2e["value"], world, "cuda"), 1)

    also = []
    details = [detail_line(w.name + " bf16", r)]
    if world == 1:
        for name in [n for n in args.also.split(",") if n]:
            wa = W.WORKLOADS[name]
            same = (wa.d, wa.E, wa.I, wa.I_shared, wa.zipf_bias, wa.seed) == \
                (w.d, w.E, w.I, w.I_shared, w.zipf_bias, w.seed)
            pa = params if same else W.make_weights(wa, device="cuda")
            n_burst = max(3, args.steps // 50)
            ra = measure(moe, W, wa, pa, n_burst, 3, 0, 1, None, smi_index, peaks)
            region_s = ra["ms"] * n_burst * 1e-3
            also.append(also_row(name, "bf16", ra,
                                 "sustained" if region_s > 1.0 else "burst"))
            details.append(detail_line(name + " bf16", ra))
            ms_burst = ra["ms"]
            del ra
            if name in SUSTAINED_FOR:
                n_sust = max(n_burst, int(SUSTAINED_S / (ms_burst * 1e-3)) + 1)
                rs = measure(moe, W, wa, pa, n_sust, 3, 0, 1, None, smi_index, peaks)
                also.append(also_row(name, "bf16", rs, "sustained"))
                details.append(detail_line(name + " bf16 sustained", rs))
                del rs
            if not same:
                del pa
            torch.cuda.empty_cache()
        for name in [n for n in args.also_single.split(",") if n]:
            wa = W.WORKLOADS[name]
            same = (wa.d, wa.E, wa.I, wa.I_shared, wa.zipf_bias, wa.seed) == \
                (w.d, w.E, w.I, w.I_shared, w.zipf_bias, w.seed)
            pa = params if same else W.make_weights(wa, device="cuda")
            n_s = max(3, args.steps // 10)
            ra = measure(moe, W, wa, pa, n_s, 3, 0, 1, None, smi_index, peaks, single_launch=True)
            also.append(also_row(name, "bf16 1-launch", ra,
                                 "sustained" if ra["ms"] * n_s * 1e-3 > 1.0 else "burst"))
            details.append(detail_line(f"{name} bf16 single launch", ra))
            del ra
            if not same:
                del pa
            torch.cuda.empty_cache()
        quant = [(n, "mxfp8") for n in args.also_mxfp8.split(",") if n] + \
            [(n, "nvfp4") for n in args.also_nvfp4.split(",") if n]
        for name, fmt in quant:
            wa = W.WORKLOADS[name]
            same = (wa.d, wa.E, wa.I, wa.I_shared, wa.zipf_bias, wa.seed) == \
                (w.d, w.E, w.I, w.I_shared, w.zipf_bias, w.seed)
            pa = params if same else W.make_weights(wa, device="cuda")
            n_q = max(3, args.steps // 10)
            ra = measure(moe, W, wa, pa, n_q, 3, 0, 1, None, smi_index, peaks,
                         mxfp8=fmt == "mxfp8", nvfp4=fmt == "nvfp4")
            region_s = ra["ms"] * n_q * 1e-3
            also.append(also_row(name, fmt, ra, "sustained" if region_s > 1.0 else "burst"))
            details.append(detail_line(f"{name} {fmt}", ra))
            del ra
            if not same:
                del pa
            torch.cuda.empty_cache()
        for name in [n for n in args.also_mxfp8_act.split(",") if n]:
            wa = W.WORKLOADS[name]
            same = (wa.d, wa.E, wa.I, wa.I_shared, wa.zipf_bias, wa.seed) == \
                (w.d, w.E, w.I, w.I_shared, w.zipf_bias, w.seed)
            pa = params if same else W.make_weights(wa, device="cuda")
            n_q = max(3, args.steps // 10)
            ra = measure(moe, W, wa, pa, n_q, 3, 0, 1, None, smi_index, peaks, mxfp8=True,
                         act_mxfp8=True)
            also.append(also_row(name, "mxfp8 w8a8", ra,
                                 "sustained" if ra["ms"] * n_q * 1e-3 > 1.0 else "burst"))
            details.append(detail_line(f"{name} mxfp8 w8a8", ra))
            del ra
            if not same:
                del pa
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(W, w, params, r["x"])

    if rank == 0:
        r["roofline"]["peak_source"] = peak_src
        line = {
            "metric": METRIC, "value": round(r["tokens_per_s"], 1), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(r["ms"], 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if args.weights == "bf16" else
            ("mxfp8 tokens and expert weights" if args.weights == "mxfp8-act" else
             f"bf16 activations, {args.weights} expert weights"),
            "data": "synthetic (seeded Gaussian x and weights)",
            "config": bench_config(w, world),
            "clocks": r["clocks"], "e2e": e2e, "gpu_launches": r["launches"],
            "roofline": r["roofline"], "cpu_baseline": cpu, "layer": r["layer"],
            "also_fields": ALSO_FIELDS, "also": also,
        }
        for dl in details:
            print(dl, file=sys.stderr, flush=True)
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
