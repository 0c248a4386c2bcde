#!/usr/bin/env python3
"""Benchmark: Q4_0 x Q8_0 ggml_mul_mat on GB300.

One step = one pass of the whole hot path over the workload's projection set:
for every weight matrix, the activations are quantized to Q8_0 and multiplied
by the resident Q4_0 weights (one q4q_mul_mat call per matrix, captured once in
a CUDA graph and replayed).  Weight quantization (Q4_0 encode) happens once
before timing, as a model load would do it, and is timed separately.

Default workload: the Llama-3-8B-shaped decode projections at 1 token (q, k, v,
o, gate, up, down, lm_head; 418 MB of Q4_0 weights), seed 2: the set the 1-token
GEMV is measured on.  The same JSON line also carries the GPT-2 117M
decode-step weight set (49 small matrices, launch-latency bound) and the
tensor-core path at 512 tokens.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Prints one JSON line (rank 0).  `value` is weight GB/s (Q4_0 weight bytes
streamed per second, all ranks).  With torchrun (N > 1) every rank runs its own
replica of the workload (the path has no exchange step): weak scaling.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "Q4_0 mul_mat weight GB/s vs HBM peak (1 tok); int8 TOPS at 512 tok"
FALLBACK_HBM_GBS = 6800.0


# --------------------------------------------------------------- helpers ----

def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def _measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(kernel_file: str) -> str:
    """First 16 hex digits of the sha256 of a kernel's source file followed by the
    shared device headers it includes (any change invalidates a profile)."""
    h = hashlib.sha256()
    headers = ("q4q_gemv.cuh", "q4q_common.cuh") if kernel_file.startswith("q4q_gemv") else ("q4q_common.cuh",)
    for f in (kernel_file,) + headers:
        with open(os.path.join(ROOT, "q4_quantized_matmul_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _profile_traffic(kernel_file: str, summary: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source is
    unchanged since it was taken (the summary records kernel_source_hash)."""
    try:
        with open(os.path.join(ROOT, "profiles", summary), encoding="utf-8") as f:
            text = f.read()
        sha = kernel_source_hash(kernel_file)
        m_sha = re.search(r"source_sha256_16:\s*([0-9a-f]+)", text)
        m_tr = re.search(r"dram_bytes_per_step:\s*([0-9.eE+]+)", text)
        if m_sha and m_tr and m_sha.group(1) == sha:
            return float(m_tr.group(1))
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the GPU is busy."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 100):
        self.index = index
        self.proc = None
        self.period_ms = period_ms

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                 "-lms", str(self.period_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), sm_max=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hw_thermal=parts[6], sw_thermal=parts[7], sw_power=parts[8]))
            except ValueError:
                continue
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["sm_max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(r["power"] for r in rows)}


# ------------------------------------------------------- cross-rank logic ---

def max_over_ranks(ms: float, world: int, device=None) -> float:
    """Slowest rank's time (the job finishes when every replica has)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank_step: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job GB/s: every rank streams its own replica of the weights (weak scaling)."""
    return world * bytes_per_rank_step * steps / (max_ms * 1e-3) / 1e9


def graph_replays(k_steps: int, graph_steps: int, rest_steps: int):
    """The graph launches that run exactly k_steps steps: whole graphs of graph_steps
    steps, then the remainder as one graph of rest_steps steps when it matches, else as
    single-step graphs.  Returns a list of (kind, steps) with kind "multi", "rest" or
    "single" (steps = steps run by that launch)."""
    if graph_steps <= 1:
        return [("single", 1)] * k_steps
    out = [("multi", graph_steps)] * (k_steps // graph_steps)
    left = k_steps % graph_steps
    if left:
        out += [("rest", left)] if left == rest_steps else [("single", 1)] * left
    return out


# --------------------------------------------------------------- the arms ---

def _weights_bytes(shapes):
    return sum(n * (k // 32) * 18 for k, n in shapes)


def _workload(name):
    from q4_quantized_matmul_gb300 import workloads
    return workloads.WORKLOADS[name]


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import q4_quantized_matmul_gb300 as q4q
    from q4_quantized_matmul_gb300 import workloads

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = _workload(args.workload)
    ne11 = args.ne11 or wl.ne11[0]
    # --matrices i,j,...: only those matrices of the set (profiling one kernel at full size)
    pick = [int(t) for t in args.matrices.split(",")] if args.matrices else list(range(len(wl.shapes)))
    shapes = [wl.shapes[i] for i in pick]
    nmat = len(shapes)

    # ---- set-up (untimed): fp32 weights -> Q4_0 on the GPU, activations resident
    # the Q4_0 output is allocated outside the events: they bracket the encoder alone
    t_q = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wq, xs, dsts = [], [], []
    quant_ms, quant_in_bytes, quant_out_bytes = 0.0, 0, 0
    for i, (ne00, ne01) in zip(pick, shapes):
        w, x = workloads.problem(args.workload, i, ne11)
        wd = torch.from_numpy(w).to(dev)
        qd = torch.empty(ne01 * q4q.q4_0_row_bytes(ne00), dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()
        t_q[0].record()
        q4q.q4q_quantize_q4_0(wd, dst=qd)
        t_q[1].record()
        torch.cuda.synchronize()
        wq.append(qd)
        quant_ms += t_q[0].elapsed_time(t_q[1])
        quant_in_bytes += w.nbytes
        quant_out_bytes += qd.numel()
        del wd
        xs.append(torch.from_numpy(x).to(dev))
        dsts.append(torch.empty((ne11, ne01), dtype=torch.float32, device=dev))
    wbytes = _weights_bytes(shapes)
    # rotate weight copies so that every step reads its weights from HBM, not L2
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    copies = max(1, -(-3 * l2 // wbytes)) if wbytes < 3 * l2 else 1
    # A decode token runs every layer's projections back to back in one graph; here a
    # graph holds one step per weight copy (4 for a decode set), so the programmatic
    # dependent launch chain also runs across step boundaries inside it.
    copies = max(copies, 4 if ne11 < 8 else 2)
    wsets = [wq] + [[t.clone() for t in wq] for _ in range(copies - 1)]
    ws_bytes = max(q4q.q4q_mul_mat_workspace_size(k, n, ne11) for k, n in shapes)
    workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)

    stream = torch.cuda.Stream(device=dev)
    # calls launch with programmatic dependent launch: each may be scheduled, and start
    # streaming its (resident, read-only) weights, while the previous call finishes
    # (honoured by the GEMV and the warp-MMA kernel, ignored by the tensor-core GEMM)
    flags = q4q.Q4Q_MUL_MAT_PDL

    def step(c):
        for i, (ne00, ne01) in enumerate(shapes):
            q4q.q4q_mul_mat(wsets[c][i], ne00, ne01, xs[i], dst=dsts[i], workspace=workspace, flags=flags)

    with torch.cuda.stream(stream):
        for c in range(copies):         # first calls outside capture (one-time set-up per kernel)
            step(c)
    torch.cuda.synchronize()
    graphs = []
    for c in range(copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(c)
        graphs.append(g)
    # one step per weight copy, in order, args.graph_rounds times over (a decode token
    # chains hundreds of launches in one graph; PDL does not reach across graph launches)
    rounds = max(1, args.graph_rounds)
    multi = torch.cuda.CUDAGraph()
    with torch.cuda.graph(multi, stream=stream):
        for _ in range(rounds):
            for c in range(copies):
                step(c)
    torch.cuda.synchronize()

    graph_steps = copies * rounds if ne11 < 8 else 1

    def capture_rest(step_fn):
        """The timed region's last args.steps % graph_steps steps as one graph (so a short
        run does not turn into single-step graphs), or None."""
        rest = args.steps % graph_steps if graph_steps > 1 else 0
        if rest == 0:
            return None
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(rest):
                step_fn(k % copies)
        return g

    rest_graph = capture_rest(step)
    torch.cuda.synchronize()

    rest_steps = args.steps % graph_steps if graph_steps > 1 else 0

    def run_steps(multi_graph, single_graphs, k_steps, rest=None):
        """Exactly k_steps steps: whole multi-step graphs, then the rest (one graph)."""
        k = 0
        for kind, _ in graph_replays(k_steps, graph_steps, rest_steps if rest is not None else -1):
            if kind == "multi":
                multi_graph.replay()
            elif kind == "rest":
                rest.replay()
            else:
                single_graphs[k % copies].replay()
                k += 1

    def barrier():
        if world > 1:
            dist.barrier()

    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
    # untimed soak so the clock sampler sees the GPU under load, then the warm-up steps;
    # the soak starts with one replay of each graph the timed region uses (a graph's
    # first launch also uploads it to the device)
    t_end = time.time() + args.soak
    n = 0
    with torch.cuda.stream(stream):
        if graph_steps > 1:
            multi.replay()
            if rest_graph is not None:
                rest_graph.replay()
        while time.time() < t_end:
            graphs[n % copies].replay()
            n += 1
            if n % 200 == 0:
                stream.synchronize()
        for k in range(args.warmup):
            graphs[k % copies].replay()
    torch.cuda.synchronize()

    # ---- timed region: exactly K steps
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        run_steps(multi, graphs, args.steps, rest_graph)
        e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    clocks = sampler.stop() if sampler else None

    ms_per_step = ms / args.steps
    value = job_throughput(wbytes, args.steps, world, ms)

    # ---- per-launch durations of the mul_mat kernel (same calls, event-bracketed, L2-cold copies)
    per_ms = []
    with torch.cuda.stream(stream):
        evs = []
        # hold the stream with a spin kernel while the launches are queued, so that
        # host launch latency does not show up between an event and its kernel
        torch.cuda._sleep(int(2e8))
        for k in range(max(3, min(args.steps, 20))):
            c = k % copies
            for i, (ne00, ne01) in enumerate(shapes):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                q4q.q4q_mul_mat(wsets[c][i], ne00, ne01, xs[i], dst=dsts[i], workspace=workspace)
                b.record(stream)
                evs.append((i, a, b))
    torch.cuda.synchronize()
    per_shape = {}
    for i, a, b in evs:
        per_ms.append(a.elapsed_time(b))
        per_shape.setdefault(i, []).append(a.elapsed_time(b))
    reps = len(per_ms) // nmat
    kern_ms_per_step = sum(per_ms) / reps
    act_bytes = sum(4 * k * ne11 for k, n in shapes)
    out_bytes = sum(4 * n * ne11 for k, n in shapes)
    alg_bytes_step = wbytes + act_bytes + out_bytes
    peak, peak_kind = _measured_peaks()
    # The timed region runs nothing but this kernel (nmat launches per step), so its
    # average launch duration there is ms_per_step / nmat (PDL lets consecutive
    # launches overlap their set-up, as they do in the timed step).
    achieved = alg_bytes_step / (ms_per_step * 1e-3) / 1e9
    isolated = alg_bytes_step / (kern_ms_per_step * 1e-3) / 1e9
    traffic_step = _profile_traffic("q4q_gemv.cu", "gemv_q4_0_%s.md" % args.workload) if ne11 < 8 else None

    # ---- end to end through the public API with host buffers (pinned), graph-captured
    xh = torch.empty(act_bytes // 4, dtype=torch.float32).pin_memory()
    oh = torch.empty(out_bytes // 4, dtype=torch.float32).pin_memory()
    off = 0
    for i, (k, n) in enumerate(shapes):
        xh[off:off + k * ne11].copy_(xs[i].reshape(-1).cpu())
        off += k * ne11
    xd = torch.empty_like(xh, device=dev)
    od = torch.empty_like(oh, device=dev)
    xviews, oviews = [], []
    off_x = off_o = 0
    for (k, n) in shapes:
        xviews.append(xd[off_x:off_x + k * ne11].view(ne11, k))
        oviews.append(od[off_o:off_o + n * ne11].view(ne11, n))
        off_x += k * ne11
        off_o += n * ne11

    def e2e_step(c):
        xd.copy_(xh, non_blocking=True)
        for i, (ne00, ne01) in enumerate(shapes):
            q4q.q4q_mul_mat(wsets[c][i], ne00, ne01, xviews[i], dst=oviews[i], workspace=workspace, flags=flags)
        oh.copy_(od, non_blocking=True)

    with torch.cuda.stream(stream):
        e2e_step(0)
    torch.cuda.synchronize()
    egraphs = []
    for c in range(copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            e2e_step(c)
        egraphs.append(g)
    emulti = torch.cuda.CUDAGraph()
    with torch.cuda.graph(emulti, stream=stream):
        for _ in range(rounds):
            for c in range(copies):
                e2e_step(c)
    erest = capture_rest(e2e_step)
    with torch.cuda.stream(stream):
        if graph_steps > 1:   # first launches (graph upload) outside the timed region
            emulti.replay()
            if erest is not None:
                erest.replay()
        for k in range(args.warmup):
            egraphs[k % copies].replay()
    torch.cuda.synchronize()
    barrier()
    with torch.cuda.stream(stream):
        e0.record(stream)
        run_steps(emulti, egraphs, args.steps, erest)
        e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ems = max_over_ranks(e0.elapsed_time(e1), world, dev)
    e2e_value = job_throughput(wbytes, args.steps, world, ems)

    batched = measure_batched(dev, stream, args) if (rank == 0 and args.batched_tokens > 0) else None
    second = (measure_decode(dev, stream, args.secondary_decode)
              if (rank == 0 and args.secondary_decode not in ("", "none") and args.secondary_decode != args.workload)
              else None)
    nxt = measure_next(dev, stream) if (rank == 0 and args.next_rows) else None
    if nxt is not None and ne11 == 1 and args.workload != "gpt2_decode_step":
        # the main decode set as one chain launch, A/B against its PDL-chained calls
        nxt["chain_" + args.workload] = measure_decode(dev, stream, args.workload, steps=200)

    # ---- CPU baseline: the oracle on this host's cores, bounded sample
    cpu = cpu_baseline(args.workload, ne11, budget_s=args.cpu_seconds) if (rank == 0 and args.cpu_seconds > 0) else None

    assert q4q.q4q_device_status() == 0, "device-side error recorded during the benchmark"
    if rank != 0:
        return None
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "i8",
        "data": "synthetic",
        "config": {
            "workload": args.workload,
            "description": wl.description,
            "ne11": ne11,
            "matrices": nmat,
            "q4_0_weight_bytes_per_step": wbytes,
            "l2_policy": "inputs larger than L2: %d rotating copies of the Q4_0 weights (%.0f MB, L2 %.0f MB)" % (
                copies, copies * wbytes / 1e6, l2 / 1e6),
            "launch": "%d q4q_mul_mat calls per step; CUDA graphs of %d consecutive steps (the %d weight copies in "
                      "turn), programmatic dependent launch between all calls of a graph" % (nmat, graph_steps, copies)
                      if ne11 < 8 else "%d q4q_mul_mat calls per step, one CUDA graph per step" % nmat,
            "graph_steps": graph_steps,
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "gpu_launches": nmat * args.steps * (1 if ne11 < 8 else 2),
        "roofline": {
            "bound": "hbm",
            "kernel": "gemv_q4_0_kernel (fused Q8_0 activation quantize + Q4_0 GEMV)" if ne11 < 8 else "mul_mat",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": (traffic_step / nmat) if traffic_step else None,
            "algorithmic_bytes_per_launch": alg_bytes_step / nmat,
            "avg_launch_us": round(ms_per_step * 1e3 / nmat, 3),
            "note": "achieved = algorithmic bytes (Q4_0 weights + fp32 activations + fp32 outputs) per "
                    "launch / average launch duration in the timed region (CUDA events on the launching "
                    "stream; the region runs only this kernel, %d launches per step)" % nmat,
            "isolated": {
                "achieved": round(isolated, 1),
                "frac": round(isolated / peak, 4),
                "avg_launch_us": round(kern_ms_per_step * 1e3 / nmat, 3),
                "per_launch": [{"shape": "%d->%d" % shapes[i], "us": round(1e3 * statistics.median(v), 2),
                                "gb_s": round(_weights_bytes([shapes[i]]) / (1e-3 * statistics.median(v)) / 1e9, 1)}
                               for i, v in sorted(per_shape.items())],
                "note": "each launch alone between its own CUDA events (stream held by a spin kernel while "
                        "they are queued), no PDL overlap, L2-cold weight copies",
            },
        },
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": act_bytes,
                "d2h_bytes_per_step": out_bytes,
                "how": "every step: pinned-host -> device copy of all activations, %d q4q_mul_mat calls, "
                       "device -> pinned-host copy of all outputs, in stream order; captured like the "
                       "device-resident line (CUDA graphs of %d steps)" % (nmat, graph_steps)},
        "weight_quantize": {"gb_per_s_fp32_in": round(quant_in_bytes / (quant_ms * 1e-3) / 1e9, 1),
                            "gb_per_s_in_out": round((quant_in_bytes + quant_out_bytes) / (quant_ms * 1e-3) / 1e9, 1),
                            "frac_of_hbm": round((quant_in_bytes + quant_out_bytes) / (quant_ms * 1e-3) / 1e9 / peak,
                                                 4),
                            "ms": round(quant_ms, 3),
                            "note": "q4q_quantize_q4_0 over the set at set-up, once per matrix (first call of each "
                                    "shape), destination allocated outside the events; steady state in "
                                    "next_rows.quantize"},
        "cpu_baseline": cpu,
        "clocks": clocks,
        "batched": batched,
        "secondary_decode": second,
        "next_rows": nxt,
    }
    return line


def measure_decode(dev, stream, name, steps=300):
    """A second 1-token workload, timed like the main one: weight copies > 3 x L2,
    one CUDA graph per copy of PDL-chained q4q_mul_mat calls."""
    import torch

    import q4_quantized_matmul_gb300 as q4q
    from q4_quantized_matmul_gb300 import workloads
    wl = workloads.WORKLOADS[name]
    shapes = list(wl.shapes)
    wq, xs, ds = [], [], []
    for i, (ne00, ne01) in enumerate(shapes):
        w, x = workloads.problem(name, i, 1)
        wd = torch.from_numpy(w).to(dev)
        wq.append(q4q.q4q_quantize_q4_0(wd))
        del wd
        xs.append(torch.from_numpy(x).to(dev))
        ds.append(torch.empty((1, ne01), dtype=torch.float32, device=dev))
    wbytes = _weights_bytes(shapes)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    copies = max(2, -(-3 * l2 // wbytes))
    wsets = [wq] + [[t.clone() for t in wq] for _ in range(copies - 1)]

    def step(c):
        for i, (ne00, ne01) in enumerate(shapes):
            q4q.q4q_mul_mat(wsets[c][i], ne00, ne01, xs[i], dst=ds[i], flags=q4q.Q4Q_MUL_MAT_PDL)

    with torch.cuda.stream(stream):
        for c in range(copies):
            step(c)
    torch.cuda.synchronize()
    # one graph per step: the 49-matrix set is a whole model's decode step already
    graphs = []
    for c in range(copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(c)
        graphs.append(g)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for k in range(10):
            graphs[k % copies].replay()
        e0.record(stream)
        for k in range(steps):
            graphs[k % copies].replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    peak, kind = _measured_peaks()
    gbs = wbytes / (ms * 1e-3) / 1e9
    out = {"workload": name, "description": wl.description, "value": round(gbs, 1), "unit": "GB/s",
           "ms_per_step": round(ms, 5), "frac_of_hbm": round(gbs / peak, 4), "matrices": len(shapes),
           "us_per_matrix": round(ms * 1e3 / len(shapes), 3),
           "graph_steps": 1,
           "note": "dependent-chain launch (PDL), one kernel per matrix; small matrices are launch-latency bound"}
    # The same step as one q4q_mul_mat_chain launch over the same weights and inputs
    # (each link still waits for the previous one to complete everywhere before it
    # reads its activations), timed the same way right after: the A/B of the
    # persistent chain against the PDL chain of separate launches.
    wsc = torch.empty(q4q.q4q_mul_mat_chain_workspace_size(len(shapes)), dtype=torch.uint8, device=dev)
    links = [[(wsets[c][i], ne00, ne01, xs[i].reshape(-1), ds[i].reshape(-1)) for i, (ne00, ne01) in
              enumerate(shapes)] for c in range(copies)]
    with torch.cuda.stream(stream):
        for c in range(copies):
            q4q.q4q_mul_mat_chain(links[c], workspace=wsc)
    torch.cuda.synchronize()
    cgraphs = []
    for c in range(copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            q4q.q4q_mul_mat_chain(links[c], workspace=wsc)
        cgraphs.append(g)
    with torch.cuda.stream(stream):
        for k in range(10):
            cgraphs[k % copies].replay()
        e0.record(stream)
        for k in range(steps):
            cgraphs[k % copies].replay()
        e1.record(stream)
    torch.cuda.synchronize()
    cms = e0.elapsed_time(e1) / steps
    cgbs = wbytes / (cms * 1e-3) / 1e9
    out["chain"] = {"value": round(cgbs, 1), "unit": "GB/s", "ms_per_step": round(cms, 5),
                    "frac_of_hbm": round(cgbs / peak, 4), "us_per_matrix": round(cms * 1e3 / len(shapes), 3),
                    "speedup_vs_pdl_launches": round(ms / cms, 3),
                    "note": "one cooperative q4q_mul_mat_chain launch per step (memset of its counters + kernel)"}
    del wsets, wq, xs, ds, cgraphs, links
    torch.cuda.empty_cache()
    return out


def measure_batched(dev, stream, args):
    """The other half of the metric: int8-equivalent TOPS (2*M*N*K per second) of
    the tensor-core path on the Llama-3-8B-shaped projection set at args.batched_tokens
    tokens (seed 3 workload), weights resident, activations quantized inside each call."""
    import torch

    import q4_quantized_matmul_gb300 as q4q
    from q4_quantized_matmul_gb300 import workloads
    name, ne11 = "llama3_8b_batched", args.batched_tokens
    shapes = list(workloads.WORKLOADS[name].shapes)
    wq, xs, ds = [], [], []
    for i, (ne00, ne01) in enumerate(shapes):
        w, x = workloads.problem(name, i, ne11)
        wd = torch.from_numpy(w).to(dev)
        wq.append(q4q.q4q_quantize_q4_0(wd))
        del wd
        xs.append(torch.from_numpy(x).to(dev))
        ds.append(torch.empty((ne11, ne01), dtype=torch.float32, device=dev))
    ws = torch.empty(max(q4q.q4q_mul_mat_workspace_size(k, n, ne11) for k, n in shapes), dtype=torch.uint8,
                     device=dev)

    def step():
        for i, (ne00, ne01) in enumerate(shapes):
            q4q.q4q_mul_mat(wq[i], ne00, ne01, xs[i], dst=ds[i], workspace=ws)

    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    steps = 10
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    ops = sum(2.0 * k * n * ne11 for k, n in shapes)
    # per-launch durations of each call (activation quantize + tensor-core GEMM)
    per = []
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(2e8))
        evs = []
        for i, (ne00, ne01) in enumerate(shapes):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            q4q.q4q_mul_mat(wq[i], ne00, ne01, xs[i], dst=ds[i], workspace=ws)
            b.record(stream)
            evs.append((i, a, b))
    torch.cuda.synchronize()
    for i, a, b in evs:
        k, n = shapes[i]
        per.append({"shape": "%d->%d" % (k, n), "us": round(a.elapsed_time(b) * 1e3, 1),
                    "tops": round(2.0 * k * n * ne11 / (a.elapsed_time(b) * 1e-3) / 1e12, 1)})
    peak = _measured_bf16()
    tops = ops / (ms * 1e-3) / 1e12
    out = {"workload": name, "ne11": ne11, "ms_per_step": round(ms, 4), "int8_equiv_tops": round(tops, 1),
           "unit": "TOPS (2*M*N*K/s)", "roofline": {"bound": "tensor", "achieved": round(tops, 1),
                                                      "peak": peak[0], "peak_kind": peak[1], "unit": "TFLOP/s",
                                                      "frac": round(tops / peak[0], 4),
                                                      "note": "fp16 exact-integer operands on tcgen05 kind::f16; "
                                                              "peak = dense f16/bf16"},
           "per_launch": per}
    del xs, ds, ws
    torch.cuda.empty_cache()
    if args.sweep_tokens:
        out["token_sweep"] = measure_token_sweep(dev, stream, shapes, wq,
                                                 [int(t) for t in args.sweep_tokens.split(",") if t],
                                                 max(1, args.graph_rounds))
    del wq
    torch.cuda.empty_cache()
    return out


def measure_token_sweep(dev, stream, shapes, wq, tokens, rounds):
    """One step over the Llama-3-8B-shaped projection set (the 8 q4q_mul_mat calls) at
    each token count of `tokens`: weights resident in 4 rotating copies (more than 3 x
    L2, so every step reads them from HBM), activations N(0, 1) (seed 5), every call
    with the workspace q4q_mul_mat_workspace_size asks for and the PDL flag.  As for the
    1-token line, one CUDA graph holds `rounds` passes over the copies (rounds x 4 steps
    in order; PDL does not reach across graph launches).  The roofline time of a step
    is the larger of its Q4_0 weight bytes over the measured HBM bandwidth and its
    2*M*N*K ops over the measured dense bf16 rate; frac = that time / the measured
    time."""
    import torch

    import q4_quantized_matmul_gb300 as q4q
    hbm, hbm_kind = _measured_peaks()
    bf16, bf16_kind = _measured_bf16()
    copies = 4
    wsets = [wq] + [[t.clone() for t in wq] for _ in range(copies - 1)]
    wbytes = _weights_bytes(shapes)
    gen = torch.Generator(device="cpu").manual_seed(5)
    rows = []
    for ne11 in tokens:
        xs = {k: torch.randn((ne11, k), generator=gen).to(dev) for k in sorted(set(k for k, _ in shapes))}
        ds = [torch.empty((ne11, n), dtype=torch.float32, device=dev) for _, n in shapes]
        ws = torch.empty(max(q4q.q4q_mul_mat_workspace_size(k, n, ne11) for k, n in shapes), dtype=torch.uint8,
                         device=dev)

        def step(c):
            for i, (ne00, ne01) in enumerate(shapes):
                q4q.q4q_mul_mat(wsets[c][i], ne00, ne01, xs[ne00], dst=ds[i], workspace=ws,
                                flags=q4q.Q4Q_MUL_MAT_PDL)

        def steps():
            for _ in range(rounds):
                for c in range(copies):
                    step(c)

        graph = _capture(stream, steps)
        per_graph = rounds * copies
        reps = max(1, -(-24 // per_graph))   # graph replays timed: at least 24 steps
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for k in range(max(1, -(-12 // per_graph))):
                graph.replay()
            e0.record(stream)
            for k in range(reps):
                graph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (reps * per_graph)
        ops = sum(2.0 * k * n * ne11 for k, n in shapes)
        t_bytes = wbytes / (hbm * 1e3)             # us
        t_ops = ops / (bf16 * 1e6)                 # us
        path = ("GEMV (q, k, v, o) and warp-MMA kernel" if 2 <= ne11 <= 3 else "warp-MMA kernel" if ne11 <= 32
                else "tensor-core GEMM")
        rows.append({"ne11": ne11, "us_per_step": round(us, 1), "weights_gb_s": round(wbytes / us / 1e3, 1),
                     "int8_equiv_tops": round(ops / us / 1e6, 1), "path": path,
                     "roofline_us": round(max(t_bytes, t_ops), 1),
                     "roofline_bound": "hbm" if t_bytes >= t_ops else "tensor",
                     "frac": round(max(t_bytes, t_ops) / us, 4)})
        del graph, xs, ds, ws
        torch.cuda.empty_cache()
    del wsets
    torch.cuda.empty_cache()
    return {"workload": "llama3_8b_batched shapes (8 projections, one layer + lm_head)", "rows": rows,
            "peaks": {"hbm_gb_s": hbm, "hbm_kind": hbm_kind, "bf16_tflops": bf16, "bf16_kind": bf16_kind},
            "graph_steps": rounds * copies,
            "note": "us per step of 8 q4q_mul_mat calls; 1 token is the main line"}


def _replay_ms(stream, graph, reps, calls_per_replay):
    """Average ms per call of `graph` (calls_per_replay calls) over `reps` replays, after 3 warm-ups."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for _ in range(3):
            graph.replay()
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (reps * calls_per_replay)


def _capture(stream, fn):
    import torch
    with torch.cuda.stream(stream):
        fn()                       # first call outside capture (one-time set-up per kernel)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    torch.cuda.synchronize()
    return g


def measure_next(dev, stream):
    """The operations next to the matmul, each timed on its own with weights rotated
    over more than 3 x L2 (CUDA graphs, CUDA events on the launching stream):
      * swiglu: the Llama-3-8B gate and up projections (4096 -> 14336, Q4_0) at one
        token through q4q_mul_mat_swiglu (one dual-weight GEMV), against the two
        plain q4q_mul_mat calls it replaces;
      * gpt2_bias_gelu: the GPT-2 117M decode-step set (49 matrices) with a bias on
        every projection but the lm_head and GELU on c_mlp_fc (q4q_mul_mat_bias_act);
      * get_rows: the Llama-3-8B-shaped token embedding (4096 x 128256, Q4_0): 512
        token ids, and the whole-table decode (HBM-bound);
      * q8_0_decode: the Llama-3-8B decode set with Q8_0 weights at one token
        (q4q_mul_mat_q8_0), PDL-chained like the main workload, and the same
        weights at 512 tokens on the tensor-core path (q8_0_batched_512);
      * llama3_8b_decode_fused: the main workload's weights with q/k/v as one
        group launch and gate/up as one SwiGLU launch (5 launches per step)."""
    import torch

    import q4_quantized_matmul_gb300 as q4q
    from q4_quantized_matmul_gb300 import workloads
    peak, kind = _measured_peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    PDL = q4q.Q4Q_MUL_MAT_PDL
    out = {}

    # ---- one pass over the Llama set: Q8_0 copies of all 8, Q4_0 gate / up / lm_head
    llama = list(workloads.WORKLOADS["llama3_8b_decode"].shapes)
    w8, xs, q4 = [], [], {}
    for i, (ne00, ne01) in enumerate(llama):
        w, x = workloads.problem("llama3_8b_decode", i)
        wd = torch.from_numpy(w).to(dev)
        w8.append(q4q.q4q_quantize_q8_0(wd))
        if i in (4, 5, 7):
            q4[i] = q4q.q4q_quantize_q4_0(wd)
        del wd
        xs.append(torch.from_numpy(x).to(dev))

    # ---- SwiGLU: gate + up fused vs two plain calls
    ne00, ne01 = llama[4]
    wb = 2 * q4[4].numel()
    copies = max(2, -(-3 * l2 // wb))
    gates = [q4[4]] + [q4[4].clone() for _ in range(copies - 1)]
    ups = [q4[5]] + [q4[5].clone() for _ in range(copies - 1)]
    x = xs[4]
    y = torch.empty((1, ne01), dtype=torch.float32, device=dev)
    yg = torch.empty_like(y)
    ws = torch.empty(q4q.q4q_mul_mat_swiglu_workspace_size(ne00, ne01, 1), dtype=torch.uint8, device=dev)
    reps = 50
    g_f = _capture(stream, lambda: [q4q.q4q_mul_mat_swiglu(gates[c], ups[c], ne00, ne01, x, dst=y, workspace=ws,
                                                           flags=PDL)
                                    for c in range(copies)])
    ms_f = _replay_ms(stream, g_f, reps, copies)
    g_u = _capture(stream, lambda: [(q4q.q4q_mul_mat(gates[c], ne00, ne01, x, dst=yg, workspace=ws, flags=PDL),
                                     q4q.q4q_mul_mat(ups[c], ne00, ne01, x, dst=y, workspace=ws, flags=PDL))
                                    for c in range(copies)])
    ms_u = _replay_ms(stream, g_u, reps, copies)
    alg = wb + 4 * ne00 + 4 * ne01
    out["swiglu"] = {
        "shape": "gate, up %d->%d (Q4_0), 1 token" % (ne00, ne01), "kernel": "gemv_q4_0_swiglu_kernel",
        "us_per_call": round(ms_f * 1e3, 2), "unfused_us_per_pair": round(ms_u * 1e3, 2),
        "roofline": {"bound": "hbm", "achieved": round(alg / (ms_f * 1e-3) / 1e9, 1), "peak": peak,
                     "peak_kind": kind, "unit": "GB/s", "frac": round(alg / (ms_f * 1e-3) / 1e9 / peak, 4),
                     "algorithmic_bytes_per_launch": alg},
        "note": "graph of %d PDL-chained calls over rotating weight copies; the unfused figure is two "
                "q4q_mul_mat calls (gate, up) without the elementwise SwiGLU" % copies}
    del gates, ups, g_f, g_u

    # ---- get_rows on the token embedding
    ne00, ne01 = llama[7]
    table = q4[7]
    rng = np.random.default_rng(5)
    ids = torch.from_numpy(rng.integers(0, ne01, size=512).astype(np.int32)).to(dev)
    rows = torch.empty((512, ne00), dtype=torch.float32, device=dev)
    g_r = _capture(stream, lambda: [q4q.q4q_get_rows_q4_0(table, ne00, ne01, ids=ids, dst=rows) for _ in range(20)])
    ms_r = _replay_ms(stream, g_r, 20, 20)
    full = torch.empty((ne01, ne00), dtype=torch.float32, device=dev)
    g_a = _capture(stream, lambda: q4q.q4q_get_rows_q4_0(table, ne00, ne01, dst=full))
    ms_a = _replay_ms(stream, g_a, 10, 1)
    rb = ne00 // 32 * 18
    alg_a = ne01 * rb + 4 * ne01 * ne00
    out["get_rows"] = {
        "table": "token embedding %d x %d Q4_0 (%.1f MB)" % (ne01, ne00, ne01 * rb / 1e6), "kernel": "get_rows_kernel",
        "ids_512": {"us_per_call": round(ms_r * 1e3, 2),
                    "gb_s": round((512 * rb + 512 * ne00 * 4) / (ms_r * 1e-3) / 1e9, 1)},
        "whole_table": {"us_per_call": round(ms_a * 1e3, 1),
                        "roofline": {"bound": "hbm", "achieved": round(alg_a / (ms_a * 1e-3) / 1e9, 1),
                                     "peak": peak, "peak_kind": kind, "unit": "GB/s",
                                     "frac": round(alg_a / (ms_a * 1e-3) / 1e9 / peak, 4),
                                     "algorithmic_bytes_per_launch": alg_a}},
        "note": "512 random ids: 20 calls per graph, launch-latency bound; whole table: Q4_0 read + fp32 write"}
    del full, rows, g_r, g_a, q4

    # ---- Q8_0-weight decode set
    wb8 = sum(t.numel() for t in w8)
    copies = max(2, -(-3 * l2 // wb8))
    sets = [w8] + [[t.clone() for t in w8] for _ in range(copies - 1)]
    ys = [torch.empty((1, n), dtype=torch.float32, device=dev) for _, n in llama]
    ws = torch.empty(max(q4q.q4q_mul_mat_q8_0_workspace_size(k, n, 1) for k, n in llama), dtype=torch.uint8,
                     device=dev)
    g_8 = _capture(stream, lambda: [q4q.q4q_mul_mat_q8_0(sets[c][i], k, n, xs[i], dst=ys[i], workspace=ws,
                                                         flags=PDL)
                                    for c in range(copies) for i, (k, n) in enumerate(llama)])
    ms_8 = _replay_ms(stream, g_8, 100, copies)
    alg8 = wb8 + sum(4 * k + 4 * n for k, n in llama)
    out["q8_0_decode"] = {
        "workload": "llama3_8b_decode with Q8_0 weights (%.1f MB)" % (wb8 / 1e6), "kernel": "gemv_q8_0_kernel",
        "ms_per_step": round(ms_8, 5), "weight_gb_s": round(wb8 / (ms_8 * 1e-3) / 1e9, 1),
        "roofline": {"bound": "hbm", "achieved": round(alg8 / (ms_8 * 1e-3) / 1e9, 1), "peak": peak,
                     "peak_kind": kind, "unit": "GB/s", "frac": round(alg8 / (ms_8 * 1e-3) / 1e9 / peak, 4),
                     "algorithmic_bytes_per_launch": alg8 / len(llama)},
        "note": "8 PDL-chained q4q_mul_mat_q8_0 calls per step, graph of %d steps over weight copies" % copies}
    del sets, g_8, ys

    # ---- Q8_0 weights at 512 tokens: the tensor-core GEMM with the Q8_0 dequantizer
    ne11b = 512
    xb = [torch.from_numpy(workloads.gen_acts("normal", ne11b, k, 3, i)).to(dev) for i, (k, n) in enumerate(llama)]
    yb = [torch.empty((ne11b, n), dtype=torch.float32, device=dev) for _, n in llama]
    wsb = torch.empty(max(q4q.q4q_mul_mat_q8_0_workspace_size(k, n, ne11b) for k, n in llama), dtype=torch.uint8,
                      device=dev)
    g_8b = _capture(stream, lambda: [q4q.q4q_mul_mat_q8_0(w8[i], k, n, xb[i], dst=yb[i], workspace=wsb)
                                     for i, (k, n) in enumerate(llama)])
    ms_8b = _replay_ms(stream, g_8b, 10, 1)
    ops = sum(2.0 * k * n * ne11b for k, n in llama)
    tops = ops / (ms_8b * 1e-3) / 1e12
    bf16 = _measured_bf16()
    out["q8_0_batched_512"] = {
        "workload": "llama3_8b_decode weights as Q8_0, 512 tokens (activations N(0,1))", "kernel": "mma_gemm_kernel<128, 0, 1>",
        "ms_per_step": round(ms_8b, 4), "int8_equiv_tops": round(tops, 1),
        "roofline": {"bound": "tensor", "achieved": round(tops, 1), "peak": bf16[0], "peak_kind": bf16[1],
                     "unit": "TFLOP/s", "frac": round(tops / bf16[0], 4)},
        "note": "8 q4q_mul_mat_q8_0 calls per step (activation operands + tcgen05 GEMM), one graph"}
    del w8, xb, yb, wsb, g_8b

    # ---- the Llama decode set with the fused launches: q, k, v as one group launch, o,
    #      gate and up as one SwiGLU launch, down, lm_head (5 launches instead of 8); the
    #      q/k/v group shares one input and the SwiGLU reads both gate and up, as in a layer
    q4s = []
    for i, (k, n) in enumerate(llama):
        w, _ = workloads.problem("llama3_8b_decode", i)
        wd = torch.from_numpy(w).to(dev)
        q4s.append(q4q.q4q_quantize_q4_0(wd))
        del wd
    wb4 = _weights_bytes(llama)
    copies = max(4, -(-3 * l2 // wb4))
    fsets = [q4s] + [[t.clone() for t in q4s] for _ in range(copies - 1)]
    h, f = llama[0][0], llama[4][1]
    xq = xs[0]
    outs = [torch.empty((1, n), dtype=torch.float32, device=dev) for _, n in llama]
    ws = torch.empty(max(q4q.q4q_mul_mat_swiglu_workspace_size(k, n, 1) for k, n in llama), dtype=torch.uint8,
                     device=dev)

    def fused_step(c):
        W = fsets[c]
        q4q.q4q_mul_mat_group([W[0], W[1], W[2]], [llama[0][1], llama[1][1], llama[2][1]], h, xq,
                              dsts=outs[0:3], workspace=ws, flags=PDL)
        q4q.q4q_mul_mat(W[3], h, llama[3][1], xs[3], dst=outs[3], workspace=ws, flags=PDL)
        q4q.q4q_mul_mat_swiglu(W[4], W[5], h, f, xs[4], dst=outs[4], workspace=ws, flags=PDL)
        q4q.q4q_mul_mat(W[6], llama[6][0], llama[6][1], xs[6], dst=outs[6], workspace=ws, flags=PDL)
        q4q.q4q_mul_mat(W[7], h, llama[7][1], xs[7], dst=outs[7], workspace=ws, flags=PDL)

    g_fs = _capture(stream, lambda: [fused_step(c) for c in range(copies)])
    ms_fs = _replay_ms(stream, g_fs, 250, copies)
    out["llama3_8b_decode_fused"] = {
        "workload": "llama3_8b_decode weights (%.1f MB Q4_0) with q/k/v grouped (one input) and gate/up fused "
                    "into SwiGLU: 5 launches per step" % (wb4 / 1e6),
        "kernels": "gemv_q4_0_group_kernel, gemv_q4_0_kernel, gemv_q4_0_swiglu_kernel",
        "ms_per_step": round(ms_fs, 5), "weight_gb_s": round(wb4 / (ms_fs * 1e-3) / 1e9, 1),
        "frac_of_hbm": round(wb4 / (ms_fs * 1e-3) / 1e9 / peak, 4),
        "note": "same weight bytes as the main workload; graph of %d PDL-chained steps over weight copies" % copies}
    del fsets, q4s, g_fs, outs, xs

    # ---- GPT-2 decode step with bias (+ GELU on c_mlp_fc)
    name = "gpt2_decode_step"
    shapes = list(workloads.WORKLOADS[name].shapes)
    wq, gx, bs, ds, acts = [], [], [], [], []
    for i, (ne00, ne01) in enumerate(shapes):
        w, xx = workloads.problem(name, i, 1)
        wd = torch.from_numpy(w).to(dev)
        wq.append(q4q.q4q_quantize_q4_0(wd))
        del wd
        gx.append(torch.from_numpy(xx).to(dev))
        last = i == len(shapes) - 1
        bs.append(None if last else torch.from_numpy(workloads.gen_bias(ne01, 1, i)).to(dev))
        acts.append(q4q.Q4Q_ACT_GELU if (not last and i % 4 == 2) else q4q.Q4Q_ACT_NONE)
        ds.append(torch.empty((1, ne01), dtype=torch.float32, device=dev))
    wbg = _weights_bytes(shapes)
    copies = max(2, -(-3 * l2 // wbg))
    wsets = [wq] + [[t.clone() for t in wq] for _ in range(copies - 1)]
    ws = torch.empty(max(q4q.q4q_mul_mat_workspace_size(k, n, 1) for k, n in shapes), dtype=torch.uint8, device=dev)
    g_b = _capture(stream, lambda: [q4q.q4q_mul_mat_bias_act(wsets[c][i], k, n, gx[i], bias=bs[i], act=acts[i],
                                                             dst=ds[i], workspace=ws, flags=PDL)
                                    for c in range(copies) for i, (k, n) in enumerate(shapes)])
    ms_b = _replay_ms(stream, g_b, 50, copies)
    # the same calls without the epilogue, in the same graph structure
    g_p = _capture(stream, lambda: [q4q.q4q_mul_mat(wsets[c][i], k, n, gx[i], dst=ds[i], workspace=ws, flags=PDL)
                                    for c in range(copies) for i, (k, n) in enumerate(shapes)])
    ms_p = _replay_ms(stream, g_p, 50, copies)
    out["gpt2_bias_gelu"] = {
        "workload": "gpt2_decode_step with bias on 48 projections and GELU on the 12 c_mlp_fc",
        "kernel": "gemv_q4_0_epi_kernel (bias / GELU in the output write)",
        "ms_per_step": round(ms_b, 5), "weight_gb_s": round(wbg / (ms_b * 1e-3) / 1e9, 1),
        "us_per_matrix": round(ms_b * 1e3 / len(shapes), 3),
        "plain_us_per_matrix": round(ms_p * 1e3 / len(shapes), 3),
        "note": "49 PDL-chained q4q_mul_mat_bias_act calls per step, graph of %d steps over weight copies; "
                "plain = the same calls as q4q_mul_mat (no bias, no GELU) in the same graphs" % copies}
    del wsets, wq, gx, bs, ds, g_b, g_p
    torch.cuda.empty_cache()
    out["quantize"] = measure_quantizers(dev, stream)
    return out


def measure_quantizers(dev, stream, reps=5):
    """The two block encoders in steady state, each on an input larger than L2, the
    destination allocated beforehand: Q4_0 of the Llama-3-8B lm_head weights
    (128256 x 4096 fp32, 2.1 GB in, 295 MB out) and Q8_0 of 8192 activation rows of
    14336 (470 MB in, 125 MB out).  Algorithmic bytes = fp32 read + blocks written."""
    import torch

    import q4_quantized_matmul_gb300 as q4q
    peak, kind = _measured_peaks()
    out = {}
    cases = [("q4_0_lm_head_weights", q4q.q4q_quantize_q4_0, (128256, 4096), q4q.q4_0_row_bytes),
             ("q8_0_activations", q4q.q4q_quantize_q8_0, (8192, 14336), q4q.q8_0_row_bytes)]
    for name, fn, (rows, cols), row_bytes in cases:
        g = torch.Generator(device=dev).manual_seed(5)
        src = torch.randn((rows, cols), device=dev, generator=g) * 0.02
        dst = torch.empty(rows * row_bytes(cols), dtype=torch.uint8, device=dev)
        with torch.cuda.stream(stream):
            fn(src, dst=dst)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                fn(src, dst=dst)
            e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        nbytes = src.numel() * 4 + dst.numel()
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"shape": [rows, cols], "us": round(ms * 1e3, 1), "gb_s": round(gbs, 1),
                     "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "peak_kind": kind,
                                  "unit": "GB/s", "frac": round(gbs / peak, 4)}}
        del src, dst
        torch.cuda.empty_cache()
    return out


def _measured_bf16():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured burst"
    except Exception:
        return 1900.0, "fallback"


def cpu_baseline(workload, ne11, budget_s=10.0, reps_min=1):
    """The oracle (as it stands) on this host's cores, timed on a bounded sample:
    all matrices of the workload, a seeded subset of rows when the full set would
    take longer than the budget.  Returns the same metric (weight GB/s)."""
    import oracle
    from q4_quantized_matmul_gb300 import workloads
    wl = workloads.WORKLOADS[workload]
    threads = os.cpu_count() or 1
    # prepare the sample: every matrix, rows subsampled to at most `cap` per matrix
    cap = 4096
    items = []
    for i, (ne00, ne01) in enumerate(wl.shapes):
        if workload == "gpt2_decode_step" and i >= 4 and i < len(wl.shapes) - 1:
            items.append(items[i % 4])      # the 12 layers repeat 4 shapes; reuse the data
            continue
        w, x = workloads.problem(workload, i, ne11)
        rows = np.arange(ne01) if ne01 <= cap else np.sort(np.random.default_rng(i).choice(ne01, cap, replace=False))
        wq = oracle.quantize_q4_0(w[rows])
        items.append((ne00, rows.size, wq, x))
    done_bytes = 0
    t0 = time.perf_counter()
    passes = 0
    while True:
        for ne00, nr, wq, x in items:
            oracle.mul_mat(wq, ne00, nr, x, nthreads=threads, with_scale=False)
            done_bytes += nr * (ne00 // 32) * 18
        passes += 1
        el = time.perf_counter() - t0
        if passes >= reps_min and el >= budget_s:
            break
        if el > 3 * budget_s:
            break
    el = time.perf_counter() - t0
    sampled = sum(nr * (k // 32) for k, nr, _, _ in items) * 18
    full = _weights_bytes(wl.shapes)
    return {"value": round(done_bytes / el / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": "%d passes over all %d matrices of %s at %d token(s), rows capped at %d per matrix "
                      "(%.1f%% of the weight bytes), incl. Q8_0 quantization of the activations; %.1f s wall"
                      % (passes, len(items), workload, ne11, cap, 100.0 * sampled / full, el)}


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle, as it stands, on this host's cores."""
    if rank != 0:
        return None
    import oracle
    from q4_quantized_matmul_gb300 import workloads
    wl = workloads.WORKLOADS[args.workload]
    ne11 = args.ne11 or wl.ne11[0]
    threads = os.cpu_count() or 1
    # one step = the oracle over every matrix of the workload on a seeded row sample
    frac = 1.0
    items = []
    for i, (ne00, ne01) in enumerate(wl.shapes):
        if args.workload == "gpt2_decode_step" and 4 <= i < len(wl.shapes) - 1:
            items.append(items[i % 4])
            continue
        w, x = workloads.problem(args.workload, i, ne11)
        items.append((ne00, ne01, oracle.quantize_q4_0(w), x))

    def one_step(fr):
        nbytes = 0
        for ne00, ne01, wq, x in items:
            nr = max(1, int(round(ne01 * fr)))
            oracle.mul_mat(wq[:nr], ne00, nr, x, nthreads=threads, with_scale=False)
            nbytes += nr * (ne00 // 32) * 18
        return nbytes

    t0 = time.perf_counter()
    one_step(frac)
    t1 = time.perf_counter() - t0
    budget = 120.0
    total_steps = args.steps + args.warmup
    if t1 * total_steps > budget:
        frac = max(1e-4, budget / (t1 * total_steps))
    for _ in range(args.warmup):
        one_step(frac)
    t0 = time.perf_counter()
    nbytes = 0
    for _ in range(args.steps):
        nbytes += one_step(frac)
    el = time.perf_counter() - t0
    value = nbytes / el / 1e9
    sample = ("each step: the oracle over all %d matrices of %s at %d token(s), first %.4g%% of each "
              "matrix's rows, incl. Q8_0 quantization of the activations" % (len(items), args.workload, ne11,
                                                                             100 * frac))
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(el * 1e3 / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "i8",
        "data": "synthetic",
        "config": {"workload": args.workload, "ne11": ne11, "matrices": len(items)},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama3_8b_decode")
    ap.add_argument("--secondary-decode", default="gpt2_decode_step",
                    help="also time this 1-token workload (empty = skip)")
    ap.add_argument("--ne11", type=int, default=0, help="override the workload's token count")
    ap.add_argument("--soak", type=float, default=1.5, help="seconds of untimed load before warm-up")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU-baseline budget (0 = skip)")
    ap.add_argument("--batched-tokens", type=int, default=512,
                    help="also measure the tensor-core path on the Llama-3-8B set at this many tokens (0 = skip)")
    ap.add_argument("--matrices", default="", help="comma-separated indices: only those matrices of the set")
    ap.add_argument("--graph-rounds", type=int, default=7,
                    help="decode steps: rounds over the 4 weight copies captured in one CUDA graph (7: 28 "
                         "steps, 224 launches, about one Llama-3-8B token of 32 layers x 7 projections "
                         "+ lm_head)")
    ap.add_argument("--sweep-tokens", default="2,4,7,8,16,32,64",
                    help="token counts of the batched-shape sweep (empty = skip)")
    ap.add_argument("--next-rows", type=int, default=1,
                    help="also time SwiGLU, bias/GELU, get_rows and Q8_0 weights (0 = skip)")
    ap.add_argument("--probe", default="", choices=["", "quantize", "batched", "decode-chain"],
                    help="run only this one measurement on GPU 0 and print its JSON (for profiling runs): "
                         "quantize = both block encoders; batched = the tensor-core path at --batched-tokens; "
                         "decode-chain = the --workload step as PDL launches and as one chain launch")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.probe:
        import torch

        import __graft_entry__
        __graft_entry__.build()
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        stream = torch.cuda.Stream(device=dev)
        if args.probe == "quantize":
            res = measure_quantizers(dev, stream)
        elif args.probe == "batched":
            res = measure_batched(dev, stream, args)
        else:
            res = measure_decode(dev, stream, args.workload, steps=args.steps)
        print(json.dumps({"probe": args.probe, "result": res}), flush=True)
        return

    world = _env_int("WORLD_SIZE", 1)
    rank = _env_int("RANK", 0)
    local_rank = _env_int("LOCAL_RANK", 0)

    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    import __graft_entry__
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if world > 1:
        import torch
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        dist.barrier()
        if rank != 0:
            __graft_entry__.build()
    line = run_ours(args, rank, world, local_rank)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
