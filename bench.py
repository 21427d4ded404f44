"""Forward-convolution benchmark (conv fprop TFLOP/s, direct-convolution FLOPs).

The headline line times the OverFeat-style stack (N=128, BF16, NHWC, FP32
output; the largest configuration that fits one GPU); its ``configs`` key
holds the same fields for the tiny FP32 layer, the AlexNet-style stack, the
ResNet-50-style layer set and the TF32 NCHW speech stack.  Every workload's
layers run on their own seeded synthetic inputs through the C ABI.  The
metric counts only direct-convolution FLOPs 2*N*K*P*Q*C*R*S (maxDNN page,
method and findings sections).

One step runs the workload's whole stack ``reps_per_step`` times back to
back (a fixed count per workload, so that the timed region of the default
steps lasts about a second and clock samplers see the GPU busy); L2 is
flushed (256 MiB write) between steps, outside the timed events, and one pass
over a stack touches more than the 129 MB L2 (except the tiny layer, which is
latency-bound and makes no roofline claim beyond that).  A step is timed by
CUDA events at its start and end.  Its passes go in blocks of eight: one pass
launched directly with an event after every launch (the per-layer times and
the dominant kernel's roofline fraction come from these), then a CUDA graph of
the other seven passes, captured once before the timed region from the same
library calls, replayed.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload overfeat|alexnet|resnet50|speech|tiny] [--no-configs]

--impl reference times the CPU oracle (FP64 direct convolution) on the host
cores on a bounded sample of the same workload.  Under torchrun with N > 1
every rank runs its own replica (the layer has no exchange step) and rank 0
prints the aggregate.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "conv fprop TFLOP/s (direct-conv FLOPs) and % of GB300 dense tensor-core peak"
L2_FLUSH_BYTES = 256 << 20
L2_BYTES = 129e6
HEADLINE = "overfeat"
CONFIG_ORDER = ["tiny", "alexnet", "overfeat", "resnet50", "speech"]
# Passes over the stack per step: about 40-60 ms of GPU work per step on
# GB300, so 20 steps keep the GPU busy for about a second.
REPS_PER_STEP = {"tiny": 2000, "alexnet": 200, "overfeat": 80, "resnet50": 40, "speech": 8}
# FP32 FFMA peak of the strict-FP32 path (bound "alu"): 152 SMs x 128 FP32
# lanes x 2 FLOP per fused multiply-add x 2.07 GHz.
FFMA_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def env_rank():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def aggregate_over_ranks(total_ms, step_flops, steps, world, device="cpu"):
    """The slowest rank's timed total (one MAX all-reduce across the ranks of
    the default process group) and the whole-job throughput in TFLOP/s: every
    rank runs the full workload (replicas), so the job does world x the FLOPs."""
    if world > 1:
        import torch
        t = torch.tensor([total_ms], device=device, dtype=torch.float64)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
    return total_ms, step_flops * world * steps / (total_ms * 1e-3) / 1e12


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# The sources each kernel's device code is built from (beside the shared
# headers): a DRAM-traffic figure in profiles/traffic.json stays valid while
# these files are unchanged.
KERNEL_SOURCES = {
    "tc_im2col_pair": ["conv_pair.cu"],
    "tc_im2col": ["conv_tc.cu"], "tc_gather_runs": ["conv_tc.cu"], "tc_gather": ["conv_tc.cu"],
    "tc_window": ["conv_window.cu"],
    "tc_rowstack": ["conv_rowstack.cu"],
    "ffma": ["conv_ffma.cu"],
    "tc_wgrad": ["conv_wgrad.cu"], "direct": ["conv_bwd.cu"],
    "pool_nhwc": ["pool_act.cu"], "flat": ["pool_act.cu"],
}
SHARED_SOURCES = ["ptx.cuh", "internal.h"]


def kernel_source_hash(kernel=None):
    """Hash of the sources of `kernel` and the shared headers (all sources when
    the kernel is not listed)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "deep_learning_convolution_gb300", "csrc")
    files = sorted(os.listdir(csrc))
    if kernel in KERNEL_SOURCES:
        files = sorted(set(KERNEL_SOURCES[kernel] + SHARED_SOURCES))
    for f in files:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def layer_geometry(layer, P, Q):
    """FLOPs and algorithmic bytes (x, w read once, y written once)."""
    esz = 2 if layer.dtype == "bf16" else 4
    flops = 2 * layer.N * layer.K * P * Q * layer.C * layer.R * layer.S
    # activation bytes actually touched (a 1x1 strided layer reads only the sampled pixels)
    if layer.R == 1 and layer.S == 1 and (layer.u > 1 or layer.v > 1):
        x_bytes = layer.N * layer.C * P * Q * esz
    else:
        x_bytes = layer.N * layer.C * layer.H * layer.W * esz
    w_bytes = layer.K * layer.C * layer.R * layer.S * esz
    y_bytes = layer.N * layer.K * P * Q * 4
    return flops, x_bytes + w_bytes + y_bytes


def layer_output_dims(layer):
    P = (layer.H + layer.pad_top + layer.pad_bottom - (layer.dil_h * (layer.R - 1) + 1)) // layer.u + 1
    Q = (layer.W + layer.pad_left + layer.pad_right - (layer.dil_w * (layer.S - 1) + 1)) // layer.v + 1
    return P, Q


def reps_for(workload, override=None):
    return int(override) if override else REPS_PER_STEP[workload]


# Passes of a step that carry per-launch events: one in INST_EVERY.  An event
# recorded between two launches keeps the second kernel from starting while
# the first drains (programmatic dependent launch); with one after every
# launch the stacks ran 1-6 % slower.  The other passes run as a user's would.
INST_EVERY = 8
TIMING_DIRECT = (f"step: start and end CUDA events; every pass launched directly, one in "
                 f"{INST_EVERY} with a CUDA event after every launch (the per-layer times)")
TIMING = (f"step: start and end CUDA events; of every {INST_EVERY} passes one is launched "
          f"directly with a CUDA event after every launch (the per-layer times) and "
          f"{INST_EVERY - 1} are replayed as one captured CUDA graph")


def instrumented_passes(reps):
    return [r for r in range(reps) if r % INST_EVERY == INST_EVERY // 2] or [reps // 2]


def capture_passes(launchers, stream, handle, n):
    """A CUDA graph of `n` passes over `launchers` captured on `stream`, and
    the library launches it holds (the handle's count over the capture); or
    (None, 0) when the capture fails, and the steps launch every pass."""
    import torch
    try:
        g = torch.cuda.CUDAGraph()
        l0 = handle.launches()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(n):
                for launch in launchers:
                    launch()
        per = handle.launches() - l0
        with torch.cuda.stream(stream):
            g.replay()  # the first replay uploads the graph
        torch.cuda.synchronize()
        return g, per
    except Exception:
        torch.cuda.synchronize()
        return None, 0


def time_steps(K, reps, launchers, flush, stream, graph=None):
    """Runs K steps of `reps` passes over `launchers` (one call per layer),
    L2 flushed before each step outside its timed events.  With `graph` (a
    capture of INST_EVERY - 1 passes; reps a multiple of INST_EVERY) each block
    of INST_EVERY passes is one pass launched with an event after every launch,
    then the graph; otherwise every pass is launched, one in INST_EVERY with
    those events.  Returns the summed step time in ms (each step's start and
    end events), the per-launcher time summed over the instrumented passes,
    how many passes that was, and how many graph replays ran."""
    import torch
    if graph is not None and reps % INST_EVERY == 0:
        blocks = reps // INST_EVERY
        nl = len(launchers)
        ev_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(K)]
        ev_pass = [[[torch.cuda.Event(enable_timing=True) for _ in range(nl + 1)]
                    for _ in range(blocks)] for _ in range(K)]
        with torch.cuda.stream(stream):
            for i in range(K):
                flush.fill_(float(i))
                ev_step[i][0].record(stream)
                for b in range(blocks):
                    ev = ev_pass[i][b]
                    ev[0].record(stream)
                    for j, launch in enumerate(launchers):
                        launch()
                        ev[j + 1].record(stream)
                    graph.replay()
                ev_step[i][1].record(stream)
        torch.cuda.synchronize()
        total_ms = sum(a.elapsed_time(b) for a, b in ev_step)
        per = [0.0] * nl
        for i in range(K):
            for ev in ev_pass[i]:
                for j in range(nl):
                    per[j] += ev[j].elapsed_time(ev[j + 1])
        return total_ms, per, K * blocks, K * blocks
    inst = instrumented_passes(reps)
    slot = {r: i for i, r in enumerate(inst)}
    nl = len(launchers)
    ev_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
    ev_pass = [[[torch.cuda.Event(enable_timing=True) for _ in range(nl + 1)] for _ in inst]
               for _ in range(K)]
    for i in range(K):
        flush.fill_(float(i))
        ev_step[i][0].record(stream)
        for r in range(reps):
            ev = ev_pass[i][slot[r]] if r in slot else None
            if ev is not None:
                ev[0].record(stream)
            for j, launch in enumerate(launchers):
                launch()
                if ev is not None:
                    ev[j + 1].record(stream)
        ev_step[i][1].record(stream)
    torch.cuda.synchronize()
    total_ms = sum(a.elapsed_time(b) for a, b in ev_step)
    per = [0.0] * nl
    for i in range(K):
        for ev in ev_pass[i]:
            for j in range(nl):
                per[j] += ev[j].elapsed_time(ev[j + 1])
    return total_ms, per, K * len(inst), 0


def workload_config(workload, world, reps=None):
    """The `config` both arms print: the workload and how a step is timed."""
    from deep_learning_convolution_gb300 import synth
    layers = synth.WORKLOADS[workload]
    reps = reps_for(workload, reps)
    geo = [layer_geometry(l, *layer_output_dims(l)) for l in layers]
    pass_flops = sum(g[0] for g in geo)
    pass_bytes = sum(g[1] for g in geo)
    l2 = (f"one pass touches {pass_bytes / 1e6:.0f} MB (> {L2_BYTES / 1e6:.0f} MB L2); "
          if pass_bytes > L2_BYTES else
          f"one pass touches {pass_bytes / 1e6:.2f} MB (resident in L2; latency-bound); ")
    l2 += "L2 flushed between steps (256 MiB write, untimed)"
    return {"workload": f"{workload}_stack", "layers": [l.name for l in layers],
            "batch": layers[0].N, "layout": layers[0].layout,
            "math": {"bf16": "bf16", "tf32": "tf32", "f32": "fp32"}[layers[0].dtype],
            "output": "fp32", "l2": l2,
            "parallelism": f"replicas{world}" if world > 1 else "single_gpu",
            "reps_per_step": reps, "flops_per_pass": pass_flops,
            "flops_per_step": pass_flops * reps}


# ---------------------------------------------------------------------------
# clocks sampling
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, interval_ms: int = 20):
        self.proc = None
        self.dev = device_index
        self.interval = interval_ms

    def query_once(self):
        try:
            out = subprocess.run(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                                  "-i", str(self.dev)], capture_output=True, text=True, timeout=20)
            return [l for l in out.stdout.splitlines() if l.strip()]
        except Exception:
            return []

    def start(self):
        self.before = self.query_once()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                 "-i", str(self.dev), "-lms", str(self.interval)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=10)
                lines = [l for l in out.splitlines() if l.strip()]
            except Exception:
                self.proc.kill()
        after = self.query_once()
        return self.summarise(lines, self.before + after)

    @staticmethod
    def _parse(line):
        f = [x.strip() for x in line.split(",")]
        if len(f) < 9:
            return None
        try:
            sm = float(f[1].split()[0])
            smax = float(f[2].split()[0])
        except ValueError:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = [n for n, v in zip(names, f[5:9]) if v.lower().startswith("active")]
        return sm, smax, reasons

    def summarise(self, during, around):
        parsed = [p for p in map(self._parse, during) if p]
        source = "during timed region"
        if not parsed:
            parsed = [p for p in map(self._parse, around) if p]
            source = "around timed region (no sample landed inside)"
        if not parsed:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "source": "nvidia-smi unavailable"}
        reasons = sorted({r for p in parsed for r in p[2]})
        return {"sm_mhz": statistics.median(p[0] for p in parsed),
                "sm_max_mhz": max(p[1] for p in parsed), "reasons": reasons,
                "samples": len(parsed), "source": source}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def _peak_for(workload, peaks):
    """(peak, unit-of-peak description) of a workload's arithmetic: the BF16
    tensor-core peak measured as a burst at the maximum SM clock (the
    convolution kernels keep the clock at its maximum through the timed
    region, where the seconds-long GEMM loop behind the sustained figure ran
    power-capped at a lower clock, so the burst figure is the stricter
    denominator), half of it for TF32 (only BF16 was measured; TF32 runs at
    half the BF16 rate), the FFMA peak for the strict-FP32 layer."""
    math = workload_config(workload, 1)["math"]
    bf16 = peaks["bf16_tflops"]
    src = f"{peaks['source']} bf16 burst"
    if math == "tf32":
        return bf16 / 2, src + " x 1/2 (tf32)"
    if math == "fp32":
        return FFMA_PEAK_TFLOPS, "FFMA: 152 SMs x 128 lanes x 2 FLOP x 2.07 GHz (derived)"
    return bf16, src


def run_workload(args, workload, handle, stream, dev, rank, world, local_rank, headline):
    """Times `steps` steps of `workload` (each `reps_per_step` passes over its
    stack); returns the JSON fields of one bench line."""
    import torch
    from deep_learning_convolution_gb300 import api, synth
    layers = synth.WORKLOADS[workload]
    reps = reps_for(workload, args.reps_per_step if headline else None)
    probs = []
    for j, layer in enumerate(layers):
        x, w, _ = synth.make_inputs(layer, synth.workload_seed(workload, j))
        xt, wt = api.layer_tensors(layer, x, w, dev)
        conv, y = api.layer_problem(handle, layer, xt, wt)
        n, k, p, q = conv.output_dim()
        flops, nbytes = layer_geometry(layer, p, q)
        probs.append(dict(layer=layer, x=xt, w=wt, y=y, conv=conv, flops=flops, bytes=nbytes,
                          kernel=conv.kernel(xt, wt, y)))
        del x, w
    pass_flops = sum(pr["flops"] for pr in probs)
    step_flops = pass_flops * reps
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    for _ in range(args.warmup):
        for _ in range(max(1, reps // 4)):
            for pr in probs:
                pr["conv"](pr["x"], pr["w"], pr["y"])
    torch.cuda.synchronize()
    handle.synchronize()

    K = args.steps
    # step time from each step's start and end events on the launch stream;
    # per-layer times from per-launch events in one pass of every INST_EVERY
    launchers = [(lambda pr=pr: pr["conv"](pr["x"], pr["w"], pr["y"])) for pr in probs]
    graph, per_graph = (capture_passes(launchers, stream, handle, INST_EVERY - 1)
                        if reps % INST_EVERY == 0 else (None, 0))
    sampler = ClockSampler(local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = handle.launches()
    sampler.start()
    time.sleep(0.05)
    total_ms, per_layer_ms, n_launch, replays = time_steps(K, reps, launchers, flush, stream, graph)
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    # direct launches counted by the handle, plus the kernels of every replay
    launches = handle.launches() - launches0 + replays * per_graph
    handle.synchronize()  # raises if a kernel recorded a device error

    total_ms, value = aggregate_over_ranks(total_ms, step_flops, K, world, dev)
    ms_per_step = total_ms / K

    peaks = load_peaks()
    peak_tf, peak_src = _peak_for(workload, peaks)
    layer_rows = []
    by_kernel = {}
    for j, pr in enumerate(probs):
        t_s = per_layer_ms[j] / n_launch * 1e-3
        tflops = pr["flops"] / t_s / 1e12
        gbs = pr["bytes"] / t_s / 1e9
        roof = min(peak_tf, pr["flops"] / pr["bytes"] * peaks["hbm_gbs"] / 1e3)
        layer_rows.append({"layer": pr["layer"].name, "kernel": pr["kernel"],
                           "us": round(t_s * 1e6, 2), "tflops": round(tflops, 1),
                           "hbm_gbs": round(gbs, 1),
                           "bound": ("alu" if workload == "tiny" else "tensor")
                           if roof >= peak_tf else "hbm",
                           "roofline_tflops": round(roof, 1),
                           "frac_of_roofline": round(tflops / roof, 4)})
        kk = by_kernel.setdefault(pr["kernel"], {"flops": 0, "bytes": 0, "ms": 0.0, "launches": 0})
        kk["flops"] += pr["flops"]
        kk["bytes"] += pr["bytes"]
        kk["ms"] += per_layer_ms[j]
        kk["launches"] += n_launch
    dom_name, dom = max(by_kernel.items(), key=lambda kv: kv[1]["ms"])
    avg_launch_s = dom["ms"] / dom["launches"] * 1e-3
    per_pass = dom["launches"] / n_launch          # launches of this kernel per pass
    flops_per_launch = dom["flops"] / per_pass
    bytes_per_launch = dom["bytes"] / per_pass
    ai = flops_per_launch / bytes_per_launch
    compute_bound = ai * peaks["hbm_gbs"] / 1e3 >= peak_tf
    traffic = None
    tfile = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tfile):
        with open(tfile) as f:
            td = json.load(f)
        ent = td.get(workload, {}).get(dom_name)
        if ent and ent.get("kernel_sha") == kernel_source_hash(dom_name):
            traffic = ent.get("dram_bytes_per_launch")
    if compute_bound:
        achieved = flops_per_launch / avg_launch_s / 1e12
        roofline = {"bound": "alu" if workload == "tiny" else "tensor",
                    "achieved": round(achieved, 1), "peak": round(peak_tf, 1),
                    "unit": "TFLOP/s", "frac": round(achieved / peak_tf, 4), "traffic": traffic,
                    "kernel": dom_name, "peak_source": peak_src}
    else:
        achieved = bytes_per_launch / avg_launch_s / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                    "traffic": traffic, "kernel": dom_name,
                    "peak_source": f"{peaks['source']} copy bandwidth"}

    # end to end: pinned host buffers -> device -> conv -> host, every step
    e2e = run_e2e(args, probs, handle, stream, dev, pass_flops, world)
    dtype = {"bf16": "bf16", "tf32": "tf32", "f32": "f32"}[layers[0].dtype]
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype,
        "data": "synthetic",
        "config": workload_config(workload, world, reps),
        "timing": TIMING if graph is not None else TIMING_DIRECT,
        "roofline": roofline,
        "layers": layer_rows,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(workload, budget_s=args.cpu_seconds if headline
                                           else args.cpu_seconds_config)
    for pr in probs:
        pr["conv"].close()
    del probs, flush
    torch.cuda.empty_cache()
    return res


# Backward routines and the pooling/activation primitives, timed like the
# forward workloads (steps of reps_per_step passes; per-launch CUDA events in
# one pass of every INST_EVERY).
EXTRA_REPS = {"overfeat_bwd_data": 40, "overfeat_bwd_filter": 24, "alexnet_pool_act": 304}


def _bwd_layers():
    from deep_learning_convolution_gb300 import synth
    # the tensor-core layers of the headline stack (layer 1 reads the 3-channel image)
    return [l for l in synth.WORKLOADS["overfeat"] if l.C % 8 == 0]


def _extra_ops(name, handle, dev):
    """[(label, launch(), flops, bytes, kernel, bound)] for one extra workload."""
    import numpy as np
    import torch
    from deep_learning_convolution_gb300 import api, synth
    ops = []
    if name in ("overfeat_bwd_data", "overfeat_bwd_filter"):
        for j, layer in enumerate(synth.WORKLOADS["overfeat"]):
            if layer not in _bwd_layers():
                continue
            x, w, _ = synth.make_inputs(layer, synth.workload_seed("overfeat", j))
            P, Q = layer_output_dims(layer)
            rng = np.random.default_rng(j)
            dy = synth.round_values(rng.standard_normal((layer.N, layer.K, P, Q), dtype=np.float32), "bf16")
            xt, wt = api.layer_tensors(layer, x, w, dev)
            dyt = api.layer_tensors(layer, dy, w[:1], dev)[0]
            kw = dict(pads=(layer.pad_top, layer.pad_bottom, layer.pad_left, layer.pad_right),
                      stride=(layer.u, layer.v), dilation=(layer.dil_h, layer.dil_w))
            flops = 2 * layer.N * layer.K * P * Q * layer.C * layer.R * layer.S
            if name == "overfeat_bwd_data":
                dx = torch.empty_like(xt, dtype=torch.float32)
                op = api.Conv2dBackwardData(handle, wt, dyt, dx, w_axes="KRSC", dy_axes="NHWC",
                                            dx_axes="NHWC", math="bf16", **kw)
                nbytes = dyt.numel() * 2 + wt.numel() * 2 + dx.numel() * 4
                ops.append((layer.name + "_dgrad", (lambda op=op, a=wt, b=dyt, c=dx: op(a, b, c)),
                            flops, nbytes, op.kernel(wt, dyt, dx), "tensor", op))
            else:
                dw = torch.empty(wt.shape, dtype=torch.float32, device=dev)
                op = api.Conv2dBackwardFilter(handle, xt, dyt, dw, x_axes="NHWC", dy_axes="NHWC",
                                              dw_axes="KRSC", math="bf16", **kw)
                nbytes = xt.numel() * 2 + dyt.numel() * 2 + dw.numel() * 4
                ops.append((layer.name + "_wgrad", (lambda op=op, a=xt, b=dyt, c=dw: op(a, b, c)),
                            flops, nbytes, op.kernel(xt, dyt, dw), "tensor", op))
    elif name == "alexnet_pool_act":
        rng = np.random.default_rng(5)
        x = synth.round_values(rng.standard_normal((128, 64, 55, 55), dtype=np.float32), "bf16")
        xt = api.layer_tensors(synth.Layer("a", 128, 64, 55, 55, 1, 1, 1), x, x[:1, :1], dev)[0]
        y = torch.empty((128, 27, 27, 64), dtype=torch.bfloat16, device=dev)
        pool = api.Pool2dForward(handle, xt, y, window=(3, 3), mode="max", stride=(2, 2),
                                 x_axes="NHWC", y_axes="NHWC")
        ops.append(("alex1_out_maxpool_3x3s2", (lambda: pool(xt, y)), 0,
                    xt.numel() * 2 + y.numel() * 2, pool.kernel(xt, y), "hbm", pool))
        ya = torch.empty_like(xt)
        relu = api.ActivationForward(handle, xt, ya, mode="relu", x_axes="NHWC", y_axes="NHWC")
        ops.append(("alex1_out_relu", (lambda: relu(xt, ya)), 0, xt.numel() * 4, "flat", "hbm", relu))
    return ops


def run_extra(args, name, handle, stream, dev, local_rank, world):
    """The bench fields of one extra workload (backward routines or the
    pooling and activation primitives)."""
    import torch
    ops = _extra_ops(name, handle, dev)
    reps = EXTRA_REPS[name]
    for _ in range(args.warmup):
        for _ in range(max(1, reps // 4)):
            for o in ops:
                o[1]()
    torch.cuda.synchronize()
    handle.synchronize()
    K = args.steps
    nl = len(ops)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    graph, per_graph = (capture_passes([o[1] for o in ops], stream, handle, INST_EVERY - 1)
                        if reps % INST_EVERY == 0 else (None, 0))
    sampler = ClockSampler(local_rank)
    torch.cuda.synchronize()
    launches0 = handle.launches()
    sampler.start()
    time.sleep(0.05)
    total_ms, per_ms, n_launch, replays = time_steps(K, reps, [o[1] for o in ops], flush, stream, graph)
    clocks = sampler.stop()
    launches = handle.launches() - launches0 + replays * per_graph
    handle.synchronize()
    pass_flops = sum(o[2] for o in ops)
    pass_bytes = sum(o[3] for o in ops)
    hbm_bound = pass_flops == 0
    # TFLOP/s from FLOPs, or GB/s from bytes (1e12 FLOP = 1e3 GB per unit)
    total_ms, value = aggregate_over_ranks(total_ms, pass_flops * reps if not hbm_bound
                                           else pass_bytes * reps * 1e3, K, world, dev)
    peaks = load_peaks()
    rows = []
    for j, o in enumerate(ops):
        t_s = per_ms[j] / n_launch * 1e-3
        gbs = o[3] / t_s / 1e9
        if o[5] == "hbm":
            rows.append({"layer": o[0], "kernel": o[4], "us": round(t_s * 1e6, 2),
                         "hbm_gbs": round(gbs, 1), "bound": "hbm",
                         "frac_of_roofline": round(gbs / peaks["hbm_gbs"], 4)})
        else:
            tf = o[2] / t_s / 1e12
            roof = min(peaks["bf16_tflops"], o[2] / o[3] * peaks["hbm_gbs"] / 1e3)
            rows.append({"layer": o[0], "kernel": o[4], "us": round(t_s * 1e6, 2),
                         "tflops": round(tf, 1), "hbm_gbs": round(gbs, 1),
                         "bound": "tensor" if roof >= peaks["bf16_tflops"] else "hbm",
                         "roofline_tflops": round(roof, 1), "frac_of_roofline": round(tf / roof, 4)})
    dom = max(range(nl), key=lambda j: per_ms[j])
    t_dom = per_ms[dom] / n_launch * 1e-3
    if hbm_bound:
        ach = ops[dom][3] / t_dom / 1e9
        roofline = {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4), "traffic": None,
                    "kernel": ops[dom][4], "peak_source": f"{peaks['source']} copy bandwidth"}
        unit, metric = "GB/s", "pooling/activation GB/s (x read + y written once)"
    else:
        kern = ops[dom][4]
        fl = sum(o[2] for o in ops if o[4] == kern)
        t = sum(per_ms[j] for j in range(nl) if ops[j][4] == kern) / n_launch * 1e-3
        ach = fl / t / 1e12
        roofline = {"bound": "tensor", "achieved": round(ach, 1), "peak": peaks["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": round(ach / peaks["bf16_tflops"], 4),
                    "traffic": None, "kernel": kern,
                    "peak_source": f"{peaks['source']} bf16 burst"}
        unit, metric = "TFLOP/s", "TFLOP/s (direct-conv FLOPs of the gradient)"
    res = {"what": metric, "value": round(value, 2), "unit": unit, "steps": K,
           "warmup": args.warmup, "ms_per_step": round(total_ms / K, 4), "dtype": "bf16",
           "config": {"workload": name, "layers": [o[0] for o in ops], "reps_per_step": reps,
                      "l2": "flushed between steps (256 MiB write, untimed)"},
           "timing": TIMING if graph is not None else TIMING_DIRECT,
           "roofline": roofline, "layers": rows, "gpu_launches": launches, "clocks": clocks,
           "e2e": None}
    for o in ops:
        if o[6] is not None:
            o[6].close()
    del ops, flush
    torch.cuda.empty_cache()
    return res


def run_ours(args, rank, world, local_rank):
    import torch
    from deep_learning_convolution_gb300 import api
    from deep_learning_convolution_gb300 import build as dlc_build

    dlc_build.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    # a stream of its own (the legacy default stream cannot be captured in a
    # CUDA graph), current for every torch operation of the run
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)
    handle = api.Handle(stream)
    result = run_workload(args, args.workload, handle, stream, dev, rank, world, local_rank,
                          headline=True)
    if not args.no_configs:
        configs = {}
        for wl in CONFIG_ORDER:
            if wl == args.workload:
                continue
            r = run_workload(args, wl, handle, stream, dev, rank, world, local_rank,
                             headline=False)
            r.pop("metric")
            r.pop("n_gpus")
            configs[wl] = r
        for name in EXTRA_REPS:
            configs[name] = run_extra(args, name, handle, stream, dev, local_rank, world)
        result["configs"] = configs
    handle.close()
    if world > 1:
        torch.distributed.destroy_process_group()
    return result if rank == 0 else None


def run_e2e(args, probs, handle, stream, dev, pass_flops, world):
    """End-to-end throughput: every e2e step copies one pass's inputs in from
    pinned host memory, runs the pass and copies every y back."""
    import numpy as np
    import torch
    steps = max(3, min(args.steps, args.e2e_steps))
    host = []
    h2d = d2h = 0
    for pr in probs:
        hx = torch.empty(pr["x"].shape, dtype=pr["x"].dtype, pin_memory=True)
        hx.copy_(pr["x"].cpu())
        hw = torch.empty(pr["w"].shape, dtype=pr["w"].dtype, pin_memory=True)
        hw.copy_(pr["w"].cpu())
        hy = torch.empty(pr["y"].shape, dtype=pr["y"].dtype, pin_memory=True)
        host.append((hx, hw, hy))
        h2d += hx.numel() * hx.element_size() + hw.numel() * hw.element_size()
        d2h += hy.numel() * hy.element_size()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    # The layers of a step are independent problems, so their copies overlap
    # other layers' convolutions: inputs go in on one copy stream, results
    # come out on another, and events keep each layer's buffers ordered (its
    # inputs land before its convolution; the previous step's convolution is
    # done reading them before they are overwritten; the previous read-back of
    # y is done before the convolution writes y again).  Every step still
    # moves all inputs in and all results out.
    s_in = torch.cuda.Stream(device=dev)
    s_outs = [torch.cuda.Stream(device=dev) for _ in range(args.e2e_out_streams)]
    nl = len(probs)
    ev_in = [torch.cuda.Event() for _ in range(nl)]
    ev_conv = [None] * nl
    ev_out = [[None] * len(s_outs) for _ in range(nl)]
    # each y comes back in equal contiguous parts, one per read-back stream
    # (copy engines work in parallel)
    parts = []
    for pr, (hx, hw, hy) in zip(probs, host):
        dv, hv = pr["y"].view(-1), hy.view(-1)
        n = dv.numel()
        cuts = [n * i // len(s_outs) for i in range(len(s_outs) + 1)]
        parts.append([(dv[a:b], hv[a:b]) for a, b in zip(cuts[:-1], cuts[1:])])

    def one():
        for j, (pr, (hx, hw, hy)) in enumerate(zip(probs, host)):
            with torch.cuda.stream(s_in):
                if ev_conv[j] is not None:
                    s_in.wait_event(ev_conv[j])
                pr["x"].copy_(hx, non_blocking=True)
                pr["w"].copy_(hw, non_blocking=True)
                ev_in[j].record(s_in)
            stream.wait_event(ev_in[j])
            for ev in ev_out[j]:
                if ev is not None:
                    stream.wait_event(ev)
            pr["conv"](pr["x"], pr["w"], pr["y"])
            ev_conv[j] = torch.cuda.Event()
            ev_conv[j].record(stream)
            for i, (so, (dpart, hpart)) in enumerate(zip(s_outs, parts[j])):
                with torch.cuda.stream(so):
                    so.wait_event(ev_conv[j])
                    hpart.copy_(dpart, non_blocking=True)
                    ev_out[j][i] = torch.cuda.Event()
                    ev_out[j][i].record(so)

    def join():  # the compute stream waits for every copy of the step
        for j in range(nl):
            for ev in ev_out[j]:
                stream.wait_event(ev)

    one()
    join()
    torch.cuda.synchronize()
    start.record(stream)
    s_in.wait_event(start)  # no copy of the timed steps starts before the clock
    for _ in range(steps):
        one()
    join()
    end.record(stream)
    torch.cuda.synchronize()
    ms, value = aggregate_over_ranks(start.elapsed_time(end), pass_flops, steps, world, dev)
    return {"value": round(value, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": round(ms / steps, 3)}


# ---------------------------------------------------------------------------
# CPU oracle (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------

def oracle_sample_step(workload, images=1, threads=None):
    """Runs the oracle over `images` images of every layer of the workload;
    returns (direct-conv FLOPs, seconds, threads)."""
    import numpy as np
    from deep_learning_convolution_gb300 import synth
    from oracle import oracle
    threads = threads or oracle.default_threads()
    flops = 0
    secs = 0.0
    for j, layer in enumerate(synth.WORKLOADS[workload]):
        x, w, _ = synth.make_inputs(layer, synth.workload_seed(workload, j), batch=images)
        x64, w64 = x.astype(np.float64), w.astype(np.float64)
        t0 = time.perf_counter()
        y, _ = oracle.conv2d_fprop(x64, w64, pads=(layer.pad_top, layer.pad_bottom,
                                                   layer.pad_left, layer.pad_right),
                                   stride=(layer.u, layer.v), dilation=(layer.dil_h, layer.dil_w),
                                   nthreads=threads)
        secs += time.perf_counter() - t0
        flops += 2 * images * layer.K * y.shape[2] * y.shape[3] * layer.C * layer.R * layer.S
    return flops, secs, threads


def cpu_baseline(workload, budget_s=15.0):
    from oracle import oracle
    oracle.build()
    flops, secs, threads = oracle_sample_step(workload, images=1)
    total_f, total_s, runs = flops, secs, 1
    while total_s < budget_s and runs < 64:
        f, s, _ = oracle_sample_step(workload, images=1)
        total_f += f
        total_s += s
        runs += 1
    return {"value": round(total_f / total_s / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{runs} x (1 image through every {workload} layer, all K, full P x Q), "
                      f"FP64 direct convolution, {total_s:.1f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    from oracle import oracle
    oracle.build()
    for _ in range(args.warmup):
        oracle_sample_step(args.workload, images=1)
    flops = 0
    secs = 0.0
    threads = oracle.default_threads()
    for _ in range(args.steps):
        f, s, threads = oracle_sample_step(args.workload, images=1)
        flops += f
        secs += s
    value = flops / secs / 1e12
    sample = (f"each step: 1 image of the {args.workload} stack through every layer "
              f"(all K, full P x Q), FP64 direct convolution on {threads} host threads")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": workload_config(args.workload, world, args.reps_per_step),
            "timing": "host wall clock (perf_counter) around each sampled layer",
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_profile_layer(args):
    """Launches one layer of the workload `reps` times (for ncu captures); prints
    the CUDA-event time per launch of a second batch of `reps` launches."""
    import torch
    from deep_learning_convolution_gb300 import api, synth
    from deep_learning_convolution_gb300 import build as dlc_build
    dlc_build.build()
    j = args.profile_layer
    if args.workload in EXTRA_REPS:  # one op of a backward or pooling workload
        handle = api.Handle()
        ops = _extra_ops(args.workload, handle, "cuda")
        op = ops[j]
        for _ in range(args.reps):
            op[1]()
        torch.cuda.synchronize()
        handle.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record()
        for _ in range(args.reps):
            op[1]()
        end.record()
        torch.cuda.synchronize()
        handle.synchronize()
        print(json.dumps({"layer": op[0], "kernel": op[4],
                          "us_per_launch": round(start.elapsed_time(end) * 1e3 / args.reps, 2)}))
        for o in ops:
            if o[6] is not None:
                o[6].close()
        handle.close()
        return
    layer = synth.WORKLOADS[args.workload][j]
    x, w, _ = synth.make_inputs(layer, synth.workload_seed(args.workload, j), batch=args.batch)
    handle = api.Handle()
    xt, wt = api.layer_tensors(layer, x, w, "cuda")
    conv, y = api.layer_problem(handle, layer, xt, wt)
    for _ in range(args.reps):
        conv(xt, wt, y)
    torch.cuda.synchronize()
    handle.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(args.reps):
        conv(xt, wt, y)
    end.record()
    torch.cuda.synchronize()
    handle.synchronize()
    print(json.dumps({"layer": layer.name, "kernel": conv.kernel(xt, wt, y),
                      "us_per_launch": round(start.elapsed_time(end) * 1e3 / args.reps, 2)}))
    conv.close()
    handle.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE, choices=CONFIG_ORDER + list(EXTRA_REPS),
                    help="the backward and pooling workloads only with --profile-layer")
    ap.add_argument("--reps-per-step", type=int, default=None,
                    help="passes over the stack per step (default: the workload's fixed count)")
    ap.add_argument("--no-configs", action="store_true",
                    help="time only --workload (no `configs` key with the other workloads)")
    ap.add_argument("--cpu-seconds-config", type=float, default=3.0,
                    help="oracle time budget of each non-headline workload's cpu_baseline")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--e2e-out-streams", type=int, default=1,
                    help="streams the end-to-end run reads results back on")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-layer", type=int, default=None,
                    help="launch only this layer of the workload 2*reps times (ncu captures)")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--batch", type=int, default=None, help="override N (profile mode)")
    args = ap.parse_args()
    if args.profile_layer is not None:
        run_profile_layer(args)
        return
    if args.workload in EXTRA_REPS:
        ap.error(f"--workload {args.workload} goes with --profile-layer (the bench times it in `configs`)")
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local_rank = env_rank()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, local_rank)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
