#!/usr/bin/env python
"""Throughput of the routed MoE expert layer (forward + backward) on GB300.

Default workload: the GPT-OSS-20B-shaped layer (T = 16384 tokens = 4 x 4096,
d = f = 2880, E = 32 experts, top-4), seeded synthetic inputs, bf16.

One step = the whole layer: moe_route -> moe_permute -> moe_expert_fwd ->
moe_combine -> moe_expert_bwd -> moe_combine (dx) -> moe_route_bwd, inputs
resident in HBM. W untimed warm-up steps, then K steps timed with CUDA events
between a barrier + synchronize on both sides; the slowest rank's time counts.
Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config NAME] [--no-cpu-baseline] [--no-side]

With the default workload, the line also carries "configs": the
Qwen3-30B-A3B-shaped layer, the small-M forward sweep (T = 128 ... 2048) and
the fine-grained 512-expert layer, each timed in the same run (median step,
whole-step roofline, every expert GEMM against its bound, the benchmark spec's
targets, its own clock record) and, under "forward", its inference forward
timed two ways: the five calls and the fused expert GEMMs
(moe_expert_fwd_fused), each with its bytes and roofline fraction; and the
decode workloads (1 and 8 tokens, forward) replayed as CUDA graphs, general
path and one-launch forward, against their weight-streaming bound.
ms_per_step is the median of the timed steps; value = tokens / median step.

--impl reference times the float64 CPU oracle (the deliberately slow,
obviously correct definition) on a bounded sample of the same workload on
the host cores; under torchrun only rank 0 runs it.

Several GPUs: one process per GPU under torchrun, each an independent replica
of the layer (the layer needs no exchange between GPUs on this path);
value = tokens of all ranks / the slowest rank's time, "scaling": "weak".
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "routed tokens/s per MoE layer fwd+bwd, bf16, 1 GB300; % of roofline"
UNIT = "tokens/s"
DEFAULT_CONFIG = "gptoss20b"
STEP_KERNELS = ["router_logits", "topk", "permute", "gateup_fwd", "down_fwd", "combine",
                "combine_bwd", "down_dgrad", "gateup_dgrad", "wgrad_down", "wgrad_gateup",
                "route_bwd"]
FWD_KERNELS = STEP_KERNELS[:6]
FUSED_KERNELS = ["router_logits", "topk", "permute", "fused_fwd", "combine"]


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--align", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-tokens", type=int, default=8192,
                    help="tokens in the oracle's bounded sample (cpu_baseline)")
    ap.add_argument("--ref-tokens", type=int, default=1,
                    help="tokens per step of the reference (oracle) arm")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-side", action="store_true",
                    help="time the headline workload only (not the other workloads)")
    ap.add_argument("--side-steps", type=int, default=30,
                    help="timed steps of each other workload")
    ap.add_argument("--path", choices=["auto", "general", "decode", "fused"], default="auto",
                    help="decode: the one-launch forward (moe_decode_fwd), forward-only "
                         "workloads of at most 8 tokens; fused: the inference forward with the "
                         "fused expert GEMMs (moe_expert_fwd_fused), forward only; auto: the "
                         "general path, measured faster than the one-launch forward at every "
                         "decode size")
    ap.add_argument("--graph", action="store_true",
                    help="launch each timed step as one captured CUDA graph (launch-bound sizes)")
    return ap.parse_args(argv)


# ----------------------------------------------------------------- peaks --

def load_peaks() -> dict:
    """Measured denominators (MEASURED_PEAKS.json), else the stated fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# -------------------------------------------------------------- clocks --

CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={CLOCK_QUERY}",
                 "--format=csv,noheader", "-lms", "50"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        return parse_clock_rows(rows)


def parse_clock_rows(rows) -> dict | None:
    def mhz(s):
        m = re.match(r"([0-9.]+)", s)
        return float(m.group(1)) if m else None

    sm = [mhz(r[1]) for r in rows if mhz(r[1]) is not None]
    mx = [mhz(r[2]) for r in rows if mhz(r[2]) is not None]
    if not sm:
        return None
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
    # samples under load: power draw in the upper half of the range the run saw
    pw = [mhz(r[3]) for r in rows]
    load = sm
    if all(p is not None for p in pw) and len(pw) == len(sm) and max(pw) > min(pw):
        cut = (max(pw) + min(pw)) / 2
        load = [c for c, p in zip(sm, pw) if p >= cut] or sm
    return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(mx) if mx else None,
            "samples": len(sm), "samples_under_load": len(load),
            "sm_mhz_all_samples": statistics.median(sm), "reasons": reasons,
            "period_ms": 50}


# ---------------------------------------------------------- distributed --

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float, device=None) -> float:
    """Max of a float over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ------------------------------------------------------------- oracle --

def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


def oracle_sample(inp: dict, wl, tokens: int) -> float:
    """Seconds the float64 oracle takes for forward + backward of the first
    `tokens` tokens of the workload (all experts' weights as in the layer)."""
    from oracle import moe_oracle as mo
    t0 = time.perf_counter()
    x = inp["x"][:tokens]
    fw = mo.forward(x, inp["w_router"], inp.get("bias"), inp["w_gate"], inp["w_up"],
                    inp["w_down"], wl.k)
    if wl.backward:
        mo.backward(x, inp["w_router"], inp.get("bias"), inp["w_gate"], inp["w_up"],
                    inp["w_down"], wl.k, inp["dy"][:tokens], fwd=fw)
    return time.perf_counter() - t0


# ------------------------------------------------------------- traffic --

# The source files that define each kernel (its translation unit and the
# device-code header it includes); a recorded ncu figure stays valid while
# these bytes are unchanged.
_GEMM_SOURCES = ("gemm.cu", "common.cuh")
KERNEL_SOURCES = {name: _GEMM_SOURCES for name in (
    "gateup_fwd", "down_fwd", "down_dgrad", "gateup_dgrad", "wgrad_down", "wgrad_gateup")}


def kernel_digest(kernel: str) -> str:
    """sha256 (first 16 hex digits) of the kernel's source files; all of csrc/
    for a kernel with no entry in KERNEL_SOURCES."""
    base = os.path.join(ROOT, "mixture_experts_routed_softmax_gb300", "csrc")
    files = KERNEL_SOURCES.get(kernel) or tuple(sorted(os.listdir(base)))
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(base, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, config: str):
    """DRAM bytes per launch from a committed ncu summary of the same kernel
    source (profiles/<kernel>_<config>.md), else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{config}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    s = re.search(r"kernel_sources_sha256_16:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != kernel_digest(kernel):
        return None
    return float(m.group(1))


# ---------------------------------------------------------------- ours --

# the workloads timed beside the headline one, in the same run (fwd+bwd unless
# the workload is forward-only): Qwen3-30B-A3B-shaped, the small-M sweep and
# the fine-grained 512-expert layer
SIDE_CONFIGS = ["qwen3_30b", "smallm_T128", "smallm_T512", "smallm_T1024", "smallm_T2048",
                "fine512"]
# the benchmark spec's per-workload targets: expert GEMMs bound by the tensor cores
# at >= 60% of the bf16 peak, those bound by HBM at >= 70% of its bandwidth
TARGET_TENSOR = 0.60
TARGET_HBM = 0.70
GEMM_KERNELS = ("gateup_fwd", "down_fwd", "down_dgrad", "gateup_dgrad", "wgrad_down",
                "wgrad_gateup", "fused_fwd")


def kernel_roofline(name, fl, by, ms, peaks):
    """Achieved rate of one launch against the bound its algorithmic FLOPs and
    bytes put it under (measured burst peaks; the sustained bf16 fraction too)."""
    t_tensor = fl / (peaks["bf16_tflops"] * 1e12)
    t_hbm = by / (peaks["hbm_gbs"] * 1e9)
    if t_tensor >= t_hbm:
        achieved = fl / (ms * 1e-3) / 1e12
        return {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                "peak_kind": f"bf16 burst, {peaks['source']}"}
    achieved = by / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "peak_kind": f"hbm copy, {peaks['source']}"}


def time_steps(run, steps, stream, flush_buf, dom_timer=None):
    """Times `steps` calls of run() with CUDA events on `stream`, one pair of
    events per step; with flush_buf, L2 is flushed (a write of twice its size)
    before each step, outside the step's events. Returns per-step ms and the
    span from the first step's start to the last step's end."""
    import torch
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    pairs = []
    if flush_buf is None:
        evs[0].record(stream)
        for i in range(steps):
            run()
            evs[i + 1].record(stream)
    else:
        for _ in range(steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            flush_buf.zero_()
            e0.record(stream)
            run()
            e1.record(stream)
            pairs.append((e0, e1))
    torch.cuda.synchronize()
    if flush_buf is None:
        per = [evs[i].elapsed_time(evs[i + 1]) for i in range(steps)]
        span = evs[0].elapsed_time(evs[steps])
    else:
        per = [a.elapsed_time(b) for a, b in pairs]
        span = sum(per)
    return per, span


def profile_kernels(step, kernels, lib_mod):
    """Per-launch device ms of each kernel group, from three steps each (the
    library's event timer, outside any timed region)."""
    per_kernel = {}
    for name in kernels:
        lib_mod.call("moe_timer_start", lib_mod.KERNELS[name], 8)
        for _ in range(3):
            step()
        ms, n = lib_mod.ctypes.c_float(), lib_mod.ctypes.c_int()
        lib_mod.call("moe_timer_read", lib_mod.ctypes.byref(ms), lib_mod.ctypes.byref(n))
        per_kernel[name] = ms.value / max(n.value, 1)
    return per_kernel


def forward_compare(layer, wl, x, stream, flush_buf, steps, shape, peaks):
    """The inference forward two ways on the same inputs: the five calls
    (route, permute, gate/up, down, combine; G and U kept for a backward)
    and the fused expert GEMMs (moe_expert_fwd_fused: one persistent launch,
    G and U never leave tensor memory); median of `steps` each, with their
    algorithmic bytes and whole-forward roofline fractions."""
    from mixture_experts_routed_softmax_gb300 import accounting
    b5 = layer.buffers(wl.T, backward=False)
    bf = layer.fused_buffers(wl.T)

    def five():
        layer.forward(x, b5)

    def fused():
        layer.forward_fused(x, bf)

    for _ in range(3):
        five()
        fused()
    st = layer.status()
    if st != 0:
        raise RuntimeError(f"forward comparison: device status {st}")
    out = {}
    for nm, fn, costs in (("five_call", five, accounting.kernel_costs(shape, backward=False)),
                          ("fused", fused, accounting.fused_forward_costs(shape))):
        per, _ = time_steps(fn, steps, stream, flush_buf)
        med = statistics.median(per)
        F = sum(c[0] for c in costs.values())
        B = sum(c[1] for c in costs.values())
        t_roof = accounting.roofline_seconds(F, B, peaks["bf16_tflops"], peaks["hbm_gbs"])
        out[nm] = {"ms": round(med, 4), "bytes": B, "roofline_frac": round(t_roof * 1e3 / med, 3)}
    st = layer.status()
    if st != 0:
        raise RuntimeError(f"forward comparison: device status {st}")
    out["fused_speedup"] = round(out["five_call"]["ms"] / out["fused"]["ms"], 3)
    del b5, bf
    return out


DECODE_SIDE = ["decode_T1", "decode_T8"]


def run_decode_side(name, dev, peaks, steps):
    """A decode workload (forward only, a few tokens), each step replayed as
    one captured CUDA graph with L2 flushed between steps: the general path
    (seven launches) and the one-launch decode forward, against the time the
    active experts' weights take to stream at the measured HBM rate."""
    import torch
    import workloads
    from mixture_experts_routed_softmax_gb300 import accounting
    from mixture_experts_routed_softmax_gb300.layer import MoELayer

    wl = workloads.CONFIGS[name]
    inp = workloads.generate_device(wl, dev, with_dy=False)
    layer = MoELayer(inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"], inp["w_down"],
                     wl.k, wl.align)
    x = inp["x"]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    out = {"workload": f"{wl.name}: {wl.note}", "T": wl.T, "d": wl.d, "f": wl.f, "E": wl.E,
           "k": wl.k, "steps": steps, "l2": "flushed between steps", "graph": True}
    for path, bufs, fwd in (("general", lambda: layer.buffers(wl.T, backward=False),
                             layer.forward),
                            ("one_launch", lambda: layer.decode_buffers(wl.T), layer.decode_fwd)):
        b = bufs()
        for _ in range(3):
            fwd(x, b)
        st = layer.status()
        if st != 0:
            raise RuntimeError(f"{name}/{path}: device status {st}")
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fwd(x, b)
        for _ in range(3):
            g.replay()
        per, _ = time_steps(g.replay, steps, stream, flush_buf)
        if layer.status() != 0:
            raise RuntimeError(f"{name}/{path}: device status")
        out[path + "_us"] = round(statistics.median(per) * 1e3, 2)
        if path == "general":
            e_act = int(torch.unique(b.topk_idx).numel())
    shape = accounting.Shape(T=wl.T, d=wl.d, f=wl.f, E=wl.E, k=wl.k, E_active=e_act)
    fl, by = accounting.decode_costs(shape)
    bound_us = by / (peaks["hbm_gbs"] * 1e9) * 1e6
    best = min(out["general_us"], out["one_launch_us"])
    out.update(E_active=e_act, weight_bound_us=round(bound_us, 2),
               frac_of_bound=round(bound_us / best, 3),
               path_auto="general" if out["general_us"] <= out["one_launch_us"] else "one_launch")
    del layer, inp
    torch.cuda.empty_cache()
    return out


def run_side(name, dev, local_rank, peaks, steps, warmup):
    """One of the other workloads, timed in the same run: median step, the
    whole-step roofline, every expert GEMM against its bound, the small-M
    sweep's expert-weight streaming rate, and the benchmark spec's targets."""
    import torch
    import workloads
    from mixture_experts_routed_softmax_gb300 import _lib, accounting
    from mixture_experts_routed_softmax_gb300.layer import MoELayer

    wl = workloads.CONFIGS[name]
    inp = workloads.generate_device(wl, dev, with_dy=wl.backward)
    layer = MoELayer(inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"], inp["w_down"],
                     wl.k, wl.align)
    b = layer.buffers(wl.T, backward=wl.backward)
    x = inp["x"]
    dy = inp.get("dy")

    def step():
        layer.forward(x, b)
        if wl.backward:
            layer.backward(dy, b)

    sampler = ClockSampler(local_rank).start()
    for _ in range(max(warmup, 3)):
        step()
    st = layer.status()
    if st != 0:
        raise RuntimeError(f"{name}: device status {st}: {_lib.status_str(st)}")
    kernels = STEP_KERNELS if wl.backward else FWD_KERNELS
    per_kernel = profile_kernels(step, kernels, _lib)
    shape = accounting.Shape(T=wl.T, d=wl.d, f=wl.f, E=wl.E, k=wl.k,
                             E_active=int((b.counts > 0).sum()))
    costs = accounting.kernel_costs(shape, wl.backward)
    F = sum(c[0] for c in costs.values())
    B = sum(c[1] for c in costs.values())
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = B < 4 * l2
    flush_buf = torch.empty(2 * l2, dtype=torch.uint8, device=dev) if flush else None
    stream = torch.cuda.current_stream()
    per, span = time_steps(step, steps, stream, flush_buf)
    clocks = sampler.stop()
    st = layer.status()
    if st != 0:
        raise RuntimeError(f"{name}: device status {st}: {_lib.status_str(st)}")
    med = statistics.median(per)
    t_roof = accounting.roofline_seconds(F, B, peaks["bf16_tflops"], peaks["hbm_gbs"])
    gemms = {}
    for k_ in GEMM_KERNELS:
        if k_ in per_kernel:
            r = kernel_roofline(k_, *costs[k_], per_kernel[k_], peaks)
            gemms[k_] = {"ms": round(per_kernel[k_], 4), "bound": r["bound"],
                         "achieved": round(r["achieved"], 1), "unit": r["unit"],
                         "frac": round(r["frac"], 3)}
    dominant = max(per_kernel, key=per_kernel.get)
    dom = kernel_roofline(dominant, *costs[dominant], per_kernel[dominant], peaks)
    dom.update(kernel=dominant, ms_per_launch=per_kernel[dominant])
    out = {"workload": f"{wl.name}: {wl.note}", "T": wl.T, "d": wl.d, "f": wl.f, "E": wl.E,
           "k": wl.k, "align": wl.align, "backward": wl.backward, "tau": inp.get("tau"),
           "E_active": shape.E_active, "steps": steps, "ms_per_step": med,
           "ms_per_step_mean": span / steps, "tokens_per_s": wl.T / (med * 1e-3),
           "l2": "flushed between steps" if flush else "inputs larger than L2",
           "layer_roofline": {"flops": F, "bytes": B, "t_roof_ms": t_roof * 1e3,
                              "frac": t_roof * 1e3 / med},
           "roofline": dom, "gemms": gemms,
           "kernels_ms": {k_: round(v, 4) for k_, v in per_kernel.items()}, "clocks": clocks}
    misses = [k_ for k_, g in gemms.items()
              if g["frac"] < (TARGET_TENSOR if g["bound"] == "tensor" else TARGET_HBM)]
    if not wl.backward:
        # the small-M sweep is reported as the rate the forward streams the
        # active experts' weights (Halo "Performance", §Levers that do not help here)
        wbytes = 3 * shape.E_active * wl.d * wl.f * 2
        gbs = wbytes / (med * 1e-3) / 1e9
        out["weight_stream"] = {"bytes": wbytes, "gbs": gbs, "frac": gbs / peaks["hbm_gbs"]}
        if gbs / peaks["hbm_gbs"] < TARGET_HBM:
            misses.append("weight_stream")
    out["targets"] = {"tensor_bound_gemm_frac": TARGET_TENSOR, "hbm_bound_frac": TARGET_HBM,
                      "met": not misses, "missed": misses}
    del b
    out["forward"] = forward_compare(layer, wl, x, stream, flush_buf, steps, shape, peaks)
    del layer, inp
    torch.cuda.empty_cache()
    return out


def run_ours(args, rank, world, local_rank):
    import torch
    import workloads
    from mixture_experts_routed_softmax_gb300 import _lib, accounting
    from mixture_experts_routed_softmax_gb300.layer import MoELayer

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = workloads.CONFIGS[args.config]
    if args.align:
        wl = wl.with_(align=args.align)
    fused = args.path == "fused"
    if fused:
        wl = wl.with_(backward=False)
    inp = workloads.generate(wl, with_dy=wl.backward)
    layer = MoELayer.from_inputs(inp, wl.k, wl.align, device=dev)
    decode = args.path == "decode"
    if decode and (wl.backward or wl.T > 8):
        raise SystemExit("the decode path runs forward-only workloads of at most 8 tokens")
    if decode:
        new_buffers = lambda: layer.decode_buffers(wl.T)  # noqa: E731
        fwd = layer.decode_fwd
    elif fused:
        new_buffers = lambda: layer.fused_buffers(wl.T)  # noqa: E731
        fwd = layer.forward_fused
    else:
        new_buffers = lambda: layer.buffers(wl.T, backward=wl.backward)  # noqa: E731
        fwd = layer.forward
    b = new_buffers()
    x = inp["x"].to(dev)
    dy = inp["dy"].to(dev) if wl.backward else None
    lib = _lib.load()
    peaks = load_peaks()

    def step():
        fwd(x, b)
        if wl.backward:
            layer.backward(dy, b)

    def active_experts():
        if decode:
            return int(torch.unique(b.topk_idx).numel())
        return int((b.counts > 0).sum())

    # SM clocks and throttle reasons are sampled from the first warm-up step to
    # the end of the timed region
    sampler = ClockSampler(local_rank).start()
    for _ in range(max(args.warmup, 3)):
        step()
    status = layer.status()
    if status != 0:
        raise RuntimeError(f"device status {status}: {_lib.status_str(status)}")

    kernels = (["decode"] if decode else FUSED_KERNELS if fused
               else STEP_KERNELS if wl.backward else FWD_KERNELS)
    per_kernel = profile_kernels(step, kernels, _lib)
    # "combine" fires twice per step (y and dx); the timer averaged both
    dominant = max(per_kernel, key=per_kernel.get)

    # ------------------------------------------------------ timed region --
    stream = torch.cuda.current_stream()
    run = step
    graph_launches = 0
    if args.graph:
        # the whole step captured once (its kernels become graph nodes) and
        # replayed; the library's launch counter sees the capture only
        g = torch.cuda.CUDAGraph()
        c0 = int(lib.moe_kernel_launches())
        with torch.cuda.graph(g):
            step()
        graph_launches = int(lib.moe_kernel_launches()) - c0
        torch.cuda.synchronize()
        run = g.replay
        for _ in range(3):
            run()
    else:
        # the dominant kernel's own launches are timed live, on the stream the
        # library launches them on, inside the timed region
        _lib.call("moe_timer_start", _lib.KERNELS[dominant], args.steps * 2)
    # A step that moves less than four L2s of data would find its weights in
    # L2 again on the next step: then L2 is flushed (a write of twice its
    # size) between steps, outside each step's own pair of events.
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    shape = accounting.Shape(T=wl.T, d=wl.d, f=wl.f, E=wl.E, k=wl.k, E_active=active_experts())
    if decode:
        costs = {"decode": accounting.decode_costs(shape)}
    elif fused:
        costs = accounting.fused_forward_costs(shape)
    else:
        costs = accounting.kernel_costs(shape, wl.backward)
    step_bytes = sum(c[1] for c in costs.values())
    flush = step_bytes < 4 * l2_bytes
    flush_buf = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev) if flush else None
    launches0 = int(lib.moe_kernel_launches())
    barrier()
    torch.cuda.synchronize()
    per_step, span_ms = time_steps(run, args.steps, stream, flush_buf)
    barrier()
    launches = int(lib.moe_kernel_launches()) - launches0 + graph_launches * args.steps
    clocks = sampler.stop()
    if args.graph:
        dom_ms = per_kernel[dominant]        # from the single-kernel timer steps above
    else:
        ms, n = _lib.ctypes.c_float(), _lib.ctypes.c_int()
        _lib.call("moe_timer_read", _lib.ctypes.byref(ms), _lib.ctypes.byref(n))
        dom_ms = ms.value / max(n.value, 1)
    status = layer.status()
    if status != 0:
        raise RuntimeError(f"device status {status}: {_lib.status_str(status)}")
    # the median step (the survey's protocol); the slowest rank's counts
    med_ms = max_over_ranks(statistics.median(per_step), dev)
    span_ms = max_over_ranks(span_ms, dev)

    # --------------------------------------------------------- end to end --
    # Every step copies its inputs (x, dY) from pinned host memory and its
    # results (y, dx) back, through the same public calls. Two sets of device
    # buffers alternate, and the copies run on two copy streams, so step i's
    # copies overlap the neighbouring steps' kernels, as a training loop that
    # prefetches its next batch does; the timed region starts before the first
    # upload and ends when the last result has reached the host.
    e2e = None
    if not args.no_e2e:
        x_h = inp["x"].pin_memory()
        dy_h = inp["dy"].pin_memory() if wl.backward else None
        y_h = [torch.empty_like(inp["x"]).pin_memory() for _ in range(2)]
        dx_h = [torch.empty_like(inp["x"]).pin_memory() for _ in range(2)] if wl.backward else None
        bi = x_h.numel() * 2 + (dy_h.numel() * 2 if wl.backward else 0)
        bo = y_h[0].numel() * 2 + (dx_h[0].numel() * 2 if wl.backward else 0)
        bufs = [b, new_buffers()]
        xs = [torch.empty_like(x) for _ in range(2)]
        dys = [torch.empty_like(dy) for _ in range(2)] if wl.backward else None
        up = torch.cuda.Stream(device=dev)       # host -> device
        down = torch.cuda.Stream(device=dev)     # device -> host
        h2d = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        d2h = [torch.cuda.Event() for _ in range(2)]
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)

        def upload(j):
            with torch.cuda.stream(up):
                xs[j].copy_(x_h, non_blocking=True)
                if wl.backward:
                    dys[j].copy_(dy_h, non_blocking=True)
                h2d[j].record(up)

        for j in range(2):
            d2h[j].record(down)                  # nothing pending on either set yet
        barrier()
        torch.cuda.synchronize()
        ev0.record(stream)
        up.wait_stream(stream)
        down.wait_stream(stream)
        for j in range(min(2, args.steps)):
            upload(j)
        for i in range(args.steps):
            j = i & 1
            stream.wait_event(h2d[j])            # step i's inputs are in set j
            stream.wait_event(d2h[j])            # step i-2's results have left set j
            fwd(xs[j], bufs[j])
            if wl.backward:
                layer.backward(dys[j], bufs[j])
            done[j].record(stream)
            down.wait_event(done[j])
            with torch.cuda.stream(down):
                y_h[j].copy_(bufs[j].y, non_blocking=True)
                if wl.backward:
                    dx_h[j].copy_(bufs[j].dx, non_blocking=True)
                d2h[j].record(down)
            if i + 2 < args.steps:               # step i+2's inputs, once step i has read set j
                up.wait_event(done[j])
                upload(j)
        stream.wait_stream(down)
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier()
        e2e_ms = max_over_ranks(ev0.elapsed_time(ev1), dev)
        assert torch.equal(y_h[(args.steps - 1) & 1], bufs[(args.steps - 1) & 1].y.cpu())
        e2e = {"value": world * wl.T * args.steps / (e2e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
               "overlap": "uploads and downloads on two copy streams, two buffer sets"}

    # ----------------------------------------------------------- roofline --
    fl, by = costs[dominant]
    roof = kernel_roofline(dominant, fl, by, dom_ms, peaks)
    roof["kernel"] = dominant
    roof["ms_per_launch"] = dom_ms
    roof["algorithmic_flops_per_launch"] = fl
    roof["algorithmic_bytes_per_launch"] = by
    roof["traffic"] = recorded_traffic(dominant, args.config)

    F = sum(c[0] for c in costs.values())
    B = sum(c[1] for c in costs.values())
    t_roof = accounting.roofline_seconds(F, B, peaks["bf16_tflops"], peaks["hbm_gbs"])
    value = world * wl.T / (med_ms / 1e3)
    gemms = {}
    for k_ in GEMM_KERNELS:
        if k_ in per_kernel:
            r = kernel_roofline(k_, *costs[k_], per_kernel[k_], peaks)
            gemms[k_] = {"ms": round(per_kernel[k_], 4), "bound": r["bound"],
                         "achieved": round(r["achieved"], 1), "unit": r["unit"],
                         "frac": round(r["frac"], 3)}
    misses = [k_ for k_, g in gemms.items()
              if g["frac"] < (TARGET_TENSOR if g["bound"] == "tensor" else TARGET_HBM)]

    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": med_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{wl.name}: {wl.note}", "T": wl.T, "d": wl.d, "f": wl.f,
                   "E": wl.E, "k": wl.k, "align": wl.align, "backward": wl.backward,
                   "tau": inp.get("tau"), "seed": wl.seed,
                   "l2": ("L2 flushed between timed steps (a step moves less than four L2s)"
                          if flush else
                          "inputs larger than L2 (no flush): one step moves several GB"),
                   "graph": bool(args.graph),
                   "path": ("decode (one launch)" if decode else
                            "fused expert GEMMs (inference)" if fused else "general"),
                   "parallelism": f"replicas x{world}"},
        "timing": {"ms_per_step": "median of the timed steps (one event pair each)",
                   "ms_per_step_mean": span_ms / args.steps,
                   "ms_min": min(per_step), "ms_max": max(per_step)},
        "roofline": roof,
        "layer_roofline": {"flops": F, "bytes": B, "t_roof_ms": t_roof * 1e3,
                           "frac": t_roof * 1e3 / med_ms,
                           "peaks": f"bf16 {peaks['bf16_tflops']} TFLOP/s burst, "
                                    f"HBM {peaks['hbm_gbs']} GB/s, {peaks['source']}",
                           "tflops_achieved": F / (med_ms * 1e-3) / 1e12,
                           "E_active": shape.E_active},
        "gemms": gemms,
        "targets": {"tensor_bound_gemm_frac": TARGET_TENSOR, "hbm_bound_frac": TARGET_HBM,
                    "met": not misses, "missed": misses},
        "pairs_per_s": value * wl.k,
        "kernels_ms": {k_: round(v, 4) for k_, v in per_kernel.items()},
        "gpu_launches": launches,
        "clocks": clocks,
        "e2e": e2e,
    }
    if not args.no_side and not decode and not fused and args.config == DEFAULT_CONFIG:
        # the other workloads, each timed in this same run (their own clock record)
        del b
        torch.cuda.empty_cache()
        out["configs"] = {n: run_side(n, dev, local_rank, peaks, args.side_steps, 3)
                          for n in SIDE_CONFIGS}
        for n in DECODE_SIDE:
            out["configs"][n] = run_decode_side(n, dev, peaks, 5 * args.side_steps)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:   # the oracle beside N = 1 only
        tokens = min(args.cpu_tokens, wl.T)
        secs = oracle_sample(inp, wl, tokens)
        out["cpu_baseline"] = {"value": tokens / secs, "unit": UNIT, "cores": blas_threads(),
                               "kind": "oracle",
                               "sample": f"first {tokens} of {wl.T} tokens, all {wl.E} experts, "
                                         f"{'fwd+bwd' if wl.backward else 'fwd'}, float64 numpy",
                               "seconds": secs}
        one = oracle_single_core_tiny()
        if one is not None:
            out["cpu_baseline"]["tiny_single_core"] = one
    return out


def oracle_single_core_tiny():
    """The float64 oracle on the tiny workload (T = 256, d = 128, f = 256,
    E = 8, top-2), fwd+bwd, on one core: a child process whose BLAS is held
    to one thread by the environment. Returns its tokens/s record or None."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1")
    code = ("import sys, time; sys.path.insert(0, %r)\n"
            "import workloads\n"
            "from oracle import moe_oracle as mo\n"
            "wl = workloads.CONFIGS['tiny']; inp = workloads.generate(wl)\n"
            "def go():\n"
            "    fw = mo.forward(inp['x'], inp['w_router'], inp['bias'], inp['w_gate'], inp['w_up'],"
            " inp['w_down'], wl.k)\n"
            "    mo.backward(inp['x'], inp['w_router'], inp['bias'], inp['w_gate'], inp['w_up'],"
            " inp['w_down'], wl.k, inp['dy'], fwd=fw)\n"
            "go(); t0 = time.perf_counter(); n = 5\n"
            "for _ in range(n): go()\n"
            "print((time.perf_counter() - t0) / n)\n" % ROOT)
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                           timeout=300)
        secs = float(r.stdout.strip().splitlines()[-1])
    except Exception:
        return None
    return {"value": 256 / secs, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "tiny workload (T = 256, d = 128, f = 256, E = 8, top-2), fwd+bwd, "
                      "float64 numpy, BLAS on one thread, mean of 5 passes",
            "seconds": secs}


# ----------------------------------------------------------- reference --

def run_reference(args):
    import workloads
    wl = workloads.CONFIGS[args.config]
    inp = workloads.generate(wl, with_dy=wl.backward)
    tokens = min(args.ref_tokens, wl.T)
    for _ in range(args.warmup):
        oracle_sample(inp, wl, tokens)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample(inp, wl, tokens)
    secs = time.perf_counter() - t0
    value = tokens * args.steps / secs
    sample = (f"first {tokens} of {wl.T} tokens per step, all {wl.E} experts, "
              f"{'fwd+bwd' if wl.backward else 'fwd'}, float64 numpy")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{wl.name}: {wl.note}", "T": wl.T, "d": wl.d, "f": wl.f,
                   "E": wl.E, "k": wl.k, "align": wl.align, "backward": wl.backward},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    out = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
