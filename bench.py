"""Benchmark of the MoE layer (forward + backward) on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the whole layer over one batch of synthetic tokens:
router, schedule, dispatch, GEMM1+SwiGLU, GEMM2, combine, then the backward
(reverse combine, dgrad GEMMs with the SwiGLU backward, reverse dispatch,
router backward, weight-gradient GEMMs). The default workload is the largest
one, the ring workload: T=16384 tokens, H=7168, E=16 experts, k=8, F=2048,
MXFP8 operands, through a 256 MiB ring at the wave-rule minibatch
(workloads.py). The balanced, skewed and MXFP8 workloads are measured after it
and reported under "other_workloads" (--only-headline skips them).

Prints ONE JSON line (rank 0). `value` is whole-job tokens/s of fwd+bwd with
inputs resident in HBM; L2 is flushed (256 MiB write) between timed steps and
each step is timed with its own CUDA events on the launch stream. Under
torchrun every rank runs an independent replica (weak scaling; the layer has
no cross-GPU exchange) and the time is the max over ranks.

--impl reference times the CPU float64 oracle (the only other implementation
of this layer) on bounded token samples of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as WL  # noqa: E402

METRIC = "MoE layer tokens/s fwd & fwd+bwd on 1 GB300; grouped-GEMM % of TC peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def committed_traffic(name, workload):
    """DRAM bytes per launch of kernel `name` on `workload` from the committed ncu table, if the
    kernel sources are unchanged since the capture; else None."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("workload") != workload:
        return None
    csrc = os.path.join(ROOT, "mixture_experts_layer_sum_gb300", "csrc")
    for f, sha in d.get("sources_sha1", {}).items():
        if hashlib.sha1(open(os.path.join(csrc, f), "rb").read()).hexdigest() != sha:
            return None
    return d.get("traffic_bytes_per_launch", {}).get(name)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def max_over_ranks(values, device=None):
    """Per-entry maximum over every rank of the default process group (the slowest
    replica sets the job's time); the values themselves when running alone."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_tokens_per_s(world_size, tokens_per_rank, steps, ms):
    """Whole-job throughput: the tokens every replica processed over the slowest time."""
    return world_size * tokens_per_rank * steps / (ms * 1e-3)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ------------------------------------------------------------------ CPU oracle timing

def oracle_inputs(inp):
    from oracle import moe_oracle as O
    return {k: (O.bf16_to_f64(v) if k != "bias" and v is not None else v) for k, v in inp.items()}


def oracle_step(w, o, ntok, caches):
    """fwd+bwd of the oracle on the first ntok tokens (all weights). `caches` keep the weight
    copies between steps: like the GPU's weight quantisation (once per weight update), the
    oracle's is made by the first, untimed, call and left out of the timed steps."""
    from oracle import moe_oracle as O
    x, dout = o["x"][:ntok], o["dout"][:ntok]
    t0 = time.perf_counter()
    f = O.forward(x, o["Wr"], o["bias"], o["W1"], o["W3"], o["W2"], w.k, precision=w.precision,
                  weight_cache=caches[0])
    O.backward(f, dout, x, o["Wr"], o["W1"], o["W3"], o["W2"], weight_cache=caches[1])
    return time.perf_counter() - t0


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(w, inp, target_s=15.0):
    o = oracle_inputs(inp)
    caches = ({}, {})
    oracle_step(w, o, 32, caches)                 # weight copies (W0), untimed
    t_small = oracle_step(w, o, 128, caches)
    per_tok = t_small / 128
    ntok = int(min(w.T, max(128, target_s / max(per_tok, 1e-9))))
    ntok = max(128, ntok // 128 * 128)
    t = oracle_step(w, o, ntok, caches)
    # a workload smaller than the time budget is passed over again until about 10 s of CPU work
    passes = 1
    while t < 10.0 and passes < 16:
        t += oracle_step(w, o, ntok, caches)
        passes += 1
    return {"value": ntok * passes / t, "unit": "tokens/s", "cores": cpu_threads(), "kind": "oracle",
            "sample": f"{passes} x fwd+bwd of the first {ntok} of {w.T} tokens of {w.name}, all weights "
                      f"(their {w.precision} copies made once, untimed, as the GPU's W0), float64 numpy "
                      f"(BLAS threads = host cores), {t:.1f} s"}


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    inp = WL.make_inputs(w)
    o = oracle_inputs(inp)
    ntok = 128 if w.precision == "mxfp8" else 256
    caches = ({}, {})
    for _ in range(args.warmup):
        oracle_step(w, o, ntok, caches)
    times = [oracle_step(w, o, ntok, caches) for _ in range(args.steps)]
    tot = sum(times)
    value = ntok * args.steps / tot
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "H": w.H, "F": w.F, "E": w.E, "k": w.k,
                   "precision": w.precision, "sample_tokens_per_step": ntok},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_threads(), "kind": "oracle",
                         "sample": f"fwd+bwd of the first {ntok} of {w.T} tokens per step, all weights "
                                   f"(weight copies made in the warm-up steps, as the GPU's W0)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm

class NvmlClockSampler:
    """Reads SM clock and clock-event reasons through NVML every 10 ms on a
    background thread (read-only queries; no setting is changed)."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, pci_bus_id):
        import ctypes
        import threading
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        self.c = ctypes
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML handle for " + pci_bus_id)
        mx = ctypes.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
        self.max_mhz = mx.value
        self.fn_reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.samples = []
        self.stop_evt = threading.Event()
        self.t = threading.Thread(target=self.run, daemon=True)
        self.t.start()

    def run(self):
        c = self.c
        while not self.stop_evt.is_set():
            mhz, rs = c.c_uint(), c.c_ulonglong()
            self.lib.nvmlDeviceGetClockInfo(self.h, 1, c.byref(mhz))
            self.fn_reasons(self.h, c.byref(rs))
            self.samples.append((mhz.value, rs.value))
            self.stop_evt.wait(0.01)

    def stop(self):
        self.stop_evt.set()
        self.t.join()
        self.lib.nvmlShutdown()
        sm = [m for m, _ in self.samples]
        reasons = sorted({name for _, r in self.samples for bit, name in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(sm), "source": "NVML, 10 ms period, during the timed loops"}


def start_clocks(local_rank):
    f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
    try:
        p = subprocess.Popen(["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                              "-lms", "200", "-i", str(local_rank)], stdout=f, stderr=subprocess.DEVNULL)
    except Exception:
        p = None
    return p, f.name


def stop_clocks(p, path):
    if p is None:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
    p.terminate()
    try:
        p.wait(5)
    except Exception:
        p.kill()
    rows = []
    for line in open(path):
        parts = [s.strip() for s in line.split(",")]
        if len(parts) >= 9:
            rows.append(parts)
    os.unlink(path)
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
    sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
    smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
            "reasons": reasons, "samples": len(rows)}


def kernel_bytes(w, name, combine_tokens=None):
    """Algorithmic HBM bytes per step of the memory-bound kernels. combine_tokens: tokens the
    combine kernel itself handles (the persistent forward combines every macrobatch but the last
    inside its own launch); None = all T."""
    T, H, F, R, E, k = w.T, w.H, w.F, w.R, w.E, w.k
    qh, qf = R * H * 33 // 32, R * F * 33 // 32   # one MXFP8 copy of R rows (codes + scales)
    if name == "combine" and combine_tokens is not None:
        T, R = combine_tokens, combine_tokens * k
    return {"decode_ffn": 3 * E * H * F * 2,   # every expert's weights streamed once (few tokens)
            "dispatch": T * H * 2 + R * H * 2, "dispatch_replay": T * H * 2 + R * H * 2,
            "dispatch_mxfp8": T * H * 2 + qh,
            "reverse_combine": T * H * 2 + R * H * 2, "combine": R * H * 2 + T * H * 2 + R * 8,
            "router_topk": T * H * 2 + T * E * 4 + T * k * 8,
            "reverse_dispatch": R * H * 2 + T * H * 2 + T * E * 4,
            "router_wgrad": T * H * 2 + T * E * 4,
            # MXFP8 backward: dout gathered once into dY along H and along the tokens; x along
            # the tokens; h.w, da, db (bf16 rows) along the tokens
            "quantize_dy": T * H * 2 + 2 * qh, "quantize_x_tokens": T * H * 2 + qh,
            "quantize_hw_tokens": R * F * 2 + qf, "quantize_da_tokens": R * F * 2 + qf,
            "quantize_db_tokens": R * F * 2 + qf}.get(name)


def gemm_flops(w, name):
    """GEMM flops per step; the persistent forward and the decode kernel run both expert GEMMs."""
    R, H, F = w.R, w.H, w.F
    return {"forward_persistent": 6 * R * H * F, "decode_ffn": 6 * R * H * F,
            "grouped_gemm_fwd1_swiglu": 4 * R * H * F, "grouped_gemm_fwd2": 2 * R * H * F,
            "grouped_gemm_bwd2_swiglu": 2 * R * H * F, "grouped_gemm_bwd1": 4 * R * H * F,
            "grouped_gemm_wgrad2": 2 * R * H * F, "grouped_gemm_wgrad13": 4 * R * H * F}.get(name)


def gemm_bytes(w, name):
    """Algorithmic HBM bytes per step of each grouped GEMM: operands read once, outputs written
    once (R = routed rows; the ring round trip of the dispatched rows is not counted). bf16
    operands; MXFP8 operands carry H*33/32 (or F*33/32) bytes per row instead of 2*H."""
    T, H, F, E, R = w.T, w.H, w.F, w.E, w.R
    W = E * H * F * 2   # one bf16 weight matrix of all experts
    return {"forward_persistent": T * H * 2 + 3 * W + 3 * R * F * 2 + R * H * 2,   # GEMM1 + GEMM2 operands
            "grouped_gemm_fwd1_swiglu": T * H * 2 + 2 * W + 3 * R * F * 2,
            "grouped_gemm_fwd2": R * F * 2 + W + R * H * 2,
            "grouped_gemm_bwd2_swiglu": R * H * 2 + W + 2 * R * F * 2 + 3 * R * F * 2,
            "grouped_gemm_bwd1": 2 * R * F * 2 + 2 * W + R * H * 2,
            "grouped_gemm_wgrad2": R * F * 2 + R * H * 2 + E * F * H * 4,
            "grouped_gemm_wgrad13": R * H * 2 + 2 * R * F * 2 + 2 * E * H * F * 4}.get(name)


GEMMS = ["grouped_gemm_fwd1_swiglu", "grouped_gemm_fwd2", "grouped_gemm_bwd2_swiglu", "grouped_gemm_bwd1",
         "grouped_gemm_wgrad2", "grouped_gemm_wgrad13"]
GEMM_KERNELS = ("grouped_gemm", "forward_persistent")   # kernels whose time is expert-GEMM time


def tensor_peak(w, peaks, peak_src, loop_s):
    """Dense tensor peak for GEMMs timed inside a loop of loop_s seconds: the burst bf16 figure
    for a loop shorter than a second, the sustained (seconds-long, power-capped) one otherwise;
    MXFP8 takes 2x the bf16 figure (the nominal fp8 / bf16 ratio, 4.5 vs 2.25 PFLOP/s)."""
    burst = loop_s < 1.0 or "bf16_tflops_sustained" not in peaks
    tf = peaks["bf16_tflops"] if burst else peaks["bf16_tflops_sustained"]
    src = f"{peak_src} {'bf16_tflops (burst' if burst else 'bf16_tflops_sustained (sustained'}; timed loop {loop_s:.2f} s)"
    if w.precision == "mxfp8":
        tf, src = 2 * tf, src + " x 2 (nominal fp8/bf16 ratio)"
    return tf, src


def layer_roofline(w, tf, hbm, step_ms):
    """Layer roofline time: the GEMMs' flops at the tensor peak plus the memory-bound stages'
    algorithmic bytes at the HBM copy bandwidth, run back to back; frac = roofline / measured."""
    mem = ["dispatch", "combine", "router_topk", "reverse_combine", "reverse_dispatch", "router_wgrad"]
    if w.precision == "mxfp8":
        mem = ["dispatch_mxfp8", "combine", "router_topk", "quantize_dy", "quantize_x_tokens",
               "quantize_hw_tokens", "quantize_da_tokens", "quantize_db_tokens", "reverse_dispatch",
               "router_wgrad"]
    t_gemm = sum(gemm_flops(w, n) for n in GEMMS) / (tf * 1e12)
    t_mem = sum(kernel_bytes(w, n) for n in mem) / (hbm * 1e9)
    t = (t_gemm + t_mem) * 1e3
    return {"time_ms": t, "gemm_ms": t_gemm * 1e3, "hbm_ms": t_mem * 1e3, "frac": t / step_ms,
            "note": "sum of GEMM flops / peak tensor rate and memory-stage algorithmic bytes / HBM copy bandwidth"}


def combine_tokens_of(w, plan):
    """Tokens the combine kernel handles with the persistent forward: the last macrobatch's."""
    nM, Mb = plan
    return w.T - (nM - 1) * Mb


def rate_kernels(w, kernels, steps, prof_ms, peaks, peak_src, loop_s, combine_tokens=None):
    """Per-kernel rates of a profiled run, the dominant kernel's roofline and the grouped GEMMs'
    fraction of the tensor peak. kernels: [(name, launches, total ms)] over `steps` steps.
    combine_tokens: see kernel_bytes."""
    tf, tf_src = tensor_peak(w, peaks, peak_src, loop_s)
    hbm = peaks.get("hbm_gbs")
    kt = sorted(kernels, key=lambda r: -r[2])
    rows = []
    for nm, n_, ms_ in kt:
        row = {"name": nm, "launches": n_, "ms_per_step": ms_ / steps, "share": ms_ / prof_ms}
        if gemm_flops(w, nm) and nm != "decode_ffn":
            row["tflops"] = gemm_flops(w, nm) * steps / (ms_ * 1e-3) / 1e12
            row["frac_of_tensor_peak"] = row["tflops"] / tf
        if kernel_bytes(w, nm) and hbm:
            row["gbs"] = kernel_bytes(w, nm, combine_tokens) * steps / (ms_ * 1e-3) / 1e9
            row["frac_of_hbm"] = row["gbs"] / hbm
        rows.append(row)
    # dominant kernel: the largest share of the profiled step; a kernel may launch several
    # times per step (once per macrobatch), so per-launch work = per-step work / launches per step
    name, n, ms = kt[0]
    per_launch_ms = ms / n
    per_step = n / steps
    roof = None
    if gemm_flops(w, name) and name != "decode_ffn":
        fl = gemm_flops(w, name) / per_step
        ach = fl / (per_launch_ms * 1e-3) / 1e12
        roof = {"kernel": name, "bound": "tensor", "achieved": ach, "peak": tf, "unit": "TFLOP/s",
                "frac": ach / tf, "traffic": committed_traffic(name, w.name), "algorithmic_per_launch": fl,
                "peak_source": tf_src}
        if w.precision == "bf16" and hbm and gemm_bytes(w, name) is not None:
            gb = gemm_bytes(w, name) / per_step
            roof["hbm_rating"] = {"algorithmic_bytes_per_launch": gb,
                                  "achieved_gbs": gb / (per_launch_ms * 1e-3) / 1e9,
                                  "frac_of_hbm": gb / (per_launch_ms * 1e-3) / 1e9 / hbm}
    elif kernel_bytes(w, name) is not None and hbm:
        gb = kernel_bytes(w, name, combine_tokens) / per_step
        ach = gb / (per_launch_ms * 1e-3) / 1e9
        roof = {"kernel": name, "bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                "frac": ach / hbm, "traffic": committed_traffic(name, w.name), "algorithmic_per_launch": gb,
                "peak_source": f"{peak_src} hbm_gbs (copy bandwidth)"}
    gemm_ms = sum(ms_ for nm, _, ms_ in kernels if nm.startswith(GEMM_KERNELS))
    gemm_fl = sum(gemm_flops(w, nm) * steps for nm, _, _ in kernels if nm.startswith(GEMM_KERNELS))
    gg = None
    if gemm_ms:
        t = gemm_fl / (gemm_ms * 1e-3) / 1e12
        gg = {"tflops": t, "frac_of_peak": t / tf, "peak": tf, "peak_source": tf_src,
              "share_of_step": gemm_ms / prof_ms}
    return rows, roof, gg, tf


class Gpu:
    """The device-side pieces of one measured workload: inputs in HBM, the layer, its output buffers."""

    def __init__(self, w, dev, rank, M, MoeLayer, torch):
        self.w, self.dev, self.torch = w, dev, torch
        self.inp = WL.make_inputs(w.with_(seed=w.seed + rank))
        self.d = {k: self.to_dev(v) for k, v in self.inp.items() if k != "bias" and v is not None}
        self.bias = torch.from_numpy(self.inp["bias"]).to(dev) if self.inp["bias"] is not None else None
        self.layer = MoeLayer(w.T, w.H, w.F, w.E, w.k, w.precision, device=dev, ring_bytes=w.ring_bytes)
        self.stream = torch.cuda.Stream(device=dev)
        bf, f32 = torch.bfloat16, torch.float32
        self.out = torch.empty(w.T, w.H, dtype=bf, device=dev)
        self.ids = torch.empty(w.T, w.k, dtype=torch.int32, device=dev)
        self.wts = torch.empty(w.T, w.k, dtype=f32, device=dev)
        self.dx = torch.empty(w.T, w.H, dtype=bf, device=dev)
        self.dWr = torch.empty(w.H, w.E, dtype=f32, device=dev)
        self.dW1 = torch.empty(w.E, w.H, w.F, dtype=f32, device=dev)
        self.dW3 = torch.empty_like(self.dW1)
        self.dW2 = torch.empty(w.E, w.F, w.H, dtype=f32, device=dev)
        if w.precision in ("mxfp8", "nvfp4"):
            self.quantize()

    def to_dev(self, a):
        t = self.torch
        return t.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(t.bfloat16).to(self.dev)

    def quantize(self):
        d = self.d
        self.layer.quantize_weights(d["W1"], d["W3"], d["W2"], stream=self.stream)

    def fwd(self, layer=None, x=None, out=None):
        d = self.d
        (layer or self.layer).forward(d["x"] if x is None else x, d["Wr"], self.bias, d["W1"], d["W3"], d["W2"],
                                      self.out if out is None else out, self.ids, self.wts, stream=self.stream)

    def bwd(self, layer=None, x=None, dout=None, dx=None):
        d = self.d
        (layer or self.layer).backward(d["dout"] if dout is None else dout, d["x"] if x is None else x, d["Wr"],
                                       d["W1"], d["W3"], d["W2"], self.dx if dx is None else dx, self.dWr,
                                       self.dW1, self.dW3, self.dW2, stream=self.stream)

    def step(self, layer=None):
        self.fwd(layer)
        self.bwd(layer)


def timed(g, flush, fn, k):
    torch = g.torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(k)]
    with torch.cuda.stream(g.stream):
        for a, b in evs:
            flush.fill_(1)                # evict L2 between timed steps (untimed)
            a.record(g.stream)
            fn()
            b.record(g.stream)
    g.stream.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs)


def e2e_ms(g, steps):
    """End to end through the public API with host buffers: every step copies its x and dout
    from pinned host memory to the device and reads its out and dx back. The copies run on their
    own streams and the device buffers are double-buffered, so step i+1's inputs arrive while
    step i computes, out leaves during the backward and dx during the next step (the usual
    input/output pipeline of a training or serving loop). The timed region runs from the first
    host-to-device copy to the end of the last device-to-host copy."""
    torch, dev, w, d = g.torch, g.dev, g.w, g.d
    hx = torch.empty(w.T, w.H, dtype=torch.bfloat16, pin_memory=True)
    hd = torch.empty_like(hx, pin_memory=True)
    hx.copy_(d["x"].cpu())
    hd.copy_(d["dout"].cpu())
    NB = 2
    hout = [torch.empty_like(hx, pin_memory=True) for _ in range(NB)]
    hdx = [torch.empty_like(hx, pin_memory=True) for _ in range(NB)]
    xin = [torch.empty_like(d["x"]) for _ in range(NB)]
    din = [torch.empty_like(d["dout"]) for _ in range(NB)]
    outb = [torch.empty_like(g.out) for _ in range(NB)]
    dxb = [torch.empty_like(g.dx) for _ in range(NB)]
    h2d = torch.cuda.Stream(device=dev)
    d2h = torch.cuda.Stream(device=dev)
    stream = g.stream

    def run(k):
        ev = lambda: torch.cuda.Event()
        used = [None] * NB      # compute done with slot b (inputs free)
        drained = [None] * NB   # outputs of slot b read back (output buffers free)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(h2d)
        for i in range(k):
            b = i % NB
            with torch.cuda.stream(h2d):
                if used[b] is not None:
                    h2d.wait_event(used[b])
                xin[b].copy_(hx, non_blocking=True)
                ex = ev(); ex.record(h2d)
                din[b].copy_(hd, non_blocking=True)
                ed = ev(); ed.record(h2d)
            stream.wait_event(ex)
            if drained[b] is not None:
                stream.wait_event(drained[b])
            g.fwd(x=xin[b], out=outb[b])
            ef = ev(); ef.record(stream)
            with torch.cuda.stream(d2h):
                d2h.wait_event(ef)
                hout[b].copy_(outb[b], non_blocking=True)
            stream.wait_event(ed)
            g.bwd(x=xin[b], dout=din[b], dx=dxb[b])
            eb = ev(); eb.record(stream)
            used[b] = eb
            with torch.cuda.stream(d2h):
                d2h.wait_event(eb)
                hdx[b].copy_(dxb[b], non_blocking=True)
                dr = ev(); dr.record(d2h)
            drained[b] = dr
        d2h.wait_event(t0)
        t1.record(d2h)
        torch.cuda.synchronize(dev)
        return t0.elapsed_time(t1)

    run(2)
    return run(steps)


def decode_entries(args, dev, rank, M, MoeLayer, torch, flush):
    """Decode-sized forward (64 tokens of the balanced shape), bf16 and NVFP4 weights: every
    expert's weights stream once, so the floor is their bytes at the HBM copy bandwidth."""
    out = []
    for prec in ("bf16", "nvfp4"):
        wd = WL.BALANCED.with_(T=64, precision=prec, name=f"{WL.BALANCED.name}@T64/{prec}")
        gd = Gpu(wd, dev, rank, M, MoeLayer, torch)
        with torch.cuda.stream(gd.stream):
            for _ in range(args.warmup):
                gd.fwd()
        t_fwd = timed(gd, flush, gd.fwd, args.steps)
        M.moe_profile_begin()
        timed(gd, flush, gd.fwd, args.steps)
        kern = M.moe_profile_end()
        gd.layer.status(gd.stream)
        hbm_d = load_peaks()[0]["hbm_gbs"]
        wbytes = kernel_bytes(wd, "decode_ffn") * (1.0 if prec == "bf16" else (0.5 + 1 / 16) / 2)
        floor_us = wbytes / (hbm_d * 1e9) * 1e6
        dk = {nm: ms_ / args.steps * 1e3 for nm, _, ms_ in kern}
        kname = "decode_ffn" if prec == "bf16" else "decode_ffn_nvfp4"
        out.append({
            "workload": wd.name, "precision": prec, "T": wd.T, "H": wd.H, "F": wd.F, "E": wd.E, "k": wd.k,
            "fwd": {"value": wd.T * args.steps / (t_fwd * 1e-3), "unit": "tokens/s",
                    "us_per_step": t_fwd / args.steps * 1e3},
            "weight_bytes": wbytes, "weight_stream_floor_us": floor_us,
            "fwd_over_floor": t_fwd / args.steps * 1e3 / floor_us,
            kname: {"us": dk.get(kname), "frac_of_hbm": floor_us / dk[kname] if dk.get(kname) else None},
            "kernels_us": dk})
        del gd
        torch.cuda.empty_cache()
    return out


def run_decode_only(args):
    """Only the decode entries (one GPU): a short command for profiling the decode kernels."""
    import torch
    torch.cuda.set_device(0)
    from mixture_experts_layer_sum_gb300 import build_ext
    build_ext.build()
    import mixture_experts_layer_sum_gb300.moe as M
    from mixture_experts_layer_sum_gb300.layer import MoeLayer
    dev = torch.device("cuda", 0)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    print(json.dumps({"decode": decode_entries(args, dev, 0, M, MoeLayer, torch, flush)}))


def run_ours(args, w):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    from mixture_experts_layer_sum_gb300 import build_ext
    build_ext.build()
    import mixture_experts_layer_sum_gb300.moe as M
    from mixture_experts_layer_sum_gb300.layer import MoeLayer
    dev = torch.device("cuda", local)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    g = Gpu(w, dev, rank, M, MoeLayer, torch)
    plan = (g.layer.plan.num_macrobatches, g.layer.plan.macrobatch_tokens, g.layer.plan.minibatch_rows)

    def barrier():
        torch.cuda.synchronize(dev)
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    props = torch.cuda.get_device_properties(dev)
    try:
        bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
        sampler = NvmlClockSampler(bus)
        clk_p = clk_path = None
    except Exception:
        sampler = None
        clk_p, clk_path = start_clocks(local)
    with torch.cuda.stream(g.stream):
        for _ in range(args.warmup):
            g.step()
    g.layer.status(g.stream)
    barrier()
    total_ms = timed(g, flush, g.step, args.steps)
    w0_ms = None
    if w.precision == "mxfp8":
        # weight quantisation runs once per weight update, outside the step; timed on its own
        w0_ms = timed(g, flush, g.quantize, args.steps)
        w0_ms, = max_over_ranks([w0_ms], device=dev)   # every rank has the same precision
    barrier()
    fwd_ms = timed(g, flush, g.fwd, args.steps)
    g.layer.status(g.stream)
    total_ms, fwd_ms = max_over_ranks([total_ms, fwd_ms], device=dev)

    # per-kernel breakdown: the same steps with events around every launch
    M.moe_profile_begin()
    prof_ms = timed(g, flush, g.step, args.steps)
    kernels = M.moe_profile_end()
    launches = sum(n for _, n, _ in kernels)

    e2e = e2e_ms(g, args.steps)
    e2e, = max_over_ranks([e2e], device=dev)
    g.layer.status(g.stream)

    sweep = None
    if args.minibatch_sweep and w.minibatch_rows:
        sweep = []
        for mbr in w.minibatch_rows:
            lay = MoeLayer(w.T, w.H, w.F, w.E, w.k, w.precision, device=dev, ring_bytes=w.ring_bytes,
                           minibatch_rows=mbr)
            if w.precision == "mxfp8":
                lay.quantize_weights(g.d["W1"], g.d["W3"], g.d["W2"], stream=g.stream)
            with torch.cuda.stream(g.stream):
                for _ in range(2):
                    g.step(lay)
            k = max(2, args.steps // 4)
            fm = timed(g, flush, lambda: g.fwd(lay), k)
            sm = timed(g, flush, lambda: g.step(lay), k)
            lay.status(g.stream)
            sweep.append({"minibatch_rows": mbr, "fwd_ms": fm / k, "fwd_bwd_ms": sm / k,
                          "macrobatches": lay.plan.num_macrobatches, "macrobatch_tokens": lay.plan.macrobatch_tokens})
            del lay
            torch.cuda.empty_cache()

    # the other workloads (single GPU): the same step, its forward and its per-kernel rates
    others = []
    if ws == 1 and not args.only_headline:
        headline_inp = g.inp
        del g
        torch.cuda.empty_cache()
        for name in OTHER_WORKLOADS:
            if name == w.name:
                continue
            wo = WL.WORKLOADS[name]
            go = Gpu(wo, dev, rank, M, MoeLayer, torch)
            with torch.cuda.stream(go.stream):
                for _ in range(args.warmup):
                    go.step()
            go.layer.status(go.stream)
            t_step = timed(go, flush, go.step, args.steps)
            t_fwd = timed(go, flush, go.fwd, args.steps)
            M.moe_profile_begin()
            t_prof = timed(go, flush, go.step, args.steps)
            kern = M.moe_profile_end()
            go.layer.status(go.stream)
            pl = go.layer.plan
            rows, roof_o, gg_o, tf_o = rate_kernels(wo, kern, args.steps, t_prof, *load_peaks(), t_step * 1e-3,
                                                    combine_tokens_of(wo, (pl.num_macrobatches, pl.macrobatch_tokens)))
            others.append({
                "workload": wo.name, "precision": wo.precision, "T": wo.T, "H": wo.H, "F": wo.F, "E": wo.E,
                "k": wo.k, "fwd_bwd": {"value": wo.T * args.steps / (t_step * 1e-3), "unit": "tokens/s",
                                       "ms_per_step": t_step / args.steps},
                "fwd": {"value": wo.T * args.steps / (t_fwd * 1e-3), "unit": "tokens/s",
                        "ms_per_step": t_fwd / args.steps},
                "grouped_gemm": gg_o, "roofline": roof_o,
                "layer_roofline": layer_roofline(wo, tf_o, load_peaks()[0]["hbm_gbs"], t_step / args.steps),
                "gpu_launches": sum(n for _, n, _ in kern),
                "kernels": [{k_: r[k_] for k_ in ("name", "launches", "ms_per_step", "share", "tflops",
                                                  "frac_of_tensor_peak", "gbs", "frac_of_hbm") if k_ in r}
                            for r in rows]})
            del go
            torch.cuda.empty_cache()
        others += decode_entries(args, dev, rank, M, MoeLayer, torch, flush)
        inp = headline_inp
    else:
        inp = g.inp
    clocks = sampler.stop() if sampler is not None else stop_clocks(clk_p, clk_path)

    if rank != 0:
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
            dist.destroy_process_group()
        return
    peaks, peak_src = load_peaks()
    rows, roof, gg, tf = rate_kernels(w, kernels, args.steps, prof_ms, peaks, peak_src, total_ms * 1e-3,
                                      combine_tokens_of(w, plan[:2]))
    value = job_tokens_per_s(ws, w.T, args.steps, total_ms)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.precision == "bf16" else "mxfp8",
        "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "H": w.H, "F": w.F, "E": w.E, "k": w.k,
                   "precision": w.precision, "step": "forward+backward",
                   "ring_bytes": w.ring_bytes or None, "macrobatches": plan[0], "macrobatch_tokens": plan[1],
                   "minibatch_rows": plan[2],
                   "l2": "flushed (256 MiB write) between timed steps",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "w0": None if w0_ms is None else {
            "ms": w0_ms / args.steps,
            "fwd_bwd_value_incl_w0": job_tokens_per_s(ws, w.T, args.steps, total_ms + w0_ms),
            "note": "MXFP8 weight copies, once per weight update; excluded from value"},
        "fwd": {"value": job_tokens_per_s(ws, w.T, args.steps, fwd_ms), "unit": "tokens/s",
                "ms_per_step": fwd_ms / args.steps},
        "roofline": roof,
        "grouped_gemm": gg,
        "kernels": rows,
        "layer_roofline": layer_roofline(w, tf, peaks["hbm_gbs"], total_ms / args.steps),
        "gpu_launches": launches,
        "e2e": {"value": job_tokens_per_s(ws, w.T, args.steps, e2e), "unit": "tokens/s",
                "h2d_bytes_per_step": 2 * w.T * w.H * 2, "d2h_bytes_per_step": 2 * w.T * w.H * 2,
                "pipelined": "copy streams, double-buffered inputs/outputs; no L2 flush (weights exceed L2)"},
        "clocks": clocks,
    }
    if sweep is not None:
        line["minibatch_sweep"] = sweep
    if others:
        line["other_workloads"] = others
    if ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, inp)
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


OTHER_WORKLOADS = [WL.BALANCED.name, WL.SKEWED.name, WL.MXFP8.name]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=WL.RING.name, choices=sorted(WL.WORKLOADS))
    ap.add_argument("--only-headline", action="store_true", help="skip the other workloads")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=0, help="override T (small cases for ncu captures)")
    ap.add_argument("--experts", type=int, default=0, help="override E, keeping k <= E (small cases for ncu captures)")
    ap.add_argument("--decode-only", action="store_true",
                    help="time only the 64-token decode forward (bf16 and NVFP4 weights) and print it")
    ap.add_argument("--minibatch-sweep", action="store_true",
                    help="also time fwd and fwd+bwd for each minibatch size of the workload (ring workload)")
    args = ap.parse_args()
    assert args.warmup >= 3 or args.impl == "reference" or args.steps < 3, "need >= 3 warm-up steps"
    w = WL.WORKLOADS[args.workload]
    if args.tokens:
        w = w.with_(T=args.tokens, name=f"{w.name}@T{args.tokens}")
    if args.experts:
        w = w.with_(E=args.experts, k=min(w.k, args.experts), name=f"{w.name}@E{args.experts}")
    if args.decode_only:
        run_decode_only(args)
    elif args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
