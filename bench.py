"""Benchmark of the MoE layer (forward + backward) on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the whole layer over one batch of synthetic tokens:
router, schedule, dispatch, GEMM1+SwiGLU, GEMM2, combine, then the backward
(reverse combine, dgrad GEMMs with the SwiGLU backward, reverse dispatch,
router backward, weight-gradient GEMMs). The default workload is the balanced
BF16 shape T=4096, H=2048, E=32, k=4, F=1024 (workloads.py).

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


def committed_traffic(name):
    """DRAM bytes per launch of `name` from the committed ncu table, if the
    kernel sources are unchanged since the capture; else None."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
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

def oracle_step(w, inp, ntok):
    """fwd+bwd of the oracle on the first ntok tokens (all weights)."""
    from oracle import moe_oracle as O
    o = {k: (O.bf16_to_f64(v) if k != "bias" and v is not None else v) for k, v in inp.items()}
    x, dout = o["x"][:ntok], o["dout"][:ntok]
    t0 = time.perf_counter()
    f = O.forward(x, o["Wr"], o["bias"], o["W1"], o["W3"], o["W2"], w.k, precision=w.precision)
    O.backward(f, dout, x, o["Wr"], o["W1"], o["W3"], o["W2"])
    return time.perf_counter() - t0


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(w, inp, target_s=15.0):
    t_small = oracle_step(w, inp, 256)
    per_tok = t_small / 256
    ntok = int(min(w.T, max(256, target_s / max(per_tok, 1e-9))))
    ntok = max(256, ntok // 256 * 256)
    t = oracle_step(w, inp, ntok)
    # a workload smaller than the time budget is passed over again until about 10 s of CPU work
    passes = 1
    while t < 10.0 and passes < 16:
        t += oracle_step(w, inp, ntok)
        passes += 1
    return {"value": ntok * passes / t, "unit": "tokens/s", "cores": cpu_threads(), "kind": "oracle",
            "sample": f"{passes} x fwd+bwd of the first {ntok} of {w.T} tokens of {w.name}, all weights, "
                      f"float64 numpy (BLAS threads = host cores), {t:.1f} s"}


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    inp = WL.make_inputs(w)
    ntok = 256
    for _ in range(args.warmup):
        oracle_step(w, inp, ntok)
    times = [oracle_step(w, inp, ntok) for _ in range(args.steps)]
    tot = sum(times)
    value = ntok * args.steps / tot
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "H": w.H, "F": w.F, "E": w.E, "k": w.k,
                   "precision": w.precision, "sample_tokens_per_step": ntok},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_threads(), "kind": "oracle",
                         "sample": f"fwd+bwd of the first {ntok} of {w.T} tokens per step, all weights"},
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


def kernel_bytes(w, name):
    """Algorithmic HBM bytes per step of the memory-bound kernels."""
    T, H, F, R, E, k = w.T, w.H, w.F, w.R, w.E, w.k
    qh, qf = R * H * 33 // 32, R * F * 33 // 32   # one MXFP8 copy of R rows (codes + scales)
    return {"dispatch": T * H * 2 + R * H * 2, "dispatch_replay": T * H * 2 + R * H * 2,
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
    R, H, F = w.R, w.H, w.F
    return {"grouped_gemm_fwd1_swiglu": 4 * R * H * F, "grouped_gemm_fwd2": 2 * R * H * F,
            "grouped_gemm_bwd2_swiglu": 2 * R * H * F, "grouped_gemm_bwd1": 4 * R * H * F,
            "grouped_gemm_wgrad2": 2 * R * H * F, "grouped_gemm_wgrad13": 4 * R * H * F}.get(name)


def gemm_bytes(w, name):
    """Algorithmic HBM bytes per step of each grouped GEMM: operands read once, outputs written
    once (R = routed rows; the ring round trip of the dispatched rows is not counted)."""
    T, H, F, E, R = w.T, w.H, w.F, w.E, w.R
    W = E * H * F * 2   # one bf16 weight matrix of all experts
    return {"grouped_gemm_fwd1_swiglu": T * H * 2 + 2 * W + 3 * R * F * 2,
            "grouped_gemm_fwd2": R * F * 2 + W + R * H * 2,
            "grouped_gemm_bwd2_swiglu": R * H * 2 + W + 2 * R * F * 2 + 3 * R * F * 2,
            "grouped_gemm_bwd1": 2 * R * F * 2 + 2 * W + R * H * 2,
            "grouped_gemm_wgrad2": R * F * 2 + R * H * 2 + E * F * H * 4,
            "grouped_gemm_wgrad13": R * H * 2 + 2 * R * F * 2 + 2 * E * H * F * 4}.get(name)


def layer_roofline(w, peaks, step_ms):
    """Layer roofline time: the GEMMs' flops at the tensor peak plus the memory-bound stages'
    algorithmic bytes at the HBM copy bandwidth, run back to back; frac = roofline / measured."""
    tf = peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops"))
    hbm = peaks.get("hbm_gbs")
    if not tf or not hbm:
        return None
    if w.precision == "mxfp8":
        tf = 2 * tf
    gemm = ["grouped_gemm_fwd1_swiglu", "grouped_gemm_fwd2", "grouped_gemm_bwd2_swiglu", "grouped_gemm_bwd1",
            "grouped_gemm_wgrad2", "grouped_gemm_wgrad13"]
    mem = ["dispatch", "combine", "router_topk", "reverse_combine", "reverse_dispatch", "router_wgrad"]
    if w.precision == "mxfp8":
        mem = ["dispatch_mxfp8", "combine", "router_topk", "quantize_dy", "quantize_x_tokens",
               "quantize_hw_tokens", "quantize_da_tokens", "quantize_db_tokens", "reverse_dispatch",
               "router_wgrad"]
    t_gemm = sum(gemm_flops(w, n) for n in gemm) / (tf * 1e12)
    t_mem = sum(kernel_bytes(w, n) for n in mem) / (hbm * 1e9)
    t = (t_gemm + t_mem) * 1e3
    return {"time_ms": t, "gemm_ms": t_gemm * 1e3, "hbm_ms": t_mem * 1e3, "frac": t / step_ms,
            "note": "sum of GEMM flops / peak tensor rate and memory-stage algorithmic bytes / HBM copy bandwidth"}


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

    inp = WL.make_inputs(w.with_(seed=w.seed + rank))
    dev = torch.device("cuda", local)

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    d = {k: to_dev(v) for k, v in inp.items() if k != "bias" and v is not None}
    bias = torch.from_numpy(inp["bias"]).to(dev) if inp["bias"] is not None else None
    layer = MoeLayer(w.T, w.H, w.F, w.E, w.k, w.precision, device=dev, ring_bytes=w.ring_bytes)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = torch.empty(w.T, w.H, dtype=torch.bfloat16, device=dev)
    ids = torch.empty(w.T, w.k, dtype=torch.int32, device=dev)
    wts = torch.empty(w.T, w.k, dtype=torch.float32, device=dev)
    dx = torch.empty(w.T, w.H, dtype=torch.bfloat16, device=dev)
    dWr = torch.empty(w.H, w.E, dtype=torch.float32, device=dev)
    dW1 = torch.empty(w.E, w.H, w.F, dtype=torch.float32, device=dev)
    dW3 = torch.empty_like(dW1)
    dW2 = torch.empty(w.E, w.F, w.H, dtype=torch.float32, device=dev)

    if w.precision == "mxfp8":
        layer.quantize_weights(d["W1"], d["W3"], d["W2"], stream=stream)

    def fwd():
        layer.forward(d["x"], d["Wr"], bias, d["W1"], d["W3"], d["W2"], out, ids, wts, stream=stream)

    def step():
        fwd()
        layer.backward(d["dout"], d["x"], d["Wr"], d["W1"], d["W3"], d["W2"], dx, dWr, dW1, dW3, dW2,
                       stream=stream)

    def barrier():
        torch.cuda.synchronize(dev)
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    def timed(fn, k):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(k)]
        with torch.cuda.stream(stream):
            for a, b in evs:
                flush.fill_(1)                # evict L2 between timed steps (untimed)
                a.record(stream)
                fn()
                b.record(stream)
        stream.synchronize()
        return sum(a.elapsed_time(b) for a, b in evs)

    props = torch.cuda.get_device_properties(dev)
    try:
        bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
        sampler = NvmlClockSampler(bus)
        clk_p = clk_path = None
    except Exception:
        sampler = None
        clk_p, clk_path = start_clocks(local)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    layer.status(stream)
    barrier()
    total_ms = timed(step, args.steps)
    w0_ms = None
    if w.precision == "mxfp8":
        # weight quantisation runs once per weight update, outside the step; timed on its own
        w0_ms = timed(lambda: layer.quantize_weights(d["W1"], d["W3"], d["W2"], stream=stream), args.steps)
        w0_ms, = max_over_ranks([w0_ms], device=dev)   # every rank has the same precision
    barrier()
    fwd_ms = timed(fwd, args.steps)
    layer.status(stream)
    total_ms, fwd_ms = max_over_ranks([total_ms, fwd_ms], device=dev)

    # per-kernel breakdown: the same steps with events around every launch
    M.moe_profile_begin()
    prof_ms = timed(step, args.steps)
    kernels = M.moe_profile_end()
    launches = sum(n for _, n, _ in kernels)

    # end to end through the public API with host buffers: every step copies its x and dout
    # from pinned host memory to the device and reads its out and dx back. The copies run on
    # their own streams and the device buffers are double-buffered, so step i+1's inputs
    # arrive while step i computes, out leaves during the backward and dx during the next
    # step (the usual input/output pipeline of a training or serving loop). The timed region
    # runs from the first host-to-device copy to the end of the last device-to-host copy.
    hx = torch.empty(w.T, w.H, dtype=torch.bfloat16, pin_memory=True)
    hd = torch.empty_like(hx, pin_memory=True)
    hx.copy_(d["x"].cpu())
    hd.copy_(d["dout"].cpu())
    NB = 2
    hout = [torch.empty_like(hx, pin_memory=True) for _ in range(NB)]
    hdx = [torch.empty_like(hx, pin_memory=True) for _ in range(NB)]
    xin = [torch.empty_like(d["x"]) for _ in range(NB)]
    din = [torch.empty_like(d["dout"]) for _ in range(NB)]
    outb = [torch.empty_like(out) for _ in range(NB)]
    dxb = [torch.empty_like(dx) for _ in range(NB)]
    h2d = torch.cuda.Stream(device=dev)
    d2h = torch.cuda.Stream(device=dev)

    def e2e_run(k):
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
            layer.forward(xin[b], d["Wr"], bias, d["W1"], d["W3"], d["W2"], outb[b], ids, wts, stream=stream)
            ef = ev(); ef.record(stream)
            with torch.cuda.stream(d2h):
                d2h.wait_event(ef)
                hout[b].copy_(outb[b], non_blocking=True)
            stream.wait_event(ed)
            layer.backward(din[b], xin[b], d["Wr"], d["W1"], d["W3"], d["W2"], dxb[b], dWr, dW1, dW3, dW2,
                           stream=stream)
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

    e2e_run(2)
    e2e_ms = e2e_run(args.steps)
    e2e_ms, = max_over_ranks([e2e_ms], device=dev)
    layer.status(stream)
    clocks = sampler.stop() if sampler is not None else stop_clocks(clk_p, clk_path)

    if rank != 0:
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
            dist.destroy_process_group()
        return
    peaks, peak_src = load_peaks()
    # dominant kernel: largest share of the profiled step
    kt = sorted(kernels, key=lambda r: -r[2])
    name, n, ms = kt[0]
    per_launch_ms = ms / n
    # gemm_flops / kernel_bytes are per step; a kernel may launch several times
    # per step (one launch per macrobatch)
    per_step = n / args.steps
    fl = gemm_flops(w, name)
    fl = None if fl is None else fl / per_step
    roof = None
    if fl is not None:
        peak = peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops"))
        if w.precision == "mxfp8":
            peak = 2 * peak     # fp8 dense = 2x bf16 (nominal 4.5 vs 2.25 PFLOP/s)
        gb = gemm_bytes(w, name) / per_step
        if w.precision == "mxfp8":
            gb = None           # operand bytes differ per operand in MXFP8; rated on the tensor pipe
        hbm = peaks.get("hbm_gbs")
        traffic = committed_traffic(name) if w.name == WL.BALANCED.name else None
        if gb is not None and hbm and gb / (hbm * 1e9) > fl / (peak * 1e12):
            # the kernel's roofline is HBM: its algorithmic bytes take longer than its flops
            ach = gb / (per_launch_ms * 1e-3) / 1e9
            roof = {"kernel": name, "bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                    "frac": ach / hbm, "traffic": traffic, "algorithmic_per_launch": gb,
                    "tensor_frac": fl / (per_launch_ms * 1e-3) / 1e12 / peak,
                    "peak_source": f"{peak_src} hbm_gbs (copy bandwidth)"}
        else:
            ach = fl / (per_launch_ms * 1e-3) / 1e12
            roof = {"kernel": name, "bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                    "frac": ach / peak, "traffic": traffic, "algorithmic_per_launch": fl,
                    "algorithmic_bytes_per_launch": gb,
                    "peak_source": f"{peak_src} bf16_tflops_sustained (kernel timed inside the step loop)"
                                   + (" x 2 (nominal fp8/bf16 ratio)" if w.precision == "mxfp8" else "")}
    elif kernel_bytes(w, name) is not None:
        peak = peaks.get("hbm_gbs")
        ach = kernel_bytes(w, name) / per_step / (per_launch_ms * 1e-3) / 1e9
        roof = {"kernel": name, "bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s",
                "frac": ach / peak, "traffic": None, "algorithmic_per_launch": kernel_bytes(w, name) / per_step,
                "peak_source": f"{peak_src} hbm_gbs"}
    gemm_ms = sum(ms_ for nm, _, ms_ in kernels if nm.startswith("grouped_gemm"))
    gemm_fl = sum(gemm_flops(w, nm) * args.steps for nm, n_, _ in kernels if nm.startswith("grouped_gemm"))
    value = job_tokens_per_s(ws, w.T, args.steps, total_ms)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.precision == "bf16" else "mxfp8",
        "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "H": w.H, "F": w.F, "E": w.E, "k": w.k,
                   "precision": w.precision, "step": "forward+backward",
                   "l2": "flushed (256 MiB write) between timed steps",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "w0": None if w0_ms is None else {
            "ms": w0_ms / args.steps,
            "fwd_bwd_value_incl_w0": job_tokens_per_s(ws, w.T, args.steps, total_ms + w0_ms),
            "note": "MXFP8 weight copies, once per weight update; excluded from value"},
        "fwd": {"value": job_tokens_per_s(ws, w.T, args.steps, fwd_ms), "unit": "tokens/s",
                "ms_per_step": fwd_ms / args.steps},
        "roofline": roof,
        "grouped_gemm": {"tflops": gemm_fl / (gemm_ms * 1e-3) / 1e12 if gemm_ms else None,
                         "frac_of_peak": (gemm_fl / (gemm_ms * 1e-3) / 1e12) /
                         (peaks.get("bf16_tflops_sustained", 1700.0) * (2 if w.precision == "mxfp8" else 1))
                         if gemm_ms else None,
                         "share_of_step": gemm_ms / prof_ms if prof_ms else None},
        "kernels": [dict({"name": nm, "launches": n_, "ms_per_step": ms_ / args.steps,
                          "share": ms_ / prof_ms},
                         **({"tflops": gemm_flops(w, nm) * args.steps / (ms_ * 1e-3) / 1e12} if gemm_flops(w, nm) else {}),
                         **({"gbs": kernel_bytes(w, nm) * args.steps / (ms_ * 1e-3) / 1e9,
                             "frac_of_hbm": kernel_bytes(w, nm) * args.steps / (ms_ * 1e-3) / 1e9 / peaks["hbm_gbs"]}
                            if kernel_bytes(w, nm) and peaks.get("hbm_gbs") else {}))
                    for nm, n_, ms_ in kt],
        "layer_roofline": layer_roofline(w, peaks, total_ms / args.steps),
        "gpu_launches": launches,
        "e2e": {"value": job_tokens_per_s(ws, w.T, args.steps, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": 2 * w.T * w.H * 2, "d2h_bytes_per_step": 2 * w.T * w.H * 2,
                "pipelined": "copy streams, double-buffered inputs/outputs; no L2 flush (weights exceed L2)"},
        "clocks": clocks,
    }
    if args.minibatch_sweep and w.minibatch_rows:
        sweep = []
        del layer
        torch.cuda.empty_cache()
        for mbr in w.minibatch_rows:
            lay = MoeLayer(w.T, w.H, w.F, w.E, w.k, w.precision, device=dev, ring_bytes=w.ring_bytes,
                           minibatch_rows=mbr)
            if w.precision == "mxfp8":
                lay.quantize_weights(d["W1"], d["W3"], d["W2"], stream=stream)

            def f1(lay=lay):
                lay.forward(d["x"], d["Wr"], bias, d["W1"], d["W3"], d["W2"], out, ids, wts, stream=stream)

            def s1(lay=lay):
                f1()
                lay.backward(d["dout"], d["x"], d["Wr"], d["W1"], d["W3"], d["W2"], dx, dWr, dW1, dW3, dW2,
                             stream=stream)
            with torch.cuda.stream(stream):
                for _ in range(2):
                    s1()
            k = max(2, args.steps // 4)
            fm, sm = timed(f1, k), timed(s1, k)
            lay.status(stream)
            sweep.append({"minibatch_rows": mbr, "fwd_ms": fm / k, "fwd_bwd_ms": sm / k,
                          "macrobatches": lay.plan.num_macrobatches, "macrobatch_tokens": lay.plan.macrobatch_tokens})
            del lay
            torch.cuda.empty_cache()
        line["minibatch_sweep"] = sweep
    if ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, inp)
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=WL.BALANCED.name, choices=sorted(WL.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=0, help="override T (small cases for ncu captures)")
    ap.add_argument("--experts", type=int, default=0, help="override E, keeping k <= E (small cases for ncu captures)")
    ap.add_argument("--minibatch-sweep", action="store_true",
                    help="also time fwd and fwd+bwd for each minibatch size of the workload (ring workload)")
    args = ap.parse_args()
    assert args.warmup >= 3 or args.impl == "reference" or args.steps < 3, "need >= 3 warm-up steps"
    w = WL.WORKLOADS[args.workload]
    if args.tokens:
        w = w.with_(T=args.tokens, name=f"{w.name}@T{args.tokens}")
    if args.experts:
        w = w.with_(E=args.experts, k=min(w.k, args.experts), name=f"{w.name}@E{args.experts}")
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
