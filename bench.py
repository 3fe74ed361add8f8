#!/usr/bin/env python3
"""Benchmark: exact attention forward + backward on one GB300 (or N independent replicas).

One step = fa_fwd + fa_bwd (preprocess, main, postprocess) over the dense causal
workload B=2, s=8192, h=16, d=128, bf16 — the shape the throughput target is quoted on.
The metric is attention TFLOPS of the forward+backward pass with the pages' convention:
4 * d FLOPs per allowed (query, key) pair for the forward, 2.5x that for the backward,
3.5x for both.  Inputs are seeded synthetic draws already resident in HBM; L2 is flushed
(a 256 MiB write) between timed steps.

--impl reference times the fp64 CPU oracle on a bounded sample of the same workload.
Under torchrun every rank runs its own replica (the path has no exchange step); the
step time is the maximum over ranks and the value counts all ranks' work.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from exact_attention_bwd_gb300 import inputs, metrics  # noqa: E402

METRIC = "attention TFLOPS fwd+bwd (bf16, d=128, causal)"
UNIT = "TFLOP/s"
WORKLOAD = "sweep_s8192_causal"
# dram__bytes_read.sum + dram__bytes_write.sum of one bwd_main launch, from the ncu
# capture summarised in profiles/ (None until a capture of the current kernel exists)
BWD_MAIN_DRAM_BYTES = 623929344  # dram read + write of one launch on this workload (ncu --set full)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the other prefill workloads")
    ap.add_argument("--decode-only", default=None, help="time one decode workload and exit")
    ap.add_argument("--decode-batch", type=int, default=None, help="batch override for --decode-only")
    ap.add_argument("--paged", action="store_true", help="--decode-only over a paged cache")
    ap.add_argument("--fp8-only", default=None, help="time the e4m3 forward of one workload and exit")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            j = json.load(f)
        return dict(hbm=j["hbm_gbs"], bf16=j["bf16_tflops"], bf16_sus=j["bf16_tflops_sustained"], src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


class _Nvml:
    """Read-only NVML queries through ctypes (libnvidia-ml ships with the driver): the SM
    clock, its maximum and the active clock-event reasons of one GPU, found by PCI id."""
    CLOCK_SM = 1
    # nvmlClocksEventReasons bits of the four reasons the timing rules name
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, pci_bus_id: str):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(self.h)) != 0:
            raise OSError(f"no NVML device at {pci_bus_id}")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        if self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.CLOCK_SM, ctypes.byref(mx)) != 0:
            raise OSError("nvmlDeviceGetMaxClockInfo failed")
        self.max_mhz = float(mx.value)

    def sample(self):
        sm, rs = self.ct.c_uint(), self.ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM, self.ct.byref(sm)) != 0:
            return None
        if self.reasons_fn(self.h, self.ct.byref(rs)) != 0:
            return None
        return float(sm.value), {nm for bit, nm in self.REASONS.items() if rs.value & bit}


def _pci_bus_id(dev_index: int) -> str:
    import torch
    pr = torch.cuda.get_device_properties(dev_index)
    return f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0"


class ClockSampler:
    """SM clocks and clock-event reasons sampled DURING the timed region: every 2 ms by a
    thread reading NVML (the timed region is tens of milliseconds), else every 200 ms by
    nvidia-smi.  The GPU is the CUDA device's own (matched by PCI id)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.out = None
        self.nvml = None
        self.samples = []
        self.stop = threading.Event()
        self.thread = None
        try:
            self.pci = _pci_bus_id(index)
        except Exception:  # noqa: BLE001 - an older torch without PCI properties
            self.pci = None
        try:
            self.nvml = _Nvml(self.pci) if self.pci else None
        except (OSError, AttributeError):
            self.nvml = None

    def _poll(self):
        while not self.stop.is_set():
            x = self.nvml.sample()
            if x is not None:
                self.samples.append(x)
            self.stop.wait(0.002)

    def __enter__(self):
        if self.nvml is not None:
            self.nvml.sample()  # first read before the region: the library is then warm
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return self
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.pci or self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader", "-lms", "200"], stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.thread is not None:
            self.stop.set()
            self.thread.join(timeout=5)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.nvml is not None:
            if not self.samples:
                return None
            reasons = set().union(*(r for _, r in self.samples))
            return {"sm_mhz": statistics.median(m for m, _ in self.samples), "sm_max_mhz": self.nvml.max_mhz,
                    "reasons": sorted(reasons), "samples": len(self.samples), "source": "nvml, every 2 ms"}
        if self.out is None:
            return None
        self.out.flush()
        self.out.seek(0)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1].split()[0]))
                mx = float(parts[2].split()[0])
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        os.unlink(self.out.name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm),
                "source": "nvidia-smi, every 200 ms"}


# ----------------------------------------------------------------------------------------------
# the GPU arm
# ----------------------------------------------------------------------------------------------

def aggregate(total_ms_local, flops_per_step, steps, world, device=None):
    """Whole-job throughput of N replicas: the timed region ends when the slowest rank
    does, so the step time is the maximum over ranks and the value counts every rank's
    work.  Returns (max total ms, TFLOP/s).  Backend-agnostic (nccl on GPUs, gloo on CPU)."""
    total = float(total_ms_local)
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([total], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total = float(t.item())
    return total, world * flops_per_step * steps / (total * 1e-3) / 1e12

def run_ours(args):
    import torch
    import torch.distributed as dist
    from exact_attention_bwd_gb300 import binding as fa

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = inputs.make(inputs.workload(args.workload))
    fl_fwd = metrics.fwd_flops(w)
    fl_bwd = metrics.bwd_flops(w)

    def up(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    q, k, v, dout = up(w["q"]), up(w["k"]), up(w["v"]), up(w["dout"])
    # sinks and packed offsets for the workloads that have them (one offsets array serves
    # queries and keys, which are packed alike)
    sinks = None if w["sinks"] is None else torch.from_numpy(w["sinks"]).to(dev)
    cu = None if w["cu_q"] is None else torch.from_numpy(w["cu_q"]).to(dev)
    kw = dict(causal=w["causal"], window=w["window"], softmax_scale=w["scale"], sinks=sinks, cu_q=cu, cu_k=cu)
    o, lse, ws_f = fa.forward(q, k, v, **kw)
    dq, dk, dv, dsk, ws_b = fa.backward(q, k, v, o, lse, dout, **kw)
    grads = (dq, dk, dv, dsk)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        fa.forward(q, k, v, **kw, out=o, lse=lse, workspace=ws_f)
        fa.backward(q, k, v, o, lse, dout, **kw, workspace=ws_b, grads=grads)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if fa.device_status(ws_f) != 0 or fa.device_status(ws_b) != 0:
        raise RuntimeError("device status nonzero after warm-up")

    fa.fa_profile_enable(True)
    kern = {n: [] for n in ("fwd", "bwd_pre", "bwd_main", "bwd_post")}
    times = []
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for _ in range(args.steps):
            flush.zero_()
            ev0.record(stream)
            step()
            ev1.record(stream)
            ev1.synchronize()
            times.append(ev0.elapsed_time(ev1))
            for n in kern:
                rc, ms = fa.fa_profile_read(n)
                if rc == 0:
                    kern[n].append(ms)
    torch.cuda.synchronize()
    fa.fa_profile_enable(False)
    clocks = clk.summary()
    total_ms, value = aggregate(sum(times), fl_fwd + fl_bwd, args.steps, world, dev)
    ms_step = total_ms / args.steps

    # ---- end to end: pinned host inputs in, results out, through the same public API ----
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, fa, kw, (q, k, v, dout), (o, lse, ws_f, ws_b), fl_fwd + fl_bwd, world, dev)

    pk = peaks()
    main_ms = statistics.mean(kern["bwd_main"]) if kern["bwd_main"] else None
    fwd_ms = statistics.mean(kern["fwd"]) if kern["fwd"] else None
    long_region = total_ms > 1000.0
    peak = pk["bf16_sus"] if long_region else pk["bf16"]
    roof = None
    if main_ms:
        ach = fl_bwd / (main_ms * 1e-3) / 1e12
        roof = {"kernel": "bwd_main", "bound": "tensor", "achieved": round(ach, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(ach / peak, 4), "traffic": BWD_MAIN_DRAM_BYTES,
                "peak_kind": f"{pk['src']} bf16 {'sustained' if long_region else 'burst'}",
                "algorithmic_flops": fl_bwd}
    per_kernel = {n: round(statistics.mean(x), 4) for n, x in kern.items() if x}
    fwd_tf = fl_fwd / (fwd_ms * 1e-3) / 1e12 if fwd_ms else None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16)",
        "config": {"workload": args.workload, "B": w["B"], "s_q": w["s_q"], "s_kv": w["s_kv"], "h_q": w["h_q"],
                   "h_kv": w["h_kv"], "d": w["d"], "causal": w["causal"], "window": list(w["window"]),
                   "l2": "flushed between timed steps (256 MiB write)", "parallelism": f"replicas x{world}"},
        "fwd_tflops": round(fwd_tf, 1) if fwd_tf else None,
        "fwd_frac_of_peak": round(fwd_tf / pk["bf16"], 4) if fwd_tf else None,
        "kernel_ms": per_kernel,
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": 4 * args.steps,
        "clocks": clocks,
        "step_ms": {"median": statistics.median(times), "mean": statistics.mean(times),
                    "std": statistics.pstdev(times), "min": min(times), "max": max(times)},
    }
    if not args.no_decode:
        line["decode"] = {n: measure_decode(dev, n) for n in
                          ("decode_d128_sq1", "decode_d128_sq64", "decode_d256_sq1", "decode_d256_sq64")}
        line["decode"].update({n + "_paged": measure_decode(dev, n, paged=True) for n in
                               ("decode_d128_sq1", "decode_d256_sq1", "decode_d128_sq64")})
    if not args.no_sweep:
        line["workloads"] = {n: measure_workload(dev, n) for n in SWEEP + OTHER}
        line["deterministic_bwd"] = {n: measure_workload(dev, n, bwd_flags=fa.FA_FLAG_DETERMINISTIC)
                                     for n in ("sweep_s8192_causal", "sweep_s2048", "gqa_window_causal", "varlen",
                                               "d256_s8192_causal")}
        line["f16"] = {n: measure_workload(dev, n, dtype="f16")
                       for n in ("sweep_s8192_causal", "sweep_s8192", "sweep_s2048", "gqa_window_causal", "varlen")}
        line["e4m3_fwd"] = {n: measure_fp8(dev, n) for n in ("sweep_s8192_causal", "sweep_s8192", "sweep_s16384",
                                                              "sweep_s2048", "decode_d128_sq64")}
    if not args.no_sweep:
        line["d256"] = measure_d256(dev)
    if "decode" in line:
        # the decode targets' figures once more, compactly, near the end of the line
        line["decode_frac_hbm"] = {n: r.get("frac_hbm") for n, r in line["decode"].items()}
    if rank == 0 and not args.no_cpu and w["cu_q"] is None:
        line["cpu_baseline"] = oracle_sample(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_e2e(args, fa, kw, ins, outs, flops, world, dev):
    """End-to-end throughput: every step copies its inputs (Q, K, V, dO) from pinned host
    memory, runs fa_fwd + fa_bwd, and copies its results (O, LSE, dQ, dK, dV) back to pinned
    host memory.  Steps are pipelined the way a serving or training loop would run them:
    copies on their own streams, two device sets of inputs and outputs, so step i+1's input
    copy and step i-1's result copy overlap step i's kernels; within a step the forward
    starts once Q, K, V have landed (dO gates the backward) and O, LSE leave while the
    backward runs.  The timed region runs from
    the first step's first input copy to the last step's last result copy (pipeline fill
    and drain included)."""
    import torch
    q, k, v, dout = ins
    o, lse, ws_f, ws_b = outs
    host_in = [t.cpu().pin_memory() for t in (q, k, v, dout)]
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (o, lse, q, k, v)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    dev_in = [[torch.empty_like(t) for t in (q, k, v, dout)] for _ in range(2)]
    dev_out = [[torch.empty_like(o), torch.empty_like(lse), torch.empty_like(q), torch.empty_like(k),
                torch.empty_like(v)] for _ in range(2)]
    dsk = None if kw.get("sinks") is None else torch.empty_like(kw["sinks"])
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_qkv = [torch.cuda.Event() for _ in range(2)]  # Q, K, V of the set have landed
    ev_in = [torch.cuda.Event() for _ in range(2)]   # ... and dO
    ev_fwd = [torch.cuda.Event() for _ in range(2)]  # the forward has written O, LSE
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def run(n, t0=None, t1=None):
        for it in range(n):
            b = it % 2
            with torch.cuda.stream(s_in):
                if it >= 2:
                    s_in.wait_event(ev_cmp[b])  # step it-2 has consumed this input set
                if it == 0 and t0 is not None:
                    t0.record(s_in)
                for dst, src in zip(dev_in[b][:3], host_in[:3]):
                    dst.copy_(src, non_blocking=True)
                ev_qkv[b].record(s_in)
                dev_in[b][3].copy_(host_in[3], non_blocking=True)
                ev_in[b].record(s_in)
            with torch.cuda.stream(s_cmp):
                # the forward needs Q, K, V only; dO (the last input copy) gates the backward
                s_cmp.wait_event(ev_qkv[b])
                if it >= 2:
                    s_cmp.wait_event(ev_out[b])  # step it-2's results have left this output set
                qb, kb, vb, dob = dev_in[b]
                ob, lb, dqb, dkb, dvb = dev_out[b]
                fa.forward(qb, kb, vb, **kw, out=ob, lse=lb, workspace=ws_f)
                ev_fwd[b].record(s_cmp)
                s_cmp.wait_event(ev_in[b])
                fa.backward(qb, kb, vb, ob, lb, dob, **kw, workspace=ws_b, grads=(dqb, dkb, dvb, dsk))
                ev_cmp[b].record(s_cmp)
            with torch.cuda.stream(s_out):
                # O and LSE leave while the backward runs; the gradients after it
                s_out.wait_event(ev_fwd[b])
                for dst, src in zip(host_out[:2], dev_out[b][:2]):
                    dst.copy_(src, non_blocking=True)
                s_out.wait_event(ev_cmp[b])
                for dst, src in zip(host_out[2:], dev_out[b][2:]):
                    dst.copy_(src, non_blocking=True)
                ev_out[b].record(s_out)
                if it == n - 1 and t1 is not None:
                    t1.record(s_out)

    run(max(args.warmup, 2))
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    run(args.steps, t0, t1)
    torch.cuda.synchronize()
    if fa.device_status(ws_f) != 0 or fa.device_status(ws_b) != 0:
        raise RuntimeError("device status nonzero after the end-to-end steps")
    tot, value = aggregate(t0.elapsed_time(t1), flops, args.steps, world, dev)
    return {"value": value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": tot / args.steps,
            "how": "pinned host buffers; copies on their own streams, double-buffered device sets, "
                   "fill and drain inside the timed region"}


# ----------------------------------------------------------------------------------------------
# every other workload: forward and forward+backward TFLOPS (context beside the headline)
# ----------------------------------------------------------------------------------------------

def measure_workload(dev, name, steps=5, warmup=2, bwd_flags=0, dtype="bf16", check_status=False):
    """fwd and fwd+bwd of one prefill workload with seeded on-device inputs (the same recipe
    seeds, drawn by torch's generator); L2 flushed before every timed step.  bwd_flags:
    fa_params flags of the backward (FA_FLAG_DETERMINISTIC for the fixed-order dQ sums);
    dtype: "bf16" or "f16" inputs (the same draws, rounded to that type)."""
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    w = inputs.workload(name)
    sd = lambda t: inputs.seed_of(w["wid"], w.get("variant", 0), t)  # noqa: E731
    if w.get("varlen"):
        lengths = inputs.varlen_lengths(sd(inputs.LENGTHS), n=w["B"], total=w["T"])
        cu = inputs.cu_seqlens(lengths)
        wf = dict(w, cu_q=cu, cu_k=cu)
        qs, ks = (w["T"], w["h_q"], w["d"]), (w["T"], w["h_kv"], w["d"])
        cu_d = torch.from_numpy(cu).to(dev)
    else:
        wf = dict(w)
        qs, ks = (w["B"], w["s_q"], w["h_q"], w["d"]), (w["B"], w["s_kv"], w["h_kv"], w["d"])
        cu_d = None
    draw = inputs.normal_f16_torch if dtype == "f16" else inputs.normal_bf16_torch
    q = draw(sd(inputs.Q), qs, dev)
    k = draw(sd(inputs.K), ks, dev)
    v = draw(sd(inputs.V), ks, dev)
    do = draw(sd(inputs.DO), qs, dev)
    sinks = None
    if w.get("sinks"):
        g = torch.Generator(device=dev)
        g.manual_seed(sd(inputs.SINKS))
        sinks = torch.randn(w["h_q"], generator=g, device=dev, dtype=torch.float32)
    kw = dict(causal=w["causal"], window=w["window"], softmax_scale=1.0 / math.sqrt(w["d"]), sinks=sinks,
              cu_q=cu_d, cu_k=cu_d)
    o, lse, wsf = fa.forward(q, k, v, **kw)
    dq, dk, dv, ds, wsb = fa.backward(q, k, v, o, lse, do, **kw, flags=bwd_flags)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    tf, tb = [], []
    for it in range(warmup + steps):
        flush.zero_()
        e0.record(stream)
        fa.forward(q, k, v, **kw, out=o, lse=lse, workspace=wsf)
        e1.record(stream)
        fa.backward(q, k, v, o, lse, do, **kw, workspace=wsb, grads=(dq, dk, dv, ds), flags=bwd_flags)
        e2.record(stream)
        e2.synchronize()
        if it >= warmup:
            tf.append(e0.elapsed_time(e1))
            tb.append(e1.elapsed_time(e2))
    if check_status and (fa.device_status(wsf) != 0 or fa.device_status(wsb) != 0):
        raise RuntimeError(f"{name}: device status nonzero after the timed steps")
    ff = metrics.fwd_flops(wf)
    mf, mb = statistics.mean(tf), statistics.mean(tb)
    del q, k, v, do, o, lse, wsf, dq, dk, dv, wsb
    torch.cuda.empty_cache()
    pk = peaks()
    # both roofs: the tensor rate and the HBM rate of the algorithmic bytes (for the shapes
    # near the ridge point, e.g. the grouped-query sliding-window workloads)
    fgb = metrics.fwd_bytes(wf) / (mf * 1e-3) / 1e9
    bgb = metrics.bwd_bytes(wf) / (mb * 1e-3) / 1e9
    return {"fwd_ms": round(mf, 4), "bwd_ms": round(mb, 4), "fwd_TFLOPS": round(ff / (mf * 1e-3) / 1e12, 1),
            "fwd_bwd_TFLOPS": round(3.5 * ff / ((mf + mb) * 1e-3) / 1e12, 1),
            "fwd_frac_tensor": round(ff / (mf * 1e-3) / 1e12 / pk["bf16"], 4),
            "fwd_GB_per_s": round(fgb, 1), "fwd_frac_hbm": round(fgb / pk["hbm"], 4),
            "bwd_GB_per_s": round(bgb, 1), "bwd_frac_hbm": round(bgb / pk["hbm"], 4)}


def measure_d256(dev):
    """fwd and fwd+bwd at head dims 256 and 192 (the wide-head kernels), with the backward's
    own rate against the bf16 peak.  Run last among the GPU sections; a failure is recorded
    in the section, not raised."""
    from exact_attention_bwd_gb300 import binding as fa
    pk = peaks()
    out = {}
    for name in ("d256_s8192_causal", "d256_s4096", "d192_s8192_causal"):
        try:
            r = measure_workload(dev, name, check_status=True)
            ff = metrics.fwd_flops(inputs.workload(name))
            bt = 2.5 * ff / (r["bwd_ms"] * 1e-3) / 1e12
            r.update(bwd_TFLOPS=round(bt, 1), bwd_frac_of_peak=round(bt / pk["bf16"], 4),
                     fwd_frac_of_peak=round(r["fwd_TFLOPS"] / pk["bf16"], 4))
            out[name] = r
        except (RuntimeError, fa.FaError) as e:
            out[name] = {"error": f"{type(e).__name__}: {e}"[:300]}
    return out


def measure_fp8(dev, name, steps=8, warmup=3):
    """Forward with e4m3 inputs (same shapes; stored values N(0, 32^2) rounded to e4m3 with
    per-(batch, kv head) descales): the whole fa_fwd call by CUDA events and the kernel
    alone by the library's own events, L2 flushed before every timed call; TFLOPS with the
    same FLOP convention."""
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    w = inputs.workload(name)
    B, s_q, s_kv, h_q, h_kv, d = w["B"], w["s_q"], w["s_kv"], w["h_q"], w["h_kv"], w["d"]
    sd = lambda t: inputs.seed_of(w["wid"], w["variant"], t)  # noqa: E731

    def draw(seed, shape):
        x = inputs.normal_bf16_torch(seed, shape, dev).float() * 32.0
        return x.to(torch.float8_e4m3fn).view(torch.uint8)
    q = draw(sd(inputs.Q), (B, s_q, h_q, d))
    k = draw(sd(inputs.K), (B, s_kv, h_kv, d))
    v = draw(sd(inputs.V), (B, s_kv, h_kv, d))
    ds = tuple(torch.full((B * h_kv,), 1.0 / 32.0, dtype=torch.float32, device=dev) for _ in range(3))
    kw = dict(causal=w["causal"], window=w["window"], softmax_scale=1.0 / math.sqrt(d), descale=ds)
    o, lse, ws = fa.forward(q, k, v, **kw)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    fa.fa_profile_enable(True)
    ts, tk = [], []
    for it in range(warmup + steps):
        flush.zero_()
        e0.record(stream)
        fa.forward(q, k, v, **kw, out=o, lse=lse, workspace=ws)
        e1.record(stream)
        e1.synchronize()
        if it >= warmup:
            ts.append(e0.elapsed_time(e1))
            rc, ms = fa.fa_profile_read("fwd")
            if rc == 0:
                tk.append(ms)
    fa.fa_profile_enable(False)
    if fa.device_status(ws) != 0:
        raise RuntimeError("device status nonzero after the e4m3 forward")
    ff = metrics.fwd_flops(dict(w, varlen=False))
    mf = statistics.mean(ts)
    del q, k, v, o, lse, ws
    torch.cuda.empty_cache()
    return {"fwd_ms": round(mf, 4), "fwd_TFLOPS": round(ff / (mf * 1e-3) / 1e12, 1),
            "kernel_ms": round(statistics.mean(tk), 4) if tk else None,
            "kernel_TFLOPS": round(ff / (statistics.mean(tk) * 1e-3) / 1e12, 1) if tk else None}


SWEEP = [f"sweep_s{s}{c}" for s in (512, 1024, 2048, 4096, 8192, 16384) for c in ("", "_causal")]
OTHER = ["gqa_window_causal", "gqa_window_2sided", "varlen"]


# ----------------------------------------------------------------------------------------------
# decode / chunked prefill against a long cache: HBM-bound, reported as GB/s
# ----------------------------------------------------------------------------------------------

PAGE_SIZE = 256  # keys per page of the paged-cache decode measurement


def measure_decode(dev, name, steps=10, warmup=3, batch=None, paged=False):
    """Forward of one decode workload: algorithmic bytes (K and V read once, Q read, O and
    LSE written) per launch over the CUDA-event time of the whole forward (split kernel +
    combine), L2 flushed between launches; per-kernel times from the library's hooks.
    paged: the cache is a pool of 256-key pages in a seeded random order, addressed
    through a block table (the table's reads are not counted as algorithmic bytes)."""
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    w = inputs.workload(name) if batch is None else inputs.workload(name, B=batch)
    B, s_q, s_kv, h_q, h_kv, d = w["B"], w["s_q"], w["s_kv"], w["h_q"], w["h_kv"], w["d"]
    sd = lambda t: inputs.seed_of(w["wid"], w["variant"], t)  # noqa: E731
    q = inputs.normal_bf16_torch(sd(inputs.Q), (B, s_q, h_q, d), dev)
    kw = dict(causal=True, softmax_scale=1.0 / math.sqrt(d))
    if paged:
        max_blocks = -(-s_kv // PAGE_SIZE)
        kshape = (B * max_blocks, PAGE_SIZE, h_kv, d)
        table = inputs.page_table(sd(7), B, max_blocks, B * max_blocks)
        kw.update(block_table=torch.from_numpy(table).to(dev), s_kv=s_kv)
    else:
        kshape = (B, s_kv, h_kv, d)
    k = inputs.normal_bf16_torch(sd(inputs.K), kshape, dev)
    v = inputs.normal_bf16_torch(sd(inputs.V), kshape, dev)
    o, lse, ws = fa.forward(q, k, v, **kw)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(warmup):
        fa.forward(q, k, v, **kw, out=o, lse=lse, workspace=ws)
    fa.fa_profile_enable(True)
    times, kern = [], {}
    for _ in range(steps):
        flush.zero_()
        e0.record(stream)
        fa.forward(q, k, v, **kw, out=o, lse=lse, workspace=ws)
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
        for n in ("fwd", "decode", "combine"):
            rc, ms = fa.fa_profile_read(n)
            if rc == 0:
                kern.setdefault(n, []).append(ms)
    fa.fa_profile_enable(False)
    torch.cuda.synchronize()
    nbytes = 2 * (2 * B * s_kv * h_kv * d) + 2 * (2 * B * s_q * h_q * d) + 4 * B * h_q * s_q
    ms = statistics.mean(times)
    gbs = nbytes / (ms * 1e-3) / 1e9
    pk = peaks()
    flops = metrics.fwd_flops(dict(w, varlen=False))
    del q, k, v, o, lse, ws
    torch.cuda.empty_cache()
    return {"ms": round(ms, 4), "GB_per_s": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm"], 4),
            "hbm_peak": pk["hbm"], "TFLOPS": round(flops / (ms * 1e-3) / 1e12, 1), "algorithmic_bytes": nbytes,
            "kernel_ms": {n: round(statistics.mean(x), 4) for n, x in kern.items()}}


# ----------------------------------------------------------------------------------------------
# the oracle on a bounded sample of the workload
# ----------------------------------------------------------------------------------------------

def oracle_sample(w, rows=256):
    """fp64 oracle fwd+bwd on the last `rows` query rows of batch element 0 (all heads,
    every key they see), timed on the host cores; TFLOPS with the same convention."""
    import oracle
    b = 0
    s_q, s_kv = w["s_q"], w["s_kv"]
    i0 = s_q - rows
    q = inputs.bf16_to_f64(w["q"][b:b + 1, i0:])
    kend = s_kv if not w["causal"] else s_kv  # the last rows see every key up to s_kv
    k = inputs.bf16_to_f64(w["k"][b:b + 1, :kend])
    v = inputs.bf16_to_f64(w["v"][b:b + 1, :kend])
    do = inputs.bf16_to_f64(w["dout"][b:b + 1, i0:])
    kw = dict(scale=w["scale"], causal=w["causal"], window=w["window"])
    sub = dict(w, B=1, s_q=rows, s_kv=kend, cu_q=None, cu_k=None, varlen=False)
    flops = 3.5 * metrics.fwd_flops(sub)
    t0 = time.perf_counter()
    oracle.fwd(q, k, v, **kw)
    oracle.bwd(q, k, v, do, **kw)
    dt = time.perf_counter() - t0
    return {"value": round(flops / dt / 1e12, 6), "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
            "seconds": round(dt, 2),
            "sample": f"batch 0, all {w['h_q']} heads, last {rows} of {s_q} query rows with all keys they see "
                      f"(fwd+bwd, fp64, {flops / 1e9:.1f} GFLOP)"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = inputs.make(inputs.workload(args.workload))
    vals = []
    cb = None
    for it in range(args.warmup + args.steps):
        r = oracle_sample(w, rows=64)
        if it >= args.warmup:
            vals.append(r["value"])
            cb = r
    val = statistics.mean(vals)
    cb = dict(cb, value=round(val, 6))
    line = {"impl": "reference", "metric": METRIC, "value": round(val, 6), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1) bf16)",
            "config": {"workload": args.workload, "B": w["B"], "s_q": w["s_q"], "s_kv": w["s_kv"],
                       "h_q": w["h_q"], "h_kv": w["h_kv"], "d": w["d"], "causal": w["causal"]},
            "cpu_baseline": cb,
            "e2e": {"value": round(val, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.fp8_only:
        import torch
        torch.cuda.set_device(0)
        r = measure_fp8(torch.device("cuda", 0), args.fp8_only, steps=args.steps, warmup=args.warmup)
        print(json.dumps({"workload": args.fp8_only, "dtype": "e4m3", **r}), flush=True)
        return
    if args.decode_only:
        import torch
        torch.cuda.set_device(0)
        r = measure_decode(torch.device("cuda", 0), args.decode_only, steps=args.steps, warmup=args.warmup,
                           batch=args.decode_batch, paged=args.paged)
        print(json.dumps({"workload": args.decode_only, "batch": args.decode_batch, "paged": args.paged, **r}),
              flush=True)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
