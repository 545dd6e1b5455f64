#!/usr/bin/env python3
"""Benchmark of the GEMM hot path on GB300.

One step is one pass over every kernel family of the library, each on its
headline workload, all inputs resident in HBM:

  bf16   C[4096x4096] = A B, bf16 in/out, fp32 accumulate  (tcgen05 kernel)
  fp32   C = 1.5 A B + 0.5 C at 4096^3                      (FP32 SIMT kernel)
  decode C = X W + C, X with M in {1, 4, 16} rows, W the six LLaMA-7B weight
         shapes (qkv, o, gate, up, down, LM head)            (split-K kernel)

value = FLOPs of the step / device time of the step, in TFLOP/s.  Each part is
also reported with its own roofline: TFLOP/s against the tensor or FP32 peak
for the two square GEMMs, HBM GB/s for the decode GEMMs (their arithmetic
intensity is about M FLOP/byte).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --case bf16_8192 --reps 3      (one workload, for profiling)

Under torchrun every rank runs the same step on its own GPU (replicas, weak
scaling); time is the max over ranks.  ``--impl reference`` times the CPU
oracle on a bounded sample of the same step instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s (bf16 TC & fp32) at 4096³, % of roofline; decode GEMM HBM GB/s"
UNIT = "TFLOP/s"
WEIGHTS = ("qkv", "o", "gate", "up", "down", "lm")
DECODE_MS = (1, 4, 16)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}

# DRAM bytes per call measured by ncu (dram__bytes_read.sum + dram__bytes_write.sum,
# summed over the call's launches) for each kernel source file, valid only while
# the file hashes to `sha256`.
NCU_TRAFFIC = {
    # profiles/sgemm_tma_kernel_fp32_4096.md: whole-wave launch 316.0 MB read + 42.6 MB
    # written, stream-K tail 58.9 MB read + 3.5 MB written
    "gemm_f32_simt.cu": {"sha256": "dd99dbeb51e4db62de7256f586ff96e5df0a3ba2678d869a6287fb46beb76e3a",
                         "bytes_per_call": 315973376 + 42619136 + 58884864 + 3521024},
}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_sha(fname):
    p = os.path.join(ROOT, "roofline_driven_optimisation_gb300", "csrc", fname)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def traffic_for(fname):
    t = NCU_TRAFFIC.get(fname)
    if t and t["sha256"] == kernel_sha(fname):
        return t["bytes_per_call"]
    return None


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML (read-only)
    every few milliseconds while running."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x2: "applications_clocks_setting"}

    def __init__(self, device_index):
        self.samples, self.reasons, self.ok = [], set(), False
        self.max_mhz = None
        self._stop = threading.Event()
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if self.nv.nvmlDeviceGetHandleByIndex_v2(device_index, ctypes.byref(self.h)) != 0:
                return
            mx = ctypes.c_uint()
            if self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self.ok = True
        except OSError:
            self.ok = False

    def _run(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) == 0:
                self.samples.append(clk.value)
            if self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(rs)) == 0:
                for bit, name in self.REASONS.items():
                    if rs.value & bit:
                        self.reasons.add(name)
            time.sleep(0.002)

    def __enter__(self):
        if self.ok:
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *exc):
        if self.ok:
            self._stop.set()
            self.t.join()

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                    "samples": len(self.samples)}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples)}


# ----------------------------------------------------------------- the step
def build_step(torch):
    """Operands of one step, drawn on the CPU by the seeded-input module."""
    from roofline_driven_optimisation_gb300 import inputs
    parts = []
    c = inputs.make("bf16_4096")
    parts.append(dict(name="bf16_4096", kernel="gemm_bf16_tc.cu", fn="bf16", M=4096, N=4096, K=4096,
                      alpha=1.0, beta=0.0, A=c.A, B=c.B, C0=None, out=torch.bfloat16,
                      in_bytes=2, out_bytes=2, bound="tensor"))
    c = inputs.make("fp32_4096")
    parts.append(dict(name="fp32_4096", kernel="gemm_f32_simt.cu", fn="f32", M=4096, N=4096, K=4096,
                      alpha=1.5, beta=0.5, A=c.A, B=c.B, C0=c.C0, out=torch.float32,
                      in_bytes=4, out_bytes=4, bound="alu"))
    # one copy of each weight (the M = 16 case's), shared by the three M values;
    # activations and the residual C come from each (M, weight) case
    weights = {w: inputs.make(f"decode_m16_{w}").B for w in WEIGHTS}
    for m in DECODE_MS:
        for w in WEIGHTS:
            c = inputs.make(f"decode_m{m}_{w}")
            parts.append(dict(name=f"decode_m{m}_{w}", kernel="gemm_skinny.cu", fn="bf16", M=m,
                              N=c.spec.N, K=c.spec.K, alpha=1.0, beta=1.0, A=c.A, B=weights[w],
                              C0=c.C0, out=torch.bfloat16, in_bytes=2, out_bytes=2, bound="hbm"))
            del c
    return parts


def launch(g, p, A, B, C, stream):
    M, N, K = p["M"], p["N"], p["K"]
    fn = g.gemm_bf16 if p["fn"] == "bf16" else g.gemm_f32
    fn(M, N, K, p["alpha"], A.data_ptr(), K, B.data_ptr(), N, p["beta"], C.data_ptr(), N, stream)


def run_ours(args):
    import torch
    import torch.distributed as dist
    import roofline_driven_optimisation_gb300 as g
    from roofline_driven_optimisation_gb300 import replicas
    from roofline_driven_optimisation_gb300 import roofline as R

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    g.load()

    parts = build_step(torch)
    for p in parts:
        p["A_d"] = p["A"].to(dev)
        p["B_d"] = p["B"].to(dev)
        p["C_d"] = (p["C0"].to(dev) if p["C0"] is not None
                    else torch.zeros((p["M"], p["N"]), dtype=p["out"], device=dev))
    stream = torch.cuda.current_stream(dev)
    s = stream.cuda_stream
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    # label each part with the kernel source the dispatcher actually runs
    files = {g.PATH_F32_SIMT: "gemm_f32_simt.cu", g.PATH_SKINNY: "gemm_skinny.cu",
             g.PATH_GENERIC: "gemm_generic.cu"}
    for p in parts:
        launch(g, p, p["A_d"], p["B_d"], p["C_d"], s)
        path = g.last_path()
        # kernel launches per call: the FP32 SIMT call adds a second launch
        # when it splits the tiles of its partial last wave
        p["kernels"] = 2 if path == g.PATH_F32_SIMT and g.last_k_split() > 1 else 1
        if path == g.PATH_BF16_TC:
            p["kernel"] = "gemm_bf16_tc2.cu" if g.last_tc_pair() == 2 else "gemm_bf16_tc.cu"
        else:
            p["kernel"] = files[path]
    torch.cuda.synchronize(dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    # the step in three groups, timed at group boundaries only: events between
    # the back-to-back decode launches would break their launch overlap
    groups = [("bf16_4096", [p for p in parts if p["name"] == "bf16_4096"]),
              ("fp32_4096", [p for p in parts if p["name"] == "fp32_4096"]),
              ("decode", [p for p in parts if p["bound"] == "hbm"])]

    def step(evs=None):
        for gi, (_, plist) in enumerate(groups):
            if evs is not None:
                evs[gi][0].record(stream)
            for p in plist:
                launch(g, p, p["A_d"], p["B_d"], p["C_d"], s)
            if evs is not None:
                evs[gi][1].record(stream)

    for _ in range(args.warmup):
        step()
    barrier()
    status, where = g.device_status(s)
    if status != 0:
        raise RuntimeError(f"device status {status} at {where} after warm-up")

    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in groups] for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    with ClockSampler(local) as clocks:
        t0.record(stream)
        for k in range(args.steps):
            step(evs[k])
        t1.record(stream)
        barrier()
    elapsed_ms = t0.elapsed_time(t1)
    status, where = g.device_status(s)
    if status != 0:
        raise RuntimeError(f"device status {status} at {where} in the timed region")
    elapsed_ms = replicas.max_over_ranks(elapsed_ms, dist if world > 1 else None, device=dev)

    # per-group average durations, from events on the launching stream
    pk, src = peaks()
    hbm = pk["hbm_gbs"] * 1e9
    bf16_peak = pk["bf16_tflops"] * 1e12
    sm_max = pk.get("sm_max_mhz", 2070.0)
    fp32_peak = R.fp32_peak(n_sm, sm_max * 1e6)
    part_out = {}
    flops_step = 0
    bytes_by_kernel, time_by_kernel, flops_by_kernel, launches_by_kernel = {}, {}, {}, {}
    for gi, (gname, plist) in enumerate(groups):
        ms = sum(evs[k][gi][0].elapsed_time(evs[k][gi][1]) for k in range(args.steps)) / args.steps
        fl = sum(R.gemm_flops(p["M"], p["N"], p["K"]) for p in plist)
        by = sum(R.gemm_bytes(p["M"], p["N"], p["K"], p["in_bytes"], p["out_bytes"], p["beta"] != 0)
                 for p in plist)
        flops_step += fl
        kern = plist[0]["kernel"]
        bytes_by_kernel[kern] = bytes_by_kernel.get(kern, 0) + by
        flops_by_kernel[kern] = flops_by_kernel.get(kern, 0) + fl
        time_by_kernel[kern] = time_by_kernel.get(kern, 0.0) + ms
        launches_by_kernel[kern] = launches_by_kernel.get(kern, 0) + len(plist)
        ent = {"ms": round(ms, 5), "calls": len(plist), "launches": sum(p["kernels"] for p in plist),
               "tflops": round(fl / (ms * 1e-3) / 1e12, 2),
               "gbs": round(by / (ms * 1e-3) / 1e9, 1), "ai": round(fl / by, 2)}
        bound = plist[0]["bound"]
        if bound == "hbm":
            ent["frac_hbm"] = round(by / (ms * 1e-3) / hbm, 4)
        elif bound == "tensor":
            ent["frac_tensor"] = round(fl / (ms * 1e-3) / bf16_peak, 4)
            ent["frac_tensor_nominal_2250"] = round(fl / (ms * 1e-3) / 2.25e15, 4)
        else:
            ent["frac_fp32"] = round(fl / (ms * 1e-3) / fp32_peak, 4)
        part_out[gname] = ent

    # per-shape decode times, isolated (events around every launch, after the
    # timed region; the weights of the 18 GEMMs are distinct, so L2 is cold).
    # A hold kernel keeps the stream busy while the host enqueues each batch,
    # so no launch waits for the host and every interval is device time.  The
    # same batch times two floors: a read-only pass over each weight's bytes
    # and an empty launch.
    import bench_probe
    bench_probe.build()
    dec = groups[2][1]
    sink = torch.zeros(4, dtype=torch.int32, device=dev)
    iso = {p["name"]: [] for p in dec}
    floor = {p["name"]: [] for p in dec}
    empty = []

    def timed(fn, into):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        into.append((e0, e1))

    for _ in range(5):
        bench_probe.probe_hold(20_000_000, s)
        for p in dec:
            timed(lambda: launch(g, p, p["A_d"], p["B_d"], p["C_d"], s), iso[p["name"]])
        for p in dec:
            timed(lambda: bench_probe.probe_read_stream(p["B_d"].data_ptr(), p["B_d"].numel() * 2,
                                                        sink.data_ptr(), s), floor[p["name"]])
        for _ in range(4):
            timed(lambda: bench_probe.probe_empty(s), empty)
        torch.cuda.synchronize(dev)
    shapes = {}
    for p in dec:
        ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in iso[p["name"]])
        fl_ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in floor[p["name"]])
        by = R.gemm_bytes(p["M"], p["N"], p["K"], 2, 2, True)
        shapes[p["name"]] = {"ms": round(ms, 5), "gbs": round(by / (ms * 1e-3) / 1e9, 1),
                             "frac_hbm": round(by / (ms * 1e-3) / hbm, 4),
                             "read_only_floor_ms": round(fl_ms, 5),
                             "vs_floor": round(fl_ms / ms, 4)}
    shapes["empty_launch_ms"] = round(statistics.median(e0.elapsed_time(e1) for e0, e1 in empty), 5)
    part_out["decode"]["isolated"] = shapes

    dom = max(time_by_kernel, key=time_by_kernel.get)
    dom_parts = [p for p in parts if p["kernel"] == dom]
    launches = launches_by_kernel[dom]
    avg_ms = time_by_kernel[dom] / launches
    bound = dom_parts[0]["bound"]
    if bound == "hbm":
        achieved = bytes_by_kernel[dom] / launches / (avg_ms * 1e-3) / 1e9
        peak, unit, rb = pk["hbm_gbs"], "GB/s", "hbm"
    elif bound == "tensor":
        achieved = flops_by_kernel[dom] / launches / (avg_ms * 1e-3) / 1e12
        peak, unit, rb = pk["bf16_tflops"], "TFLOP/s", "tensor"
    else:
        achieved = flops_by_kernel[dom] / launches / (avg_ms * 1e-3) / 1e12
        peak, unit, rb = fp32_peak / 1e12, "TFLOP/s", "alu"
    tr = traffic_for(dom)
    roofline = {"bound": rb, "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": unit,
                "frac": round(achieved / peak, 4),
                "traffic": (tr if tr is None else int(tr)),
                "kernel": dom, "peak_source": src if rb != "alu" else
                f"{n_sm} SMs x 128 FP32 lanes x 2 FLOP x {sm_max:.0f} MHz",
                # one call of the dominant kernel's GEMM (its launches back to back)
                "launches_per_call": dom_parts[0]["kernels"],
                "algorithmic_bytes_per_call": int(bytes_by_kernel[dom] / launches),
                "algorithmic_flops_per_call": int(flops_by_kernel[dom] / launches)}

    ms_step = elapsed_ms / args.steps
    value = replicas.whole_job_rate(flops_step, world, ms_step * 1e-3) / 1e12
    e2e = run_e2e(args, g, torch, dev, parts, s, world)
    fused_ffn = measure_fused_ffn(g, torch, dev, s, hbm, bf16_peak) if rank == 0 else None
    fma_probe = measure_fp32_fma(g, torch, dev, fp32_peak / 1e12) if rank == 0 else None
    graph = measure_graph_step(g, torch, dev, parts, flops_step) if rank == 0 else None
    configs = measure_configs(g, torch, dev, pk["bf16_tflops"], hbm) if rank == 0 else None
    fp8 = measure_fp8(g, torch, dev, pk["bf16_tflops"]) if rank == 0 else None
    int4_dq = measure_int4_dequant(g, torch, dev, hbm) if rank == 0 else None
    w4 = measure_w4_decode(g, torch, dev, hbm) if rank == 0 else None
    attn = measure_attention(g, torch, dev, pk["bf16_tflops"]) if rank == 0 else None

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16/f32",
        "data": "synthetic",
        "config": {"workload": "bf16 4096^3 + fp32 4096^3 (alpha 1.5, beta 0.5) + decode M{1,4,16} x "
                               "LLaMA-7B weights (qkv,o,gate,up,down,lm), beta 1",
                   "parallelism": f"replicas x{world}",
                   "l2": "no flush: step working set ~0.92 GB > 129 MB L2; each input is touched "
                         "once per step"},
        "roofline": roofline,
        "parts": part_out,
        "graph_step": graph,
        "bf16_configs": configs,
        "fused_ffn_swiglu": fused_ffn,
        "fp32_fma_probe": fma_probe,
        "fp8_gemm": fp8,
        "int4_dequant": int4_dq,
        "w4a16_decode": w4,
        "attention": attn,
        "e2e": e2e,
        "gpu_launches": sum(p["kernels"] for p in parts) * args.steps,
        "clocks": clocks.summary(),
    }
    if rank == 0:
        result["cpu_baseline"] = cpu_baseline(parts, args.cpu_seconds)
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def measure_graph_step(g, torch, dev, parts, flops_step, reps=20):
    """The same step captured once as a CUDA graph (stream capture of the same
    C-ABI calls) and replayed: no host launch work inside the replays."""
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        cs = torch.cuda.current_stream(dev).cuda_stream
        for p in parts:
            launch(g, p, p["A_d"], p["B_d"], p["C_d"], cs)
    for _ in range(3):
        gr.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        gr.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    status, where = g.device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} at {where} in the graph replays")
    ms = e0.elapsed_time(e1) / reps
    return {"ms_per_step": round(ms, 4), "tflops": round(flops_step / (ms * 1e-3) / 1e12, 2),
            "replays": reps}


def run_e2e(args, g, torch, dev, parts, s, world):
    """Same step through the public API with host buffers: every step copies
    its inputs host->device from pinned memory and reads its results back.
    Copies in, GEMMs and copies out run on three streams ordered by events,
    so part i+1's inputs travel while part i computes and part i-1's result
    comes back (a copy into a part's buffers waits for that part's previous
    read-back)."""
    host = []
    h2d = d2h = 0
    for p in parts:
        hA = p["A"].pin_memory()
        hB = p["B"].pin_memory()
        hC0 = p["C0"].pin_memory() if p["C0"] is not None else None
        hC = torch.empty((p["M"], p["N"]), dtype=p["out"]).pin_memory()
        host.append((hA, hB, hC0, hC))
        h2d += hA.numel() * hA.element_size() + hB.numel() * hB.element_size()
        if hC0 is not None:
            h2d += hC0.numel() * hC0.element_size()
        d2h += hC.numel() * hC.element_size()
    comp = torch.cuda.current_stream(dev)
    cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    done_out = [None] * len(parts)

    def step():
        for i, (p, (hA, hB, hC0, hC)) in enumerate(zip(parts, host)):
            with torch.cuda.stream(cin):
                if done_out[i] is not None:
                    cin.wait_event(done_out[i])      # last step's read-back of this part
                p["A_d"].copy_(hA, non_blocking=True)
                p["B_d"].copy_(hB, non_blocking=True)
                if hC0 is not None:
                    p["C_d"].copy_(hC0, non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(cin)
            comp.wait_event(ready)
            launch(g, p, p["A_d"], p["B_d"], p["C_d"], comp.cuda_stream)
            computed = torch.cuda.Event()
            computed.record(comp)
            with torch.cuda.stream(cout):
                cout.wait_event(computed)
                hC.copy_(p["C_d"], non_blocking=True)
                done_out[i] = torch.cuda.Event()
                done_out[i].record(cout)

    def join():
        # the timed region ends when all three streams are done
        for st in (cin, cout):
            ev = torch.cuda.Event()
            ev.record(st)
            comp.wait_event(ev)

    steps = max(1, min(args.steps, 20))
    for _ in range(max(1, args.warmup)):
        step()
    join()
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(comp)
    cin.wait_event(t0)
    cout.wait_event(t0)
    for _ in range(steps):
        step()
    join()
    t1.record(comp)
    torch.cuda.synchronize(dev)
    ms = t0.elapsed_time(t1) / steps
    flops = sum(2 * p["M"] * p["N"] * p["K"] for p in parts)
    return {"value": round(world * flops / (ms * 1e-3) / 1e12, 2), "unit": UNIT,
            "ms_per_step": round(ms, 4), "steps": steps,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "streams": "copies in, GEMMs, copies out on three streams, ordered by events"}


def measure_fp32_fma(g, torch, dev, formula_tflops, iters=16000, reps=3):
    """Measured FP32 FMA rate with scalar and packed (f32x2) FMAs, against
    the SMs x 128 lanes x 2 x clock peak the FP32 roofline uses."""
    import bench_probe
    bench_probe.build()
    stream = torch.cuda.current_stream(dev)
    sink = torch.zeros(1, dtype=torch.float32, device=dev)
    out = {"formula_tflops": round(formula_tflops, 2)}
    for name, packed in (("scalar", False), ("packed_f32x2", True)):
        bench_probe.probe_fp32_fma(packed, iters, sink.data_ptr(), stream.cuda_stream)   # warm-up
        best = 0.0
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            flops = bench_probe.probe_fp32_fma(packed, iters, sink.data_ptr(), stream.cuda_stream)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            best = max(best, flops / (e0.elapsed_time(e1) * 1e-3) / 1e12)
        out[f"{name}_tflops"] = round(best, 2)
        out[f"{name}_frac_of_formula"] = round(best / formula_tflops, 4)
    return out


def measure_configs(g, torch, dev, bf16_peak_tflops, hbm, reps=7):
    """The bf16 workloads the step leaves out, each timed alone: 4096^3 with
    fp32 C, 8192^3 with bf16 and fp32 C (seed 2), and the LLaMA-7B prefill
    GEMMs at M = 2048 tokens (seed 3, bf16 C).  Events around each call, L2
    flushed by a read pass before every call, median of `reps`.  Fraction of
    min(measured bf16 peak, AI x measured HBM bandwidth).  Not part of the
    step."""
    from roofline_driven_optimisation_gb300 import inputs
    from roofline_driven_optimisation_gb300 import roofline as R
    stream = torch.cuda.current_stream(dev)
    flush = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    cases = [("bf16_4096_f32out", "bf16_4096", torch.float32), ("bf16_8192", "bf16_8192", torch.bfloat16),
             ("bf16_8192_f32out", "bf16_8192", torch.float32)]
    cases += [(f"prefill_m2048_{w}", f"prefill_{w}", torch.bfloat16) for w in WEIGHTS]
    out = {"peak_tflops": round(bf16_peak_tflops, 1)}
    made = {}
    for name, wl, odt in cases:
        if wl not in made:
            made.clear()
            c = inputs.make(wl)
            made[wl] = (c.A.to(dev), c.B.to(dev))
        A, B = made[wl]
        M, K = A.shape
        N = B.shape[1]
        C = torch.empty((M, N), dtype=odt, device=dev)
        g.gemm(A, B, C, 1.0, 0.0)
        path, pair, bn = g.last_path(), g.last_tc_pair(), g.last_tile_n()
        evs = []
        for _ in range(reps):
            flush.sum()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.gemm(A, B, C, 1.0, 0.0)
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize(dev)
        ms = statistics.median(a.elapsed_time(b) for a, b in evs)
        fl = R.gemm_flops(M, N, K)
        by = R.gemm_bytes(M, N, K, 2, C.element_size(), False)
        roof = min(bf16_peak_tflops * 1e12, fl / by * hbm)
        out[name] = {"M": M, "N": N, "K": K, "ms": round(ms, 5), "tflops": round(fl / (ms * 1e-3) / 1e12, 1),
                     "frac_roofline": round(fl / (ms * 1e-3) / roof, 4), "ai": round(fl / by, 1),
                     "kernel": g.PATH_NAMES[path] + (f" pair x{pair} BN {bn}" if path == g.PATH_BF16_TC else "")}
        del C
    made.clear()
    status, where = g.device_status(stream.cuda_stream)
    if status != 0:
        raise RuntimeError(f"device status {status} at {where} in the config measurement")
    return out


def measure_fp8(g, torch, dev, bf16_peak_tflops, reps=7):
    """FP8 (E4M3) GEMM, bf16 C, at 4096^3 and 8192^3 against the FP8 dense
    peak taken as the measured bf16 peak x 2 (the nominal FP8 : bf16 ratio,
    4.5 : 2.25 PFLOP/s).  Events around each call, L2 flushed by a read pass
    before every call, median of `reps`.  Not part of the step."""
    from roofline_driven_optimisation_gb300 import inputs
    stream = torch.cuda.current_stream(dev)
    flush = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    peak = 2.0 * bf16_peak_tflops
    out = {"peak_tflops": round(peak, 1), "peak_source": "measured bf16 x 2 (nominal ratio)"}
    for n in (4096, 8192):
        c = inputs.make_fp8(n, n, n, inputs.FP8_E4M3, inputs.FP8_E4M3, seed=7)
        A, B = c.A.to(dev), c.B.to(dev)
        C = torch.empty((n, n), dtype=torch.bfloat16, device=dev)
        g.gemm_fp8_tensors(A, 0, B, 0, C, c.alpha)
        evs = []
        for _ in range(reps):
            flush.sum()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.gemm_fp8_tensors(A, 0, B, 0, C, c.alpha)
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize(dev)
        ms = statistics.median(a.elapsed_time(b) for a, b in evs)
        tf = 2 * n ** 3 / (ms * 1e-3) / 1e12
        out[f"e4m3_{n}"] = {"ms": round(ms, 5), "tflops": round(tf, 1), "frac": round(tf / peak, 4),
                            "frac_nominal_4500": round(tf / 4500.0, 4)}
        del A, B, C
    status, where = g.device_status(stream.cuda_stream)
    if status != 0:
        raise RuntimeError(f"device status {status} at {where} in the FP8 measurement")
    return out


def measure_int4_dequant(g, torch, dev, hbm, reps=7):
    """INT4 dequantisation of a 16384 x 16384 weight (group 128, zero point 8)
    to bf16 and to fp32, in HBM GB/s of algorithmic bytes (codes read once,
    scales once, output written once; more than L2, so no flush).  Not part
    of the step."""
    from roofline_driven_optimisation_gb300 import inputs
    stream = torch.cuda.current_stream(dev)
    n = 16384
    c = inputs.make_int4(n, n, group=128, zero=8, seed=8)
    q, sc = c.q.to(dev), c.scales.to(dev)
    out = {}
    for name, dt in (("bf16_out", torch.bfloat16), ("f32_out", torch.float32)):
        W = torch.empty((n, n), dtype=dt, device=dev)
        g.int4_dequant(q, sc, n, 128, 8, W)
        evs = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.int4_dequant(q, sc, n, 128, 8, W)
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize(dev)
        ms = statistics.median(a.elapsed_time(b) for a, b in evs)
        by = q.numel() + sc.numel() * 2 + W.numel() * W.element_size()
        out[name] = {"ms": round(ms, 4), "gbs": round(by / (ms * 1e-3) / 1e9, 1),
                     "frac_hbm": round(by / (ms * 1e-3) / hbm, 4), "bytes": int(by)}
        del W
    return out


def measure_w4_decode(g, torch, dev, hbm, iters=20):
    """INT4-weight decode GEMMs (group 128, zero point 8, bf16 X and C, beta 1)
    on the six LLaMA-7B weight shapes at M = 1, 4, 16: the 18 calls back to
    back, events around the run, median of `iters`.  Algorithmic bytes: codes
    (K*N/2) and scales once, X, C read and written.  Not part of the step."""
    from roofline_driven_optimisation_gb300 import inputs
    stream = torch.cuda.current_stream(dev)
    s = stream.cuda_stream
    weights = {}
    for w in WEIGHTS:
        K, N = inputs.LLAMA7B_WEIGHTS[w]
        c = inputs.make_int4(K, N, group=128, zero=8, seed=20 + len(weights))
        weights[w] = (K, N, g.int4_repack(c.q.to(dev), K, N), c.scales.to(dev))
    gen = torch.Generator().manual_seed(21)
    calls, by = [], 0
    for m in DECODE_MS:
        for w in WEIGHTS:
            K, N, qk, sc = weights[w]
            X = torch.randn((m, K), generator=gen).to(torch.bfloat16).to(dev)
            C = torch.randn((m, N), generator=gen).to(torch.bfloat16).to(dev)
            calls.append((m, N, K, X, qk, sc, C))
            by += K * N // 2 + sc.numel() * 2 + 2 * m * K + 4 * m * N

    def run():
        for m, N, K, X, qk, sc, C in calls:
            g.gemm_w4a16(m, N, K, 1.0, X.data_ptr(), K, qk.data_ptr(), sc.data_ptr(), N, 128, 8, 1.0,
                         C.data_ptr(), N, s)

    for _ in range(3):
        run()
    evs = []
    for _ in range(iters):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize(dev)
    status, where = g.device_status(s)
    if status != 0:
        raise RuntimeError(f"device status {status} at {where} in the INT4 decode measurement")
    ms = statistics.median(a.elapsed_time(b) for a, b in evs)
    return {"launches": len(calls), "ms": round(ms, 5), "bytes": int(by),
            "gbs": round(by / (ms * 1e-3) / 1e9, 1), "frac_hbm": round(by / (ms * 1e-3) / hbm, 4),
            "flops": int(sum(2 * m * N * K for m, N, K, *_ in calls))}


def measure_attention(g, torch, dev, bf16_peak_tflops, reps=7, batch=8):
    """Attention forward: one LLaMA-7B layer's prefill (32 heads of 128, 2048
    tokens, causal) and a 4096-token non-causal case.  FLOPs = 4 * D * (the
    query-key pairs a query sees), i.e. both products; against the measured
    bf16 peak.  Events around each call, median of `reps` (each call pays a
    launch from an idle stream); and `back_to_back`: `batch` calls queued
    behind a hold kernel with events around the batch, per call (as the
    layers of a model's forward pass run).  Not part of the step."""
    import bench_probe
    from roofline_driven_optimisation_gb300 import inputs
    bench_probe.build()
    stream = torch.cuda.current_stream(dev)
    out = {"peak_tflops": round(bf16_peak_tflops, 1)}
    for name, S, causal in (("llama7b_prefill_2048_causal", 2048, True), ("s4096_noncausal", 4096, False)):
        c = inputs.make_attention(B=1, Hq=32, Hkv=32, Sq=S, Sk=S, D=128, seed=9)
        Q, K, V = c.Q.to(dev), c.K.to(dev), c.V.to(dev)
        O = torch.empty_like(Q)
        g.attention(Q, K, V, O, causal=causal)
        evs = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.attention(Q, K, V, O, causal=causal)
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize(dev)
        ms = statistics.median(a.elapsed_time(b) for a, b in evs)
        bb = []
        for _ in range(3):
            bench_probe.probe_hold(5_000_000, stream.cuda_stream)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(batch):
                g.attention(Q, K, V, O, causal=causal)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            bb.append(e0.elapsed_time(e1) / batch)
        ms_bb = min(bb)
        pairs = S * (S + 1) // 2 if causal else S * S
        flops = 4 * 32 * 128 * pairs
        tf = flops / (ms * 1e-3) / 1e12
        tf_bb = flops / (ms_bb * 1e-3) / 1e12
        out[name] = {"ms": round(ms, 4), "tflops": round(tf, 1), "frac": round(tf / bf16_peak_tflops, 4),
                     "back_to_back": {"ms": round(ms_bb, 4), "tflops": round(tf_bb, 1),
                                      "frac": round(tf_bb / bf16_peak_tflops, 4), "calls": batch}}
        del Q, K, V, O
    status, where = g.device_status(stream.cuda_stream)
    if status != 0:
        raise RuntimeError(f"device status {status} at {where} in the attention measurement")
    return out


def measure_fused_ffn(g, torch, dev, s, hbm, bf16_peak, reps=7):
    """The fused FFN gate/up pair, C = silu(X Wg) * (X Wu) with the LLaMA-7B
    shapes (K = 4096, N = 11008), against the two plain GEMMs it replaces
    (which still leave the elementwise pass undone).  Timed with events
    around each call, L2 flushed before every call by reading a buffer twice
    its size (a read leaves only clean lines, so no write-back lands in the
    timed call), median of `reps`.  Decode sizes are also timed back to back
    over three distinct weight pairs (30 calls, events around the run), as a
    decode loop launches them.  Not part of the step."""
    from roofline_driven_optimisation_gb300 import inputs
    stream = torch.cuda.current_stream(dev)
    flush = torch.ones(64 << 20, dtype=torch.float32, device=dev)   # 256 MB, 2x the L2
    out = {}
    for M in (1, 4, 16, 2048):
        c = inputs.make_swiglu(M)
        A, Bg, Bu = c.A.to(dev), c.Bgate.to(dev), c.Bup.to(dev)
        K, N = A.shape[1], Bg.shape[1]
        C, G, U = (torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(3))

        def fused():
            g.gemm_bf16_swiglu(M, N, K, A.data_ptr(), K, Bg.data_ptr(), Bu.data_ptr(), N,
                               C.data_ptr(), N, s)

        def two_gemms():
            g.gemm_bf16(M, N, K, 1.0, A.data_ptr(), K, Bg.data_ptr(), N, 0.0, G.data_ptr(), N, s)
            g.gemm_bf16(M, N, K, 1.0, A.data_ptr(), K, Bu.data_ptr(), N, 0.0, U.data_ptr(), N, s)

        times = {"fused": [], "two": []}
        for fn in (fused, two_gemms):
            fn()
        for _ in range(reps):
            for key, fn in (("fused", fused), ("two", two_gemms)):
                flush.sum()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                times[key].append((e0, e1))
        torch.cuda.synchronize(dev)
        status, where = g.device_status(s)
        if status != 0:
            raise RuntimeError(f"device status {status} at {where} in the fused FFN measurement")
        ms = {k: statistics.median(a.elapsed_time(b) for a, b in v) for k, v in times.items()}
        flops = 2 * 2 * M * N * K
        by = 2 * M * K + 2 * 2 * K * N + 2 * M * N
        ent = {"M": M, "N": N, "K": K, "fused_ms": round(ms["fused"], 5),
               "two_gemms_ms": round(ms["two"], 5),
               "speedup_vs_two_gemms": round(ms["two"] / ms["fused"], 3),
               "fused_gbs": round(by / (ms["fused"] * 1e-3) / 1e9, 1),
               "fused_tflops": round(flops / (ms["fused"] * 1e-3) / 1e12, 2)}
        if M <= 16:
            ent["frac_hbm"] = round(by / (ms["fused"] * 1e-3) / hbm, 4)
            # back to back over three weight pairs (1.1 GB, beyond L2)
            gen = torch.Generator(device=dev)
            gen.manual_seed(105)
            copies = [(Bg, Bu)] + [tuple((torch.randn(w.shape, generator=gen, device=dev) * 0.02)
                                         .to(w.dtype) for w in (Bg, Bu)) for _ in range(2)]
            for wg, wu in copies:
                g.gemm_bf16_swiglu(M, N, K, A.data_ptr(), K, wg.data_ptr(), wu.data_ptr(), N,
                                   C.data_ptr(), N, s)
            flush.sum()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(30):
                wg, wu = copies[i % 3]
                g.gemm_bf16_swiglu(M, N, K, A.data_ptr(), K, wg.data_ptr(), wu.data_ptr(), N,
                                   C.data_ptr(), N, s)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            b2b = e0.elapsed_time(e1) / 30
            ent["back_to_back_ms"] = round(b2b, 5)
            ent["back_to_back_gbs"] = round(by / (b2b * 1e-3) / 1e9, 1)
            ent["back_to_back_frac_hbm"] = round(by / (b2b * 1e-3) / hbm, 4)
            del copies
        else:
            ent["frac_tensor"] = round(flops / (ms["fused"] * 1e-3) / bf16_peak, 4)
        out[f"m{M}"] = ent
        del A, Bg, Bu, C, G, U
    return out


# ----------------------------------------------------------------- CPU oracle
def oracle_sample_step(parts, frac, threads):
    """One bounded sample of the step on the CPU oracle: the first rows of each
    square GEMM and the first columns of each decode GEMM. Returns FLOPs."""
    import oracle
    flops = 0
    for p in parts:
        M, N, K = p["M"], p["N"], p["K"]
        if p["bound"] == "hbm":
            n = max(1, int(N * frac))
            C0 = p["C0"][:, :n] if p["C0"] is not None else None
            oracle.gemm(p["A"], p["B"][:, :n], p["alpha"], p["beta"], C0, threads)
            flops += 2 * M * n * K
        else:
            r = max(1, int(M * frac))
            C0 = p["C0"][:r] if p["C0"] is not None else None
            oracle.gemm(p["A"][:r], p["B"], p["alpha"], p["beta"], C0, threads)
            flops += 2 * r * N * K
    return flops


def _calibrate(parts, threads, target_s):
    """Row fraction whose oracle sample takes about target_s seconds (two
    rounds: the first run is dominated by fixed per-call costs)."""
    frac = 1.0 / 256
    for _ in range(2):
        t = time.perf_counter()
        oracle_sample_step(parts, frac, threads)
        dt = max(time.perf_counter() - t, 1e-3)
        frac = min(1.0, frac * target_s / dt) if _ == 1 else min(1.0, frac * min(8.0, target_s / dt))
    return frac


def cpu_baseline(parts, target_s=15.0):
    import oracle
    threads = oracle.default_threads()
    frac = _calibrate(parts, threads, target_s)
    t = time.perf_counter()
    fl = oracle_sample_step(parts, frac, threads)
    dt = time.perf_counter() - t
    # the smallest workload (fp32 256^3, alpha 1, beta 0) in full, on one core and on all
    from roofline_driven_optimisation_gb300 import inputs
    c = inputs.make("fp32_256")
    small = {}
    for label, th in (("one_core", 1), ("all_cores", threads)):
        t1 = time.perf_counter()
        oracle.gemm(c.A, c.B, 1.0, 0.0, None, th)
        small[label + "_gflops"] = round(2 * 256 ** 3 / (time.perf_counter() - t1) / 1e9, 3)
    return {"value": round(fl / dt / 1e12, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"fp64 oracle on the first {frac:.4%} of the rows of the two 4096^3 GEMMs and of "
                      f"the columns of the 18 decode GEMMs ({fl / 1e9:.1f} GFLOP, {dt:.1f} s)",
            "fp32_256_full": small}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch
    import oracle
    parts = build_step(torch)
    threads = oracle.default_threads()
    budget = float(os.environ.get("BENCH_REFERENCE_SECONDS", "150"))
    frac = _calibrate(parts, threads, budget / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample_step(parts, frac, threads)
    t = time.perf_counter()
    fl = 0
    for _ in range(args.steps):
        fl += oracle_sample_step(parts, frac, threads)
    dt = time.perf_counter() - t
    value = fl / dt / 1e12
    sample = (f"each step: fp64 oracle on the first {frac:.4%} of the rows of the two 4096^3 GEMMs "
              f"and of the columns of the 18 decode GEMMs ({fl / args.steps / 1e9:.2f} GFLOP)")
    print(json.dumps({
        "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": "bf16 4096^3 + fp32 4096^3 (alpha 1.5, beta 0.5) + decode M{1,4,16} x "
                               "LLaMA-7B weights (qkv,o,gate,up,down,lm), beta 1",
                   "parallelism": "CPU oracle, rank 0 only"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ---------------------------------------------------------------- profiling cases
# ``python bench.py --case <workload>`` (or --swiglu/--fp8/--attention/--int4/--w4)
# runs one workload through the C ABI a few times and prints the kernel family
# and the CUDA-event time of each call: the commands the ncu summaries under
# profiles/ are taken with.  Workload names are those of
# ``roofline_driven_optimisation_gb300.inputs``.

CASE_ARGS = ("case", "swiglu", "fp8", "attention", "int4", "w4")


def run_case(a):
    import torch
    import roofline_driven_optimisation_gb300 as g
    from roofline_driven_optimisation_gb300 import inputs

    g.load()
    if a.tc_pair:
        g.force_tc_pair(a.tc_pair)
    if a.tile_n:
        g.force_tile_n(a.tile_n)
    if a.swiglu is not None:
        return case_swiglu(g, torch, inputs, a)
    if a.fp8 is not None:
        return case_fp8(g, torch, inputs, a)
    if a.attention is not None:
        return case_attention(g, torch, inputs, a)
    if a.int4 is not None:
        return case_int4(g, torch, inputs, a)
    if a.w4 is not None:
        return case_w4(g, torch, inputs, a)
    c = inputs.make(a.case, M=a.M, N=a.N, K=a.K)
    sp = c.spec
    if sp.in_dtype == "f32":
        out = torch.float32
    else:
        out = torch.float32 if a.out == "f32" else torch.bfloat16
    A, B = c.A.cuda(), c.B.cuda()
    C = c.C0.to(out).cuda() if c.C0 is not None else torch.zeros((sp.M, sp.N), dtype=out, device="cuda")
    for i in range(a.reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.gemm(A, B, C, sp.alpha, sp.beta)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        print(f"{a.case} M={sp.M} N={sp.N} K={sp.K} path={g.PATH_NAMES[g.last_path()]} "
              f"call {i}: {ms:.4f} ms, {2 * sp.M * sp.N * sp.K / ms / 1e9:.1f} TFLOP/s")
    status, where = g.device_status()
    if status != 0:
        raise SystemExit(f"device status {status} at site {where}")


def case_swiglu(g, torch, inputs, a):
    kw = {k: v for k, v in (("N", a.N), ("K", a.K)) if v is not None}
    c = inputs.make_swiglu(a.swiglu, **kw)
    A, Bg, Bu = c.A.cuda(), c.Bgate.cuda(), c.Bup.cuda()
    M, K = A.shape
    N = Bg.shape[1]
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    for i in range(a.reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.swiglu(A, Bg, Bu, C)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        by = 2 * M * K + 4 * K * N + 2 * M * N
        print(f"swiglu M={M} N={N} K={K} path={g.PATH_NAMES[g.last_path()]} call {i}: {ms:.4f} ms, "
              f"{4 * M * N * K / ms / 1e9:.1f} TFLOP/s, {by / ms / 1e6:.1f} GB/s")
    status, where = g.device_status()
    if status != 0:
        raise SystemExit(f"device status {status} at site {where}")


def case_fp8(g, torch, inputs, a):
    n = a.fp8
    c = inputs.make_fp8(n, n, n, inputs.FP8_E4M3, inputs.FP8_E4M3, seed=7)
    A, B = c.A.cuda(), c.B.cuda()
    C = torch.empty((n, n), dtype=torch.bfloat16, device="cuda")
    for i in range(a.reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.gemm_fp8_tensors(A, 0, B, 0, C, c.alpha)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        print(f"fp8 e4m3 n={n} path={g.PATH_NAMES[g.last_path()]} call {i}: {ms:.4f} ms, "
              f"{2 * n ** 3 / ms / 1e9:.1f} TFLOP/s")
    status, where = g.device_status()
    if status != 0:
        raise SystemExit(f"device status {status} at site {where}")


def _case_status(g):
    status, where = g.device_status()
    if status != 0:
        raise SystemExit(f"device status {status} at site {where}")


def _case_timed(torch, fn):
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def case_attention(g, torch, inputs, a):
    S = a.attention
    causal = not a.noncausal
    c = inputs.make_attention(B=1, Hq=32, Hkv=32, Sq=S, Sk=S, D=128, seed=9)
    Q, K, V = c.Q.cuda(), c.K.cuda(), c.V.cuda()
    O = torch.empty_like(Q)
    pairs = S * (S + 1) // 2 if causal else S * S
    for i in range(a.reps):
        ms = _case_timed(torch, lambda: g.attention(Q, K, V, O, causal=causal))
        print(f"attention S={S} causal={causal} path={g.PATH_NAMES[g.last_path()]} call {i}: {ms:.4f} ms, "
              f"{4 * 32 * 128 * pairs / ms / 1e9:.1f} TFLOP/s")
    _case_status(g)


def case_int4(g, torch, inputs, a):
    n = a.int4
    c = inputs.make_int4(n, n, group=128, zero=8, seed=8)
    q, sc = c.q.cuda(), c.scales.cuda()
    out = torch.float32 if a.out == "f32" else torch.bfloat16
    W = torch.empty((n, n), dtype=out, device="cuda")
    by = q.numel() + sc.numel() * 2 + W.numel() * W.element_size()
    for i in range(a.reps):
        ms = _case_timed(torch, lambda: g.int4_dequant(q, sc, n, 128, 8, W))
        print(f"int4 dequant n={n} out={a.out} path={g.PATH_NAMES[g.last_path()]} call {i}: {ms:.4f} ms, "
              f"{by / ms / 1e6:.1f} GB/s")
    _case_status(g)


def case_w4(g, torch, inputs, a):
    M, K, N = a.w4, a.K or 4096, a.N or 32000
    c = inputs.make_int4(K, N, group=128, zero=8, seed=1)
    qk = g.int4_repack(c.q.cuda(), K, N)
    X = torch.randn((M, K), generator=torch.Generator().manual_seed(4)).to(torch.bfloat16).cuda()
    C = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    sc = c.scales.cuda()
    by = K * N // 2 + sc.numel() * 2 + 2 * M * K + 2 * M * N
    for i in range(a.reps):
        ms = _case_timed(torch, lambda: g.w4a16(X, qk, sc, 128, 8, C))
        print(f"w4a16 M={M} N={N} K={K} path={g.PATH_NAMES[g.last_path()]} call {i}: {ms:.4f} ms, "
              f"{by / ms / 1e6:.1f} GB/s")
    _case_status(g)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    # profiling cases (one workload, a few calls; no JSON line)
    ap.add_argument("--case", help="a workload of roofline_driven_optimisation_gb300.inputs")
    ap.add_argument("--swiglu", type=int, metavar="M",
                    help="fused silu(X Wg) * (X Wu) with M rows and the LLaMA-7B gate/up shapes")
    ap.add_argument("--fp8", type=int, metavar="n", help="E4M3 GEMM of size n^3, bf16 C")
    ap.add_argument("--attention", type=int, metavar="S", help="causal attention, 32 heads of 128")
    ap.add_argument("--noncausal", action="store_true", help="attention without the causal mask")
    ap.add_argument("--int4", type=int, metavar="n", help="INT4 dequantisation of an n x n weight (group 128)")
    ap.add_argument("--w4", type=int, metavar="M",
                    help="INT4-weight decode GEMM with M rows (K 4096, N 32000 unless given; group 128)")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--out", default="auto", choices=["auto", "bf16", "f32"])
    ap.add_argument("--tc-pair", type=int, choices=[1, 2],
                    help="pin the tensor-core kernel to single CTAs (1) or CTA pairs (2)")
    ap.add_argument("--tile-n", type=int, help="pin the C tile width (gemm_force_tile_n)")
    ap.add_argument("--M", type=int)
    ap.add_argument("--N", type=int)
    ap.add_argument("--K", type=int)
    args = ap.parse_args()
    n_case = sum(getattr(args, k) is not None for k in CASE_ARGS)
    if n_case > 1:
        ap.error("give at most one of --case, --swiglu, --fp8, --attention, --int4 and --w4")
    if n_case == 1:
        run_case(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
