#!/usr/bin/env python3
"""Benchmark of the fp8 training Linear (libfp8lin) on GB300.

One step = one forward + backward of the 4096->4096 Linear at M = 65536
tokens with tensorwise dynamic scaling: amax, scale, e4m3/e5m2 casts with
transposed copies, and the three FP8 GEMMs (y = x W^T, dX = dY W,
dW = dY^T x).  The workload is the largest row of the single-linear table of
"Integrate float8nocompile, an experimental feature for high performance"
(pytorch/torchtitan PR 778), with inputs that exceed L2 (x and dY are
512 MiB each), so no L2 flush is needed between steps.

Prints ONE JSON line: value = TFLOP/s of the whole job (6 M N K per step),
plus the GEMM kernel's roofline (tensor pipe vs measured peak), the cast
kernel's HBM roofline, an end-to-end figure through the host-buffer API,
the oracle timed on the host cores, SM clocks sampled during the timed
region, and a sweep of the other workloads (M = 16 / 256 / 4096, GPT-1.5B
block Linears with delayed scaling, Llama-3-8B FFN Linears, cast-only
bandwidth).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
  python -m torch.distributed.run --nproc-per-node N bench.py --gpus N ...

With N > 1 every rank runs an independent replica on its own GPU (the path
has no exchange step); value is the sum over ranks, time the max over ranks.
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

METRIC = "FP8 Linear fwd+bwd µs & TFLOP/s (vs FP8 peak); amax+cast GB/s vs HBM"
HEADLINE = "linear4096_m65536"
L2_BYTES = 129 * 1024 * 1024
FP8_OVER_BF16 = 2.0      # nominal dense fp8 / bf16 tensor rate (4.5 / 2.25 PFLOP/s)


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--full-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--workload", default=HEADLINE)
    return ap.parse_args(argv)


# ------------------------------------------------------------------ helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def device_code_sha(kernel: str) -> str:
    """sha256[:16] of a kernel's device code: its own header and the PTX
    helpers it inlines (the host-side launchers live in other files)."""
    import hashlib
    csrc = os.path.join(ROOT, "quantised_gemm_gb300", "csrc")
    h = hashlib.sha256()
    for name in ({"gemm": "gemm_kernels.cuh", "cast": "cast_kernels.cuh"}[kernel], "ptx.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic(kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current source of the kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = device_code_sha(kernel)
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line.startswith("{"):
                rec = json.loads(line)
                if rec.get("kernel") == kernel and rec.get("src_sha") == sha:
                    return rec
    return None


class ClockSampler:
    """nvidia-smi clock / throttle samples every 100 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), smax=float(f[2]),
                                 power=float(f[3]) if f[3] not in ("[N/A]", "N/A") else None,
                                 hw=f[5], hwt=f[6], swt=f[7], swp=f[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        loaded = [r for r in rows if r["power"] is None or r["power"] > 300] or rows
        reasons = set()
        for r in loaded:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded),
                "sm_max_mhz": max(r["smax"] for r in rows), "reasons": sorted(reasons),
                "samples": len(loaded)}


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(torch, value, world, device):
    """The largest `value` over all ranks (one process per GPU): the whole
    job's step time is the slowest rank's."""
    if world <= 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flop_per_rank_step, ms_step, world):
    """Throughput of all ranks together: every rank does the same step (the
    replicas of a weak-scaling run), the job takes the slowest rank's time."""
    return world * flop_per_rank_step / (ms_step * 1e-3) / 1e12


# ------------------------------------------------------------------ native arm

def make_inputs(name, idx=0, step=0):
    import synth_inputs as si
    return si.workload_inputs(name, idx, step=step)


def to_dev(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def time_region(fn, steps, flush=None):
    """Device time (ms) of `steps` calls of fn on the current stream.  With a
    flush function, each step is timed alone and the flush runs between."""
    import torch
    stream = torch.cuda.current_stream()
    if flush is None:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1)
    evs = []
    for _ in range(steps):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        evs.append((a, b))
    evs[-1][1].synchronize()
    return sum(a.elapsed_time(b) for a, b in evs)


def graphed(torch, fn):
    """Capture fn (already warmed up) into a CUDA graph; returns its replay."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    with torch.cuda.graph(g):
        fn()
    for _ in range(2):
        g.replay()
    return g.replay


def linear_sweep_entry(q, torch, dev, name, steps, warmup, flush, use_graph=True,
                       cache_weight=False):
    """fwd+bwd time of every Linear of a workload (sum over its Linears).
    cache_weight: W is cast once and reused by every step, as over the
    micro-batches of one optimizer step (not the full step of the headline)."""
    import synth_inputs as si
    wl = si.WORKLOADS[name]
    delayed = wl.get("delayed", False)
    total_ms, total_flop = 0.0, 0.0
    for idx, (M, K, N) in enumerate(wl["shapes"]):
        x, w, dy = make_inputs(name, idx)
        xd, wd, dyd = to_dev(x, dev), to_dev(w, dev), to_dev(dy, dev)
        del x, w, dy
        lin = q.Fp8Linear(M, K, N, scaling="delayed" if delayed else "dynamic",
                          history_len=wl.get("history_len", 16), cache_weight=cache_weight,
                          device=dev)

        def step():
            lin.forward(xd, wd)
            lin.backward(dyd)
            lin.sync_scales()

        for _ in range(warmup):
            step()
        fn = graphed(torch, step) if use_graph else step
        torch.cuda.synchronize()
        ms = time_region(fn, steps, flush)
        q.check(lin.ws)
        total_ms += ms / steps
        total_flop += 6.0 * M * N * K
        del lin, xd, wd, dyd
        torch.cuda.empty_cache()
    return {"workload": name + (" (W cast once, reused: micro-batches of one optimizer step)"
                                if cache_weight else ""),
            "us_per_fwd_bwd": round(total_ms * 1e3, 2),
            "tflops": round(total_flop / (total_ms * 1e-3) / 1e12, 1),
            "scaling": "delayed" if delayed else "dynamic",
            "l2": "flushed between steps" if flush else "inputs larger than L2",
            "cuda_graph": use_graph}


def library_gemm_entry(q, torch, dev, M, N, K, fmt_a, rounds=3, iters=10):
    """The FP8 GEMM of this library against cuBLASLt's (torch._scaled_mm,
    tensorwise scales) on the same operands: D[M,N] = A[M,K] B[N,K]^T, bf16
    out.  Both read operands larger than L2.  The two alternate ABBA over
    `rounds` rounds so clock drift under the power cap favours neither; the
    medians are reported, with the largest |difference| of the two outputs
    (the accumulation order may differ)."""
    import statistics
    fp8 = {0: torch.float8_e4m3fn, 1: torch.float8_e5m2}
    g = torch.Generator(device=dev).manual_seed(7)
    a = (torch.randn(M, K, device=dev, generator=g) * 4).to(fp8[fmt_a])
    b = (torch.randn(N, K, device=dev, generator=g) * 4).to(torch.float8_e4m3fn)
    one = torch.ones((), device=dev)
    inv = torch.ones(1, device=dev)
    d = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ws = q.Workspace()

    def lib():
        return torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)

    def ours():
        q.gemm(a.view(torch.uint8), b.view(torch.uint8), fmt_a, 0, inv, inv, d, ws)

    try:
        ref = lib()
    except Exception as e:  # a torch build without FP8 matmul for this GPU
        return {"shape": [M, N, K], "unavailable": repr(e)[:200]}
    ours()
    torch.cuda.synchronize()
    q.check(ws)
    diff = (ref.float() - d.float()).abs().max().item()
    del ref
    s = torch.cuda.current_stream()

    def timed(fn):
        fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(iters):
            fn()
        e1.record(s)
        e1.synchronize()
        return e0.elapsed_time(e1) / iters

    tl, to = [], []
    for _ in range(rounds):
        tl.append(timed(lib))
        to.append(timed(ours))
        to.append(timed(ours))
        tl.append(timed(lib))
    fl = 2.0 * M * N * K
    ml, mo = statistics.median(tl), statistics.median(to)
    return {"shape": [M, N, K], "a": "e4m3" if fmt_a == 0 else "e5m2", "b": "e4m3",
            "cublaslt_ms": round(ml, 4), "cublaslt_tflops": round(fl / (ml * 1e-3) / 1e12, 1),
            "ours_ms": round(mo, 4), "ours_tflops": round(fl / (mo * 1e-3) / 1e12, 1),
            "ours_over_cublaslt": round(ml / mo, 3), "max_abs_diff": diff,
            "ours_kernel": q.gemm_describe(M, N, K)}


def chain_sweep_entry(q, torch, dev, name, steps, warmup, flush, rounds=3):
    """Two Linears of a workload's shape in a chain (the second consumes the
    first's y, the first's grad_output is the second's dX), fwd+bwd of both,
    with the amax of y and dX taken in the GEMM epilogues (link_linears: those
    two casts read their tensor once) and with separate amax passes.  The two
    variants alternate over `rounds` rounds (median reported), so clock drift
    under the power cap does not favour either; a profiled pass of each gives
    its time per kernel kind."""
    import statistics
    import synth_inputs as si
    M, K, N = si.WORKLOADS[name]["shapes"][0]
    assert K == N, "a chain of square Linears"
    x, w, dy = make_inputs(name, 0)
    xd, wd, dyd = to_dev(x, dev), to_dev(w, dev), to_dev(dy, dev)
    del x, w, dy
    variants = {}
    for linked in (False, True):
        l1, l2 = q.Fp8Linear(M, K, N, device=dev), q.Fp8Linear(M, N, N, device=dev)
        if linked:
            q.link_linears(l1, l2)

        def step(l1=l1, l2=l2):
            l1.forward(xd, wd)
            l2.forward(l1.y, wd)
            l2.backward(dyd)
            l1.backward(l2.dx)

        for _ in range(warmup):
            step()
        q.profile_enable(True)
        for _ in range(2):
            step()
        prof = q.profile_collect()
        q.profile_enable(False)
        variants["fused_amax" if linked else "separate_amax"] = {
            "step": step, "graph": graphed(torch, step), "lins": (l1, l2), "ms": [],
            "kernel_us_per_step": {k: round(v[0] * 1e3 / 2, 1) for k, v in prof.items()
                                   if v[1] > 0}}
    torch.cuda.synchronize()
    for _ in range(rounds):
        for v in variants.values():
            v["ms"].append(time_region(v["graph"], steps, flush) / steps)
    res = {"workload": "2 x %s chained" % name, "l2": "flushed between steps" if flush else
           "inputs larger than L2", "cuda_graph": True, "rounds": rounds}
    for key, v in variants.items():
        for lin in v["lins"]:
            q.check(lin.ws)
        ms = statistics.median(v["ms"])
        res[key] = {"us_per_fwd_bwd": round(ms * 1e3, 2),
                    "tflops": round(2 * 6.0 * M * N * K / (ms * 1e-3) / 1e12, 1),
                    "kernel_us_per_step": v["kernel_us_per_step"]}
    res["saved_us"] = round(res["separate_amax"]["us_per_fwd_bwd"] -
                            res["fused_amax"]["us_per_fwd_bwd"], 2)
    del variants, xd, wd, dyd
    torch.cuda.empty_cache()
    return res


def cast_sweep(q, torch, dev, peaks, full):
    """amax + scale + cast (+T) of [R, 4096] / [4096, R] tensors: GB/s of the
    algorithmic bytes (2 B read + 1 B per fp8 copy) and fraction of HBM."""
    import synth_inputs as si
    sizes = [1 << 20, 1 << 22, 1 << 24, 1 << 26, 1 << 28, 1 << 30] if full else \
        [1 << 20, 1 << 24, 1 << 28]
    fmts = [q.E4M3, q.E5M2] if full else [q.E4M3]
    shapes = ["rows", "cols"] if full else ["rows"]
    ws = q.Workspace(device=dev)
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    out = []
    for n in sizes:
        for shp in shapes:
            R = n // 4096
            rows, cols = (R, 4096) if shp == "rows" else (4096, R)
            x = si.normal_bf16((rows, cols), 1.0, 0, 1)
            xd = to_dev(x, dev)
            del x
            o = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
            ot = torch.empty((cols, rows), dtype=torch.uint8, device=dev)
            for fmt in fmts:
                for trans in (True, False):
                    for algo in (q.AMAX_ATOMIC, q.AMAX_REDUCTION, q.AMAX_SINGLE_PASS):
                        if algo == q.AMAX_SINGLE_PASS and n > q.single_pass_max_elems():
                            continue
                        if algo == q.AMAX_REDUCTION and not full:
                            continue
                        st = q.ScalingState(fmt, q.DYNAMIC, amax_algo=algo, device=dev)
                        call = lambda: q.cast_dynamic(xd, st, o, ot if trans else None, ws)  # noqa
                        for _ in range(3):
                            call()
                        fn = graphed(torch, call)
                        flush = (lambda: flush_buf.zero_()) if n * 2 < 2 * L2_BYTES else None
                        steps = 20 if n >= (1 << 28) else 50
                        torch.cuda.synchronize()
                        ms = time_region(fn, steps, flush) / steps
                        q.check(ws)
                        alg_bytes = n * (2 + 1 + (1 if trans else 0))
                        gbs = alg_bytes / (ms * 1e-3) / 1e9
                        out.append({"elems": n, "shape": [rows, cols], "cuda_graph": True,
                                    "fmt": "e4m3" if fmt == q.E4M3 else "e5m2",
                                    "transpose": trans,
                                    "amax": {0: "atomic", 1: "reduction", 2: "single_pass"}[algo],
                                    "us": round(ms * 1e3, 2), "gbs": round(gbs, 1),
                                    "frac_hbm": round(gbs / peaks["hbm_gbs"], 3)})
            del xd, o, ot
            torch.cuda.empty_cache()
    return out


def cpu_baseline_sample(name, budget_s=12.0):
    """The oracle, as it stands, on host cores: fwd+bwd of the workload's
    Linear on its first Ms tokens (doubling Ms until the budget is used).
    Returns (TFLOP/s, description, threads)."""
    import oracle
    import synth_inputs as si
    oracle.build()
    wl = si.WORKLOADS[name]
    M, K, N = wl["shapes"][0]
    w = si.weight(K, N, w_init=wl["w_init"], w_std=wl.get("w_std", 0.02))
    Ms, spent, flop, elapsed = 64, 0.0, 0.0, 0.0
    while True:
        x = si.normal_bf16((Ms, K), 1.0, 0, si.STREAM_X)
        dy = si.normal_bf16((Ms, N), 1e-3, 0, si.STREAM_DY)
        t0 = time.perf_counter()
        sx = oracle.scale_dynamic(oracle.amax(x), oracle.E4M3)[0]
        sw = oracle.scale_dynamic(oracle.amax(w), oracle.E4M3)[0]
        sd = oracle.scale_dynamic(oracle.amax(dy), oracle.E5M2)[0]
        oracle.linear_fwd_bwd(x, w, dy, sx, sw, sd)
        dt = time.perf_counter() - t0
        spent += dt
        flop, elapsed = 6.0 * Ms * N * K, dt
        if spent > budget_s or Ms >= M or dt > budget_s / 3:
            break
        Ms *= 2
    desc = ("oracle fwd+bwd (C casts + numpy fp64 GEMMs) of the %dx%d Linear on the first %d "
            "of %d tokens, %.2f s" % (K, N, Ms, M, elapsed))
    return flop / elapsed / 1e12, desc, oracle.num_threads()


def end_to_end(q, lin, x, w, dy, M, K, N, world, flop_step, steps):
    """The same step through the host-buffer API (Fp8Linear.step_host):
    pinned host inputs copied in and y, dX, dW copied out every step."""
    import torch
    hx = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
    hw = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16).pin_memory()
    hdy = torch.from_numpy(dy.view(np.int16)).view(torch.bfloat16).pin_memory()
    hy = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    hdx = torch.empty((M, K), dtype=torch.bfloat16).pin_memory()
    hdw = torch.empty((N, K), dtype=torch.bfloat16).pin_memory()
    n = max(3, min(20, steps // 10))
    lanes = os.environ.get("FP8LIN_COPY_LANES")
    if lanes:
        lin.copy_lanes = int(lanes)
    for _ in range(2):
        lin.step_host(hx, hw, hdy, hy, hdx, hdw)
    torch.cuda.synchronize()
    # Pipelined steps: each step's compute may run while the previous step's
    # downloads finish; the last downloads complete inside the timed region.
    # The host link is shared with the rest of the machine, so three blocks of
    # n steps are timed and the median block is reported.
    cur = torch.cuda.current_stream()
    blocks = []
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        for _ in range(n):
            lin.step_host(hx, hw, hdy, hy, hdx, hdw, wait=False)
        lin.finish_host(cur)
        e1.record(cur)
        e1.synchronize()
        blocks.append(max_over_ranks(torch, e0.elapsed_time(e1) / n, world, lin.y.device))
    ms = sorted(blocks)[1]
    h2d = 2 * (M * K + N * K + M * N)
    d2h = 2 * (M * N + M * K + N * K)
    link = host_link_rates(torch, hx, lin.y.device)
    floor_ms = max(h2d / (link["h2d_gbs"] * 1e9), d2h / (link["d2h_gbs"] * 1e9),
                   (h2d + d2h) / (link["both_gbs"] * 1e9)) * 1e3
    return {"value": round(whole_job_tflops(flop_step, ms, world), 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3),
            "steps": n, "blocks_ms_per_step": [round(b, 3) for b in blocks],
            "copy_lanes": lin.copy_lanes,
            "api": "Fp8Linear.step_host(wait=False) + finish_host (pinned host buffers)",
            "host_link": link, "copy_floor_ms": round(floor_ms, 3),
            "frac_of_copy_floor": round(floor_ms / ms, 3)}


def host_link_rates(torch, host, dev):
    """Copy rate of the host link with pinned buffers (GB/s): host -> device,
    device -> host, and both at once on two streams (the rate the step's
    copies can reach at best)."""
    nbytes = host.numel() * host.element_size()
    d = torch.empty_like(host, device=dev)
    back = torch.empty_like(host).pin_memory()
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def timed(fn, reps=3):
        fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s1)
        for _ in range(reps):
            fn()
        s1.wait_stream(s2)
        b.record(s1)
        b.synchronize()
        return a.elapsed_time(b) / reps

    def up():
        with torch.cuda.stream(s1):
            d.copy_(host, non_blocking=True)

    def down():
        with torch.cuda.stream(s1):
            back.copy_(d, non_blocking=True)

    def both():
        s2.wait_stream(s1)
        with torch.cuda.stream(s1):
            d.copy_(host, non_blocking=True)
        with torch.cuda.stream(s2):
            back.copy_(d2, non_blocking=True)

    d2 = torch.empty_like(d)
    t_up, t_down, t_both = timed(up), timed(down), timed(both)
    torch.cuda.synchronize()
    del d, d2, back
    return {"h2d_gbs": round(nbytes / (t_up * 1e-3) / 1e9, 1),
            "d2h_gbs": round(nbytes / (t_down * 1e-3) / 1e9, 1),
            "both_gbs": round(2 * nbytes / (t_both * 1e-3) / 1e9, 1),
            "bytes": nbytes}


def run_native(args):
    import torch
    import quantised_gemm_gb300 as q
    import synth_inputs as si

    world, rank, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    wl = si.WORKLOADS[args.workload]
    M, K, N = wl["shapes"][0]

    x, w, dy = make_inputs(args.workload, 0)
    xd, wd, dyd = to_dev(x, dev), to_dev(w, dev), to_dev(dy, dev)
    lin = q.Fp8Linear(M, K, N, device=dev)

    def step():
        lin.forward(xd, wd)
        lin.backward(dyd)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    q.check(lin.ws)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = q.launch_count()
    q.profile_enable(True)
    sampler.mark("t0")
    ms = time_region(step, args.steps)
    sampler.mark("t1")
    torch.cuda.synchronize()
    prof = q.profile_collect()
    q.profile_enable(False)
    launches = q.launch_count() - launches0
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    q.check(lin.ws)
    ms_step = max_over_ranks(torch, ms / args.steps, world, dev)
    flop_step = 6.0 * M * N * K
    value = whole_job_tflops(flop_step, ms_step, world)

    gemm_ms, gemm_n = prof["gemm"]
    gemm_avg = gemm_ms / max(1, gemm_n)
    gemm_flop = 2.0 * M * N * K          # each of the three GEMMs of this square Linear
    achieved = gemm_flop / (gemm_avg * 1e-3) / 1e12
    peak = peaks["bf16_tflops_sustained"] * FP8_OVER_BF16
    tr = load_traffic("gemm")
    roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak, 1),
                "unit": "TFLOP/s", "frac": round(achieved / peak, 3),
                "traffic": tr["bytes_per_launch"] if tr else None,
                "kernel": q.gemm_describe(M, N, K).split(":")[0] +
                          " (tcgen05, e4m3/e5m2 x e4m3 -> bf16)",
                "schedule": {"y = x8.W8^T": q.gemm_describe(M, N, K),
                             "dX = dY8.W8t^T": q.gemm_describe(M, K, N),
                             "dW = dY8t.x8t^T": q.gemm_describe(N, K, M)},
                "launch_us": round(gemm_avg * 1e3, 1),
                "peak_basis": "%s bf16 sustained %.1f TFLOP/s x %.0f (nominal fp8/bf16)" % (
                    peaks["source"], peaks["bf16_tflops_sustained"], FP8_OVER_BF16)}
    # Casts of the step: x [M,K], W [N,K], dY [M,N], each 2 B read + 1 B + 1 B
    # (transposed) written per element.  Tensors that fit on chip run as the
    # single-pass kernel (kind "cast_fused", amax included); the others as
    # amax + cast_stream_kernel (kind "cast").
    cap = q.single_pass_max_elems()
    two_pass = [n for n in (M * K, N * K, M * N) if n > cap]
    one_pass = [n for n in (M * K, N * K, M * N) if n <= cap]
    cast_ms = prof["cast"][0] / args.steps
    fused_ms = prof["cast_fused"][0] / args.steps
    amax_ms = prof["amax"][0] / args.steps
    if two_pass and cast_ms > 0:
        kernel_bytes = 4.0 * sum(two_pass)
        cast_gbs = kernel_bytes / (cast_ms * 1e-3) / 1e9
        cast_kernel = "cast_stream_kernel (+transpose, TMA ring), two-pass casts"
    else:
        kernel_bytes = 4.0 * sum(one_pass)
        cast_gbs = kernel_bytes / (max(fused_ms, 1e-9) * 1e-3) / 1e9
        cast_kernel = "cast_single_pass_kernel (+transpose)"
    trc = load_traffic("cast")
    cast_roofline = {"bound": "hbm", "achieved": round(cast_gbs, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(cast_gbs / peaks["hbm_gbs"], 3),
                     "traffic": trc["bytes_per_launch"] if trc else None,
                     "kernel": cast_kernel, "bytes_per_step": round(kernel_bytes)}
    # The whole amax + scale + cast stage against its algorithmic bytes (one
    # read, one write per fp8 copy): a second read by two-pass amax counts as
    # time, not as bytes.
    stage_bytes = 4.0 * (M * K + N * K + M * N)
    stage_ms = cast_ms + fused_ms + amax_ms + prof["scale"][0] / args.steps
    amax_cast_stage = {"bound": "hbm", "unit": "GB/s", "peak": peaks["hbm_gbs"],
                       "achieved": round(stage_bytes / (stage_ms * 1e-3) / 1e9, 1),
                       "frac": round(stage_bytes / (stage_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 3),
                       "us_per_step": round(stage_ms * 1e3, 1),
                       "algorithmic_bytes_per_step": round(stage_bytes)}
    kernel_ms = {k: round(v[0] / args.steps, 4) for k, v in prof.items()}

    e2e = None
    if not args.no_e2e:
        e2e = end_to_end(q, lin, x, w, dy, M, K, N, world, flop_step, args.steps)
    del x, w, dy
    del lin, xd, wd, dyd
    torch.cuda.empty_cache()

    sweep = None
    if not args.no_sweep:
        flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
        flush = lambda: flush_buf.zero_()  # noqa: E731
        sweep = {"linears": [], "chains": None, "cast": None, "gemm_vs_cublaslt": None}
        for name in ("linear4096_m16", "linear4096_m256", "linear4096_m4096",
                     "gpt1.5b_linears_m12288", "llama3_8b_ffn_m8192"):
            small = si.WORKLOADS[name]["shapes"][0][0] <= 4096
            sweep["linears"].append(linear_sweep_entry(
                q, torch, dev, name, steps=50 if small else 20, warmup=5,
                flush=flush if small else None))
        for name in ("linear4096_m16", "linear4096_m256"):
            sweep["linears"].append(linear_sweep_entry(
                q, torch, dev, name, steps=50, warmup=5, flush=flush, cache_weight=True))
        sweep["chains"] = [
            chain_sweep_entry(q, torch, dev, "linear4096_m4096", steps=50, warmup=5, flush=flush),
            chain_sweep_entry(q, torch, dev, "linear4096_m65536", steps=10, warmup=3, flush=None)]
        del flush_buf
        torch.cuda.empty_cache()
        sweep["cast"] = cast_sweep(q, torch, dev, peaks, args.full_sweep)
        # the three products of the 65536-token step: y, dX (e5m2 A), dW (long K)
        sweep["gemm_vs_cublaslt"] = [library_gemm_entry(q, torch, dev, 65536, 4096, 4096, 0),
                                     library_gemm_entry(q, torch, dev, 65536, 4096, 4096, 1),
                                     library_gemm_entry(q, torch, dev, 4096, 4096, 65536, 1)]
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, desc, cores = cpu_baseline_sample(args.workload)
        cpu = {"value": round(v, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": desc}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup),
            "ms_per_step": round(ms_step, 4), "us_per_fwd_bwd": round(ms_step * 1e3, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp8",
            "data": "synthetic",
            "config": {"workload": "%s: Linear 4096->4096, M=%d tokens, dynamic tensorwise "
                                   "scaling, x~N(0,1)+0.1%% N(0,50) outliers, W~U(+-1/64), "
                                   "dY~N(0,1e-3)" % (args.workload, M),
                       "M": M, "K": K, "N": N, "l2": "inputs larger than L2 (x, dY 512 MiB)",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": roofline, "cast_roofline": cast_roofline,
            "amax_cast_stage": amax_cast_stage,
            "kernel_ms_per_step": kernel_ms,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": int(launches), "clocks": clocks, "peaks": peaks,
            "sweep": sweep,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ------------------------------------------------------------------ reference arm

REF_BUDGET_S = 60.0


def ref_sample_tokens(t16: float, t128: float, n_steps: int,
                      budget_s: float = REF_BUDGET_S) -> int:
    """Tokens per reference step: the largest multiple of 16 up to 128 for
    which n_steps steps fit in budget_s, at least 16.  A step costs
    a + b * tokens: the weight's amax and casts are the fixed part, so the
    line through the probe times of 16 and 128 tokens gives the cost."""
    b = max(0.0, (t128 - t16) / 112.0)
    a = max(0.0, t16 - 16.0 * b)
    for ms in range(128, 15, -16):
        if (a + b * ms) * n_steps <= budget_s:
            return ms
    return 16


def run_reference(args):
    """The oracle on host cores, same metric / unit / config, each step a
    bounded sample of the workload (the first Ms tokens of the Linear).  It
    runs exactly `warmup` untimed and `steps` timed steps; Ms (a multiple of
    16, at most 128) is chosen from two untimed probe steps so that the whole
    run takes about REF_BUDGET_S seconds where that is possible."""
    world, rank, _ = dist_info()
    if rank != 0:
        return
    import oracle
    import synth_inputs as si
    oracle.build()
    wl = si.WORKLOADS[args.workload]
    M, K, N = wl["shapes"][0]
    w = si.weight(K, N, w_init=wl["w_init"], w_std=wl.get("w_std", 0.02))

    def sample(ms):
        return (si.normal_bf16((ms, K), 1.0, 0, si.STREAM_X),
                si.normal_bf16((ms, N), 1e-3, 0, si.STREAM_DY))

    def step(x, dy):
        sx = oracle.scale_dynamic(oracle.amax(x), oracle.E4M3)[0]
        sw = oracle.scale_dynamic(oracle.amax(w), oracle.E4M3)[0]
        sd = oracle.scale_dynamic(oracle.amax(dy), oracle.E5M2)[0]
        oracle.linear_fwd_bwd(x, w, dy, sx, sw, sd)

    steps, warmup = max(1, args.steps), max(0, args.warmup)
    probe = {}
    for ms in (16, 128):
        x, dy = sample(ms)
        t0 = time.perf_counter()
        step(x, dy)
        probe[ms] = time.perf_counter() - t0
    Ms = ref_sample_tokens(probe[16], probe[128], steps + warmup)
    if Ms != 128:
        x, dy = sample(Ms)
    for _ in range(warmup):
        step(x, dy)
    t0 = time.perf_counter()
    for _ in range(steps):
        step(x, dy)
    dt = (time.perf_counter() - t0) / steps
    value = 6.0 * Ms * N * K / dt / 1e12
    sample = ("oracle fwd+bwd of the %dx%d Linear on the first %d of %d tokens per step" %
              (K, N, Ms, M))
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": world, "steps": steps, "warmup": warmup,
            "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "%s: Linear 4096->4096, M=%d tokens (sampled %d)" %
                                   (args.workload, M, Ms), "M": M, "K": K, "N": N},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "kind": "oracle",
                             "cores": oracle.num_threads(), "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
