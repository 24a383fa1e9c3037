#!/usr/bin/env python3
"""Benchmark of the fp8 training Linear (libfp8lin) on GB300.

One step = one forward + backward of the 4096->4096 Linear at M = 65536
tokens with tensorwise dynamic scaling: amax, scale, e4m3/e5m2 casts with
transposed copies, and the three FP8 GEMMs (y = x W^T, dX = dY W,
dW = dY^T x).  The workload is the largest row of the single-linear table of
"Integrate float8nocompile, an experimental feature for high performance"
(pytorch/torchtitan PR 778), with inputs that exceed L2 (x and dY are
512 MiB each), so no L2 flush is needed between steps.

Prints ONE compact JSON line: value = TFLOP/s of the whole job (6 M N K per
step, timed without instrumentation), the GEMM kernel's roofline (tensor pipe
vs the measured peak), the cast kernel's HBM roofline, the amax + cast stage
against its algorithmic bytes, an end-to-end figure through the host-buffer
API, the oracle timed on the host cores, SM clocks sampled during the timed
region, and one entry per other workload (M = 16 / 256 / 4096, GPT-1.5B block
Linears with delayed scaling, Llama-3-8B FFN Linears, cast-only bandwidth),
each with its fraction of the roofline that bounds it.  Per-kernel times come
from a separate profiled pass (an event pair around every launch) run right
after the timed region.  ``--detail PATH`` also writes every figure behind
the line to PATH.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
  python -m torch.distributed.run --nproc-per-node N bench.py --gpus N ...

With N > 1 the Linear is split over the tokens: every rank runs M tokens on
its own GPU with the whole job's tensorwise scales (one all-reduce(max) of
the amax of x and of dY per step, quantised_gemm_gb300.sharded); value is the
sum over ranks, time the max over ranks.
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
BURST_LIMIT_S = 2.0      # timed regions shorter than this are held to the burst peak


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--detail", default=None, help="write every figure behind the line here")
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


def fp8_peak(peaks, region_s):
    """Dense fp8 peak for a timed region of region_s seconds: the burst figure
    for short regions, the sustained one (power cap) for long ones; nominal
    fp8 / bf16 ratio applied to the measured bf16 figure."""
    burst = region_s < BURST_LIMIT_S
    bf = peaks["bf16_tflops"] if burst else peaks["bf16_tflops_sustained"]
    basis = "%s bf16 %s %.1f x %.0f" % (peaks["source"], "burst" if burst else "sustained", bf,
                                        FP8_OVER_BF16)
    return bf * FP8_OVER_BF16, basis


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


def load_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current source of the kernel for this workload (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = device_code_sha(kernel)
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line.startswith("{"):
                rec = json.loads(line)
                if (rec.get("kernel") == kernel and rec.get("src_sha") == sha
                        and rec.get("workload") == workload):
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

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

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


def step_bytes(M, K, N, cast_w=True):
    """Algorithmic HBM bytes of one fwd+bwd: every cast reads its bf16 tensor
    once and writes two fp8 copies (2 + 1 + 1 B per element); each GEMM reads
    its two fp8 operands once and writes its bf16 output."""
    casts = 4 * (M * K + M * N + (N * K if cast_w else 0))
    gemms = (M * K + N * K + 2 * M * N) + (M * N + N * K + 2 * M * K) + (M * N + M * K + 2 * N * K)
    return casts + gemms


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


def gemm_roofline(M, N, K, gemm_each, peak, kernel, traffic):
    """The step's GEMMs against the tensor peak: y, dX and dW (2MNK flops
    each) over the summed time (ms) of the step's GEMM launches -- three, or
    two when the backward runs dX and dW as one grouped launch."""
    achieved = 3 * 2.0 * M * N * K / (sum(gemm_each) * 1e-3) / 1e12
    if len(gemm_each) == 2:
        kernel += "; dX + dW: one grouped launch (gemm_fp8_pair2_kernel)"
    return {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak, 1),
            "unit": "TFLOP/s", "frac": round(achieved / peak, 3), "traffic": traffic,
            "kernel": kernel}


def profiled(q, torch, step, n, flush=None):
    """Per-kernel device times of n un-graphed steps (an event pair around
    every launch).  Returns (per-kind ms per step, GEMM ms per step in launch
    order within a step, launches per step)."""
    torch.cuda.synchronize()
    q.profile_enable(True)
    for _ in range(n):
        if flush is not None:
            flush()
        step()
    torch.cuda.synchronize()
    recs = q.profile_launches()
    q.profile_enable(False)
    kinds = {}
    for k, ms in recs:
        kinds[k] = kinds.get(k, 0.0) + ms / n
    # the products of a step, in order: GEMM launches, and the few-token
    # launches that fuse a product with its casts
    gemms = [ms for k, ms in recs if k in ("gemm", "small_m")]
    per = len(gemms) // n if n else 0
    gemm_each = [sum(gemms[i + j * per] for j in range(n)) / n for i in range(per)]
    return kinds, gemm_each, len(recs) // max(1, n)


def linear_sweep_entry(q, torch, dev, name, steps, warmup, flush, peak_fp8, peaks,
                       cache_weight=False):
    """fwd+bwd time of every Linear of a workload (sum over its Linears),
    graph-replayed, with its fraction of the roofline: the tensor peak for
    the GEMMs (per GEMM kernel, from a profiled pass), HBM for the whole step
    on its algorithmic bytes.  cache_weight: W is cast once and reused by
    every step, as over the micro-batches of one optimizer step."""
    import synth_inputs as si
    wl = si.WORKLOADS[name]
    delayed = wl.get("delayed", False)
    total_ms = flop = gemm_ms = nbytes = warm_ms = 0.0
    kinds = {}
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
        fn = graphed(torch, step)
        torch.cuda.synchronize()
        ms = time_region(fn, steps, flush) / steps
        if flush is not None:  # the same replays back to back: L2 warm
            warm_ms += time_region(fn, steps) / steps
        kk, gemm_each, _ = profiled(q, torch, step, 5, flush)
        q.check(lin.ws)
        total_ms += ms
        flop += 6.0 * M * N * K
        gemm_ms += sum(gemm_each)
        nbytes += step_bytes(M, K, N, cast_w=not cache_weight)
        for k, v in kk.items():
            kinds[k] = kinds.get(k, 0.0) + v
        del lin, xd, wd, dyd
        torch.cuda.empty_cache()
    tf = flop / (total_ms * 1e-3) / 1e12
    gemm_tf = flop / (gemm_ms * 1e-3) / 1e12
    hbm = nbytes / (total_ms * 1e-3) / 1e9
    return {"workload": name + (" (W cast once, reused)" if cache_weight else ""),
            "us": round(total_ms * 1e3, 2), "tf": round(tf, 1),
            "frac": round(tf / peak_fp8, 3),
            "gemm_us": round(gemm_ms * 1e3, 2), "gemm_tf": round(gemm_tf, 1),
            "gemm": round(gemm_tf / peak_fp8, 3),
            "bytes": int(nbytes), "hbm_gbs": round(hbm, 1),
            "hbm": round(hbm / peaks["hbm_gbs"], 3),
            "kernel_us": {k: round(v * 1e3, 2) for k, v in kinds.items()},
            "scaling": "delayed" if delayed else "dynamic",
            "l2": "flushed between steps" if flush else "inputs larger than L2",
            "us_warm": round(warm_ms * 1e3, 2) if flush is not None else None,
            "cuda_graph": True}


def library_gemm_entry(q, torch, dev, M, N, K, fmt_a, rounds=3, iters=10):
    """The FP8 GEMM of this library against cuBLASLt's (torch._scaled_mm,
    tensorwise scales) on the same operands: D[M,N] = A[M,K] B[N,K]^T, bf16
    out.  Both read operands larger than L2.  The two alternate ABBA over
    `rounds` rounds so clock drift under the power cap favours neither; the
    medians are reported, with the largest |difference| of the two outputs
    (the accumulation order may differ)."""
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
    under the power cap does not favour either."""
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
        kk, _, _ = profiled(q, torch, step, 2)
        variants["fused_amax" if linked else "separate_amax"] = {
            "graph": graphed(torch, step), "lins": (l1, l2), "ms": [],
            "kernel_us_per_step": {k: round(v * 1e3, 1) for k, v in kk.items()}}
    torch.cuda.synchronize()
    order = list(variants.values())
    for r in range(rounds):  # ABBA: neither variant always runs first
        for v in (order if r % 2 == 0 else order[::-1]):
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


CAST_ALGOS = ("atomic", "reduction", "single_pass", "delayed")


def cast_sweep(q, torch, dev, peaks):
    """amax + scale + cast (+T) of [R, 4096] / [4096, R] bf16 N(0,1) tensors,
    R * 4096 = 2^20 ... 2^30, e4m3 and e5m2, with and without the transposed
    copy, for each amax algorithm: two-pass ATOMIC and REDUCTION, the
    single pass where the tensor fits on chip, and delayed scaling's cast
    (stored scale, amax recorded in the same pass: one read).  GB/s of the
    algorithmic bytes (2 B read + 1 B per fp8 copy), so a second read by a
    two-pass amax counts as time.  Inputs are drawn on the device (seeded):
    this is a measurement, the parity of these casts is in the tests."""
    sizes = [1 << 20, 1 << 22, 1 << 24, 1 << 26, 1 << 28, 1 << 30]
    ws = q.Workspace(device=dev)
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    gen = torch.Generator(device=dev)
    out = []
    for n in sizes:
        for shp in ("rows", "cols"):
            R = n // 4096
            rows, cols = (R, 4096) if shp == "rows" else (4096, R)
            gen.manual_seed(n + (shp == "cols"))
            xd = torch.randn((rows, cols), device=dev, generator=gen).to(torch.bfloat16)
            o = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
            ot = torch.empty((cols, rows), dtype=torch.uint8, device=dev)
            for fmt in (q.E4M3, q.E5M2):
                for trans in (True, False):
                    for algo in CAST_ALGOS:
                        if algo == "single_pass" and n > q.single_pass_max_elems():
                            continue
                        if algo == "delayed":
                            st = q.ScalingState(fmt, q.DELAYED, history_len=16, device=dev)
                            call = lambda st=st: q.cast_delayed(  # noqa: E731
                                xd, st, o, ot if trans else None, ws)
                        else:
                            a = {"atomic": q.AMAX_ATOMIC, "reduction": q.AMAX_REDUCTION,
                                 "single_pass": q.AMAX_SINGLE_PASS}[algo]
                            st = q.ScalingState(fmt, q.DYNAMIC, amax_algo=a, device=dev)
                            call = lambda st=st: q.cast_dynamic(  # noqa: E731
                                xd, st, o, ot if trans else None, ws)
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
                        out.append({"elems": n, "shape": [rows, cols],
                                    "fmt": "e4m3" if fmt == q.E4M3 else "e5m2",
                                    "transpose": trans, "amax": algo,
                                    "us": round(ms * 1e3, 2), "gbs": round(gbs, 1),
                                    "frac_hbm": round(gbs / peaks["hbm_gbs"], 3)})
            del xd, o, ot
            torch.cuda.empty_cache()
    del flush_buf
    torch.cuda.empty_cache()
    return out


def cast_sweep_summary(rows):
    """Per size: [median, min] fraction of HBM over the 8 format x shape x
    transpose cases, per amax algorithm (None where it does not apply)."""
    res = {}
    for n in sorted({r["elems"] for r in rows}):
        ent = []
        for algo in CAST_ALGOS:
            f = [r["frac_hbm"] for r in rows if r["elems"] == n and r["amax"] == algo]
            ent.append([round(statistics.median(f), 3), round(min(f), 3)] if f else None)
        res["2^%d" % (n.bit_length() - 1)] = ent
    return res


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
    desc = ("oracle fwd+bwd (C casts, numpy fp64 GEMMs), %dx%d Linear, first %d of %d tokens, "
            "%.2f s" % (K, N, Ms, M, elapsed))
    return flop / elapsed / 1e12, desc, oracle.num_threads()


def host_cpu():
    """The host CPU's model name and its logical CPU count."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith("model name"):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    import platform
    return "%s (%d logical CPUs, %s)" % (model or "unknown model", os.cpu_count() or 0,
                                         platform.machine())


def cpu_baseline_one_core(name, budget_s=5.0):
    """cpu_baseline_sample on one core: a child process whose OpenMP and BLAS
    pools have one thread (set before the oracle and numpy load).  Returns
    (TFLOP/s, description, threads) or None if the child failed."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import json, sys; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench.cpu_baseline_sample(%r, %r)))" % (ROOT, name, budget_s))
    try:
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                           env=env, cwd=ROOT, timeout=300)
        return tuple(json.loads(r.stdout.strip().splitlines()[-1])) if r.returncode == 0 else None
    except (OSError, subprocess.SubprocessError, ValueError, IndexError):
        return None


def end_to_end(q, lin, x, w, dy, M, K, N, world, flop_step):
    """The same step through the C ABI's host-buffer entry point
    (fp8lin_step_host, called by Fp8Linear.step_host): pinned host inputs
    copied in and y, dX, dW copied out every step."""
    import torch
    hx = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
    hw = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16).pin_memory()
    hdy = torch.from_numpy(dy.view(np.int16)).view(torch.bfloat16).pin_memory()
    hy = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    hdx = torch.empty((M, K), dtype=torch.bfloat16).pin_memory()
    hdw = torch.empty((N, K), dtype=torch.bfloat16).pin_memory()
    # Blocks of 12 steps whatever --steps says: the two device slots make the
    # copies of one step overlap the compute of the next, a pipeline that
    # needs several steps to reach its steady state (blocks of 3 measured
    # 7.64 ms per step where blocks of 20 measured 6.65 ms on the same box).
    n = 12
    for _ in range(2):
        lin.step_host(hx, hw, hdy, hy, hdx, hdw)
    torch.cuda.synchronize()
    # Pipelined steps: each step's compute may run while the previous step's
    # downloads finish; the last downloads complete inside the timed region.
    # The host link is shared with the rest of the machine, so five blocks of
    # n steps are timed and the median block is reported.
    cur = torch.cuda.current_stream()
    blocks = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        for _ in range(n):
            lin.step_host(hx, hw, hdy, hy, hdx, hdw, wait=False)
        lin.finish_host(cur)
        e1.record(cur)
        e1.synchronize()
        blocks.append(max_over_ranks(torch, e0.elapsed_time(e1) / n, world, lin.y.device))
    ms = sorted(blocks)[2]
    h2d = 2 * (M * K + N * K + M * N)
    d2h = 2 * (M * N + M * K + N * K)
    link = host_link_rates(torch, hx, lin.y.device)
    floor_ms = max(h2d / (link["h2d_gbs"] * 1e9), d2h / (link["d2h_gbs"] * 1e9),
                   (h2d + d2h) / (link["both_gbs"] * 1e9)) * 1e3
    return {"value": round(whole_job_tflops(flop_step, ms, world), 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3),
            "steps": n, "blocks_ms_per_step": [round(b, 3) for b in blocks],
            "api": "fp8lin_step_host via Fp8Linear.step_host(wait=False) + finish_host "
                   "(pinned host buffers, two device slots)",
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


def few_token_roofline(M, K, N, product_ms, peaks):
    """HBM roofline of the slower few-token product of a step (M <= 32).
    Algorithmic bytes of each launch: the forward reads x and W (2 B) and
    writes x8, x8^T, W8, W8^T (1 B each) and y (2 B); the backward reads dY
    (2 B) and W8^T (1 B), writes dY8, dY8^T (1 B) and dX (2 B), and with dW
    fused (two products per step) also reads x8^T (1 B) and writes dW (2 B)."""
    fwd = 4.0 * N * K + 4.0 * M * K + 2.0 * M * N
    with_dw = len(product_ms) == 2
    bwd = 1.0 * N * K + 4.0 * M * N + 2.0 * M * K + (2.0 * N * K + 1.0 * M * K if with_dw else 0)
    names = ["small_m_kernel<cast W> (x, W casts; y)",
             "small_m_kernel<dW> (dY cast; dX, dW)" if with_dw else "small_m_kernel (dY cast; dX)"]
    i = 0 if product_ms[0] >= product_ms[1] else 1
    gbs = (fwd, bwd)[i] / (product_ms[i] * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(gbs / peaks["hbm_gbs"], 3), "traffic": None, "kernel": names[i],
            "peak_basis": "measured HBM copy (of measured)" if peaks["source"] == "measured"
            else "HBM copy (of fallback)"}


SHORT = {"linear4096_m16": "m16", "linear4096_m256": "m256", "linear4096_m4096": "m4096",
         "gpt1.5b_linears_m12288": "gpt1.5b_delayed", "llama3_8b_ffn_m8192": "llama3_ffn"}


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
    if world > 1:
        # M-sharded over the ranks (weak scaling: M tokens per rank) with one
        # tensorwise scale for the whole job: the amaxes of x and dY are
        # all-reduced (max) before their casts.  dW stays per rank: its sum
        # is the data-parallel gradient reduction, outside the Linear.
        from quantised_gemm_gb300.sharded import ShardedFp8Linear
        sharded = ShardedFp8Linear(M, K, N, reduce_dw=False, device=dev)
        lin = sharded.lin
        layer = sharded
    else:
        lin = layer = q.Fp8Linear(M, K, N, device=dev)

    def step():
        layer.forward(xd, wd)
        layer.backward(dyd)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    q.check(lin.ws)

    # ---- timed region: plain launches, no instrumentation
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = q.launch_count()
    ms = time_region(step, args.steps)
    launches = q.launch_count() - launches0
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    q.check(lin.ws)
    ms_step = max_over_ranks(torch, ms / args.steps, world, dev)
    flop_step = 6.0 * M * N * K
    value = whole_job_tflops(flop_step, ms_step, world)
    region_s = ms_step * args.steps * 1e-3
    peak, basis = fp8_peak(peaks, region_s)

    # ---- per-kernel split: a profiled pass of the same steps, right after
    n_prof = max(3, min(args.steps, 40))
    kinds, gemm_each, per_step = profiled(q, torch, step, n_prof)
    q.check(lin.ws)
    if kinds.get("small_m", 0.0) > 0:
        # A few tokens: the products are fused with their casts and bound by
        # their bytes; the slower of the two against HBM.
        roofline = few_token_roofline(M, K, N, gemm_each, peaks)
        roofline["kernel_time"] = ("mean of %d launches, profiled pass of %d steps after the "
                                   "timed region" % (n_prof, n_prof))
    else:
        tr = load_traffic("gemm", args.workload)
        roofline = gemm_roofline(M, N, K, gemm_each, peak,
                                 q.gemm_describe(M, N, K).split(":")[0],
                                 tr["bytes_per_launch"] if tr else None)
        roofline["peak_basis"] = (basis + " (of measured)" if peaks["source"] == "measured" else
                                  basis + " (of fallback)")
        roofline["kernel_time"] = ("the step's GEMM flops over the summed time of its %d GEMM "
                                   "launches, profiled pass of %d steps after the timed region"
                                   % (len(gemm_each), n_prof))
    # Casts of the step: x [M,K], W [N,K], dY [M,N], each 2 B read + 1 B + 1 B
    # (transposed) written per element.  Tensors that fit on chip run as the
    # single-pass kernel (kind "cast_fused", amax included); the others as
    # amax + cast_stream_kernel (kind "cast").
    cap = q.single_pass_max_elems()
    two_pass = [n for n in (M * K, N * K, M * N) if n > cap]
    one_pass = [n for n in (M * K, N * K, M * N) if n <= cap]
    cast_ms, fused_ms = kinds.get("cast", 0.0), kinds.get("cast_fused", 0.0)
    amax_ms, scale_ms = kinds.get("amax", 0.0), kinds.get("scale", 0.0)
    cast_roofline = None
    if two_pass and cast_ms > 0:
        kernel_bytes, kernel_ms, cast_kernel = 4.0 * sum(two_pass), cast_ms, "cast_stream_kernel"
    elif fused_ms > 0:
        kernel_bytes, kernel_ms, cast_kernel = 4.0 * sum(one_pass), fused_ms, "cast_single_pass_kernel"
    else:                     # (a few-token step runs its casts inside the products)
        kernel_ms = 0.0
    if kernel_ms > 0:
        cast_gbs = kernel_bytes / (kernel_ms * 1e-3) / 1e9
        trc = load_traffic("cast", args.workload)
        cast_roofline = {"bound": "hbm", "achieved": round(cast_gbs, 1), "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": round(cast_gbs / peaks["hbm_gbs"], 3),
                         "traffic": trc["bytes_per_launch"] if trc else None,
                         "kernel": cast_kernel}
    # The whole amax + scale + cast stage against its algorithmic bytes (one
    # read, one write per fp8 copy); a second read by two-pass amax counts as
    # time.  Two-pass dynamic scaling moves 6 B per element for 4 algorithmic
    # ones, so its ceiling is 2/3 of HBM.
    stage_bytes = 4.0 * (M * K + N * K + M * N)
    stage_ms = cast_ms + fused_ms + amax_ms + scale_ms
    stage = None
    if stage_ms > 0:          # (a few-token step runs its casts inside the products)
        stage_frac = stage_bytes / (stage_ms * 1e-3) / 1e9 / peaks["hbm_gbs"]
        stage = {"us": round(stage_ms * 1e3, 1), "frac": round(stage_frac, 3),
                 "of_two_pass_ceiling": round(stage_frac / (4.0 / 6.0), 3)}
    labels = ("y", "dx", "dw") if len(gemm_each) == 3 else ("y", "dx_dw")
    kernel_us = {k: round(v * 1e3, 1) for k, v in zip(labels, gemm_each)}
    kernel_us.update({"cast": round(cast_ms * 1e3, 1), "cast_fused": round(fused_ms * 1e3, 1),
                      "amax": round(amax_ms * 1e3, 1), "scale": round(scale_ms * 1e3, 1)})

    e2e = None
    if not args.no_e2e:
        e2e = end_to_end(q, lin, x, w, dy, M, K, N, world, flop_step)
    del x, w, dy
    del lin, xd, wd, dyd
    torch.cuda.empty_cache()

    detail = {"headline_kernels_ms_per_step": kinds, "headline_gemm_ms": gemm_each,
              "launches_per_step": per_step}
    configs, cast_sum, vs_lt, chains = None, None, None, None
    if not args.no_sweep:
        flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
        flush = lambda: flush_buf.zero_()  # noqa: E731
        entries = []
        for name in ("linear4096_m16", "linear4096_m256", "linear4096_m4096",
                     "gpt1.5b_linears_m12288", "llama3_8b_ffn_m8192"):
            small = si.WORKLOADS[name]["shapes"][0][0] <= 4096
            entries.append((SHORT[name], linear_sweep_entry(
                q, torch, dev, name, steps=50 if small else 20, warmup=5,
                flush=flush if small else None, peak_fp8=peak, peaks=peaks)))
        for name in ("linear4096_m16", "linear4096_m256"):
            entries.append((SHORT[name] + "_cachedW", linear_sweep_entry(
                q, torch, dev, name, steps=50, warmup=5, flush=flush, peak_fp8=peak,
                peaks=peaks, cache_weight=True)))
        detail["linears"] = dict(entries)
        configs = {}
        for key, e in entries:
            c = {"us": e["us"], "tf": e["tf"]}
            if e["us_warm"] is not None:
                c["us_warm"] = e["us_warm"]   # no flush between the replays
            if key.startswith(("m16", "m256")):
                c["hbm"] = e["hbm"]           # HBM-bound: the step against its bytes
            else:
                c["gemm"] = e["gemm"]         # tensor-bound: GEMM kernels vs fp8 peak
                c["frac"] = e["frac"]
            configs[key] = c
        chains = [chain_sweep_entry(q, torch, dev, "linear4096_m4096", steps=50, warmup=5,
                                    flush=flush),
                  chain_sweep_entry(q, torch, dev, "linear4096_m65536", steps=10, warmup=3,
                                    flush=None, rounds=6)]
        detail["chains"] = chains
        del flush_buf
        torch.cuda.empty_cache()
        rows = cast_sweep(q, torch, dev, peaks)
        detail["cast_sweep"] = rows
        cast_sum = cast_sweep_summary(rows)
        # the three products of the 65536-token step: y, dX (e5m2 A), dW (long K)
        lt = [library_gemm_entry(q, torch, dev, 65536, 4096, 4096, 0),
              library_gemm_entry(q, torch, dev, 65536, 4096, 4096, 1),
              library_gemm_entry(q, torch, dev, 4096, 4096, 65536, 1)]
        detail["gemm_vs_cublaslt"] = lt
        vs_lt = [e.get("ours_over_cublaslt") for e in lt]
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, desc, cores = cpu_baseline_sample(args.workload)
        cpu = {"value": round(v, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": desc, "cpu": host_cpu()}
        one = cpu_baseline_one_core(args.workload)
        if one is not None:  # (its sample, fewer tokens, in the detail file)
            cpu["one_core"] = {"value": round(one[0], 6), "threads": one[2]}
            detail["cpu_baseline_one_core"] = {"value": one[0], "threads": one[2],
                                               "sample": one[1]}

    if rank == 0:
        e2e_line = None
        if e2e is not None:
            e2e_line = {k: e2e[k] for k in ("value", "unit", "h2d_bytes_per_step",
                                            "d2h_bytes_per_step", "ms_per_step",
                                            "frac_of_copy_floor")}
            e2e_line["api"] = "fp8lin_step_host"
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup),
            "ms_per_step": round(ms_step, 4), "us_per_fwd_bwd": round(ms_step * 1e3, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp8",
            "data": "synthetic",
            "config": {"workload": "%s: Linear 4096->4096, M=%d, dynamic tensorwise" %
                                   (args.workload, M),
                       "l2": "inputs > L2",
                       "parallelism": "dp%d, M-sharded, global amax" % world if world > 1
                       else "1 GPU"},
            "roofline": roofline, "cast_roofline": cast_roofline, "amax_cast_stage": stage,
            "kernel_us": kernel_us, "cpu_baseline": cpu, "e2e": e2e_line,
            "gpu_launches": int(launches), "clocks": clocks,
            "configs": configs,
            "cast_sweep": ({"cols": "per size [median,min] frac HBM over fmt x shape x T: "
                                    "atomic, reduction, single_pass, delayed", **cast_sum}
                           if cast_sum else None),
            "vs_cublaslt_y_dx_dw": vs_lt,
            "chain_fused_amax_saved_us": [c["saved_us"] for c in chains] if chains else None,
        }
        print(json.dumps(line, separators=(",", ":"), ensure_ascii=False), flush=True)
        if args.detail:
            detail.update({"line": line, "e2e": e2e, "peaks": peaks})
            with open(args.detail, "w") as f:
                json.dump(detail, f, indent=1)
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
                             "cores": oracle.num_threads(), "sample": sample,
                             "cpu": host_cpu()},
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
