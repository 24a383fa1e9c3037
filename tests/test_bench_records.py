"""bench.py's DRAM-traffic records, on CPU: a record counts only for the device
code and the workload it was captured on, and its per-launch figure is the
captured one scaled to the benchmark's launch."""
import json
import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _records():
    with open(os.path.join(ROOT, "profiles", "dram_traffic.txt")) as f:
        return [json.loads(line) for line in f if line.strip().startswith("{")]


def test_records_are_internally_consistent():
    recs = _records()
    assert {r["kernel"] for r in recs} == {"gemm", "cast"}
    for r in recs:
        assert r["bytes_per_launch"] == pytest.approx(r["captured_bytes"] * r["scale"], rel=1e-3)
        assert len(r["src_sha"]) == 16


def test_record_applies_only_to_its_device_code(monkeypatch):
    for kernel in ("gemm", "cast"):
        rec = bench.load_traffic(kernel, bench.HEADLINE)
        if rec is not None:  # a fresh record: keyed on exactly this code
            assert rec["src_sha"] == bench.device_code_sha(kernel)
        monkeypatch.setattr(bench, "device_code_sha", lambda k: "0" * 16)
        assert bench.load_traffic(kernel, bench.HEADLINE) is None
        monkeypatch.undo()


def test_record_applies_only_to_its_workload():
    assert {r["workload"] for r in _records()} == {bench.HEADLINE}
    for kernel in ("gemm", "cast"):
        assert bench.load_traffic(kernel, "linear4096_m16") is None


def test_few_token_roofline_bytes():
    peaks = {"hbm_gbs": 1000.0, "source": "measured"}
    M, K, N = 16, 4096, 4096
    # forward: x, W read (2 B), x8, x8^T, W8, W8^T written (1 B each), y (2 B)
    fwd = 2 * M * K + 2 * N * K + 2 * M * K + 2 * N * K + 2 * M * N
    # backward with dW: dY (2 B), W8^T, x8^T read; dY8, dY8^T, dX (2 B), dW (2 B) written
    bwd = 2 * M * N + N * K + M * K + 2 * M * N + 2 * M * K + 2 * N * K
    r = bench.few_token_roofline(M, K, N, [0.02, 0.01], peaks)
    assert r["achieved"] == pytest.approx(fwd / 0.02e-3 / 1e9, rel=1e-3) and "cast W" in r["kernel"]
    r = bench.few_token_roofline(M, K, N, [0.01, 0.02], peaks)
    assert r["achieved"] == pytest.approx(bwd / 0.02e-3 / 1e9, rel=1e-3) and "dW" in r["kernel"]
    assert r["bound"] == "hbm" and r["frac"] == pytest.approx(r["achieved"] / 1000.0, abs=1e-3)


def test_hash_covers_the_inlined_ptx_helpers(tmp_path, monkeypatch):
    csrc = os.path.join(tmp_path, "quantised_gemm_gb300", "csrc")
    os.makedirs(csrc)
    for name in ("gemm_kernels.cuh", "cast_kernels.cuh", "ptx.cuh"):
        shutil.copy(os.path.join(ROOT, "quantised_gemm_gb300", "csrc", name), csrc)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    before = {k: bench.device_code_sha(k) for k in ("gemm", "cast")}
    assert before["gemm"] != before["cast"]
    with open(os.path.join(csrc, "ptx.cuh"), "a") as f:
        f.write("\n// edited\n")
    after = {k: bench.device_code_sha(k) for k in ("gemm", "cast")}
    assert all(after[k] != before[k] for k in before)


def test_reference_sample_fits_the_budget():
    # fixed 0.4 s (the weight's casts) + 1 ms per token
    t = lambda ms: 0.4 + 0.001 * ms  # noqa: E731
    assert bench.ref_sample_tokens(t(16), t(128), 10) == 128
    assert bench.ref_sample_tokens(t(16), t(128), 100, budget_s=60.0) == 128  # 52.8 s
    ms = bench.ref_sample_tokens(t(16), t(128), 120, budget_s=60.0)
    assert ms == 96 and t(ms) * 120 <= 60.0 < t(ms + 16) * 120
    assert bench.ref_sample_tokens(t(16), t(128), 410, budget_s=60.0) == 16  # fixed part alone overruns


def test_gemm_roofline_counts_the_step_flops_once():
    M, N, K = 4096, 4096, 4096
    flop = 3 * 2.0 * M * N * K
    three = bench.gemm_roofline(M, N, K, [0.05, 0.05, 0.05], 4000.0, "pair", None)
    two = bench.gemm_roofline(M, N, K, [0.05, 0.10], 4000.0, "pair", 123)
    assert three["achieved"] == pytest.approx(flop / 0.15e-3 / 1e12, rel=1e-3)
    assert two["achieved"] == three["achieved"]          # same work, same summed time
    assert "pair2" in two["kernel"] and "pair2" not in three["kernel"]
    assert two["frac"] == pytest.approx(two["achieved"] / 4000.0, abs=1e-3)
    assert two["traffic"] == 123 and two["bound"] == "tensor"


def test_cpu_baseline_reports_the_host_and_one_thread():
    """cpu_baseline's `cpu` names the host, and its one-core figure comes from
    a child whose OpenMP and BLAS pools really have one thread."""
    desc = bench.host_cpu()
    assert "logical CPUs" in desc and str(os.cpu_count()) in desc
    one = bench.cpu_baseline_one_core("linear4096_m65536", budget_s=0.3)
    assert one is not None
    value, sample, threads = one
    assert threads == 1 and value > 0
    assert "first" in sample and "of 65536 tokens" in sample
