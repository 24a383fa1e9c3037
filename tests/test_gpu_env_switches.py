"""The environment switches that choose between fused and separate launches
(read once per process, so each setting runs in a child process).  A 16-token
step with FP8LIN_SMALL_M=0 (casts and GEMMs as separate kernels), with
FP8LIN_SMALL_M_DW=0 (the fused products, dW as its own GEMM) and with neither
gives the same fp8 bytes and scales, and every output within the oracle's
bound; dW with and without its fusion is equal value for value.  A
few-hundred-token forward with FP8LIN_PAIR_CAST=0 casts x and W in two
launches instead of one paired single pass: the same bits, one launch more."""
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
import synth_inputs as si
from helpers import assert_within_bound

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
M, K, N = 16, 784, 1040

CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1])
import quantised_gemm_gb300 as q, synth_inputs as si
M, K, N = (int(v) for v in sys.argv[3].split(",")) if len(sys.argv) > 3 else (%d, %d, %d)
x, w, dy = si.linear_inputs(M, K, N, w_init="uniform64", outlier_frac=1e-2, seed=83)
dev = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
lin = q.Fp8Linear(M, K, N)
n0 = q.launch_count()
lin.forward(dev(x), dev(w))
lin.backward(dev(dy))
q.check(lin.ws)
launches = q.launch_count() - n0
out = {name: getattr(lin, name).cpu().numpy() for name in ("x8", "x8t", "w8", "w8t", "dy8", "dy8t")}
for name in ("y", "dx", "dw"):
    out[name] = getattr(lin, name).cpu().view(torch.int16).numpy()
for st in ("sx", "sw", "sdy"):
    out[st] = getattr(lin, st).scale.cpu().numpy()
out["launches"] = np.array([launches])
np.savez(sys.argv[2], **out)
""" % (M, K, N)


def _run(tmp_path, name, env, mkn=None):
    path = os.path.join(tmp_path, name + ".npz")
    e = dict(os.environ)
    e.update(env)
    args = [sys.executable, "-c", CHILD, ROOT, path] + ([",".join(map(str, mkn))] if mkn else [])
    subprocess.run(args, env=e, check=True, timeout=600)
    return dict(np.load(path))


def bf16_to_f64_bits(bits):
    return (bits.astype(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_few_token_switches(tmp_path):
    base = {"FP8LIN_SMALL_M": "1", "FP8LIN_SMALL_M_DW": "1"}
    runs = {"fused": _run(tmp_path, "fused", base),
            "no_dw_fusion": _run(tmp_path, "no_dw", dict(base, FP8LIN_SMALL_M_DW="0")),
            "separate": _run(tmp_path, "separate", dict(base, FP8LIN_SMALL_M="0"))}
    assert int(runs["fused"]["launches"][0]) == 2          # forward product, backward product
    assert int(runs["no_dw_fusion"]["launches"][0]) == 3   # ... and dW's GEMM
    assert int(runs["separate"]["launches"][0]) > 3        # casts and GEMMs one by one
    x, w, dy = si.linear_inputs(M, K, N, w_init="uniform64", outlier_frac=1e-2, seed=83)
    sx = oracle.scale_dynamic(oracle.amax(x), oracle.E4M3)[0]
    sw = oracle.scale_dynamic(oracle.amax(w), oracle.E4M3)[0]
    sd = oracle.scale_dynamic(oracle.amax(dy), oracle.E5M2)[0]
    ref = oracle.linear_fwd_bwd(x, w, dy, sx, sw, sd)
    for label, r in runs.items():
        for name in ("x8", "x8t", "w8", "w8t", "dy8", "dy8t"):
            assert np.array_equal(r[name], ref[name]), (label, name)
        for st, s in (("sx", sx), ("sw", sw), ("sdy", sd)):
            assert np.float32(r[st][0]) == np.float32(s), (label, st)
        for name, sref in (("y", "sy"), ("dx", "sdx"), ("dw", "sdw")):
            assert_within_bound(bf16_to_f64_bits(r[name]), ref[name], ref[sref], label + " " + name)
    # dW fused into the backward product equals the GEMM kernel's (zeros may differ in sign).
    assert np.array_equal(bf16_to_f64_bits(runs["fused"]["dw"]),
                          bf16_to_f64_bits(runs["no_dw_fusion"]["dw"]))
    # Only the fusion of dW differs between these two: y and dX are the same bits.
    for name in ("y", "dx"):
        assert np.array_equal(runs["fused"][name], runs["no_dw_fusion"][name]), name


@pytest.mark.parametrize("mkn", [(256, 4096, 4096), (208, 1552, 784)])
def test_paired_forward_cast_switch(tmp_path, mkn):
    paired = _run(tmp_path, "paired", {"FP8LIN_PAIR_CAST": "1"}, mkn)
    apart = _run(tmp_path, "apart", {"FP8LIN_PAIR_CAST": "0"}, mkn)
    assert int(apart["launches"][0]) == int(paired["launches"][0]) + 1
    for name in ("x8", "x8t", "w8", "w8t", "dy8", "dy8t", "y", "dx", "dw", "sx", "sw", "sdy"):
        assert np.array_equal(paired[name], apart[name]), name
