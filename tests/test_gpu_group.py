"""The backward's two GEMMs (dX and dW) in one launch of the grouped pair
kernel, against two launches of the pair kernel: FP8LIN_GROUP (read once per
process, so each setting runs in a child process) 0 never groups, 2 always
groups when both GEMMs run on 256-wide pair tiles.  Same fp8 bytes and scales,
every output within the oracle's bound, one launch fewer when grouped, and dX
and dW the same bits wherever the separate launch runs whole tiles (no K
split: the same accumulation order).  The grouped launch also delivers
max |dX| from its epilogue; with both amaxes asked for, the two GEMMs run as
two launches.  The shapes cover one round, several rounds with the long
tiles' pairs taking d short ones, and ragged edges, plus three seeded random
ones."""
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
SHAPES = [(4096, 2048, 1024), (2064, 1552, 784), (1040, 784, 2000), (3008, 1200, 4992),
          (2064, 2064, 1552)]  # the last: 144 tiles of 13 and 17 K blocks, four epilogue warps
# and three seeded random ones, every size a multiple of 16 above 128 (both
# products on 256-wide pair tiles), mostly ragged
_g = np.random.default_rng(53)
SHAPES += [tuple(int(v) * 16 for v in _g.integers(9, 200, 3)) for _ in range(3)]

CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1])
import quantised_gemm_gb300 as q, synth_inputs as si
out = {}
for i, (M, K, N) in enumerate(%r):
    x, w, dy = si.linear_inputs(M, K, N, w_init="uniform64", outlier_frac=1e-3, seed=91 + i)
    dev = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    lin = q.Fp8Linear(M, K, N)
    lin.dx_amax_to = torch.zeros(1, dtype=torch.float32, device="cuda")  # max |dX| from the epilogue
    lin.forward(dev(x), dev(w))
    torch.cuda.synchronize()
    n0 = q.launch_count()
    lin.backward(dev(dy))
    q.check(lin.ws)
    out["launches%%d" %% i] = np.array([q.launch_count() - n0])
    out["dxamax%%d" %% i] = lin.dx_amax_to.cpu().numpy()
    # Both amaxes asked for: never one launch (it publishes one); same dX and dW.
    amx = torch.zeros(2, dtype=torch.float32, device="cuda")
    dx2, dw2 = torch.empty_like(lin.dx), torch.empty_like(lin.dw)
    n0 = q.launch_count()
    q.backward(dev(dy), lin.x8t, lin.w8t, lin.sx, lin.sw, lin.sdy, lin.dy8, lin.dy8t, dx2, dw2,
               lin.ws, dx_amax=amx[0:1], dw_amax=amx[1:2])
    q.check(lin.ws)
    out["launches_both%%d" %% i] = np.array([q.launch_count() - n0])
    out["amax_both%%d" %% i] = amx.cpu().numpy()
    out["dx_both%%d" %% i] = dx2.cpu().view(torch.int16).numpy()
    out["dw_both%%d" %% i] = dw2.cpu().view(torch.int16).numpy()
    for name in ("x8", "w8", "dy8", "dy8t"):
        out[name + "%%d" %% i] = getattr(lin, name).cpu().numpy()
    for name in ("y", "dx", "dw"):
        out[name + "%%d" %% i] = getattr(lin, name).cpu().view(torch.int16).numpy()
    for st in ("sx", "sw", "sdy"):
        out[st + "%%d" %% i] = getattr(lin, st).scale.cpu().numpy()
    out["desc_dx%%d" %% i] = np.array(q.gemm_describe(M, K, N))
    out["desc_dw%%d" %% i] = np.array(q.gemm_describe(N, K, M))
np.savez(sys.argv[2], **out)
""" % (SHAPES,)


def _run(tmp_path, mode):
    path = os.path.join(tmp_path, "group%s.npz" % mode)
    env = dict(os.environ, FP8LIN_GROUP=mode)
    subprocess.run([sys.executable, "-c", CHILD, ROOT, path], env=env, check=True, timeout=900)
    return dict(np.load(path))


def bf16_to_f64_bits(bits):
    return (bits.astype(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_grouped_backward_matches_separate(tmp_path):
    sep, grp = _run(tmp_path, "0"), _run(tmp_path, "2")
    for i, (M, K, N) in enumerate(SHAPES):
        assert int(sep["launches%d" % i][0]) - int(grp["launches%d" % i][0]) == 1, (M, K, N)
        x, w, dy = si.linear_inputs(M, K, N, w_init="uniform64", outlier_frac=1e-3, seed=91 + i)
        sx = oracle.scale_dynamic(oracle.amax(x), oracle.E4M3)[0]
        sw = oracle.scale_dynamic(oracle.amax(w), oracle.E4M3)[0]
        sd = oracle.scale_dynamic(oracle.amax(dy), oracle.E5M2)[0]
        ref = oracle.linear_fwd_bwd(x, w, dy, sx, sw, sd)
        for label, r in (("separate", sep), ("grouped", grp)):
            for name in ("x8", "w8", "dy8", "dy8t"):
                assert np.array_equal(r[name + str(i)], ref[name]), (label, name, M, K, N)
            for st, s in (("sx", sx), ("sw", sw), ("sdy", sd)):
                assert np.float32(r[st + str(i)][0]) == np.float32(s), (label, st)
            for name, sref in (("y", "sy"), ("dx", "sdx"), ("dw", "sdw")):
                assert_within_bound(bf16_to_f64_bits(r[name + str(i)]), ref[name], ref[sref],
                                    "%s %s %s" % (label, name, (M, K, N)))
        assert np.array_equal(sep["y%d" % i], grp["y%d" % i])
        for label, r in (("separate", sep), ("grouped", grp)):
            # the epilogue's max |dX| is that of the stored bf16 dX, exactly
            dx = bf16_to_f64_bits(r["dx%d" % i])
            assert np.float32(r["dxamax%d" % i][0]) == np.float32(np.abs(dx).max()), label
            # with both amaxes asked for, dX and dW run as two launches in either mode
            assert int(r["launches_both%d" % i][0]) == int(sep["launches%d" % i][0]), label
            dw = bf16_to_f64_bits(r["dw_both%d" % i])
            assert np.float32(r["amax_both%d" % i][1]) == np.float32(np.abs(dw).max()), label
            assert np.float32(r["amax_both%d" % i][0]) == np.float32(
                np.abs(bf16_to_f64_bits(r["dx_both%d" % i])).max()), label
        for name in ("dx", "dw"):
            if str(sep["desc_%s%d" % (name, i)]).endswith("whole tiles"):
                assert np.array_equal(sep[name + str(i)], grp[name + str(i)]), (name, M, K, N)
