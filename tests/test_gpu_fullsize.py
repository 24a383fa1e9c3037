"""Full-size parity of the fp8 Linear against the oracle, at the sizes and in
the launch configuration the benchmark times.

Every fp8 byte (x8, x8^T, W8, W8^T, dY8, dY8^T) is compared with the oracle's
cast, and amax, scale and inverse scale exactly.  The three GEMM outputs are
compared on whole tiles: the first and last row bands, the N-edge column
band, every tile the planner runs as K slices (the tail of the 65536-deep dW
product), and random entries; small products in full (tests/fullsize.py).

Workloads: the 4096 -> 4096 Linear of the single-linear table of "Integrate
float8nocompile, an experimental feature for high performance" (torchtitan
PR 778) at M = 16, 256, 4096 and 65536 with dynamic scaling; the Llama-3-8B
FFN Linears (that PR's training table) at M = 8192; the GPT-1.5B block
Linears of "[float8] FP8 GPT 1.5B Delayed Scaling 2x Slower than BF16"
(pytorch/ao issue 1297) at M = 12 x 1024 with delayed scaling, H = 16, over
20 steps, checked in full at steps 0, 1, 15 and 19 and on the scalars at
every step."""
import numpy as np
import pytest
import torch

import oracle
import quantised_gemm_gb300 as q
import synth_inputs as si
from fullsize import check_linear
from helpers import dev_f32_bits, f32_bits, to_dev_bf16

pytestmark = pytest.mark.gpu

E4M3, E5M2 = oracle.E4M3, oracle.E5M2


def _dynamic_full(name, idx):
    M, K, N = si.WORKLOADS[name]["shapes"][idx]
    x, w, dy = si.workload_inputs(name, idx)
    lin = q.Fp8Linear(M, K, N)              # the benchmark's configuration (AMAX_AUTO)
    lin.forward(to_dev_bf16(x), to_dev_bf16(w))
    lin.backward(to_dev_bf16(dy))
    q.check(lin.ws)
    sx, ix = oracle.scale_dynamic(oracle.amax(x), E4M3)
    sw, iw = oracle.scale_dynamic(oracle.amax(w), E4M3)
    sd, idy = oracle.scale_dynamic(oracle.amax(dy), E5M2)
    for st, s, inv, src in ((lin.sx, sx, ix, x), (lin.sw, sw, iw, w), (lin.sdy, sd, idy, dy)):
        assert dev_f32_bits(st.amax) == f32_bits(oracle.amax(src))
        assert dev_f32_bits(st.scale) == f32_bits(s)
        assert dev_f32_bits(st.inv_scale) == f32_bits(inv)
    check_linear(lin, q, x, w, dy, sx, sw, sd, E4M3, E5M2, seed=idx)
    del lin
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["linear4096_m16", "linear4096_m256", "linear4096_m4096",
                                  "linear4096_m65536"])
def test_linear4096_every_byte(name):
    _dynamic_full(name, 0)


@pytest.mark.parametrize("idx", [0, 1, 2])
def test_llama3_ffn_every_byte(idx):
    _dynamic_full("llama3_8b_ffn_m8192", idx)


FULL_STEPS = (0, 1, 15, 19)


@pytest.mark.parametrize("idx", [0, 1, 2, 3])
def test_gpt_delayed_20_steps(idx):
    """One GPT-1.5B block Linear (qkv, out, fc, proj) over 20 steps of delayed
    scaling with amax init: the scale each step casts with comes from the
    amaxes of the steps before it (ring of 16); every step's scalars are
    exact, and steps 0, 1, 15, 19 are compared in full."""
    name = "gpt1.5b_linears_m12288"
    wl = si.WORKLOADS[name]
    M, K, N = wl["shapes"][idx]
    H, steps = wl["history_len"], wl["steps"]
    lin = q.Fp8Linear(M, K, N, scaling="delayed", history_len=H)
    _, w, _ = si.workload_inputs(name, idx, step=0)
    wd = to_dev_bf16(w)
    refs = {"x": oracle.DelayedState(H, E4M3), "w": oracle.DelayedState(H, E4M3),
            "dy": oracle.DelayedState(H, E5M2)}
    amax_w = oracle.amax(w)
    for t in range(steps):
        x, _, dy = si.workload_inputs(name, idx, step=t)
        amaxes = {"x": oracle.amax(x), "w": amax_w, "dy": oracle.amax(dy)}
        if t == 0:
            for k in refs:
                refs[k].init_from(amaxes[k])
        used = {k: (refs[k].scale, refs[k].inv_scale) for k in refs}
        lin.forward(to_dev_bf16(x), wd)
        lin.backward(to_dev_bf16(dy))
        for k, st in (("x", lin.sx), ("w", lin.sw), ("dy", lin.sdy)):
            assert dev_f32_bits(st.scale) == f32_bits(used[k][0]), (t, k)
            assert dev_f32_bits(st.inv_scale) == f32_bits(used[k][1]), (t, k)
            assert dev_f32_bits(st.amax) == f32_bits(amaxes[k]), (t, k)
        if t in FULL_STEPS:
            q.check(lin.ws)
            check_linear(lin, q, x, w, dy, used["x"][0], used["w"][0], used["dy"][0], E4M3,
                         E5M2, seed=t)
        lin.sync_scales()
        for k in refs:
            refs[k].update(amaxes[k])
    for k, st in (("x", lin.sx), ("w", lin.sw), ("dy", lin.sdy)):
        assert dev_f32_bits(st.scale) == f32_bits(refs[k].scale)
        assert np.array_equal(st.amax_history.cpu().numpy().view(np.uint32),
                              refs[k].ring.view(np.uint32))
        assert int(st.head.item()) == refs[k].head
    q.check(lin.ws)
