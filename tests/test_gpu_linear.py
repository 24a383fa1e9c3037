"""GPU parity of the whole fp8 Linear step (forward + backward, dynamic and
delayed scaling) against the oracle on small and ragged shapes, element by
element, plus the host-buffer step, chained Linears, the cached weight and
degenerate sizes.  The full workload sizes are in test_gpu_fullsize.py."""
import numpy as np
import pytest
import torch

import oracle
import quantised_gemm_gb300 as q
import synth_inputs as si
from helpers import assert_within_bound, bf16_to_f64, dev_f32_bits, f32_bits, to_dev_bf16

pytestmark = pytest.mark.gpu

E4M3, E5M2 = oracle.E4M3, oracle.E5M2


def _check_full(lin, x, w, dy, sx, sw, sd):
    ref = oracle.linear_fwd_bwd(x, w, dy, sx, sw, sd)
    for name in ("x8", "x8t", "w8", "w8t", "dy8", "dy8t"):
        assert np.array_equal(getattr(lin, name).cpu().numpy(), ref[name]), name
    for name, sname in (("y", "sy"), ("dx", "sdx"), ("dw", "sdw")):
        assert_within_bound(bf16_to_f64(getattr(lin, name)), ref[name], ref[sname], name)


@pytest.mark.parametrize("mkn", [(16, 4096, 4096), (256, 4096, 4096), (144, 272, 208),
                                 (48, 160, 96), (1040, 784, 512), (208, 1552, 784)])
@pytest.mark.parametrize("algo", [q.AMAX_ATOMIC, q.AMAX_REDUCTION, q.AMAX_SINGLE_PASS, q.AMAX_AUTO])
def test_linear_dynamic_full_compare(mkn, algo):
    M, K, N = mkn
    x, w, dy = si.linear_inputs(M, K, N, w_init="uniform64", outlier_frac=1e-3, seed=M + N)
    lin = q.Fp8Linear(M, K, N, amax_algo=algo)
    lin.forward(to_dev_bf16(x), to_dev_bf16(w))
    lin.backward(to_dev_bf16(dy))
    q.check(lin.ws)
    sx, invx = oracle.scale_dynamic(oracle.amax(x), E4M3)
    sw, _ = oracle.scale_dynamic(oracle.amax(w), E4M3)
    sd, _ = oracle.scale_dynamic(oracle.amax(dy), E5M2)
    assert dev_f32_bits(lin.sx.scale) == f32_bits(sx)
    assert dev_f32_bits(lin.sx.inv_scale) == f32_bits(invx)
    assert dev_f32_bits(lin.sw.scale) == f32_bits(sw)
    assert dev_f32_bits(lin.sdy.scale) == f32_bits(sd)
    _check_full(lin, x, w, dy, sx, sw, sd)


def _paired_cast_shapes(n, seed=47):
    """Seeded shapes whose forward casts x with W in one launch: more than 32
    tokens, W above the one-cluster cast and within the single pass (in
    128 x 128 tiles), x at most one tile for each CTA of W's launch (the
    smaller of W's tile count and 152); sizes multiples of 16, mostly ragged."""
    g = np.random.default_rng(seed)
    tiles = lambda r, c: -(-r // 128) * -(-c // 128)  # noqa: E731
    out = []
    while len(out) < n:
        M, K, N = (int(v) * 16 for v in (g.integers(3, 38), g.integers(1, 129), g.integers(1, 257)))
        if (M > 32 and N * K >= 1 << 20 and tiles(N, K) <= 152 * 7
                and tiles(M, K) <= min(tiles(N, K), 152)):
            out.append((M, K, N))
    return out


@pytest.mark.parametrize("mkn", _paired_cast_shapes(8))
def test_paired_forward_cast_random_shapes(mkn):
    """The paired single pass (W's tiles in shared memory, x's one tile per
    CTA in registers, both maxima at one grid barrier) on random ragged
    shapes: the forward is two launches, and every fp8 byte, scale and GEMM
    output matches the oracle."""
    M, K, N = mkn
    x, w, dy = si.linear_inputs(M, K, N, w_init="uniform64", outlier_frac=1e-3, seed=M + K + N)
    lin = q.Fp8Linear(M, K, N)
    torch.cuda.synchronize()
    n0 = q.launch_count()
    lin.forward(to_dev_bf16(x), to_dev_bf16(w))
    torch.cuda.synchronize()
    assert q.launch_count() - n0 == 2, mkn
    lin.backward(to_dev_bf16(dy))
    q.check(lin.ws)
    sx, invx = oracle.scale_dynamic(oracle.amax(x), E4M3)
    sw, invw = oracle.scale_dynamic(oracle.amax(w), E4M3)
    sd, _ = oracle.scale_dynamic(oracle.amax(dy), E5M2)
    for st, s, inv in ((lin.sx, sx, invx), (lin.sw, sw, invw)):
        assert dev_f32_bits(st.scale) == f32_bits(s) and dev_f32_bits(st.inv_scale) == f32_bits(inv)
    assert dev_f32_bits(lin.sdy.scale) == f32_bits(sd)
    _check_full(lin, x, w, dy, sx, sw, sd)


def _few_token_shapes(n, seed=59):
    """Seeded shapes of the few-token fused products: 16 or 32 tokens, K and N
    multiples of 16 up to 4096 with the weight in at most 152 x 7 tiles."""
    g = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        M, K, N = int(g.choice([16, 32])), int(g.integers(1, 257)) * 16, int(g.integers(1, 257)) * 16
        if -(-K // 128) * -(-N // 128) <= 152 * 7:
            out.append((M, K, N))
    return out


@pytest.mark.parametrize("mkn", _few_token_shapes(4))
def test_few_token_fused_random_shapes(mkn):
    """The two fused few-token products on random ragged shapes: one launch
    each way, every fp8 byte and scale exact, y, dX and dW within the bound."""
    M, K, N = mkn
    x, w, dy = si.linear_inputs(M, K, N, w_init="uniform64", outlier_frac=1e-2, seed=M * K + N)
    lin = q.Fp8Linear(M, K, N)
    launches = []
    for call in (lambda: lin.forward(to_dev_bf16(x), to_dev_bf16(w)),
                 lambda: lin.backward(to_dev_bf16(dy))):
        torch.cuda.synchronize()
        n0 = q.launch_count()
        call()
        torch.cuda.synchronize()
        launches.append(q.launch_count() - n0)
    q.check(lin.ws)
    assert launches == [1, 1], (mkn, launches)
    sx, _ = oracle.scale_dynamic(oracle.amax(x), E4M3)
    sw, _ = oracle.scale_dynamic(oracle.amax(w), E4M3)
    sd, _ = oracle.scale_dynamic(oracle.amax(dy), E5M2)
    for st, s in ((lin.sx, sx), (lin.sw, sw), (lin.sdy, sd)):
        assert dev_f32_bits(st.scale) == f32_bits(s)
    _check_full(lin, x, w, dy, sx, sw, sd)


@pytest.mark.parametrize("mkn", [(16, 272, 208), (32, 784, 1040), (16, 16, 16), (32, 4096, 4096),
                                 (16, 2048, 6144)])
@pytest.mark.parametrize("given_amax", [False, True])
def test_few_token_fused_path(mkn, given_amax):
    """M <= 32 tokens with dynamic scaling: x's cast, W's cast and y in one
    launch, dY's cast, dX and dW in another.  Every fp8 byte and scalar
    exact, the GEMMs within the bound, over ragged bands and K tails; with
    given_amax the token-side amaxes come from the caller (PRECOMPUTED), as a
    producing GEMM's epilogue would deliver them.  The fused dW equals the
    GEMM kernel's dW on the same fp8 operands, value for value."""
    M, K, N = mkn
    x, w, dy = si.linear_inputs(M, K, N, w_init="uniform64", outlier_frac=1e-2, seed=M + K + N)
    lin = q.Fp8Linear(M, K, N)
    if given_amax:
        lin.sx.amax_algo = lin.sdy.amax_algo = q.AMAX_PRECOMPUTED
        lin.sx.amax.fill_(oracle.amax(x))
        lin.sdy.amax.fill_(oracle.amax(dy))
    n0 = q.launch_count()
    lin.forward(to_dev_bf16(x), to_dev_bf16(w))
    lin.backward(to_dev_bf16(dy))
    assert q.launch_count() - n0 == 2              # fused forward, fused dY + dX + dW
    q.check(lin.ws)
    sx, ix = oracle.scale_dynamic(oracle.amax(x), E4M3)
    sw, iw = oracle.scale_dynamic(oracle.amax(w), E4M3)
    sd, idy = oracle.scale_dynamic(oracle.amax(dy), E5M2)
    for st, s, inv, src in ((lin.sx, sx, ix, x), (lin.sw, sw, iw, w), (lin.sdy, sd, idy, dy)):
        assert dev_f32_bits(st.amax) == f32_bits(oracle.amax(src))
        assert dev_f32_bits(st.scale) == f32_bits(s)
        assert dev_f32_bits(st.inv_scale) == f32_bits(inv)
    _check_full(lin, x, w, dy, sx, sw, sd)
    dw_gemm = torch.empty_like(lin.dw)
    q.gemm(lin.dy8t, lin.x8t, E5M2, E4M3, lin.sdy.inv_scale, lin.sx.inv_scale, dw_gemm, lin.ws)
    q.check(lin.ws)
    assert torch.equal(lin.dw.float(), dw_gemm.float())  # (zeros may differ in sign)


def test_few_token_fused_output_amaxes_and_repeat():
    """The fused few-token products deliver max |y| and max |dX| from their
    reduction, and a second call on the same workspace gives the same bits
    (the band tickets and amax words clean themselves)."""
    M, K, N = 16, 784, 1040
    lin = q.Fp8Linear(M, K, N)
    x, w, dy = si.linear_inputs(M, K, N, w_init="uniform64", seed=61)
    ya, dxa = (torch.full((1,), -1.0, device="cuda") for _ in range(2))
    outs = []
    for _ in range(2):
        q.forward(to_dev_bf16(x), to_dev_bf16(w), lin.sx, lin.sw, lin.y, lin.x8, lin.x8t, lin.w8,
                  lin.w8t, lin.ws, y_amax=ya)
        q.backward(to_dev_bf16(dy), lin.x8t, lin.w8t, lin.sx, lin.sw, lin.sdy, lin.dy8, lin.dy8t,
                   lin.dx, lin.dw, lin.ws, dx_amax=dxa)
        q.check(lin.ws)
        assert dev_f32_bits(ya) == f32_bits(oracle.amax(_bits(lin.y)))
        assert dev_f32_bits(dxa) == f32_bits(oracle.amax(_bits(lin.dx)))
        outs.append([_bits(t) for t in (lin.y, lin.dx, lin.dw)])
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("M", [16, 32])
def test_few_token_backward_variants(M):
    """The few-token backward with dW's amax asked for (dW then runs as its own
    GEMM after the fused dY / dX launch), with dX skipped (no fused launch),
    and with dW skipped: every variant's dX and dW equal the fused launch's
    value for value, and max |dW| is the stored dW's."""
    K, N = 784, 1040
    x, w, dy = si.linear_inputs(M, K, N, w_init="uniform64", seed=67)
    lin = q.Fp8Linear(M, K, N)
    lin.forward(to_dev_bf16(x), to_dev_bf16(w))
    dyd = to_dev_bf16(dy)
    n0 = q.launch_count()
    lin.backward(dyd)
    assert q.launch_count() - n0 == 1               # dY's cast, dX and dW in one launch
    dx_f, dw_f = lin.dx.clone(), lin.dw.clone()
    dwa = torch.full((1,), -1.0, device="cuda")
    q.backward(dyd, lin.x8t, lin.w8t, lin.sx, lin.sw, lin.sdy, lin.dy8, lin.dy8t, lin.dx, lin.dw,
               lin.ws, dw_amax=dwa)
    q.check(lin.ws)
    assert torch.equal(lin.dx.view(torch.int16), dx_f.view(torch.int16))
    assert torch.equal(lin.dw.float(), dw_f.float())
    assert dev_f32_bits(dwa) == f32_bits(oracle.amax(_bits(lin.dw)))
    lin.dx.fill_(5.0)
    lin.dw.zero_()
    lin.backward(dyd, need_dx=False)
    assert torch.all(lin.dx == 5.0) and torch.equal(lin.dw.float(), dw_f.float())
    lin.dw.fill_(5.0)
    lin.backward(dyd, need_dw=False)
    q.check(lin.ws)
    assert torch.all(lin.dw == 5.0)
    assert torch.equal(lin.dx.view(torch.int16), dx_f.view(torch.int16))


def test_linear_delayed_small_full_compare():
    """Delayed scaling with a stale scale can saturate; compare everything."""
    M, K, N = 144, 272, 208
    H = 3
    lin = q.Fp8Linear(M, K, N, scaling="delayed", history_len=H)
    _, w, _ = si.linear_inputs(M, K, N, w_init="kaiming", seed=5)
    refs = [oracle.DelayedState(H, f) for f in (E4M3, E4M3, E5M2)]
    for t in range(6):
        x, _, dy = si.linear_inputs(M, K, N, w_init="kaiming", x_std=4.0 ** t, seed=5, step=t)
        am = [oracle.amax(x), oracle.amax(w), oracle.amax(dy)]
        if t == 0:
            for r, a in zip(refs, am):
                r.init_from(a)
        lin.forward(to_dev_bf16(x), to_dev_bf16(w))
        lin.backward(to_dev_bf16(dy))
        _check_full(lin, x, w, dy, refs[0].scale, refs[1].scale, refs[2].scale)
        lin.sync_scales()
        for r, a in zip(refs, am):
            r.update(a)


def test_backward_without_dx_or_dw():
    M, K, N = 128, 256, 192
    x, w, dy = si.linear_inputs(M, K, N, w_init="uniform64", seed=9)
    lin = q.Fp8Linear(M, K, N)
    lin.forward(to_dev_bf16(x), to_dev_bf16(w))
    lin.dx.fill_(5.0)
    lin.backward(to_dev_bf16(dy), need_dx=False)
    assert torch.all(lin.dx == 5.0)
    lin.dw.fill_(5.0)
    lin.backward(to_dev_bf16(dy), need_dw=False)
    assert torch.all(lin.dw == 5.0)


def test_bad_arguments_raise_without_launch():
    lin = q.Fp8Linear(128, 256, 192)
    x = torch.zeros((128, 256), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((192, 256), dtype=torch.bfloat16, device="cuda")
    before = q.launch_count()
    with pytest.raises(q.Fp8linError):   # M not a multiple of 16
        q.forward(x[:100], w, lin.sx, lin.sw, lin.y[:100], lin.x8, lin.x8t, lin.w8, lin.w8t,
                  lin.ws)
    lin.sx.fmt = E5M2                     # wrong format for the input role
    with pytest.raises(q.Fp8linError):
        lin.forward(x, w)
    lin.sx.fmt = E4M3
    lin.sx.eps = 0.0
    with pytest.raises(q.Fp8linError):
        lin.forward(x, w)
    assert q.launch_count() == before


@pytest.mark.parametrize("scaling", ["dynamic", "delayed"])
def test_step_host_matches_device_path(scaling):
    """The host-buffer step (fp8lin_step_host: uploads and downloads on copy
    streams, ordered by the slot's events, two slots used in turn) returns
    the bits of the device path, over consecutive steps; with delayed
    scaling the history sync runs inside the step as well."""
    M, K, N = 560, 768, 1024
    dev_lin = q.Fp8Linear(M, K, N, scaling=scaling, history_len=4)
    host_lin = q.Fp8Linear(M, K, N, scaling=scaling, history_len=4)
    hy = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    hdx = torch.empty((M, K), dtype=torch.bfloat16).pin_memory()
    hdw = torch.empty((N, K), dtype=torch.bfloat16).pin_memory()
    for step in range(3):
        x, w, dy = si.linear_inputs(M, K, N, w_init="uniform64", seed=3, step=step)
        pin = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory()
        host_lin.step_host(pin(x), pin(w), pin(dy), hy, hdx, hdw)
        torch.cuda.current_stream().synchronize()
        dev_lin.step(to_dev_bf16(x), to_dev_bf16(w), to_dev_bf16(dy))
        torch.cuda.synchronize()
        assert torch.equal(hy.view(torch.int16), dev_lin.y.cpu().view(torch.int16)), step
        assert torch.equal(hdx.view(torch.int16), dev_lin.dx.cpu().view(torch.int16)), step
        assert torch.equal(hdw.view(torch.int16), dev_lin.dw.cpu().view(torch.int16)), step
        for a, b in ((host_lin.sx, dev_lin.sx), (host_lin.sw, dev_lin.sw),
                     (host_lin.sdy, dev_lin.sdy)):
            assert dev_f32_bits(a.scale) == dev_f32_bits(b.scale), step


def test_step_host_rejects_bad_arguments_without_launch():
    lin = q.Fp8Linear(128, 256, 192)
    good = dict(x_h=torch.empty((128, 256), dtype=torch.bfloat16),
                w_h=torch.empty((192, 256), dtype=torch.bfloat16),
                dy_h=torch.empty((128, 192), dtype=torch.bfloat16),
                y_h=torch.empty((128, 192), dtype=torch.bfloat16),
                dx_h=torch.empty((128, 256), dtype=torch.bfloat16),
                dw_h=torch.empty((192, 256), dtype=torch.bfloat16))
    before = q.launch_count()
    bad = dict(good, x_h=torch.empty((128, 256), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError):
        lin.step_host(**bad)
    lin.sdy.fmt = E4M3                    # wrong format for the grad_output role
    with pytest.raises(q.Fp8linError):
        lin.step_host(**good)
    assert q.launch_count() == before


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def test_forward_backward_output_amaxes():
    """y_amax, dx_amax and dw_amax from the GEMM epilogues equal the oracle's
    amax of the y, dX and dW the GPU stored."""
    M, K, N = 560, 768, 1024
    lin = q.Fp8Linear(M, K, N)
    ya, dxa, dwa = (torch.full((1,), -1.0, device="cuda") for _ in range(3))
    x, w, dy = si.linear_inputs(M, K, N, w_init="uniform64", seed=5)
    q.forward(to_dev_bf16(x), to_dev_bf16(w), lin.sx, lin.sw, lin.y, lin.x8, lin.x8t, lin.w8,
              lin.w8t, lin.ws, y_amax=ya)
    q.backward(to_dev_bf16(dy), lin.x8t, lin.w8t, lin.sx, lin.sw, lin.sdy, lin.dy8, lin.dy8t,
               lin.dx, lin.dw, lin.ws, dx_amax=dxa, dw_amax=dwa)
    q.check(lin.ws)
    for t, a, what in ((lin.y, ya, "y"), (lin.dx, dxa, "dX"), (lin.dw, dwa, "dW")):
        assert dev_f32_bits(a) == f32_bits(oracle.amax(_bits(t))), what


@pytest.mark.parametrize("M", [16, 560])
def test_linked_linears_match_unlinked(M):
    """Two Linears chained with link_linears (amax of y and dX from the GEMM
    epilogues, casts of y and dX in one pass) give the same bits as the same
    chain with separate amax passes, over two steps; the linked states hold
    the oracle's amax of the tensors they cast."""
    K, N1, N2 = 768, 1024, 512
    x, w1, _ = si.linear_inputs(M, K, N1, w_init="uniform64", seed=8)
    _, w2, dy2 = si.linear_inputs(M, N1, N2, w_init="uniform64", seed=9)
    xd, w1d, w2d, dy2d = (to_dev_bf16(a) for a in (x, w1, w2, dy2))

    def run(linked):
        l1, l2 = q.Fp8Linear(M, K, N1), q.Fp8Linear(M, N1, N2)
        if linked:
            q.link_linears(l1, l2)
        for _ in range(2):
            l1.forward(xd, w1d)
            l2.forward(l1.y, w2d)
            l2.backward(dy2d)
            l1.backward(l2.dx)
        q.check(l1.ws)
        q.check(l2.ws)
        outs = [_bits(t) for t in (l1.y, l2.y, l2.dx, l1.dx, l1.dw, l2.dw)]
        scalars = [dev_f32_bits(t) for t in (l2.sx.amax, l2.sx.scale, l1.sdy.amax, l1.sdy.scale)]
        if linked:
            assert scalars[0] == f32_bits(oracle.amax(outs[0]))     # amax of y1
            assert scalars[2] == f32_bits(oracle.amax(outs[2]))     # amax of dX2
        return outs, scalars

    (o1, s1), (o2, s2) = run(True), run(False)
    for i, (u, v) in enumerate(zip(o1, o2)):
        assert np.array_equal(u, v), i
    assert s1 == s2


@pytest.mark.parametrize("M", [16, 48])
def test_cached_weight_dynamic_matches_recast(M):
    """cache_weight: micro-batches with the same W skip W's cast and give the
    bits of a fresh cast; an in-place update of W makes the next forward cast
    again.  At 48 tokens the forward is two launches either way (x's cast
    with W's in one paired launch, or x's alone, then y); at 16 tokens it is
    one fused launch either way.  The skipped cast shows in W's state, which a
    cached forward leaves untouched."""
    K, N = 4096, 4096
    lc = q.Fp8Linear(M, K, N, cache_weight=True)
    lu = q.Fp8Linear(M, K, N)
    _, w, _ = si.linear_inputs(M, K, N, w_init="uniform64", seed=31)
    wd = to_dev_bf16(w)
    for step in range(4):
        x, _, dy = si.linear_inputs(M, K, N, w_init="uniform64", seed=31, step=step)
        if step == 2:
            wd.mul_(2.0)                       # an optimizer step, in place
        lc.sw.amax.fill_(-1.0)                 # only a cast of W writes it
        n0 = q.launch_count()
        lc.forward(to_dev_bf16(x), wd)
        launches = q.launch_count() - n0
        cast_w = step in (0, 2)
        assert launches == (2 if M > 32 else 1), (step, launches)
        torch.cuda.synchronize()
        assert (lc.sw.amax.item() > 0) == cast_w, step
        lc.backward(to_dev_bf16(dy))
        lu.forward(to_dev_bf16(x), wd)
        lu.backward(to_dev_bf16(dy))
        torch.cuda.synchronize()
        for a, b, what in ((lc.y, lu.y, "y"), (lc.dx, lu.dx, "dX"), (lc.dw, lu.dw, "dW")):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), (step, what)


def test_cached_weight_delayed_micro_batches():
    """Delayed scaling with cache_weight: W is cast once per optimizer step
    (sync_scales moves W's scale and drops the cache) and every micro-batch
    gives the bits of the uncached Linear."""
    M, K, N = 256, 768, 1024
    lc = q.Fp8Linear(M, K, N, scaling="delayed", history_len=4, cache_weight=True)
    lu = q.Fp8Linear(M, K, N, scaling="delayed", history_len=4)
    _, w, _ = si.linear_inputs(M, K, N, w_init="uniform64", seed=37)
    wd = to_dev_bf16(w)
    for step in range(3):
        for micro in range(3):
            x, _, dy = si.linear_inputs(M, K, N, w_init="uniform64", seed=37,
                                        step=3 * step + micro)
            for lin in (lc, lu):
                lin.forward(to_dev_bf16(x), wd)
                lin.backward(to_dev_bf16(dy))
            torch.cuda.synchronize()
            for a, b, what in ((lc.y, lu.y, "y"), (lc.dx, lu.dx, "dX"), (lc.dw, lu.dw, "dW")):
                assert torch.equal(a.view(torch.int16), b.view(torch.int16)), (step, micro, what)
        lc.sync_scales()
        lu.sync_scales()
        torch.cuda.synchronize()
        assert dev_f32_bits(lc.sw.scale) == dev_f32_bits(lu.sw.scale)


def test_linear_degenerate_sizes_and_zero_tensors():
    """M = 0 (no tokens): dW is all zeros and x's amax is 0 with scale F/eps.
    All-zero x and dY: every code is +0, y, dX, dW are zeros, and the scales
    are F/eps exactly as the oracle derives them."""
    K, N = 256, 384
    lin = q.Fp8Linear(0, K, N)
    _, w, _ = si.linear_inputs(16, K, N, w_init="uniform64", seed=41)
    lin.dw.fill_(1.0)
    lin.forward(torch.empty((0, K), dtype=torch.bfloat16, device="cuda"), to_dev_bf16(w))
    lin.backward(torch.empty((0, N), dtype=torch.bfloat16, device="cuda"))
    q.check(lin.ws)
    assert torch.count_nonzero(lin.dw.float()).item() == 0
    s0, inv0 = oracle.scale_dynamic(0.0, oracle.E4M3)
    assert lin.sx.amax.item() == 0.0 and dev_f32_bits(lin.sx.scale) == f32_bits(s0)
    assert dev_f32_bits(lin.sx.inv_scale) == f32_bits(inv0)

    M = 64
    lin = q.Fp8Linear(M, K, N)
    x = np.zeros((M, K), dtype=np.uint16)
    dy = np.zeros((M, N), dtype=np.uint16)
    lin.forward(to_dev_bf16(x), to_dev_bf16(w))
    lin.backward(to_dev_bf16(dy))
    q.check(lin.ws)
    for t in (lin.x8, lin.x8t, lin.dy8, lin.dy8t):
        assert torch.count_nonzero(t).item() == 0
    for t in (lin.y, lin.dx, lin.dw):
        assert torch.count_nonzero(t.float()).item() == 0
    s2, _ = oracle.scale_dynamic(0.0, oracle.E5M2)
    assert dev_f32_bits(lin.sx.scale) == f32_bits(s0)
    assert dev_f32_bits(lin.sdy.scale) == f32_bits(s2)


def test_step_host_pipelined_matches_device_path():
    """step_host(wait=False) over alternating device slots: four steps run
    back to back, each downloading into its own host buffers; after
    finish_host every step's y, dX, dW equal the device path's bits."""
    M, K, N = 560, 768, 1024
    dev_lin = q.Fp8Linear(M, K, N)
    host_lin = q.Fp8Linear(M, K, N)
    pin = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory()
    steps, outs, ins = 4, [], []
    for step in range(steps):
        x, w, dy = si.linear_inputs(M, K, N, w_init="uniform64", seed=5, step=step)
        ins.append((x, w, dy))
        hy = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
        hdx = torch.empty((M, K), dtype=torch.bfloat16).pin_memory()
        hdw = torch.empty((N, K), dtype=torch.bfloat16).pin_memory()
        outs.append((hy, hdx, hdw))
        host_lin.step_host(pin(x), pin(w), pin(dy), hy, hdx, hdw, wait=False)
    host_lin.finish_host()
    torch.cuda.current_stream().synchronize()
    for step, ((x, w, dy), (hy, hdx, hdw)) in enumerate(zip(ins, outs)):
        dev_lin.step(to_dev_bf16(x), to_dev_bf16(w), to_dev_bf16(dy))
        torch.cuda.synchronize()
        assert torch.equal(hy.view(torch.int16), dev_lin.y.cpu().view(torch.int16)), step
        assert torch.equal(hdx.view(torch.int16), dev_lin.dx.cpu().view(torch.int16)), step
        assert torch.equal(hdw.view(torch.int16), dev_lin.dw.cpu().view(torch.int16)), step
