"""Parity of the dynamic amax -> scale -> cast (+ transpose) at the sizes of
the cast-only bandwidth sweep: bf16 tensors of 2^20 ... 2^30 elements shaped
[R, 4096] and [4096, R], in the configurations the benchmark times
(two-pass atomic amax, and the automatic choice that takes the single pass
when the tensor fits on chip).  The amax, scale and inverse scale are
compared exactly; the fp8 bytes on sampled rows of q and the matching
columns of q^T.  Edge tensors (all-zero, +-1, +-max-finite, subnormals, one
non-zero, amax at the last element) are compared in full."""
import numpy as np
import pytest
import torch

import oracle
import quantised_gemm_gb300 as q
import synth_inputs as si
from helpers import dev_f32_bits, f32_bits, to_dev_bf16

pytestmark = pytest.mark.gpu

E4M3, E5M2 = oracle.E4M3, oracle.E5M2


@pytest.fixture(scope="module")
def ws():
    return q.Workspace()


def _check(x_host, rows, cols, fmt, algo, ws, seed):
    xd = to_dev_bf16(x_host.reshape(rows, cols))
    st = q.ScalingState(fmt, q.DYNAMIC, amax_algo=algo)
    out = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    out_t = torch.empty((cols, rows), dtype=torch.uint8, device="cuda")
    q.cast_dynamic(xd, st, out, out_t, ws)
    q.check(ws)
    xs = x_host.reshape(rows, cols)
    a = oracle.amax(xs)
    s, inv = oracle.scale_dynamic(a, fmt)
    assert dev_f32_bits(st.amax) == f32_bits(a)
    assert dev_f32_bits(st.scale) == f32_bits(s)
    assert dev_f32_bits(st.inv_scale) == f32_bits(inv)
    g = np.random.default_rng(seed)
    sel = np.unique(np.concatenate([g.integers(0, rows, 6), [0, rows - 1]]))
    ref = oracle.cast_rows(xs, sel, s, fmt)
    idx = torch.from_numpy(sel).cuda()
    assert np.array_equal(out[idx].cpu().numpy(), ref)
    assert np.array_equal(out_t[:, idx].cpu().numpy().T, ref)
    del xd, out, out_t
    torch.cuda.empty_cache()


@pytest.mark.parametrize("log2n", [20, 22, 24, 26, 28, 30])
def test_cast_sweep_sizes(log2n, ws):
    n = 1 << log2n
    x = si.normal_bf16((n,), 1.0, log2n, 1)
    fmt = E4M3 if log2n % 4 == 0 else E5M2
    R = n // 4096
    for algo in (q.AMAX_ATOMIC, q.AMAX_AUTO):
        _check(x, R, 4096, fmt, algo, ws, seed=log2n)
        _check(x, 4096, R, fmt, algo, ws, seed=log2n + 1)


@pytest.mark.parametrize("kind", si.EDGE_KINDS)
@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_cast_sweep_edge_tensors(kind, fmt, ws):
    x = si.edge_tensor(kind, 256, 4096, seed=4)
    a = oracle.amax(x)
    s, inv = oracle.scale_dynamic(a, fmt)
    qr, qtr, _ = oracle.cast(x, s, fmt, transpose=True)
    for algo in (q.AMAX_ATOMIC, q.AMAX_REDUCTION, q.AMAX_SINGLE_PASS):
        st = q.ScalingState(fmt, q.DYNAMIC, amax_algo=algo)
        out = torch.empty((256, 4096), dtype=torch.uint8, device="cuda")
        out_t = torch.empty((4096, 256), dtype=torch.uint8, device="cuda")
        q.cast_dynamic(to_dev_bf16(x), st, out, out_t, ws)
        assert dev_f32_bits(st.amax) == f32_bits(a), (kind, algo)
        assert dev_f32_bits(st.scale) == f32_bits(s), (kind, algo)
        assert dev_f32_bits(st.inv_scale) == f32_bits(inv), (kind, algo)
        assert np.array_equal(out.cpu().numpy(), qr), (kind, algo)
        assert np.array_equal(out_t.cpu().numpy(), qtr), (kind, algo)
