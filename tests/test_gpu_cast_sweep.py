"""Parity of the dynamic amax -> scale -> cast (+ transpose) at the sizes of
the cast-only bandwidth sweep: bf16 tensors of 2^20 ... 2^30 elements shaped
[R, 4096] and [4096, R], in the configurations the benchmark times
(two-pass atomic amax, and the automatic choice that takes the single pass
when the tensor fits on chip).  The amax, scale and inverse scale are
compared exactly, and every fp8 byte of q and q^T.  Edge tensors (all-zero,
+-1, +-max-finite, subnormals, one non-zero, amax at the last element) are
compared in full as well."""
import numpy as np
import pytest
import torch

import oracle
import quantised_gemm_gb300 as q
import synth_inputs as si
from fullsize import check_bytes
from helpers import dev_f32_bits, f32_bits, to_dev_bf16

pytestmark = pytest.mark.gpu

E4M3, E5M2 = oracle.E4M3, oracle.E5M2


@pytest.fixture(scope="module")
def ws():
    return q.Workspace()


def _check(x_host, rows, cols, fmt, algos, ws):
    xs = x_host.reshape(rows, cols)
    xd = to_dev_bf16(xs)
    a = oracle.amax(xs)
    s, inv = oracle.scale_dynamic(a, fmt)
    ref, ref_t, _ = oracle.cast(xs, s, fmt, transpose=True)
    out = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    out_t = torch.empty((cols, rows), dtype=torch.uint8, device="cuda")
    for algo in algos:
        st = q.ScalingState(fmt, q.DYNAMIC, amax_algo=algo)
        out.fill_(0xAA)
        out_t.fill_(0xAA)
        q.cast_dynamic(xd, st, out, out_t, ws)
        q.check(ws)
        assert dev_f32_bits(st.amax) == f32_bits(a), algo
        assert dev_f32_bits(st.scale) == f32_bits(s), algo
        assert dev_f32_bits(st.inv_scale) == f32_bits(inv), algo
        check_bytes(out, ref, "q [%d, %d] algo %d" % (rows, cols, algo))
        check_bytes(out_t, ref_t, "q^T [%d, %d] algo %d" % (cols, rows, algo))
    del xd, out, out_t, ref, ref_t
    torch.cuda.empty_cache()


@pytest.mark.parametrize("log2n", [20, 22, 24, 26, 28, 30])
def test_cast_sweep_sizes(log2n, ws):
    n = 1 << log2n
    x = si.normal_bf16((n,), 1.0, log2n, 1)
    fmt = E4M3 if log2n % 4 == 0 else E5M2
    R = n // 4096
    _check(x, R, 4096, fmt, (q.AMAX_ATOMIC, q.AMAX_AUTO), ws)
    _check(x, 4096, R, fmt, (q.AMAX_ATOMIC, q.AMAX_AUTO), ws)


@pytest.mark.parametrize("log2n", [24, 28])
def test_cast_sweep_other_format_and_reduction(log2n, ws):
    """The format the size above does not take, with the REDUCTION amax."""
    n = 1 << log2n
    x = si.normal_bf16((n,), 1.0, log2n + 100, 1)
    R = n // 4096
    _check(x, R, 4096, E5M2, (q.AMAX_REDUCTION,), ws)
    _check(x, 4096, R, E5M2, (q.AMAX_REDUCTION,), ws)


@pytest.mark.parametrize("log2n", [24, 28])
def test_delayed_cast_sweep_sizes(log2n, ws):
    """Delayed scaling's single pass (stored scale, amax recorded in the same
    read) at sweep sizes: amax init on the first call, then a cast with the
    stored scale; every byte, and the recorded amax exactly."""
    n = 1 << log2n
    R = n // 4096
    x0 = si.normal_bf16((R, 4096), 1.0, log2n + 200, 1)
    x1 = si.normal_bf16((R, 4096), 2.0, log2n + 201, 1)
    st = q.ScalingState(E4M3, q.DELAYED, history_len=16)
    out = torch.empty((R, 4096), dtype=torch.uint8, device="cuda")
    out_t = torch.empty((4096, R), dtype=torch.uint8, device="cuda")
    s0, _ = oracle.scale_dynamic(oracle.amax(x0), E4M3)
    for xh, expect_scale in ((x0, s0), (x1, s0)):      # no fp8lin_scale between: scale kept
        q.cast_delayed(to_dev_bf16(xh), st, out, out_t, ws)
        q.check(ws)
        assert st.needs_init == 0
        assert dev_f32_bits(st.scale) == f32_bits(expect_scale)
        assert dev_f32_bits(st.amax) == f32_bits(oracle.amax(xh))
        ref, ref_t, _ = oracle.cast(xh, expect_scale, E4M3, transpose=True)
        check_bytes(out, ref, "delayed q")
        check_bytes(out_t, ref_t, "delayed q^T")
        del ref, ref_t


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
