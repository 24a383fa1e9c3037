"""The allocation-free amax entry point (fp8lin_amax_noalloc).

Some callers cannot call cudaMalloc and have no workspace to pass (a plug-in
inside a framework that owns all device memory through its own pool, a tool
limited to the buffers it was handed).  fp8lin_amax_noalloc serves them by
keeping the REDUCTION amax's partial maxima in a static device array of the
library.  This test calls it through the C ABI and checks that it returns
the same bits as the workspace-based fp8lin_amax on two calls in a row --
a large tensor followed by a smaller one with a smaller maximum, so a stale
slot left by the first call would show in the second.  The file is named to
be collected last, and it passes alone in a fresh process as well as after
the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import quantised_gemm_gb300 as q
import synth_inputs as si
from helpers import to_dev_bf16

pytestmark = pytest.mark.gpu


def _reference_amax(x, ws):
    out = torch.full((1,), -1.0, device="cuda")
    q.amax(x, out, q.AMAX_REDUCTION, ws)
    return out


def _noalloc_amax(x):
    lib = q.library()
    out = torch.full((1,), -1.0, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = lib.fp8lin_amax_noalloc(ctypes.c_void_p(x.data_ptr()), x.shape[0], x.shape[1],
                                 x.stride(0), ctypes.c_void_p(out.data_ptr()),
                                 ctypes.c_void_p(stream))
    assert st == 0, lib.fp8lin_status_string(st)
    return out


def test_noalloc_amax_matches_workspace_amax_twice():
    ws = q.Workspace()
    big = si.normal_bf16((8192, 4096), 1.0, 41, 1)
    big = si.add_outliers(big, 1e-3, 50.0, 41)
    small = si.normal_bf16((272, 1552), 0.25, 42, 1)     # smaller grid, smaller maximum
    for host in (big, small):
        x = to_dev_bf16(host)
        got = _noalloc_amax(x)
        ref = _reference_amax(x, ws)
        torch.cuda.synchronize()
        assert got.view(torch.int32).item() == ref.view(torch.int32).item()
        expect = np.max(np.abs(si.bf16_bits_to_f32(host)))
        assert got.item() == float(expect)


def _noalloc_raw(x_ptr, rows, cols, ld):
    lib = q.library()
    out = torch.full((1,), -1.0, device="cuda")
    st = lib.fp8lin_amax_noalloc(ctypes.c_void_p(x_ptr), rows, cols, ld,
                                 ctypes.c_void_p(out.data_ptr()),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.fp8lin_status_string(st)
    return out


def test_noalloc_amax_empty_tensor_is_zero():
    """rows == 0 or cols == 0: the amax of an empty tensor is exactly +0.0
    (the call writes it; the -1 placed there beforehand must go)."""
    x = torch.empty((0, 4096), dtype=torch.bfloat16, device="cuda")
    for rows, cols in ((0, 4096), (64, 0)):
        got = _noalloc_raw(x.data_ptr(), rows, cols, 4096)
        torch.cuda.synchronize()
        assert got.view(torch.int32).item() == 0


def test_noalloc_amax_ignores_row_padding():
    """A strided view (row stride ld > cols): the padding columns hold values
    far above the tensor's own maximum and must not reach the amax."""
    rows, cols, ld = 1040, 784, 1024
    host = si.normal_bf16((rows, cols), 1.0, 43, 1)
    full = np.full((rows, ld), 0x7F00, dtype=np.uint16)      # bf16 1.7e38 in the padding
    full[:, :cols] = host
    x = to_dev_bf16(full)
    got = _noalloc_raw(x.data_ptr(), rows, cols, ld)
    ref = _reference_amax(x[:, :cols], q.Workspace())
    torch.cuda.synchronize()
    assert got.view(torch.int32).item() == ref.view(torch.int32).item()
    assert got.item() == float(np.max(np.abs(si.bf16_bits_to_f32(host))))
