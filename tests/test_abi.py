"""Host-side checks of the C ABI (no GPU needed): the library builds, loads,
exports every entry point include/*.h declares, and rejects bad arguments
with the documented status before touching the device."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from quantised_gemm_gb300 import build as qb
    qb.build()
    import quantised_gemm_gb300 as q
    return q.library()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(fp8lin_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_path():
    names = _declared_functions()
    for required in ("fp8lin_amax", "fp8lin_scale", "fp8lin_cast", "fp8lin_forward",
                     "fp8lin_backward", "fp8lin_gemm"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(lib):
    for code in range(5):
        assert lib.fp8lin_status_string(code).startswith(b"FP8LIN_")
    assert b"unknown" in lib.fp8lin_status_string(99)
    assert lib.fp8lin_version() == 101
    assert lib.fp8lin_workspace_bytes(65536, 4096, 4096) >= 256


def test_argument_errors_before_any_cuda_call(lib):
    import quantised_gemm_gb300._lib as L
    fake = ctypes.c_void_p(0x10000)        # never dereferenced: checks fail first
    odd = ctypes.c_void_p(0x10008)
    # amax: negative size, null input, misaligned input, columns not multiple of 16
    assert lib.fp8lin_amax(fake, -1, 16, 16, fake, 0, None, None) == L.EINVAL
    assert lib.fp8lin_amax(None, 16, 16, 16, fake, 0, None, None) == L.EINVAL
    assert lib.fp8lin_amax(odd, 16, 16, 16, fake, 0, None, None) == L.EINVAL
    assert lib.fp8lin_amax(fake, 16, 24, 24, fake, 0, None, None) == L.EUNSUPPORTED
    assert lib.fp8lin_amax(fake, 16, 16, 8, fake, 0, None, None) == L.EINVAL       # ld < cols
    assert lib.fp8lin_amax(fake, 16, 16, 16, fake, 7, None, None) == L.EUNSUPPORTED
    assert lib.fp8lin_amax(fake, 16, 16, 16, fake, 1, None, None) == L.EINVAL      # no ws
    # cast: bad format, no outputs, transposed copy needs rows % 16 == 0
    assert lib.fp8lin_cast(fake, 16, 16, 16, 5, fake, fake, None, None, None) == L.EUNSUPPORTED
    assert lib.fp8lin_cast(fake, 16, 16, 16, 0, fake, None, None, None, None) == L.EINVAL
    assert lib.fp8lin_cast(fake, 8, 16, 16, 0, fake, fake, fake, None, None) == L.EUNSUPPORTED
    # gemm: no workspace, K not multiple of 16, misaligned output
    assert lib.fp8lin_gemm(fake, fake, 16, 16, 16, 16, 16, 0, 0, fake, fake, fake, 16, None,
                           None, 0, None) == L.EINVAL
    ws = ctypes.c_void_p(0x20000)
    nb = lib.fp8lin_workspace_bytes(16, 16, 16)
    assert lib.fp8lin_gemm(fake, fake, 16, 16, 24, 32, 32, 0, 0, fake, fake, fake, 16, None,
                           ws, nb, None) == L.EUNSUPPORTED
    assert lib.fp8lin_gemm(fake, fake, 16, 16, 16, 16, 16, 0, 0, fake, fake, odd, 16, None,
                           ws, nb, None) == L.EINVAL
    assert lib.fp8lin_gemm(fake, fake, 16, 16, 16, 16, 16, 0, 0, fake, fake, fake, 16,
                           ctypes.c_void_p(0x10002), ws, nb, None) == L.EINVAL  # misaligned amax
    assert lib.fp8lin_gemm(fake, fake, 16, 16, 16, 16, 16, 0, 3, fake, fake, fake, 16, None,
                           ws, nb, None) == L.EUNSUPPORTED


def _state(fmt, kind=0, H=1, eps=1e-12, algo=0):
    import quantised_gemm_gb300._lib as L
    s = L.ScalingStateC()
    s.amax = s.scale = s.inv_scale = 0x30000
    s.amax_history = 0x40000 if kind == 1 else 0
    s.head = 0x50000 if kind == 1 else 0
    s.history_len, s.fmt, s.kind, s.amax_algo, s.needs_init, s.eps = H, fmt, kind, algo, 0, eps
    return s


def test_forward_backward_argument_errors(lib):
    import quantised_gemm_gb300._lib as L
    p = ctypes.c_void_p(0x10000)
    ws = ctypes.c_void_p(0x20000)
    nb = lib.fp8lin_workspace_bytes(128, 128, 128)
    sx, sw, sd = _state(0), _state(0), _state(1)
    fwd = lambda M, K, N, a, b, ya=None: lib.fp8lin_forward(
        p, p, M, K, N, ctypes.byref(a), ctypes.byref(b), p, ya, p, p, p, p, ws, nb, None)
    assert fwd(100, 128, 128, sx, sw) == L.EUNSUPPORTED            # M % 16
    assert fwd(-16, 128, 128, sx, sw) == L.EINVAL
    assert fwd(128, 128, 128, _state(1), sw) == L.EUNSUPPORTED     # x must be e4m3
    assert fwd(128, 128, 128, _state(0, eps=0.0), sw) == L.EINVAL  # eps must be > 0
    assert fwd(128, 128, 128, _state(0, kind=1, H=0), sw) == L.EINVAL   # delayed H >= 1
    assert fwd(128, 128, 128, _state(0, algo=9), sw) == L.EUNSUPPORTED
    # a precomputed amax is a dynamic-scaling mode only
    assert fwd(128, 128, 128, _state(0, kind=1, H=4, algo=L.AMAX_PRECOMPUTED), sw) == \
        L.EUNSUPPORTED
    assert fwd(128, 128, 128, sx, sw, ctypes.c_void_p(0x10001)) == L.EINVAL   # misaligned y_amax
    # a cached weight (w == NULL) still needs w8 / w8t, and a first delayed cast
    assert lib.fp8lin_forward(p, None, 128, 128, 128, ctypes.byref(sx), ctypes.byref(sw), p, None,
                              p, p, None, p, ws, nb, None) == L.EINVAL
    swd = _state(0, kind=1, H=4)
    swd.needs_init = 1
    assert lib.fp8lin_forward(p, None, 128, 128, 128, ctypes.byref(sx), ctypes.byref(swd), p, None,
                              p, p, p, p, ws, nb, None) == L.EINVAL
    assert lib.fp8lin_forward(p, p, 128, 128, 128, ctypes.byref(sx), ctypes.byref(sw), p, None, p,
                              p, p, p, None, nb, None) == L.EINVAL    # no workspace
    bwd = lambda d, dxa=None, dwa=None, dx=p, dw=p: lib.fp8lin_backward(
        p, 128, 128, 128, p, p, ctypes.byref(sx), ctypes.byref(sw), ctypes.byref(d), p, p, dx, dw,
        dxa, dwa, ws, nb, None)
    assert bwd(_state(0)) == L.EUNSUPPORTED                        # grad_output must be e5m2
    assert bwd(sd, dxa=p, dx=None) == L.EINVAL                     # dX amax without dX
    assert bwd(sd, dwa=p, dw=None) == L.EINVAL                     # dW amax without dW
    assert lib.fp8lin_scale(None, None) == L.EINVAL
    assert lib.fp8lin_scale(ctypes.byref(_state(0, kind=1, H=0)), None) == L.EINVAL
    # the batched update: 0..8 states, each checked as fp8lin_scale checks it
    good, bad = _state(0), _state(0, kind=1, H=0)
    arr = (L.ScalingStateC * 9)(*([good] * 9))
    assert lib.fp8lin_scale_many(None, 1, None) == L.EINVAL
    assert lib.fp8lin_scale_many(arr, -1, None) == L.EINVAL
    assert lib.fp8lin_scale_many(arr, 9, None) == L.EINVAL
    assert lib.fp8lin_scale_many(None, 0, None) == L.OK             # nothing to do
    arr[2] = bad
    assert lib.fp8lin_scale_many(arr, 3, None) == L.EINVAL
    # states whose written buffers overlap another state's buffers (checked
    # before any launch; no valid case is launched here, the pointers are fake)
    def state(base, kind=0, H=1):
        s = _state(0, kind=kind, H=H)
        s.amax, s.scale, s.inv_scale = base, base + 4, base + 8
        if kind == 1:
            s.amax_history, s.head = base + 64, base + 64 + 4 * H
        return s
    two = (L.ScalingStateC * 2)
    assert lib.fp8lin_scale_many(two(state(0x30000), state(0x30000)), 2, None) == L.EINVAL
    a, b = state(0x30000, kind=1, H=16), state(0x31000)
    b.scale = 0x30000 + 64 + 4 * 15                    # inside a's ring
    assert lib.fp8lin_scale_many(two(a, b), 2, None) == L.EINVAL
    a, b = state(0x30000), state(0x31000)
    b.inv_scale = 0x30000                              # written over a's amax
    assert lib.fp8lin_scale_many(two(a, b), 2, None) == L.EINVAL
    a, b = state(0x30000, kind=1, H=4), state(0x31000, kind=1, H=4)
    b.head = 0x30000 + 64 + 4 * 4                      # a's head
    assert lib.fp8lin_scale_many(two(a, b), 2, None) == L.EINVAL


def test_gemm_describe_argument_errors(lib):
    import quantised_gemm_gb300._lib as L
    buf = ctypes.create_string_buffer(64)
    assert lib.fp8lin_gemm_describe(16, 16, 16, None, 64) == L.EINVAL
    assert lib.fp8lin_gemm_describe(16, 16, 16, buf, 0) == L.EINVAL
    assert lib.fp8lin_gemm_describe(-16, 16, 16, buf, 64) == L.EINVAL
    # without a GPU the valid call reports a CUDA error and leaves an empty line
    st = lib.fp8lin_gemm_describe(16, 16, 16, buf, 64)
    assert st in (L.OK, L.ECUDA) and (st == L.OK or buf.value == b"")


def test_cast_delayed_step_host_and_profile_argument_errors(lib):
    import quantised_gemm_gb300._lib as L
    p = ctypes.c_void_p(0x10000)
    ws = ctypes.c_void_p(0x20000)
    nb = lib.fp8lin_workspace_bytes(128, 128, 128)
    # the delayed cast wants a delayed state, a workspace and an output
    dyn, dly = _state(0), _state(0, kind=1, H=4)
    assert lib.fp8lin_cast_delayed(p, 128, 128, 128, ctypes.byref(dyn), p, p, ws, None) == L.EINVAL
    assert lib.fp8lin_cast_delayed(p, 128, 128, 128, ctypes.byref(dly), p, p, None, None) == \
        L.EINVAL
    assert lib.fp8lin_cast_delayed(p, 128, 128, 128, ctypes.byref(dly), None, None, ws, None) == \
        L.EINVAL
    assert lib.fp8lin_cast_delayed(p, 120, 128, 128, ctypes.byref(dly), p, p, ws, None) == \
        L.EUNSUPPORTED                                              # transposed copy: rows % 16
    # the host step checks its slot, sizes, states and events before anything else
    sx, sw, sd = _state(0), _state(0), _state(1)
    slot = L.StepSlotC()
    for name in ("x", "w", "dy", "y", "dx", "dw", "x8", "x8t", "w8", "w8t", "dy8", "dy8t"):
        setattr(slot, name, 0x10000)
    slot.ws, slot.ws_bytes = 0x20000, nb
    step = lambda M, s, sdy=sd: lib.fp8lin_step_host(
        p, p, p, p, p, p, M, 128, 128, ctypes.byref(sx), ctypes.byref(sw), ctypes.byref(sdy),
        s, None, None, None, 1)
    assert step(128, None) == L.EINVAL                             # no slot
    assert step(128, ctypes.byref(slot)) == L.EINVAL               # events missing
    for i in range(5):
        slot.ev[i] = 0x60000 + 64 * i                              # never used: checks fail first
    assert step(100, ctypes.byref(slot)) == L.EUNSUPPORTED         # M % 16
    assert step(128, ctypes.byref(slot), sdy=_state(0)) == L.EUNSUPPORTED   # grad_output e5m2
    slot.dx = 0
    assert step(128, ctypes.byref(slot)) == L.EINVAL               # the step needs dX's buffer
    # the launch-ordered profile record wants both arrays
    assert lib.fp8lin_profile_launches(None, None, 4) == -L.EINVAL
