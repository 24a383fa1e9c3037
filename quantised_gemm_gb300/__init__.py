"""quantised_gemm_gb300 -- Python binding of libfp8lin, the float8 training
Linear with tensorwise scaling on GB300 (sm_103a).

Every function here only marshals arguments (torch tensors -> device
pointers, the current CUDA stream) into the C ABI declared in
``include/fp8lin.h``; every step of the path runs in the library's CUDA
kernels.  There is no CPU fallback: on a machine without the built library
or a CUDA device the calls raise.

The method (torchao's float8 training Linear as discussed in "Integrate
float8nocompile, an experimental feature for high performance",
pytorch/torchtitan PR 778, and "[float8] FP8 GPT 1.5B Delayed Scaling 2x
Slower than BF16", pytorch/ao issue 1297):

  forward   x8, x8^T = cast_e4m3(x, s_x);  W8, W8^T = cast_e4m3(W, s_w)
            y  = x8 . W8^T / (s_x s_w)
  backward  dY8, dY8^T = cast_e5m2(dY, s_dy)
            dX = dY8 . W8 / (s_dy s_w);  dW = dY8^T . x8 / (s_dy s_x)
  scales    dynamic: s = F / max(amax(t), eps) from the tensor itself;
            delayed: s from the max of an amax history updated after backward.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import (AMAX_ATOMIC, AMAX_AUTO, AMAX_PRECOMPUTED, AMAX_REDUCTION, AMAX_SINGLE_PASS,
                   DELAYED, DYNAMIC,
                   E4M3, E5M2, Fp8linError, PROF_KINDS)

__all__ = [
    "E4M3", "E5M2", "AMAX_ATOMIC", "AMAX_REDUCTION", "AMAX_SINGLE_PASS", "AMAX_AUTO",
    "AMAX_PRECOMPUTED", "DYNAMIC",
    "DELAYED",
    "Fp8linError", "ScalingState", "Workspace", "amax", "amax_noalloc", "scale", "cast", "cast_dynamic", "cast_delayed", "gemm",
    "gemm_describe", "gemm_describe_for",
    "forward", "backward", "check", "workspace_bytes", "single_pass_max_elems", "launch_count",
    "profile_enable", "profile_collect", "profile_launches", "Fp8Linear", "link_linears", "library", "Float8Linear",
    "Float8LinearConfig", "CastConfig", "convert_to_float8_training",
    "sync_float8_amax_and_scale_history",
]


def library():
    """The loaded ctypes handle of libfp8lin (raises if not built)."""
    return _lib.load()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream=None) -> int:
    if stream is None:
        if _raw_stream is not None:   # the current stream's handle, without a Stream object
            return _raw_stream(torch.cuda.current_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t: torch.Tensor | None, name: str, dtype=None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t.data_ptr()


def _bf16_2d(t: torch.Tensor, name: str):
    if t.dim() != 2:
        raise ValueError("%s must be 2-D" % name)
    if t.stride(1) != 1:
        raise ValueError("%s must have unit column stride" % name)
    return _dev(t, name, torch.bfloat16), t.shape[0], t.shape[1], max(t.stride(0), t.shape[1])


def workspace_bytes(M: int = 0, K: int = 0, N: int = 0) -> int:
    return int(library().fp8lin_workspace_bytes(M, K, N))


def single_pass_max_elems() -> int:
    return int(library().fp8lin_single_pass_max_elems())


def gemm_describe(M: int, N: int, K: int) -> str:
    """The kernel, tile shape and schedule gemm() uses for an M x N x K GEMM
    on the current device."""
    buf = ctypes.create_string_buffer(256)
    _lib.check(library().fp8lin_gemm_describe(M, N, K, buf, len(buf)), "fp8lin_gemm_describe")
    return buf.value.decode()


def gemm_group_describe_for(dx_mnk, dw_mnk, num_sms: int) -> str:
    """How backward() would run its two GEMMs (dX and dW, each an (M, N, K)
    as the GEMM sees it) on a device of num_sms SMs, computed on the host:
    "grouped" (one launch dealing the tiles of both by their K loops) or
    "separate", with the plan's figures.  No GPU needed."""
    buf = ctypes.create_string_buffer(256)
    _lib.check(library().fp8lin_gemm_group_describe_for(*dx_mnk, *dw_mnk, num_sms, buf, len(buf)),
               "fp8lin_gemm_group_describe_for")
    return buf.value.decode()


def gemm_describe_for(M: int, N: int, K: int, num_sms: int) -> str:
    """gemm_describe() for a device of num_sms SMs holding one GEMM CTA per
    SM, computed on the host: no GPU needed."""
    buf = ctypes.create_string_buffer(256)
    _lib.check(library().fp8lin_gemm_describe_for(M, N, K, num_sms, buf, len(buf)),
               "fp8lin_gemm_describe_for")
    return buf.value.decode()


class Workspace:
    """Caller-owned device workspace (zero-filled once at creation)."""

    def __init__(self, M: int = 0, K: int = 0, N: int = 0, device="cuda"):
        self.nbytes = workspace_bytes(M, K, N)
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8, device=device)

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()


class ScalingState:
    """Per-tensor scaling state with its device buffers.

    kind: DYNAMIC or DELAYED; fmt: E4M3 or E5M2; history_len: ring length
    for DELAYED; amax_algo: AMAX_ATOMIC, AMAX_REDUCTION, AMAX_SINGLE_PASS,
    AMAX_AUTO, or AMAX_PRECOMPUTED (``amax`` is written by the producing
    GEMM's epilogue before the cast).
    Delayed states start with ``needs_init`` set (amax init on the first
    cast)."""

    def __init__(self, fmt: int, kind: int = DYNAMIC, history_len: int = 16,
                 amax_algo: int = AMAX_ATOMIC, eps: float = 1e-12, device="cuda"):
        self.fmt, self.kind, self.amax_algo, self.eps = fmt, kind, amax_algo, eps
        self.history_len = history_len if kind == DELAYED else 1
        self.amax = torch.zeros(1, dtype=torch.float32, device=device)
        self.scale = torch.ones(1, dtype=torch.float32, device=device)
        self.inv_scale = torch.ones(1, dtype=torch.float32, device=device)
        self.amax_history = torch.zeros(max(1, self.history_len), dtype=torch.float32,
                                        device=device)
        self.head = torch.zeros(1, dtype=torch.int32, device=device)
        self.needs_init = 1 if kind == DELAYED else 0
        self._c = _lib.ScalingStateC()

    def c_struct(self) -> _lib.ScalingStateC:
        c = self._c
        c.amax, c.scale, c.inv_scale = (self.amax.data_ptr(), self.scale.data_ptr(),
                                        self.inv_scale.data_ptr())
        c.amax_history, c.head = self.amax_history.data_ptr(), self.head.data_ptr()
        c.history_len, c.fmt, c.kind = self.history_len, self.fmt, self.kind
        c.amax_algo, c.needs_init, c.eps = self.amax_algo, self.needs_init, self.eps
        return c

    def _pull(self):
        self.needs_init = int(self._c.needs_init)


def _ws(ws):
    if ws is None:
        raise ValueError("a Workspace is required")
    return ws.ptr, ws.nbytes


def check(ws: Workspace, stream=None):
    """Synchronise and report a device-side error recorded in the workspace."""
    _lib.check(library().fp8lin_check(ws.ptr, _stream(stream)), "fp8lin_check")


def amax(x: torch.Tensor, out: torch.Tensor, algo: int = AMAX_ATOMIC, ws: Workspace | None = None,
         stream=None):
    px, rows, cols, ld = _bf16_2d(x, "x")
    lib = library()
    st = lib.fp8lin_amax(px, rows, cols, ld, _dev(out, "out", torch.float32), algo,
                         ws.ptr if ws is not None else None, _stream(stream))
    _lib.check(st, "fp8lin_amax")
    return out


def amax_noalloc(x: torch.Tensor, out: torch.Tensor, stream=None):
    """amax with no workspace and no allocation (static scratch in the
    library; calls that overlap on the GPU race on it)."""
    px, rows, cols, ld = _bf16_2d(x, "x")
    st = library().fp8lin_amax_noalloc(px, rows, cols, ld, _dev(out, "out", torch.float32),
                                       _stream(stream))
    _lib.check(st, "fp8lin_amax_noalloc")
    return out


def scale(state: ScalingState, stream=None):
    _lib.check(library().fp8lin_scale(ctypes.byref(state.c_struct()), _stream(stream)),
               "fp8lin_scale")


def scale_many(states, stream=None):
    """scale() of each of up to 8 states in one launch (the same results)."""
    states = list(states)
    arr = (_lib.ScalingStateC * max(1, len(states)))()
    for i, st in enumerate(states):
        ctypes.memmove(ctypes.byref(arr, i * ctypes.sizeof(_lib.ScalingStateC)),
                       ctypes.byref(st.c_struct()), ctypes.sizeof(_lib.ScalingStateC))
    _lib.check(library().fp8lin_scale_many(arr, len(states), _stream(stream)),
               "fp8lin_scale_many")


def cast(x: torch.Tensor, fmt: int, scale_t: torch.Tensor, out: torch.Tensor | None,
         out_t: torch.Tensor | None = None, amax_out: torch.Tensor | None = None, stream=None):
    px, rows, cols, ld = _bf16_2d(x, "x")
    st = library().fp8lin_cast(px, rows, cols, ld, fmt, _dev(scale_t, "scale", torch.float32),
                               _dev(out, "out", torch.uint8), _dev(out_t, "out_t", torch.uint8),
                               _dev(amax_out, "amax_out", torch.float32), _stream(stream))
    _lib.check(st, "fp8lin_cast")


def cast_dynamic(x: torch.Tensor, state: ScalingState, out: torch.Tensor | None,
                 out_t: torch.Tensor | None, ws: Workspace, stream=None):
    px, rows, cols, ld = _bf16_2d(x, "x")
    st = library().fp8lin_cast_dynamic(px, rows, cols, ld, ctypes.byref(state.c_struct()),
                                       _dev(out, "out", torch.uint8),
                                       _dev(out_t, "out_t", torch.uint8), ws.ptr, _stream(stream))
    _lib.check(st, "fp8lin_cast_dynamic")


def cast_delayed(x: torch.Tensor, state: ScalingState, out: torch.Tensor | None,
                 out_t: torch.Tensor | None, ws: Workspace, stream=None):
    """Delayed scaling's cast: the stored scale, the amax recorded in the same
    pass (amax init first if the state still needs it)."""
    px, rows, cols, ld = _bf16_2d(x, "x")
    c = state.c_struct()
    st = library().fp8lin_cast_delayed(px, rows, cols, ld, ctypes.byref(c),
                                       _dev(out, "out", torch.uint8),
                                       _dev(out_t, "out_t", torch.uint8), ws.ptr, _stream(stream))
    state._pull()
    _lib.check(st, "fp8lin_cast_delayed")


def gemm(a8: torch.Tensor, b8: torch.Tensor, fmt_a: int, fmt_b: int, inv_a: torch.Tensor,
         inv_b: torch.Tensor, out: torch.Tensor, ws: Workspace, stream=None,
         amax_out: torch.Tensor | None = None):
    """out[m, n] = bf16(sum_k a8[m, k] b8[n, k] * inv_a * inv_b); amax_out
    (fp32[1], optional) receives max |out| from the epilogue."""
    if a8.dim() != 2 or b8.dim() != 2 or a8.shape[1] != b8.shape[1]:
        raise ValueError("a8 [M, K] and b8 [N, K] expected")
    M, K = a8.shape
    N = b8.shape[0]
    if tuple(out.shape) != (M, N):
        raise ValueError("out must be [M, N]")
    pw, nb = _ws(ws)
    st = library().fp8lin_gemm(_dev(a8, "a8", torch.uint8), _dev(b8, "b8", torch.uint8), M, N, K,
                               max(a8.stride(0), K), max(b8.stride(0), K), fmt_a, fmt_b,
                               _dev(inv_a, "inv_a", torch.float32),
                               _dev(inv_b, "inv_b", torch.float32),
                               _dev(out, "out", torch.bfloat16), max(out.stride(0), N),
                               _dev(amax_out, "amax_out", torch.float32), pw, nb, _stream(stream))
    _lib.check(st, "fp8lin_gemm")
    return out


def forward(x, w, sx: ScalingState, sw: ScalingState, y, x8, x8t, w8, w8t, ws: Workspace,
            stream=None, y_amax: torch.Tensor | None = None):
    """y = x W^T in fp8.  w=None reuses w8 / w8t / sw from an earlier call
    (an unchanged weight); y_amax (fp32[1], optional) receives max |y|."""
    M, K = x.shape
    N = w8.shape[0] if w is None else w.shape[0]
    for t, n in ((x, "x"), (w, "w"), (y, "y")):
        if t is not None and not t.is_contiguous():
            raise ValueError("%s must be contiguous" % n)
    pw, nb = _ws(ws)
    cx, cw = sx.c_struct(), sw.c_struct()
    st = library().fp8lin_forward(_dev(x, "x", torch.bfloat16), _dev(w, "w", torch.bfloat16), M, K,
                                  N, ctypes.byref(cx), ctypes.byref(cw),
                                  _dev(y, "y", torch.bfloat16),
                                  _dev(y_amax, "y_amax", torch.float32),
                                  _dev(x8, "x8", torch.uint8),
                                  _dev(x8t, "x8t", torch.uint8), _dev(w8, "w8", torch.uint8),
                                  _dev(w8t, "w8t", torch.uint8), pw, nb, _stream(stream))
    sx._pull()
    sw._pull()
    _lib.check(st, "fp8lin_forward")
    return y


def backward(dy, x8t, w8t, sx: ScalingState, sw: ScalingState, sdy: ScalingState, dy8, dy8t,
             dx, dw, ws: Workspace, stream=None, dx_amax: torch.Tensor | None = None,
             dw_amax: torch.Tensor | None = None):
    M, N = dy.shape
    K = x8t.shape[0] if x8t is not None else w8t.shape[0]
    if not dy.is_contiguous():
        raise ValueError("dy must be contiguous")
    pw, nb = _ws(ws)
    cd = sdy.c_struct()
    st = library().fp8lin_backward(_dev(dy, "dy", torch.bfloat16), M, K, N,
                                   _dev(x8t, "x8t", torch.uint8), _dev(w8t, "w8t", torch.uint8),
                                   ctypes.byref(sx.c_struct()), ctypes.byref(sw.c_struct()),
                                   ctypes.byref(cd), _dev(dy8, "dy8", torch.uint8),
                                   _dev(dy8t, "dy8t", torch.uint8), _dev(dx, "dx", torch.bfloat16),
                                   _dev(dw, "dw", torch.bfloat16),
                                   _dev(dx_amax, "dx_amax", torch.float32),
                                   _dev(dw_amax, "dw_amax", torch.float32), pw, nb,
                                   _stream(stream))
    sdy._pull()
    _lib.check(st, "fp8lin_backward")
    return dx, dw


def launch_count() -> int:
    return int(library().fp8lin_launch_count())


def profile_enable(on: bool = True):
    library().fp8lin_profile_enable(1 if on else 0)


def profile_collect() -> dict:
    """{kind: (milliseconds, launches)} since profile_enable(True)."""
    ms = (ctypes.c_double * len(PROF_KINDS))()
    cnt = (ctypes.c_int64 * len(PROF_KINDS))()
    _lib.check(library().fp8lin_profile_collect(ms, cnt), "fp8lin_profile_collect")
    return {k: (ms[i], cnt[i]) for i, k in enumerate(PROF_KINDS)}


def profile_launches(capacity: int = 8192) -> list:
    """[(kind, milliseconds), ...] of every launch since profile_enable(True),
    in launch order."""
    ms = (ctypes.c_double * capacity)()
    kind = (ctypes.c_int32 * capacity)()
    n = int(library().fp8lin_profile_launches(ms, kind, capacity))
    if n < 0:
        _lib.check(-n, "fp8lin_profile_launches")
    return [(PROF_KINDS[kind[i]], ms[i]) for i in range(n)]


from .linear import Fp8Linear, link_linears  # noqa: E402
from .nn import (CastConfig, Float8Linear, Float8LinearConfig,  # noqa: E402
                 convert_to_float8_training, sync_float8_amax_and_scale_history)
