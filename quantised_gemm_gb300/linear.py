"""Fp8Linear: the buffers and scaling states of one float8 training Linear,
driving libfp8lin's forward / backward / delayed-scale update.

Mirrors the user-facing flow of the pages' float8 Linear: a config per
tensor role (input, weight, grad_output) with dynamic or delayed scaling
("[float8] FP8 GPT 1.5B Delayed Scaling 2x Slower than BF16", pytorch/ao
issue 1297, repro script: Float8LinearConfig / CastConfig / ScalingType), a
forward and backward, and after backward the per-tensor history sync
(sync_float8_amax_and_scale_history).  All device memory is allocated here,
once, through PyTorch; the library itself allocates nothing.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from . import (AMAX_AUTO, AMAX_PRECOMPUTED, DELAYED, DYNAMIC, E4M3, E5M2, ScalingState,
               Workspace, _stream, backward, forward, scale, scale_many)


class Fp8Linear:
    """One Linear y = x W^T with x [M, K], W [N, K], fp8 tensorwise scaling."""

    def __init__(self, M: int, K: int, N: int, *, scaling: str = "dynamic", history_len: int = 16,
                 amax_algo: int = AMAX_AUTO, eps: float = 1e-12, cache_weight: bool = False,
                 device="cuda"):
        kind = {"dynamic": DYNAMIC, "delayed": DELAYED}[scaling]
        self.M, self.K, self.N = M, K, N
        u8 = dict(dtype=torch.uint8, device=device)
        bf = dict(dtype=torch.bfloat16, device=device)
        self.x8 = torch.empty((M, K), **u8)
        self.x8t = torch.empty((K, M), **u8)
        self.w8 = torch.empty((N, K), **u8)
        self.w8t = torch.empty((K, N), **u8)
        self.dy8 = torch.empty((M, N), **u8)
        self.dy8t = torch.empty((N, M), **u8)
        self.y = torch.empty((M, N), **bf)
        self.dx = torch.empty((M, K), **bf)
        self.dw = torch.empty((N, K), **bf)
        self.ws = Workspace(M, K, N, device=device)
        mk = lambda fmt: ScalingState(fmt, kind, history_len, amax_algo, eps, device)  # noqa: E731
        self.sx, self.sw, self.sdy = mk(E4M3), mk(E4M3), mk(E5M2)
        # Where the GEMM epilogues deliver max |y| and max |dX| (set by link_linears()).
        self.y_amax_to = None
        self.dx_amax_to = None
        # cache_weight: cast W only when it changed since the last cast (its
        # storage or its in-place version counter), e.g. once for all the
        # micro-batches of an optimizer step.
        self.cache_weight = cache_weight
        self._w_key = None

    def forward(self, x: torch.Tensor, w: torch.Tensor, stream=None) -> torch.Tensor:
        key = ((id(w), w.data_ptr(), w._version, tuple(w.shape), w.device)
               if self.cache_weight else None)
        reuse = key is not None and key == self._w_key
        forward(x, None if reuse else w, self.sx, self.sw, self.y, self.x8, self.x8t, self.w8,
                self.w8t, self.ws, stream, y_amax=self.y_amax_to)
        self._w_key = key
        return self.y

    def backward(self, dy: torch.Tensor, need_dx: bool = True, need_dw: bool = True, stream=None):
        return backward(dy, self.x8t, self.w8t, self.sx, self.sw, self.sdy, self.dy8, self.dy8t,
                        self.dx if need_dx else None, self.dw if need_dw else None, self.ws,
                        stream, dx_amax=self.dx_amax_to if need_dx else None)

    def sync_scales(self, stream=None):
        """Delayed scaling: push this step's amaxes into the histories and
        recompute the scales (a no-op for dynamic scaling).  A new delayed
        weight scale makes a cached W8 stale: the next forward casts again."""
        delayed = [st for st in (self.sx, self.sw, self.sdy) if st.kind == DELAYED]
        if delayed:
            scale_many(delayed, stream)  # one launch for the Linear's states
        if self.sw.kind == DELAYED:
            self._w_key = None

    def _step_slots(self):
        """Two device slots for step_host, created on first use: the bf16
        inputs and outputs and five events each (the fp8 copies and the
        workspace are shared: all compute runs on one stream)."""
        if getattr(self, "_slots", None) is not None:
            return self._slots
        dev = self.y.device
        cur = torch.cuda.current_stream(dev)
        mk = lambda r, c: torch.empty((r, c), dtype=torch.bfloat16, device=dev)  # noqa: E731
        slots = []
        for k in range(2):
            bufs = {"x": mk(self.M, self.K), "w": mk(self.N, self.K), "dy": mk(self.M, self.N),
                    "y": self.y if k == 0 else mk(self.M, self.N),
                    "dx": self.dx if k == 0 else mk(self.M, self.K),
                    "dw": self.dw if k == 0 else mk(self.N, self.K)}
            evs = [torch.cuda.Event() for _ in range(5)]
            for ev in evs:
                ev.record(cur)                  # creates the event (torch creates it lazily)
            c = _lib.StepSlotC()
            for name, t in bufs.items():
                setattr(c, name, t.data_ptr())
            for name in ("x8", "x8t", "w8", "w8t", "dy8", "dy8t"):
                setattr(c, name, getattr(self, name).data_ptr())
            c.ws, c.ws_bytes = self.ws.ptr, self.ws.nbytes
            for i, ev in enumerate(evs):
                c.ev[i] = ev.cuda_event
            slots.append((bufs, evs, c))
        self._slots = slots
        self._slot = 0
        self._h2d = torch.cuda.Stream(device=dev)
        self._d2h = torch.cuda.Stream(device=dev)
        return slots

    def step_host(self, x_h, w_h, dy_h, y_h, dx_h, dw_h, stream=None, wait=True):
        """End-to-end step from host buffers through fp8lin_step_host: copy x,
        W, dY in, forward + backward (+ the delayed scales' sync), copy y, dX,
        dW out.  Host tensors: bf16, contiguous, pinned for the copies to be
        asynchronous.  Uploads and downloads run on two copy streams of this
        Linear, ordered against the compute by the slot's events; the two
        device slots are used in turn, so a step's copies overlap the other
        slot's compute.  The compute runs on `stream` (default: the current
        stream).  With wait=True that stream then waits for this step's
        downloads; with wait=False the next step may start while they are in
        flight -- finish_host() makes the stream wait for all of them."""
        for t, n, shape in ((x_h, "x_h", (self.M, self.K)), (w_h, "w_h", (self.N, self.K)),
                            (dy_h, "dy_h", (self.M, self.N)), (y_h, "y_h", (self.M, self.N)),
                            (dx_h, "dx_h", (self.M, self.K)), (dw_h, "dw_h", (self.N, self.K))):
            if t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or \
                    tuple(t.shape) != shape:
                raise ValueError("%s must be a contiguous host bf16 tensor of shape %s" %
                                 (n, shape))
        slots = self._step_slots()
        bufs, evs, c = slots[self._slot]
        self._slot ^= 1
        cx, cw, cd = self.sx.c_struct(), self.sw.c_struct(), self.sdy.c_struct()
        st = _lib.load().fp8lin_step_host(
            x_h.data_ptr(), w_h.data_ptr(), dy_h.data_ptr(), y_h.data_ptr(), dx_h.data_ptr(),
            dw_h.data_ptr(), self.M, self.K, self.N, ctypes.byref(cx), ctypes.byref(cw),
            ctypes.byref(cd), ctypes.byref(c), _stream(stream), self._h2d.cuda_stream,
            self._d2h.cuda_stream, 1 if wait else 0)
        for state in (self.sx, self.sw, self.sdy):
            state._pull()
        _lib.check(st, "fp8lin_step_host")
        self.y, self.dx, self.dw = bufs["y"], bufs["dx"], bufs["dw"]
        self._w_key = None      # W was cast from the slot's copy
        return y_h, dx_h, dw_h

    def finish_host(self, stream=None):
        """Make `stream` wait until every download of step_host is complete."""
        main = stream if stream is not None else torch.cuda.current_stream()
        for _, evs, _ in getattr(self, "_slots", None) or []:
            main.wait_event(evs[4])

    def step(self, x, w, dy, stream=None):
        """One forward + backward (+ delayed sync)."""
        self.forward(x, w, stream)
        self.backward(dy, stream=stream)
        self.sync_scales(stream)
        return self.y, self.dx, self.dw


class _NullCtx:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def link_linears(prev: Fp8Linear, nxt: Fp8Linear):
    """Chain two Linears, nxt consuming prev's output: nxt's input is
    ``prev.y`` and prev's grad_output is ``nxt.dx``.  prev's forward GEMM then
    writes max |y| straight into nxt's input amax, and nxt's dX GEMM writes
    max |dX| into prev's grad_output amax, both from their epilogues; the two
    states switch to AMAX_PRECOMPUTED, so each of those casts reads its tensor
    once instead of twice.  Both states must use dynamic scaling, and the
    caller must feed exactly prev.y / nxt.dx to the linked layer."""
    if prev.N != nxt.K or prev.M != nxt.M:
        raise ValueError("prev [M, N] output must be nxt's [M, K] input")
    if nxt.sx.kind != DYNAMIC or prev.sdy.kind != DYNAMIC:
        raise ValueError("a producer-computed amax needs dynamic scaling")
    nxt.sx.amax_algo = AMAX_PRECOMPUTED
    prev.sdy.amax_algo = AMAX_PRECOMPUTED
    prev.y_amax_to = nxt.sx.amax
    nxt.dx_amax_to = prev.sdy.amax
