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

import torch

from . import (AMAX_AUTO, AMAX_PRECOMPUTED, DELAYED, DYNAMIC, E4M3, E5M2, ScalingState,
               Workspace, backward, forward, scale)


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
        for st in (self.sx, self.sw, self.sdy):
            if st.kind == DELAYED:
                scale(st, stream)
        if self.sw.kind == DELAYED:
            self._w_key = None

    copy_lanes = 1   # copy streams per direction; with more, each tensor moves in row slices

    def step_host(self, x_h, w_h, dy_h, y_h, dx_h, dw_h, stream=None, wait=True):
        """End-to-end step from host buffers (pinned, for asynchronous copies):
        copy x, W, dY in, forward + backward (+ delayed sync), copy y, dX, dW
        out.  The copies run on copy streams of their own (``copy_lanes`` per
        direction; with more than one, each moves a slice of the rows -- one
        per direction measured fastest on a 4096 x 65536 step), ordered by
        events.  Device inputs and outputs come in two slots used in turn, so
        a step's uploads need only the step two back to be done with its slot:
        dY's upload overlaps the forward, y's download the backward, and the
        next step's uploads this step's compute.

        The compute runs on `stream` (default: the current stream).  With
        wait=True it waits, at the end, for this step's downloads: the host
        buffers hold the results.  With wait=False the next step's compute may
        run while those downloads are still in flight (the host link then
        sets the pace, both directions busy at once); the host buffers are
        complete after finish_host(), and a later step overwrites them.
        Device slots and copy streams are created on the first call."""
        main = stream if stream is not None else torch.cuda.current_stream()
        n = self.copy_lanes
        if not hasattr(self, "_slots"):
            dev = self.y.device
            mk = lambda r, c: torch.empty((r, c), dtype=torch.bfloat16, device=dev)  # noqa: E731
            self._slots = []
            for k in range(2):
                sl = {"x": mk(self.M, self.K), "w": mk(self.N, self.K), "dy": mk(self.M, self.N),
                      "y": self.y if k == 0 else mk(self.M, self.N),
                      "dx": self.dx if k == 0 else mk(self.M, self.K),
                      "dw": self.dw if k == 0 else mk(self.N, self.K),
                      "fwd_done": torch.cuda.Event(), "bwd_done": torch.cuda.Event(),
                      "downloads": []}
                sl["fwd_done"].record(main)
                sl["bwd_done"].record(main)
                self._slots.append(sl)
            self._slot = 0
            self._up = [torch.cuda.Stream(device=dev) for _ in range(n)]
            self._down = [torch.cuda.Stream(device=dev) for _ in range(n)]

        def move(pairs, streams, after):
            """Copy each (dst, src) in row slices over `streams` once `after`
            has fired; returns the events marking each stream's end."""
            done = []
            for i, st in enumerate(streams):
                st.wait_event(after)
                with torch.cuda.stream(st):
                    for dst, src in pairs:
                        rows = dst.shape[0]
                        lo, hi = rows * i // len(streams), rows * (i + 1) // len(streams)
                        if hi > lo:
                            dst[lo:hi].copy_(src[lo:hi], non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(st)
                    done.append(ev)
            return done

        sl = self._slots[self._slot]
        self._slot ^= 1
        # this slot's inputs are free once the step two back has consumed them
        xw_in = move([(sl["x"], x_h), (sl["w"], w_h)], self._up, sl["fwd_done"])
        dy_in = move([(sl["dy"], dy_h)], self._up, sl["bwd_done"])
        for ev in sl["downloads"] + xw_in:        # its outputs once downloaded
            main.wait_event(ev)
        self.y, self.dx, self.dw = sl["y"], sl["dx"], sl["dw"]
        self.forward(sl["x"], sl["w"], main)
        sl["fwd_done"].record(main)
        y_out = move([(y_h, sl["y"])], self._down, sl["fwd_done"])
        for ev in dy_in:
            main.wait_event(ev)
        self.backward(sl["dy"], stream=main)
        self.sync_scales(main)
        sl["bwd_done"].record(main)
        sl["downloads"] = y_out + move([(dx_h, sl["dx"]), (dw_h, sl["dw"])], self._down,
                                       sl["bwd_done"])
        if wait:
            self.finish_host(main)
        return y_h, dx_h, dw_h

    def finish_host(self, stream=None):
        """Make `stream` wait until every download of step_host is complete."""
        main = stream if stream is not None else torch.cuda.current_stream()
        for sl in getattr(self, "_slots", []):
            for ev in sl["downloads"]:
                main.wait_event(ev)

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
