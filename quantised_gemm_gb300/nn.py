"""torch.nn front end of libfp8lin: a Float8Linear module, the module swap and
the delayed-scaling sync, mirroring the user-facing API the pages use.

  * "Why swapping nn.Linear with FP8Linear brings throughput decrease for 7B
    LLAMA2-like model?" (pytorch/ao issue 1199): nn.Linear modules are swapped
    for FP8Linear by ``convert_to_float8_training``.
  * "[float8] FP8 GPT 1.5B Delayed Scaling 2x Slower than BF16" (pytorch/ao
    issue 1297), repro script: ``Float8LinearConfig`` with a ``CastConfig``
    (scaling type) per tensor role, ``convert_to_float8_training(model,
    config=...)``, and ``sync_float8_amax_and_scale_history(model)`` after
    ``loss.backward()``.

The forward and backward of every swapped Linear run entirely in libfp8lin
(amax, scale, cast + transpose, the three FP8 GEMMs); this file only wires
them into autograd.  Inputs and weights must be bf16 (other dtypes raise: the
library takes bf16 only), and the token count (all leading dimensions
flattened) and both feature sizes must be multiples of 16.  A bias, if
present, is added by PyTorch after the FP8 GEMM; it is not part of the path.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch
from torch import nn

from . import (AMAX_ATOMIC, AMAX_AUTO, AMAX_REDUCTION, AMAX_SINGLE_PASS, DELAYED, DYNAMIC, E4M3,
               E5M2, ScalingState, Workspace, _lib, backward, forward, scale)

_KINDS = {"dynamic": DYNAMIC, "delayed": DELAYED}
_ALGOS = {"atomic": AMAX_ATOMIC, "reduction": AMAX_REDUCTION, "single_pass": AMAX_SINGLE_PASS,
          "auto": AMAX_AUTO}


@dataclass
class CastConfig:
    """Scaling of one tensor role: 'dynamic' (scale from this tensor's amax)
    or 'delayed' (scale from an amax history of ``history_len`` steps)."""
    scaling_type: str = "dynamic"
    history_len: int = 16
    amax_algo: str = "auto"


@dataclass
class Float8LinearConfig:
    cast_config_input: CastConfig = field(default_factory=CastConfig)
    cast_config_weight: CastConfig = field(default_factory=CastConfig)
    cast_config_grad_output: CastConfig = field(default_factory=CastConfig)
    eps: float = 1e-12


def _state(cc: CastConfig, fmt: int, eps: float, device) -> ScalingState:
    if cc.scaling_type not in _KINDS:
        raise ValueError("scaling_type must be 'dynamic' or 'delayed'")
    return ScalingState(fmt, _KINDS[cc.scaling_type], cc.history_len, _ALGOS[cc.amax_algo], eps,
                        device)


class _SavedScale:
    """A scaling state as the backward sees it: the forward's inverse scale,
    snapshotted, so a second forward of the same module before this
    backward (weight sharing, re-computation) cannot change it."""

    def __init__(self, state: ScalingState, inv_scale: torch.Tensor):
        self._state = state
        self.inv_scale = inv_scale

    def c_struct(self):
        src = self._state.c_struct()
        c = _lib.ScalingStateC()
        for name, _ in _lib.ScalingStateC._fields_:
            setattr(c, name, getattr(src, name))
        c.inv_scale = self.inv_scale.data_ptr()
        return c


class _Fp8LinearFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x2d, weight, mod):
        M, K = x2d.shape
        N = weight.shape[0]
        dev = x2d.device
        x8 = torch.empty((M, K), dtype=torch.uint8, device=dev)
        x8t = torch.empty((K, M), dtype=torch.uint8, device=dev)
        w8 = torch.empty((N, K), dtype=torch.uint8, device=dev)
        w8t = torch.empty((K, N), dtype=torch.uint8, device=dev)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        ws = mod._workspace(dev)
        forward(x2d, weight, mod.sx, mod.sw, y, x8, x8t, w8, w8t, ws)
        inv_x = mod.sx.inv_scale.clone()
        inv_w = mod.sw.inv_scale.clone()
        ctx.save_for_backward(x8t, w8t, inv_x, inv_w)
        ctx.mod = mod
        ctx.shape = (M, K, N)
        return y

    @staticmethod
    def backward(ctx, dy):
        x8t, w8t, inv_x, inv_w = ctx.saved_tensors
        mod = ctx.mod
        M, K, N = ctx.shape
        dev = dy.device
        dy = dy.contiguous()
        if dy.dtype != torch.bfloat16:
            raise TypeError("grad_output must be bf16, got %s" % dy.dtype)
        dy8 = torch.empty((M, N), dtype=torch.uint8, device=dev)
        dy8t = torch.empty((N, M), dtype=torch.uint8, device=dev)
        need_dx, need_dw = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        dx = torch.empty((M, K), dtype=torch.bfloat16, device=dev) if need_dx else None
        dw = torch.empty((N, K), dtype=torch.bfloat16, device=dev) if need_dw else None
        backward(dy, x8t, w8t, _SavedScale(mod.sx, inv_x), _SavedScale(mod.sw, inv_w), mod.sdy,
                 dy8, dy8t, dx, dw, mod._workspace(dev))
        return dx, dw, None


_SHARED_WS: dict = {}


class Float8Linear(nn.Module):
    """Drop-in nn.Linear whose forward and backward run as FP8 (e4m3 input
    and weight, e5m2 grad_output) with tensorwise scaling."""

    def __init__(self, in_features: int, out_features: int, bias: bool = False,
                 config: Float8LinearConfig | None = None, device=None):
        super().__init__()
        self.in_features, self.out_features = in_features, out_features
        self.config = config or Float8LinearConfig()
        dev = torch.device(device) if device is not None else torch.device("cuda")
        self.weight = nn.Parameter(torch.empty((out_features, in_features), dtype=torch.bfloat16,
                                               device=dev))
        self.bias = nn.Parameter(torch.zeros(out_features, dtype=torch.bfloat16, device=dev)) \
            if bias else None
        nn.init.kaiming_uniform_(self.weight, a=5 ** 0.5)
        c = self.config
        self.sx = _state(c.cast_config_input, E4M3, c.eps, dev)
        self.sw = _state(c.cast_config_weight, E4M3, c.eps, dev)
        self.sdy = _state(c.cast_config_grad_output, E5M2, c.eps, dev)

    def _workspace(self, device) -> Workspace:
        # One workspace per (device, stream), shared by every Float8Linear:
        # it holds only scratch and self-cleaning counters, and calls on one
        # stream never overlap on the GPU, so sharing is safe there.
        dev = torch.device(device)
        key = (dev.index if dev.index is not None else torch.cuda.current_device(),
               torch.cuda.current_stream(dev).cuda_stream)
        ws = _SHARED_WS.get(key)
        if ws is None:
            ws = _SHARED_WS[key] = Workspace(device=dev)
        return ws

    @classmethod
    def from_linear(cls, lin: nn.Linear, config: Float8LinearConfig | None = None):
        m = cls(lin.in_features, lin.out_features, bias=lin.bias is not None, config=config,
                device=lin.weight.device)
        with torch.no_grad():
            m.weight.copy_(lin.weight.to(torch.bfloat16))
            if lin.bias is not None:
                m.bias.copy_(lin.bias.to(torch.bfloat16))
        return m

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        if x.dtype != torch.bfloat16 or self.weight.dtype != torch.bfloat16:
            raise TypeError("Float8Linear takes bf16 input and weight (got %s, %s)"
                            % (x.dtype, self.weight.dtype))
        lead = x.shape[:-1]
        x2d = x.reshape(-1, self.in_features)
        if not x2d.is_contiguous():
            x2d = x2d.contiguous()
        y = _Fp8LinearFunction.apply(x2d, self.weight, self)
        y = y.reshape(*lead, self.out_features)
        if self.bias is not None:
            y = y + self.bias
        return y

    def sync_scales(self):
        for st in (self.sx, self.sw, self.sdy):
            if st.kind == DELAYED:
                scale(st)

    def extra_repr(self):
        return "in_features=%d, out_features=%d, bias=%s" % (
            self.in_features, self.out_features, self.bias is not None)


def convert_to_float8_training(model: nn.Module, config: Float8LinearConfig | None = None,
                               module_filter_fn=None) -> nn.Module:
    """Swap every nn.Linear of `model` (in place) for a Float8Linear with the
    same weights.  `module_filter_fn(module, fqn)` may exclude modules."""
    for name, child in list(model.named_children()):
        if isinstance(child, nn.Linear) and not isinstance(child, Float8Linear):
            if module_filter_fn is None or module_filter_fn(child, name):
                setattr(model, name, Float8Linear.from_linear(child, config))
        else:
            convert_to_float8_training(child, config, module_filter_fn)
    return model


def sync_float8_amax_and_scale_history(model: nn.Module) -> None:
    """After backward: push every delayed-scaling tensor's amax into its
    history and recompute its scale (a no-op for dynamic scaling)."""
    for m in model.modules():
        if isinstance(m, Float8Linear):
            m.sync_scales()
