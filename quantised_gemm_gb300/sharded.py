"""ShardedFp8Linear: the fp8 training Linear split over the tokens (M) of a
data-parallel group, with one tensorwise scale per tensor for the whole
group.

Each rank holds its own M_r tokens of x and dY and the whole weight.  A
tensorwise scale is a function of the amax of the whole tensor, so the two
token-sharded tensors need one exchange each:

  forward   a_x  = all_reduce_max(amax(x_r))          one fp32 per step
            x8_r = cast_e4m3(x_r, F / max(a_x, eps))  (AMAX_PRECOMPUTED: the cast
                                                       reads x_r once more)
            W8   = cast_e4m3(W)                       W is replicated: its amax is
                                                       the same on every rank
            y_r  = x8_r . W8^T / (s_x s_w)
  backward  a_dy = all_reduce_max(amax(dY_r)), dY8_r with that scale
            dX_r = dY8_r . W8 / (s_dy s_w)            local
            dW   = sum_r dY8_r^T . x8_r / (s_dy s_x)  all_reduce_sum in fp32 (optional:
                                                       the data-parallel gradient sum)

With delayed scaling the casts use the stored scales and record the local
amaxes in the same pass; sync_scales() takes the maximum of each recorded
amax over the group before the history update -- what
sync_float8_amax_and_scale_history does across ranks in "[float8] FP8 GPT
1.5B Delayed Scaling 2x Slower than BF16" (pytorch/ao issue 1297).  The
multi-GPU training runs of the pages ("Why swapping nn.Linear with FP8Linear
brings throughput decrease for 7B LLAMA2-like model?", pytorch/ao issue 1199:
torchrun on two GPUs; "Integrate float8nocompile ...", torchtitan PR 778:
Llama3-8B on four GPUs) are data parallel in this sense.

The collectives are torch.distributed calls on `group` (NCCL between GPUs);
every other step runs in libfp8lin's kernels.  The exchange helpers are
plain functions so the host logic can be exercised with CPU ranks.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import AMAX_ATOMIC, AMAX_PRECOMPUTED, DELAYED, DYNAMIC, amax, scale, scale_many
from .linear import Fp8Linear


def global_amax_(amax_t: torch.Tensor, group=None) -> torch.Tensor:
    """In place: the largest amax over the ranks of `group` (one fp32).  The
    maximum of non-negative floats does not depend on the order, so every
    rank ends with the same bits as the amax of the whole tensor."""
    dist.all_reduce(amax_t, op=dist.ReduceOp.MAX, group=group)
    return amax_t


def reduce_grad_(dw: torch.Tensor, group=None, out: torch.Tensor | None = None) -> torch.Tensor:
    """The sum over the ranks of `group` of each rank's bf16 dW partial, in
    fp32 (so the sum adds no rounding of its own beyond fp32's); returns the
    fp32 sum (into `out` if given)."""
    acc = out if out is not None else torch.empty(dw.shape, dtype=torch.float32, device=dw.device)
    acc.copy_(dw)
    dist.all_reduce(acc, op=dist.ReduceOp.SUM, group=group)
    return acc


class ShardedFp8Linear:
    """One rank's part of a token-sharded Linear: x_r [M_r, K], W [N, K],
    dY_r [M_r, N]; y_r, dX_r local, dW summed over the group (fp32) when
    reduce_dw is set.  Scaling 'dynamic' or 'delayed' for all three tensors."""

    def __init__(self, M_local: int, K: int, N: int, *, group=None, scaling: str = "dynamic",
                 history_len: int = 16, reduce_dw: bool = True, device="cuda"):
        self.group = group
        self.reduce_dw = reduce_dw
        self.lin = Fp8Linear(M_local, K, N, scaling=scaling, history_len=history_len,
                             device=device)
        self.dynamic = scaling == "dynamic"
        if self.dynamic:
            # x and dY take the group's amax, computed before their casts
            self.lin.sx.amax_algo = AMAX_PRECOMPUTED
            self.lin.sdy.amax_algo = AMAX_PRECOMPUTED
        self.dw_sum = (torch.empty((N, K), dtype=torch.float32, device=device)
                       if reduce_dw else None)

    def _group_amax(self, t: torch.Tensor, st):
        amax(t, st.amax, AMAX_ATOMIC, self.lin.ws)
        global_amax_(st.amax, self.group)

    def _amax_init(self, t: torch.Tensor, st):
        """Delayed scaling's first step (enable_amax_init): the scale from the
        group's amax of this tensor, the ring untouched -- the scale a single
        process holding the whole tensor would start from."""
        if st.kind == DELAYED and st.needs_init:
            self._group_amax(t, st)
            st.kind = DYNAMIC
            scale(st)                   # scale = F / max(amax, eps) from the group's amax
            st.kind = DELAYED
            st.needs_init = 0

    def forward(self, x_local: torch.Tensor, w: torch.Tensor) -> torch.Tensor:
        lin = self.lin
        if self.dynamic:
            self._group_amax(x_local, lin.sx)
        else:
            self._amax_init(x_local, lin.sx)
        return lin.forward(x_local, w)

    def backward(self, dy_local: torch.Tensor):
        """Returns (dX_r, dW): dW is the group's fp32 sum with reduce_dw, else
        this rank's bf16 partial."""
        lin = self.lin
        if self.dynamic:
            self._group_amax(dy_local, lin.sdy)
        else:
            self._amax_init(dy_local, lin.sdy)
        lin.backward(dy_local)
        if self.reduce_dw:
            return lin.dx, reduce_grad_(lin.dw, self.group, self.dw_sum)
        return lin.dx, lin.dw

    def sync_scales(self):
        """Delayed scaling: the group's maximum of each recorded amax, then the
        history update of every state (a no-op for dynamic scaling)."""
        delayed = [st for st in (self.lin.sx, self.lin.sw, self.lin.sdy) if st.kind == DELAYED]
        for st in delayed:
            global_amax_(st.amax, self.group)
        if delayed:
            scale_many(delayed)  # one launch for the three states
