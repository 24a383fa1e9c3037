"""Shared helpers of the tests: host <-> device conversion of bf16 bit arrays
and comparison of GEMM outputs against the oracle's bound."""
from __future__ import annotations

import numpy as np
import torch


def to_dev_bf16(a: np.ndarray, device="cuda") -> torch.Tensor:
    """uint16 bf16 bits (numpy) -> CUDA bfloat16 tensor with the same bits."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def f32_bits(v) -> int:
    return int(np.float32(v).view(np.uint32))


def dev_f32_bits(t: torch.Tensor) -> int:
    return int(t.view(torch.int32).item()) & 0xFFFFFFFF


def assert_within_bound(got: np.ndarray, ref: np.ndarray, s: np.ndarray, what: str):
    """|got - ref| <= 2^-7 |ref| + 1e-4 S element-wise; returns max err/bound."""
    err = np.abs(got - ref)
    bound = np.ldexp(np.abs(ref), -7) + 1e-4 * s
    bad = err > bound
    ratio = float(np.max(err / np.maximum(bound, 1e-300))) if err.size else 0.0
    if np.any(bad):
        idx = np.argwhere(bad)[:5]
        raise AssertionError("%s: %d of %d outside the bound (max err/bound %.3g); first %s" %
                             (what, int(bad.sum()), bad.size, ratio, idx.tolist()))
    return ratio
