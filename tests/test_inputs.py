"""The seeded input generators, on CPU: the recipes the workloads state
(distributions, bounds, outlier fraction), bf16 rounding, reproducibility,
and the edge tensors of the cast sweep."""
import numpy as np
import pytest
import torch

import synth_inputs as si

N_STAT = 1 << 20


def _f(bits):
    return si.bf16_bits_to_f32(bits).astype(np.float64)


def test_bf16_rounding_matches_torch():
    g = np.random.default_rng(5)
    a = np.concatenate([
        g.standard_normal(1 << 16).astype(np.float32) * np.float32(3.0),
        # exact ties between two bf16 values, both parities of the kept bit
        ((np.arange(4096, dtype=np.uint32) << 16) | 0x8000).view(np.float32),
        np.array([0.0, -0.0, 3.0e38, -3.0e38, 1e-40, -1e-40], dtype=np.float32),
    ])
    a = a[np.isfinite(a)]
    ref = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(si.f32_to_bf16_bits(a), ref)


@pytest.mark.parametrize("std", [1.0, 1e-3, 1e-4, 0.02])
def test_normal_recipe(std):
    v = _f(si.normal_bf16((N_STAT,), std, 0, si.STREAM_X))
    assert abs(v.mean()) < 5 * std / np.sqrt(N_STAT)
    assert v.std() == pytest.approx(std, rel=0.01)


@pytest.mark.parametrize("b", [1.0 / 64, 1.0 / np.sqrt(1600), 1.0 / np.sqrt(6400)])
def test_uniform_recipe(b):
    v = _f(si.uniform_bf16((N_STAT,), -b, b, 0, si.STREAM_W))
    assert v.min() >= -b * (1 + 2 ** -8) and v.max() <= b * (1 + 2 ** -8)   # bf16 rounding
    assert v.var() == pytest.approx((2 * b) ** 2 / 12, rel=0.01)
    assert abs(v.mean()) < 5 * b / np.sqrt(3 * N_STAT)


def test_outliers_replace_the_stated_fraction():
    base = si.normal_bf16((1024, 1024), 1.0, 3, si.STREAM_X)
    x = si.add_outliers(base.copy(), 1e-3, 50.0, 3)
    changed = np.flatnonzero(x.reshape(-1) != base.reshape(-1))
    count = round(x.size * 1e-3)
    # positions are drawn without replacement; a draw may round to the same bf16
    assert count - 2 <= changed.size <= count
    vals = _f(x.reshape(-1)[changed])
    assert np.abs(vals).max() > 4 * 50.0 * 0.5 and vals.std() == pytest.approx(50.0, rel=0.15)
    assert (vals < 0).any() and (vals > 0).any()   # the sign comes with the draw


def test_reproducible_and_streams_independent():
    a = si.normal_bf16((4096,), 1.0, 7, si.STREAM_X)
    assert np.array_equal(a, si.normal_bf16((4096,), 1.0, 7, si.STREAM_X))
    assert not np.array_equal(a, si.normal_bf16((4096,), 1.0, 7, si.STREAM_DY))
    assert not np.array_equal(a, si.normal_bf16((4096,), 1.0, 8, si.STREAM_X))
    # chunked generation gives the same stream as one piece
    big = si.normal_bf16((3 << 20,), 1.0, 7, si.STREAM_X)
    g = si.rng(7, si.STREAM_X)
    one = si.f32_to_bf16_bits(g.standard_normal(3 << 20, dtype=np.float32))
    assert np.array_equal(big, one)


def test_weight_fixed_across_steps_inputs_fresh():
    x0, w0, d0 = si.linear_inputs(32, 64, 48, w_init="kaiming", seed=0, step=0)
    x1, w1, d1 = si.linear_inputs(32, 64, 48, w_init="kaiming", seed=0, step=1)
    assert np.array_equal(w0, w1)
    assert not np.array_equal(x0, x1) and not np.array_equal(d0, d1)
    assert x0.shape == (32, 64) and w0.shape == (48, 64) and d0.shape == (32, 48)


def test_workload_shapes():
    shapes = {k: v["shapes"] for k, v in si.WORKLOADS.items()}
    assert shapes["linear4096_m65536"] == [(65536, 4096, 4096)]
    assert shapes["gpt1.5b_linears_m12288"] == [(12288, 1600, 4800), (12288, 1600, 1600),
                                                (12288, 1600, 6400), (12288, 6400, 1600)]
    assert shapes["llama3_8b_ffn_m8192"] == [(8192, 4096, 14336), (8192, 4096, 14336),
                                             (8192, 14336, 4096)]
    for k, v in si.WORKLOADS.items():
        for M, K, N in v["shapes"]:
            assert M % 16 == 0 and K % 16 == 0 and N % 16 == 0, k


def test_edge_tensors():
    r, c = 64, 128
    z = si.edge_tensor("zeros", r, c)
    assert not z.any()
    assert (si.edge_tensor("ones", r, c) == 0x3F80).all()
    assert (si.edge_tensor("neg_ones", r, c) == 0xBF80).all()
    m = si.edge_tensor("max_finite", r, c)
    assert ((m & 0x7FFF) == 0x7F7F).all() and (m >> 15).any() and not (m >> 15).all()
    s = si.edge_tensor("subnormal", r, c)
    assert ((s & 0x7F80) == 0).all() and ((s & 0x7F) != 0).all()
    one = si.edge_tensor("single", r, c)
    assert np.count_nonzero(one) == 1 and _f(one).min() == -5.0
    last = _f(si.edge_tensor("last", r, c)).reshape(-1)
    assert last[-1] == 50.0 and np.abs(last[:-1]).max() < 50.0
    for kind in si.EDGE_KINDS:
        assert np.isfinite(_f(si.edge_tensor(kind, r, c))).all(), kind
