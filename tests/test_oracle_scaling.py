"""Pins of the oracle's amax, scale, delayed update and cast.

amax: closed forms (known maximum at a known place, all-zero, empty),
permutation and stride invariance.  Scale: exact powers of two, and for other
values the correct-rounding property |s - F/a| <= ulp(s)/2 checked in exact
rational arithmetic.  Delayed: the hand-worked sequence in
tests/golden/delayed_h3.json.  Cast: element-wise agreement with torch's own
fp32 multiply and float8 conversion where the result is in range, the
saturation rule where it is not, and q^T == transpose(q).
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import synth_inputs as si

E4M3, E5M2 = 0, 1
F = {E4M3: 448.0, E5M2: 57344.0}
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(vals):
    return si.f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))


# ------------------------------------------------------------------ amax

def test_amax_closed_forms(oracle_mod):
    x = np.zeros((37, 48), dtype=np.uint16)
    assert oracle_mod.amax(x) == 0.0
    x[17, 5] = bf16([-3.5])[0]
    x[2, 40] = bf16([2.0])[0]
    assert oracle_mod.amax(x) == 3.5
    assert oracle_mod.amax(np.zeros((0, 16), dtype=np.uint16)) == 0.0
    assert oracle_mod.amax(np.zeros((16, 0), dtype=np.uint16)) == 0.0
    big = bf16([[-3.3895314e38, 1.0]])             # largest finite bf16 magnitude
    assert oracle_mod.amax(big) == np.float32(si.bf16_bits_to_f32(big)[0, 0] * -1)


def test_amax_invariances(oracle_mod):
    x = si.normal_bf16((64, 96), 1.0, seed=3, stream=1)
    a = oracle_mod.amax(x)
    ref = float(np.max(np.abs(si.bf16_bits_to_f32(x))))
    assert a == ref
    perm = np.random.default_rng(0).permutation(x.size)
    assert oracle_mod.amax(x.reshape(-1)[perm].reshape(96, 64)) == a
    wide = np.zeros((64, 128), dtype=np.uint16)
    wide[:, :96] = x
    wide[:, 96:] = bf16(np.full((64, 32), 1e6))   # outside the view: must be ignored
    assert oracle_mod.amax(wide[:, :96]) == a


# ------------------------------------------------------------------ scale

def _is_correctly_rounded(s, exact):
    s = np.float32(s)
    up = np.nextafter(s, np.float32(np.inf))
    dn = np.nextafter(s, np.float32(0))
    err = abs(Fraction(float(s)) - exact)
    half_up = (Fraction(float(up)) - Fraction(float(s))) / 2
    half_dn = (Fraction(float(s)) - Fraction(float(dn))) / 2
    return err <= max(half_up, half_dn) and err <= (half_up if exact > Fraction(float(s)) else half_dn)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_scale_powers_of_two_exact(oracle_mod, fmt):
    for a, expect in ((0.5, 2 * F[fmt]), (1.0, F[fmt]), (4.0, F[fmt] / 4), (2.0 ** -10, F[fmt] * 1024)):
        s, inv = oracle_mod.scale_dynamic(a, fmt)
        assert s == np.float32(expect)
        assert Fraction(float(inv)) * Fraction(float(s)) == 1 or _is_correctly_rounded(
            inv, 1 / Fraction(float(s)))


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_scale_correct_rounding(oracle_mod, fmt):
    g = np.random.default_rng(5)
    amaxes = np.exp2(g.uniform(-20, 20, 500)).astype(np.float32)
    for a in amaxes:
        s, inv = oracle_mod.scale_dynamic(float(a), fmt)
        assert _is_correctly_rounded(s, Fraction(F[fmt]) / Fraction(float(a)))
        assert _is_correctly_rounded(inv, 1 / Fraction(float(s)))


def test_scale_eps_floor(oracle_mod):
    eps32 = np.float32(1e-12)
    s, inv = oracle_mod.scale_dynamic(0.0, E4M3, eps=1e-12)
    assert np.isfinite(s)
    assert _is_correctly_rounded(s, Fraction(448) / Fraction(float(eps32)))
    s2, _ = oracle_mod.scale_dynamic(1e-15, E4M3, eps=1e-12)   # below eps: eps wins
    assert s2 == s


# ------------------------------------------------------------------ delayed

def test_delayed_hand_worked_sequence(oracle_mod):
    with open(os.path.join(GOLDEN, "delayed_h3.json")) as f:
        g = json.load(f)
    for fmt_name, fmt in (("e4m3", E4M3), ("e5m2", E5M2)):
        st = oracle_mod.DelayedState(g["history_len"], fmt)
        amaxes = g["amaxes"]
        used = []
        st.init_from(amaxes[0])                   # amax init: first tensor's own amax
        for a in amaxes:
            used.append(float(st.scale))          # scale the step casts with
            st.update(a)                          # after backward
        used.append(float(st.scale))
        expect = [F[fmt] / d for d in g["scale_divisors"]]
        assert used == expect, (fmt_name, used)
        assert list(st.ring) == g["final_ring"]
        assert st.head == g["final_head"]


def test_delayed_h1_is_previous_step_dynamic(oracle_mod):
    g = np.random.default_rng(9)
    amaxes = np.exp2(g.uniform(-8, 8, 12)).astype(np.float32)
    st = oracle_mod.DelayedState(1, E4M3)
    st.init_from(float(amaxes[0]))
    for t in range(1, len(amaxes)):
        st.update(float(amaxes[t - 1]))
        assert st.scale == oracle_mod.scale_dynamic(float(amaxes[t - 1]), E4M3)[0]


def test_delayed_rejects_empty_history(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.DelayedState(0, E4M3)


# ------------------------------------------------------------------ cast

@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_cast_matches_torch_multiply_and_convert(oracle_mod, fmt):
    x = si.normal_bf16((48, 80), 1.0, seed=11, stream=1)
    x = si.add_outliers(x, 0.02, 50.0, seed=11)
    a = oracle_mod.amax(x)
    s, _ = oracle_mod.scale_dynamic(a, fmt)
    q, qt, a2 = oracle_mod.cast(x, s, fmt)
    assert a2 == a
    xt = torch.from_numpy(si.bf16_bits_to_f32(x))
    r = xt * torch.tensor(float(s), dtype=torch.float32)       # torch's fp32 multiply
    inr = r.abs() <= F[fmt]
    ref = r.to(torch.float8_e4m3fn if fmt == E4M3 else torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(q[inr.numpy()], ref[inr.numpy()])
    # the element at amax lands on +-F or one step below it
    assert np.array_equal(qt, q.T)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_cast_saturates_with_stale_scale(oracle_mod, fmt):
    # delayed scaling can cast with a scale from a smaller history amax
    x = bf16(np.array([[1.0, -1.0, 8.0, -8.0, 1000.0, -1e30, 0.0, -0.0]], dtype=np.float32))
    s = np.float32(F[fmt])                       # as if the history amax were 1
    q, _, _ = oracle_mod.cast(x, s, fmt, transpose=False)
    maxc = 0x7E if fmt == E4M3 else 0x7B
    assert list(q[0]) == [maxc, maxc | 0x80, maxc, maxc | 0x80, maxc, maxc | 0x80, 0x00, 0x80]


def test_cast_transpose_layout(oracle_mod):
    x = si.normal_bf16((32, 48), 1.0, seed=2, stream=1)
    q, qt, _ = oracle_mod.cast(x, 10.0, E4M3)
    assert qt.shape == (48, 32)
    for i in (0, 5, 31):
        for j in (0, 7, 47):
            assert qt[j, i] == q[i, j]
