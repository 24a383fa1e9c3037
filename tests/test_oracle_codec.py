"""Pins of the oracle's fp8 codec against things other than itself.

* decode: all 256 codes of each format against torch's float8 dtypes (a
  library routine) and against hand anchors of the format definitions;
* encode: round trip, ties-to-even at every midpoint, saturation, signed
  zero, and agreement with torch's fp32 -> float8 conversion on in-range
  values (torch does not saturate, so only |r| <= F is compared there).
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

E4M3, E5M2 = 0, 1
TORCH_DT = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _torch_decode(fmt):
    codes = torch.arange(256, dtype=torch.uint8)
    return codes.view(TORCH_DT[fmt]).to(torch.float64).numpy()


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_decode_matches_torch_dtype(oracle_mod, fmt):
    ours = oracle_mod.decode_table(fmt)
    ref = _torch_decode(fmt)
    assert np.array_equal(ours, ref, equal_nan=True)


def test_decode_anchors(oracle_mod):
    with open(os.path.join(GOLDEN, "fp8_anchors.json")) as f:
        anchors = json.load(f)
    for fmt_name, fmt in (("e4m3", E4M3), ("e5m2", E5M2)):
        for code_hex, value in anchors[fmt_name].items():
            got = oracle_mod.decode(int(code_hex, 16), fmt)
            if value == "nan":
                assert np.isnan(got), (fmt_name, code_hex)
            elif value in ("inf", "-inf"):
                assert got == float(value), (fmt_name, code_hex)
            else:
                assert got == float(Fraction(value)), (fmt_name, code_hex, got)
    assert oracle_mod.fp8_max(E4M3) == 448.0
    assert oracle_mod.fp8_max(E5M2) == 57344.0


def _finite_codes(oracle_mod, fmt):
    t = oracle_mod.decode_table(fmt)
    return [c for c in range(256) if np.isfinite(t[c])], t


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_round_trip(oracle_mod, fmt):
    codes, t = _finite_codes(oracle_mod, fmt)
    for c in codes:
        assert oracle_mod.encode(np.float32(t[c]), fmt) == c, hex(c)
    # the count of finite codes fixes the special-value layout
    assert len(codes) == (254 if fmt == E4M3 else 248)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_midpoints_tie_to_even(oracle_mod, fmt):
    t = oracle_mod.decode_table(fmt)
    F = oracle_mod.fp8_max(fmt)
    pos = sorted(c for c in range(128) if np.isfinite(t[c]))
    for lo, hi in zip(pos[:-1], pos[1:]):
        mid = (t[lo] + t[hi]) / 2            # exact in fp32: one more bit
        assert np.float32(mid) == mid
        even = lo if (lo & 1) == 0 else hi
        assert oracle_mod.encode(np.float32(mid), fmt) == even
        assert oracle_mod.encode(np.float32(-mid), fmt) == (even | 0x80)
        below = np.nextafter(np.float32(mid), np.float32(0))
        above = np.nextafter(np.float32(mid), np.float32(np.inf))
        assert oracle_mod.encode(below, fmt) == lo
        assert oracle_mod.encode(above, fmt) == hi
    assert t[pos[-1]] == F


@pytest.mark.parametrize("fmt,F,maxcode,next_mid", [(E4M3, 448.0, 0x7E, 464.0),
                                                    (E5M2, 57344.0, 0x7B, 61440.0)])
def test_saturation(oracle_mod, fmt, F, maxcode, next_mid):
    over = [np.nextafter(np.float32(F), np.float32(np.inf)), np.float32(next_mid),
            np.float32(next_mid + 1), np.float32(2 * F), np.float32(3.0e38),
            np.float32(np.inf)]
    for v in over:
        assert oracle_mod.encode(v, fmt) == maxcode, v
        assert oracle_mod.encode(-v, fmt) == (maxcode | 0x80), v
    # just below the midpoint above F still rounds to F
    assert oracle_mod.encode(np.nextafter(np.float32(next_mid), np.float32(0)), fmt) == maxcode


@pytest.mark.parametrize("fmt,min_sub", [(E4M3, 2.0 ** -9), (E5M2, 2.0 ** -16)])
def test_signed_zero_and_subnormals(oracle_mod, fmt, min_sub):
    assert oracle_mod.encode(np.float32(0.0), fmt) == 0x00
    assert oracle_mod.encode(np.float32(-0.0), fmt) == 0x80
    half = np.float32(min_sub / 2)                 # tie between 0 and min_sub: even is 0
    assert oracle_mod.encode(half, fmt) == 0x00
    assert oracle_mod.encode(-half, fmt) == 0x80
    assert oracle_mod.encode(np.nextafter(half, np.float32(1)), fmt) == 0x01
    assert oracle_mod.encode(np.float32(min_sub * 1.5), fmt) == 0x02   # tie 1|2 -> 2 (even)
    assert oracle_mod.encode(np.float32(min_sub * 2.5), fmt) == 0x02   # tie 2|3 -> 2
    assert oracle_mod.encode(np.float32(min_sub * 3.5), fmt) == 0x04   # tie 3|4 -> 4


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encode_matches_torch_in_range(oracle_mod, fmt):
    F = oracle_mod.fp8_max(fmt)
    g = np.random.default_rng(1234 + fmt)
    mag = np.exp2(g.uniform(-30.0, np.log2(F), 400_000)).astype(np.float32)
    r = mag * np.where(g.random(mag.size) < 0.5, -1, 1).astype(np.float32)
    r = r[np.abs(r) <= F]
    ours = oracle_mod.encode_array(r, fmt)
    ref = torch.from_numpy(r).to(TORCH_DT[fmt]).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encode_all_bf16_in_range_matches_torch(oracle_mod, fmt):
    F = oracle_mod.fp8_max(fmt)
    f = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    f = f[np.isfinite(f) & (np.abs(f) <= F)]
    ours = oracle_mod.encode_array(f, fmt)
    ref = torch.from_numpy(f).to(TORCH_DT[fmt]).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)
