"""Pins of the oracle's GEMM and of the Linear step it assembles.

* brute force in exact rational arithmetic (fractions) on tiny, non-square
  operands, so a transposed operand or a dropped scale fails;
* the sampled-entry routine against the full product;
* the three products of the Linear (y = x W^T, dX = dY W, dW = dY^T x, the
  FP8Linear of "Why swapping nn.Linear with FP8Linear brings throughput
  decrease ..." (pytorch/ao issue 1199)) against brute force on dequantised
  operands, with W = I special cases (dX = dY, y = x up to the fp8 codes).
"""
from fractions import Fraction

import numpy as np
import pytest

import synth_inputs as si

E4M3, E5M2 = 0, 1


def _random_codes(rng, shape, oracle_mod, fmt):
    t = oracle_mod.decode_table(fmt)
    finite = np.array([c for c in range(256) if np.isfinite(t[c])], dtype=np.uint8)
    return finite[rng.integers(0, finite.size, size=shape)]


def _brute(a8, b8, fmt_a, fmt_b, sa, sb, oracle_mod):
    ta = [Fraction(float(v)) if np.isfinite(v) else None for v in oracle_mod.decode_table(fmt_a)]
    tb = [Fraction(float(v)) if np.isfinite(v) else None for v in oracle_mod.decode_table(fmt_b)]
    M, K = a8.shape
    N = b8.shape[0]
    d = Fraction(float(np.float32(sa))) * Fraction(float(np.float32(sb)))
    y = [[sum(ta[a8[m, k]] * tb[b8[n, k]] for k in range(K)) / d for n in range(N)] for m in range(M)]
    s = [[sum(abs(ta[a8[m, k]] * tb[b8[n, k]]) for k in range(K)) / d for n in range(N)]
         for m in range(M)]
    return y, s


@pytest.mark.parametrize("fmt_a,fmt_b", [(E4M3, E4M3), (E5M2, E4M3)])
def test_gemm_brute_force_tiny(oracle_mod, fmt_a, fmt_b):
    rng = np.random.default_rng(21 + fmt_a)
    a8 = _random_codes(rng, (3, 7), oracle_mod, fmt_a)
    b8 = _random_codes(rng, (5, 7), oracle_mod, fmt_b)
    sa, sb = np.float32(3.0), np.float32(0.7)
    y, s = oracle_mod.gemm(a8, b8, fmt_a, fmt_b, sa, sb)
    yb, sbr = _brute(a8, b8, fmt_a, fmt_b, sa, sb, oracle_mod)
    assert y.shape == (3, 5)
    for m in range(3):
        for n in range(5):
            assert abs(Fraction(y[m, n]) - yb[m][n]) <= abs(yb[m][n]) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 80)
            assert abs(Fraction(s[m, n]) - sbr[m][n]) <= sbr[m][n] * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 80)
            assert s[m, n] >= abs(y[m, n])


def test_gemm_entries_match_full(oracle_mod):
    rng = np.random.default_rng(4)
    a8 = _random_codes(rng, (40, 96), oracle_mod, E5M2)
    b8 = _random_codes(rng, (24, 96), oracle_mod, E4M3)
    y, s = oracle_mod.gemm(a8, b8, E5M2, E4M3, 2.5, 0.125)
    m = rng.integers(0, 40, 50)
    n = rng.integers(0, 24, 50)
    ye, se = oracle_mod.gemm_entries(a8, b8, E5M2, E4M3, 2.5, 0.125, m, n)
    np.testing.assert_allclose(ye, y[m, n], rtol=1e-13, atol=1e-300)
    np.testing.assert_allclose(se, s[m, n], rtol=1e-13, atol=1e-300)


def test_linear_products_brute_force(oracle_mod):
    """y = x W^T, dX = dY W, dW = dY^T x on the dequantised fp8 operands."""
    M, K, N = 4, 6, 5
    x = si.normal_bf16((M, K), 1.0, seed=1, stream=1)
    w = si.normal_bf16((N, K), 0.5, seed=1, stream=2)
    dy = si.normal_bf16((M, N), 1e-3, seed=1, stream=3)
    sx = oracle_mod.scale_dynamic(oracle_mod.amax(x), E4M3)[0]
    sw = oracle_mod.scale_dynamic(oracle_mod.amax(w), E4M3)[0]
    sd = oracle_mod.scale_dynamic(oracle_mod.amax(dy), E5M2)[0]
    r = oracle_mod.linear_fwd_bwd(x, w, dy, sx, sw, sd)

    def deq(q, fmt, s):
        t = oracle_mod.decode_table(fmt)
        return [[Fraction(float(t[c])) / Fraction(float(s)) for c in row] for row in q]

    X = deq(r["x8"], E4M3, sx)
    W = deq(r["w8"], E4M3, sw)
    D = deq(r["dy8"], E5M2, sd)
    tol = Fraction(1, 2 ** 48)
    for m in range(M):
        for n in range(N):
            ref = sum(X[m][k] * W[n][k] for k in range(K))
            assert abs(Fraction(r["y"][m, n]) - ref) <= tol * (abs(ref) + 1)
    for m in range(M):
        for k in range(K):
            ref = sum(D[m][n] * W[n][k] for n in range(N))
            assert abs(Fraction(r["dx"][m, k]) - ref) <= tol * (abs(ref) + Fraction(1, 10 ** 6))
    for n in range(N):
        for k in range(K):
            ref = sum(D[m][n] * X[m][k] for m in range(M))
            assert abs(Fraction(r["dw"][n, k]) - ref) <= tol * (abs(ref) + Fraction(1, 10 ** 6))
    assert r["y"].shape == (M, N) and r["dx"].shape == (M, K) and r["dw"].shape == (N, K)


def test_identity_weight(oracle_mod):
    """W = I (e4m3 code of 1.0 on the diagonal, scale 1): dX equals the
    dequantised dY exactly and y equals the dequantised x."""
    n = 32
    w8 = np.zeros((n, n), dtype=np.uint8)
    np.fill_diagonal(w8, 0x38)                        # e4m3 1.0
    rng = np.random.default_rng(8)
    dy8 = _random_codes(rng, (7, n), oracle_mod, E5M2)
    x8 = _random_codes(rng, (7, n), oracle_mod, E4M3)
    dx, _ = oracle_mod.gemm(dy8, np.ascontiguousarray(w8.T), E5M2, E4M3, 4.0, 1.0)
    assert np.array_equal(dx, oracle_mod.decode_array(dy8, E5M2) / 4.0)
    y, _ = oracle_mod.gemm(x8, w8, E4M3, E4M3, 2.0, 1.0)
    assert np.array_equal(y, oracle_mod.decode_array(x8, E4M3) / 2.0)


def test_bound_formula(oracle_mod):
    y = np.array([1.0, -2.0, 0.0])
    s = np.array([3.0, 2.0, 5.0])
    b = oracle_mod.gemm_bound(y, s)
    assert np.allclose(b, [2.0 ** -7 + 3e-4, 2.0 ** -6 + 2e-4, 5e-4])
