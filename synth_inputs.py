"""Seeded synthetic inputs for the float8 training Linear.

Shared by the tests, the benchmark and the smoke check; used to feed both the
CUDA library and the CPU oracle the same bf16 bytes.  It holds none of the
method's arithmetic: only random draws and the rounding of those draws to
bf16 (round-to-nearest-even on the fp32 bit pattern).

Streams are numpy PCG64 generators keyed by (seed, stream id), so every
tensor is reproducible on any machine with numpy 2.x.  ``N(0, s)`` below means
a normal draw with standard deviation ``s``.

Workloads (shapes and value recipes of the pages' experiments):
  * single 4096->4096 Linear (torchtitan PR 778, single-linear table):
    x ~ N(0,1), W ~ U(-1/64, 1/64), dY ~ N(0, 1e-3); optionally 0.1% of x
    replaced by N(0, 50) outliers.
  * GPT-1.5B block Linears, M = 12 x 1024 (pytorch/ao issue 1297 repro):
    W ~ U(-1/sqrt(K), 1/sqrt(K)) (nn.Linear's default init), fresh
    x ~ N(0,1) and dY ~ N(0, 1e-3) every step.
  * Llama-3-8B FFN Linears, M = 8192 (torchtitan PR 778 training table):
    W ~ N(0, 0.02), x ~ N(0, 1), dY ~ N(0, 1e-4).
  * cast-only sweep: [R, 4096] and [4096, R] of N(0,1) plus edge tensors.
"""
from __future__ import annotations

import numpy as np

STREAM_X, STREAM_W, STREAM_DY, STREAM_OUTLIER_POS, STREAM_OUTLIER_VAL = 1, 2, 3, 4, 5


def rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(seed), int(stream)]))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits.
    Inputs must be NaN-free (every generator here is)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _chunked_fill(shape, draw, chunk=1 << 24) -> np.ndarray:
    """Generate a large bf16 tensor in pieces to bound fp32 temporaries."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        out[lo:hi] = f32_to_bf16_bits(draw(hi - lo))
    return out.reshape(shape)


def normal_bf16(shape, std: float, seed: int, stream: int) -> np.ndarray:
    g = rng(seed, stream)
    return _chunked_fill(shape, lambda n: g.standard_normal(n, dtype=np.float32) * np.float32(std))


def uniform_bf16(shape, lo: float, hi: float, seed: int, stream: int) -> np.ndarray:
    g = rng(seed, stream)
    span = np.float32(hi - lo)
    return _chunked_fill(shape, lambda n: g.random(n, dtype=np.float32) * span + np.float32(lo))


def add_outliers(bits: np.ndarray, frac: float, std: float, seed: int) -> np.ndarray:
    """Replace ``frac`` of the positions (chosen without replacement) by draws
    from N(0, std); the sign comes with the draw."""
    flat = bits.reshape(-1)
    count = int(round(flat.size * frac))
    if count == 0:
        return bits
    pos = rng(seed, STREAM_OUTLIER_POS).choice(flat.size, size=count, replace=False)
    vals = rng(seed, STREAM_OUTLIER_VAL).standard_normal(count, dtype=np.float32) * np.float32(std)
    flat[pos] = f32_to_bf16_bits(vals)
    return bits


def linear_inputs(M: int, K: int, N: int, *, w_init: str, x_std: float = 1.0,
                  dy_std: float = 1e-3, w_std: float = 0.02, outlier_frac: float = 0.0,
                  outlier_std: float = 50.0, seed: int = 0, step: int = 0):
    """x [M,K], W [N,K], dY [M,N] as bf16 bits.  ``w_init``: 'uniform64'
    (U(-1/64,1/64)), 'kaiming' (U(-1/sqrt(K), 1/sqrt(K))) or 'normal'
    (N(0, w_std)).  W depends on ``seed`` only; x and dY on seed + step."""
    s = seed + step
    x = normal_bf16((M, K), x_std, s, STREAM_X)
    if outlier_frac > 0:
        x = add_outliers(x, outlier_frac, outlier_std, s)
    w = weight(K, N, w_init=w_init, w_std=w_std, seed=seed)
    dy = normal_bf16((M, N), dy_std, s, STREAM_DY)
    return x, w, dy


def weight(K: int, N: int, *, w_init: str, w_std: float = 0.02, seed: int = 0) -> np.ndarray:
    """W [N, K] as bf16 bits (see linear_inputs for the recipes)."""
    if w_init == "uniform64":
        return uniform_bf16((N, K), -1.0 / 64, 1.0 / 64, seed, STREAM_W)
    if w_init == "kaiming":
        b = 1.0 / np.sqrt(K)
        return uniform_bf16((N, K), -b, b, seed, STREAM_W)
    if w_init == "normal":
        return normal_bf16((N, K), w_std, seed, STREAM_W)
    raise ValueError(w_init)


# Named workloads: (M, K, N) per Linear and the value recipe.
WORKLOADS = {
    "linear4096_m16": dict(shapes=[(16, 4096, 4096)], w_init="uniform64", dy_std=1e-3),
    "linear4096_m256": dict(shapes=[(256, 4096, 4096)], w_init="uniform64", dy_std=1e-3,
                            outlier_frac=1e-3),
    "linear4096_m4096": dict(shapes=[(4096, 4096, 4096)], w_init="uniform64", dy_std=1e-3,
                             outlier_frac=1e-3),
    "linear4096_m16384": dict(shapes=[(16384, 4096, 4096)], w_init="uniform64", dy_std=1e-3,
                              outlier_frac=1e-3),
    "linear4096_m65536": dict(shapes=[(65536, 4096, 4096)], w_init="uniform64", dy_std=1e-3,
                              outlier_frac=1e-3),
    "gpt1.5b_linears_m12288": dict(shapes=[(12288, 1600, 4800), (12288, 1600, 1600),
                                           (12288, 1600, 6400), (12288, 6400, 1600)],
                                   w_init="kaiming", dy_std=1e-3, delayed=True,
                                   history_len=16, steps=20),
    "llama3_8b_ffn_m8192": dict(shapes=[(8192, 4096, 14336), (8192, 4096, 14336),
                                        (8192, 14336, 4096)],
                                w_init="normal", w_std=0.02, dy_std=1e-4),
}


def workload_inputs(name: str, index: int = 0, seed: int = 0, step: int = 0):
    """Inputs of Linear ``index`` of a named workload."""
    wl = WORKLOADS[name]
    M, K, N = wl["shapes"][index]
    return linear_inputs(M, K, N, w_init=wl["w_init"], dy_std=wl.get("dy_std", 1e-3),
                         w_std=wl.get("w_std", 0.02), outlier_frac=wl.get("outlier_frac", 0.0),
                         seed=seed + 1000 * index, step=step)


# Edge tensors of the cast sweep (all NaN/inf-free).
EDGE_KINDS = ("zeros", "ones", "neg_ones", "max_finite", "subnormal", "single", "last")


def edge_tensor(kind: str, rows: int, cols: int, seed: int = 0) -> np.ndarray:
    """bf16 bits of one edge tensor of shape [rows, cols]."""
    n = rows * cols
    if kind == "zeros":
        t = np.zeros(n, dtype=np.uint16)
    elif kind == "ones":
        t = np.full(n, 0x3F80, dtype=np.uint16)
    elif kind == "neg_ones":
        t = np.full(n, 0xBF80, dtype=np.uint16)
    elif kind == "max_finite":          # +-0x7F7F, the largest finite bf16
        t = np.where(rng(seed, 7).random(n) < 0.5, 0x7F7F, 0xFF7F).astype(np.uint16)
    elif kind == "subnormal":           # bf16 subnormals of both signs
        m = rng(seed, 8).integers(1, 0x80, size=n).astype(np.uint16)
        t = np.where(rng(seed, 9).random(n) < 0.5, m, m | 0x8000).astype(np.uint16)
    elif kind == "single":              # one non-zero element in the middle
        t = np.zeros(n, dtype=np.uint16)
        t[n // 2] = 0xC0A0               # -5.0
    elif kind == "last":                # amax at the very last element
        t = normal_bf16((n,), 1.0, seed, 10)
        t[-1] = 0x4248                   # 50.0
    else:
        raise ValueError(kind)
    return t.reshape(rows, cols)
