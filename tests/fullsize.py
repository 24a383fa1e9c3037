"""Helpers of the full-size parity tests: whole-tensor comparison of fp8
bytes, and GEMM outputs compared on whole tiles where large-index or
schedule faults would show.

For a GEMM D [M, N] = A [M, K] . B [N, K]^T the checked blocks are
  * the first and the last band of output rows (one tile high),
  * the last band of output columns (the N-edge tiles, all rows),
  * every tile the planner runs as K slices (named by fp8lin_gemm_describe:
    "last R tiles K split S ways", or every tile with "K split S ways"),
  * plus random single entries all over D.
Each block is compared element by element with oracle.gemm evaluated on the
block's rows of A and columns of B, within the acceptance bound.  Products of
at most `full_macs` multiply-adds are compared in full instead.
"""
from __future__ import annotations

import re

import numpy as np
import torch

import oracle
from helpers import assert_within_bound, bf16_to_f64

_DESC = re.compile(r"(?P<swap>swap-AB \(D\^T = B\.A\^T\), )?(?P<rows>\d+)x(?P<bn>\d+) tiles, "
                   r"(?P<tiles>\d+) tiles on .*?, (?P<sched>.*)$")


def plan_of(desc: str):
    """(swap, tile rows, tile cols, number of tiles, first split tile) of a
    fp8lin_gemm_describe line, in the kernel's view (swapped: rows run over
    D's columns)."""
    m = _DESC.search(desc)
    assert m, desc
    tiles = int(m.group("tiles"))
    sched = m.group("sched")
    t_split = tiles
    mm = re.match(r"last (\d+) tiles K split \d+ ways", sched)
    if mm:
        t_split = tiles - int(mm.group(1))
    elif sched.startswith("K split"):
        t_split = 0
    return bool(m.group("swap")), int(m.group("rows")), int(m.group("bn")), tiles, t_split


def split_tile_blocks(M: int, N: int, desc: str):
    """Output blocks ((r0, r1), (c0, c1)) of D [M, N] that the planner runs as
    K slices."""
    swap, rows, bn, tiles, t_split = plan_of(desc)
    km, kn = (N, M) if swap else (M, N)          # the kernel's view of D
    num_n = (kn + bn - 1) // bn
    blocks = []
    for t in range(t_split, tiles):
        mb, nb = divmod(t, num_n)
        r = (mb * rows, min(km, (mb + 1) * rows))
        c = (nb * bn, min(kn, (nb + 1) * bn))
        blocks.append((c, r) if swap else (r, c))
    return blocks


def check_bytes(dev: torch.Tensor, ref: np.ndarray, what: str):
    got = dev.cpu().numpy()
    if not np.array_equal(got, ref):
        bad = np.argwhere(got != ref)
        raise AssertionError("%s: %d of %d fp8 bytes differ; first %s" %
                             (what, len(bad), ref.size, bad[:5].tolist()))


def _check_block(d: torch.Tensor, a8, b8, fa, fb, sa, sb, rows, cols, what, col_chunk=1024):
    r0, r1 = rows
    for c0 in range(cols[0], cols[1], col_chunk):
        c1 = min(cols[1], c0 + col_chunk)
        y, s = oracle.gemm(a8[r0:r1], b8[c0:c1], fa, fb, sa, sb)
        got = bf16_to_f64(d[r0:r1, c0:c1])
        assert_within_bound(got, y, s, "%s block rows %d:%d cols %d:%d" % (what, r0, r1, c0, c1))


def check_gemm(d: torch.Tensor, a8: np.ndarray, b8: np.ndarray, fa: int, fb: int, sa, sb,
               desc: str, what: str, band: int = 256, samples: int = 256, seed: int = 0,
               full_macs: int = 1 << 34, row_chunk: int = 1024):
    """Compare D = a8 . b8^T (scaled) on the blocks listed in the module
    docstring; a8 [M, K], b8 [N, K] are the fp8 operands the GPU used."""
    M, N = d.shape
    if M * N * a8.shape[1] <= full_macs:
        for r0 in range(0, M, row_chunk):
            _check_block(d, a8, b8, fa, fb, sa, sb, (r0, min(M, r0 + row_chunk)), (0, N), what)
        return
    blocks = [((0, min(band, M)), (0, N)), ((max(0, M - band), M), (0, N))]
    c_edge = ((N - 1) // band) * band
    for r0 in range(0, M, row_chunk):
        blocks.append(((r0, min(M, r0 + row_chunk)), (c_edge, N)))
    blocks += split_tile_blocks(M, N, desc)
    for rows, cols in blocks:
        _check_block(d, a8, b8, fa, fb, sa, sb, rows, cols, what)
    g = np.random.default_rng(seed)
    m = g.integers(0, M, samples)
    n = g.integers(0, N, samples)
    y, s = oracle.gemm_entries(a8, b8, fa, fb, sa, sb, m, n)
    got = bf16_to_f64(d[torch.from_numpy(m).to(d.device), torch.from_numpy(n).to(d.device)])
    assert_within_bound(got, y, s, "%s samples" % what)


def check_linear(lin, q, x, w, dy, sx, sw, sd, E4M3, E5M2, seed=0):
    """Every fp8 byte of x8, x8^T, W8, W8^T, dY8, dY8^T against the oracle's
    cast with the given scales; the three GEMM outputs on whole tiles."""
    M, K = x.shape
    N = w.shape[0]
    for name, src, s, fmt in (("x", x, sx, E4M3), ("w", w, sw, E4M3), ("dy", dy, sd, E5M2)):
        q8, q8t, _ = oracle.cast(src, s, fmt, transpose=True)
        check_bytes(getattr(lin, name + "8"), q8, name + "8")
        check_bytes(getattr(lin, name + "8t"), q8t, name + "8t")
        del q8, q8t
    x8, x8t = lin.x8.cpu().numpy(), lin.x8t.cpu().numpy()
    w8, w8t = lin.w8.cpu().numpy(), lin.w8t.cpu().numpy()
    dy8, dy8t = lin.dy8.cpu().numpy(), lin.dy8t.cpu().numpy()
    check_gemm(lin.y, x8, w8, E4M3, E4M3, sx, sw, q.gemm_describe(M, N, K), "y", seed=seed)
    check_gemm(lin.dx, dy8, w8t, E5M2, E4M3, sd, sw, q.gemm_describe(M, K, N), "dX",
               seed=seed + 1)
    check_gemm(lin.dw, dy8t, x8t, E5M2, E4M3, sd, sx, q.gemm_describe(N, K, M), "dW",
               seed=seed + 2)
