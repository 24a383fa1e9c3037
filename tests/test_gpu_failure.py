"""A bounded wait that runs out is reported, not hung on: fp8lin_check
returns FP8LIN_ETIMEOUT, and the context and the workspace stay usable.

The failure is planted on the host, in the workspace.  The counters on which
the K slices of a split GEMM wait for each other are set so far below zero
that the slices can never all check in.  Each waiting warp gives up at the
kernel's 2 s limit, records its error code and returns.  Every load and MMA
of the kernel has completed before that wait, so nothing is left in flight.
fp8lin_check then reports ETIMEOUT and clears the counters, after which the
same GEMM is correct again."""
import time

import numpy as np
import pytest
import torch

import oracle
import quantised_gemm_gb300 as q
import synth_inputs as si
from quantised_gemm_gb300 import _lib as L
from helpers import assert_within_bound, bf16_to_f64

pytestmark = pytest.mark.gpu

# Workspace layout (quantised_gemm_gb300/csrc/internal.h): the K-split
# tickets, 4096 int32, follow the fixed part of 256 + 4 * 4096 bytes rounded
# up to 256 bytes.
TICKETS_OFFSET = 16640
TICKETS = 4096


def _operand(rows, k, fmt, seed):
    x = si.normal_bf16((rows, k), 1.0, seed, 1)
    s, inv = oracle.scale_dynamic(oracle.amax(x), fmt)
    q8, _, _ = oracle.cast(x, s, fmt, transpose=False)
    return q8, s, inv


@pytest.mark.parametrize("M,N,K,sched", [
    (16, 4096, 4096, "K split 4 ways"),
    (256, 4096, 4096, "K split 4 ways"),
    (1024, 5120, 12288, "last 4 tiles K split 8 ways"),
])
def test_split_gemm_wait_runs_out_and_the_workspace_recovers(M, N, K, sched):
    """M = 16: the one-CTA kernel; M = 256: the CTA-pair kernel, whose
    closing path then has both CTAs exchange their failure state and the even
    CTA confirm every stage's last load before either CTA leaves; M = 1024:
    the pair kernel with four epilogue warps, whose whole tiles finish and
    whose split tail tiles give up."""
    desc = q.gemm_describe(M, N, K)
    assert desc.endswith(sched), desc
    assert ("pair" in desc) == (M > 128), desc
    a8, sa, inva = _operand(M, K, oracle.E4M3, seed=71)
    b8, sb, invb = _operand(N, K, oracle.E4M3, seed=72)
    a, b = torch.from_numpy(a8).cuda(), torch.from_numpy(b8).cuda()
    ia, ib = torch.tensor([inva], device="cuda"), torch.tensor([invb], device="cuda")
    d = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ws = q.Workspace()

    ws.buf[TICKETS_OFFSET:TICKETS_OFFSET + 4 * TICKETS].view(torch.int32).fill_(-(1 << 30))
    t0 = time.time()
    q.gemm(a, b, oracle.E4M3, oracle.E4M3, ia, ib, d, ws)
    with pytest.raises(q.Fp8linError) as ei:
        q.check(ws)
    elapsed = time.time() - t0
    assert ei.value.status == L.ETIMEOUT
    assert 1.0 < elapsed < 60.0, elapsed          # the 2 s limit, not a hang
    assert torch.count_nonzero(ws.buf[TICKETS_OFFSET:TICKETS_OFFSET + 4 * TICKETS]).item() == 0

    q.gemm(a, b, oracle.E4M3, oracle.E4M3, ia, ib, d, ws)
    q.check(ws)
    y, s = oracle.gemm(a8, b8, oracle.E4M3, oracle.E4M3, sa, sb)
    assert_within_bound(bf16_to_f64(d), y, s, "after recovery")
