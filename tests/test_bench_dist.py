"""The multi-rank side of bench.py, on CPU.  With one process per GPU each
rank runs its own M tokens (the Linear's exchange, one amax per tensor, is
covered by test_sharded_dist.py); the timing shares a barrier and the
slowest rank's step time.  Two gloo ranks check that they agree on that
time, and that the whole-job throughput counts every rank's work.  A
non-zero rank of the reference arm must leave at once, without work."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    torch.distributed.init_process_group("gloo", init_method="env://")
    try:
        w, r, _ = bench.dist_info()
        ms = bench.max_over_ranks(torch, 1.0 + 0.5 * r, w, torch.device("cpu"))
        tf = bench.whole_job_tflops(6.0 * 4096 ** 3, ms, w)
        torch.distributed.barrier()
        out.put((r, w, ms, tf))
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=180) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _, _ in res] == [0, 1]
    for _, w, ms, tf in res:
        assert w == 2 and ms == 1.5                      # rank 1 is the slower one
        assert tf == pytest.approx(2 * 6.0 * 4096 ** 3 / 1.5e-3 / 1e12)


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(torch, 2.5, 1, torch.device("cpu")) == 2.5
    assert bench.whole_job_tflops(1e12, 1000.0, 1) == pytest.approx(1.0)


def test_reference_arm_other_ranks_do_nothing(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = bench.parse(["--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3"])
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""
