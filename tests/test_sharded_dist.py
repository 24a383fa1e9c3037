"""The exchange steps of the token-sharded Linear (quantised_gemm_gb300.sharded)
on two gloo ranks on CPU.  The per-rank compute is played by the oracle
here (the kernels need a GPU; tests/test_gpu_sharded.py runs them), so what
is checked is the host logic around it: after global_amax_ every rank holds
the amax of the whole tensor, hence the scale of the whole tensor bit for
bit, and each shard's fp8 bytes cast with it are the rows of the whole
tensor's cast; reduce_grad_ returns the fp32 sum of the ranks' partials."""
import os
import socket
import sys

import numpy as np
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
M, K, N, WORLD = 96, 64, 48, 2


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    import synth_inputs as si
    x, w, dy = si.linear_inputs(M, K, N, w_init="uniform64", outlier_frac=0.02, seed=17)
    return x, w, dy


def _worker(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(WORLD))
    sys.path.insert(0, ROOT)
    import oracle
    from quantised_gemm_gb300.sharded import global_amax_, reduce_grad_
    torch.distributed.init_process_group("gloo", init_method="env://")
    try:
        oracle.build()
        x, w, dy = _inputs()
        rows = slice(rank * M // WORLD, (rank + 1) * M // WORLD)
        res = {"rank": rank}
        for name, full, fmt in (("x", x, oracle.E4M3), ("dy", dy, oracle.E5M2)):
            a = torch.tensor([oracle.amax(np.ascontiguousarray(full[rows]))], dtype=torch.float32)
            global_amax_(a)
            res[name + "_amax"] = float(a.item())
            s, _ = oracle.scale_dynamic(float(a.item()), fmt)
            res[name + "_scale"] = float(s)
            q8, q8t, _ = oracle.cast(np.ascontiguousarray(full[rows]), s, fmt)
            res[name + "8"] = q8
            res[name + "8t"] = q8t
        # this rank's dW partial, rounded to bf16 as the GEMM stores it
        sx, sd = np.float32(res["x_scale"]), np.float32(res["dy_scale"])
        part, _ = oracle.gemm(res["dy8t"], res["x8t"], oracle.E5M2, oracle.E4M3, sd, sx)
        part_bf16 = torch.from_numpy(part.astype(np.float32)).to(torch.bfloat16)
        res["dw_part"] = part_bf16.float().numpy()
        res["dw_sum"] = reduce_grad_(part_bf16).numpy()
        out.put(res)
    finally:
        torch.distributed.destroy_process_group()


def test_two_ranks_share_one_tensorwise_scale_and_sum_dw(oracle_mod):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=300) for _ in range(WORLD)), key=lambda r: r["rank"])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    o = oracle_mod
    x, w, dy = _inputs()
    for name, full, fmt in (("x", x, o.E4M3), ("dy", dy, o.E5M2)):
        a = o.amax(full)
        s, _ = o.scale_dynamic(a, fmt)
        q8, q8t, _ = o.cast(full, s, fmt)
        for r in res:
            rows = slice(r["rank"] * M // WORLD, (r["rank"] + 1) * M // WORLD)
            assert np.float32(r[name + "_amax"]).view(np.uint32) == np.float32(a).view(np.uint32)
            assert np.float32(r[name + "_scale"]).view(np.uint32) == np.float32(s).view(np.uint32)
            assert np.array_equal(r[name + "8"], q8[rows])
            assert np.array_equal(r[name + "8t"], q8t[:, rows])
    expect = sum(r["dw_part"] for r in res).astype(np.float32)
    for r in res:
        assert np.array_equal(r["dw_sum"], expect)
