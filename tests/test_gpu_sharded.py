"""The token-sharded Linear (quantised_gemm_gb300.sharded) through the
library's kernels, as two ranks: two processes on this one GPU that meet
only in gloo collectives on the host (their kernels never wait for one
another).  Each rank casts its shard with the scale of the whole tensor;
the test checks, against the oracle, the scales bit for bit, every fp8 byte
of each shard, y and dX of each shard within the bound, and the group's dW
(the fp32 sum of the ranks' partials) within the sum of the partials'
bounds -- for dynamic scaling, and for delayed scaling over three steps
with the amaxes synced over the group."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from helpers import assert_within_bound

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
M, K, N, WORLD, STEPS = 544, 784, 512, 2, 3


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(step):
    import synth_inputs as si
    x, w, dy = si.linear_inputs(M, K, N, w_init="uniform64", outlier_frac=0.01, seed=23,
                                step=step)
    return x, w, dy


def _worker(rank, port, scaling, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(WORLD))
    sys.path.insert(0, ROOT)
    import quantised_gemm_gb300 as q
    from quantised_gemm_gb300.sharded import ShardedFp8Linear
    torch.cuda.set_device(0)
    torch.distributed.init_process_group("gloo", init_method="env://")
    try:
        lin = ShardedFp8Linear(M // WORLD, K, N, scaling=scaling, history_len=4)
        rows = slice(rank * M // WORLD, (rank + 1) * M // WORLD)
        res = []
        for t in range(STEPS if scaling == "delayed" else 1):
            x, w, dy = _inputs(t)
            dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(  # noqa
                torch.bfloat16).cuda()
            lin.forward(dev(x[rows]), dev(w))
            dx, dw = lin.backward(dev(dy[rows]))
            q.check(lin.lin.ws)
            L = lin.lin
            bits = lambda t: int(t.view(torch.int32).item()) & 0xFFFFFFFF  # noqa: E731
            res.append({"scales": [bits(s.scale) for s in (L.sx, L.sw, L.sdy)],
                        "x8": L.x8.cpu().numpy(), "x8t": L.x8t.cpu().numpy(),
                        "w8": L.w8.cpu().numpy(), "w8t": L.w8t.cpu().numpy(),
                        "dy8": L.dy8.cpu().numpy(), "dy8t": L.dy8t.cpu().numpy(),
                        "y": L.y.float().cpu().numpy(), "dx": dx.float().cpu().numpy(),
                        "dw": dw.cpu().numpy()})
            lin.sync_scales()
        out.put((rank, res, None))
    except Exception as e:  # report to the parent instead of hanging it
        out.put((rank, None, repr(e)))
    finally:
        torch.distributed.destroy_process_group()


@pytest.mark.parametrize("scaling", ["dynamic", "delayed"])
def test_sharded_linear_two_ranks_on_one_gpu(scaling, oracle_mod):
    o = oracle_mod
    ctx = mp.get_context("spawn")
    qu = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, scaling, qu)) for r in range(WORLD)]
    for p in procs:
        p.start()
    got = dict()
    for _ in range(WORLD):
        r, res, err = qu.get(timeout=600)
        assert err is None, "rank %d: %s" % (r, err)
        got[r] = res
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    f32 = lambda v: int(np.float32(v).view(np.uint32))  # noqa: E731
    states = [o.DelayedState(4, f) for f in (o.E4M3, o.E4M3, o.E5M2)]
    for t in range(len(got[0])):
        x, w, dy = _inputs(t)
        amaxes = [o.amax(x), o.amax(w), o.amax(dy)]       # of the whole tensors
        if scaling == "dynamic":
            scales = [o.scale_dynamic(a, f)[0] for a, f in zip(amaxes, (o.E4M3, o.E4M3, o.E5M2))]
        else:
            if t == 0:
                for s, a in zip(states, amaxes):
                    s.init_from(a)
            scales = [s.scale for s in states]
        sx, sw, sd = scales
        xq, xqt, _ = o.cast(x, sx, o.E4M3)
        wq, wqt, _ = o.cast(w, sw, o.E4M3)
        dq, dqt, _ = o.cast(dy, sd, o.E5M2)
        dw_ref = np.zeros((N, K))
        dw_abs = np.zeros((N, K))
        dw_s = np.zeros((N, K))
        for r in range(WORLD):
            rows = slice(r * M // WORLD, (r + 1) * M // WORLD)
            g = got[r][t]
            assert g["scales"] == [f32(sx), f32(sw), f32(sd)], (t, r)
            assert np.array_equal(g["x8"], xq[rows]) and np.array_equal(g["x8t"], xqt[:, rows])
            assert np.array_equal(g["w8"], wq) and np.array_equal(g["w8t"], wqt)
            assert np.array_equal(g["dy8"], dq[rows]) and np.array_equal(g["dy8t"], dqt[:, rows])
            y, s = o.gemm(xq[rows], wq, o.E4M3, o.E4M3, sx, sw)
            assert_within_bound(g["y"].astype(np.float64), y, s, "y rank %d step %d" % (r, t))
            y, s = o.gemm(dq[rows], wqt, o.E5M2, o.E4M3, sd, sw)
            assert_within_bound(g["dx"].astype(np.float64), y, s, "dX rank %d step %d" % (r, t))
            y, s = o.gemm(np.ascontiguousarray(dqt[:, rows]), np.ascontiguousarray(xqt[:, rows]),
                          o.E5M2, o.E4M3, sd, sx)
            dw_ref += y
            dw_abs += np.abs(y)
            dw_s += s
        bound = np.ldexp(dw_abs, -7) + 1e-4 * dw_s
        for r in range(WORLD):
            err = np.abs(got[r][t]["dw"].astype(np.float64) - dw_ref)
            assert np.all(err <= bound), ("dW sum", r, t, float(np.max(err / bound)))
        if scaling == "delayed":
            for s, a in zip(states, amaxes):
                s.update(a)
