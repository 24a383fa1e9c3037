"""GPU parity of amax, scale and cast (+transpose) against the oracle:
bit-exact for every amax, scale, inverse scale and fp8 byte."""
import numpy as np
import pytest
import torch

import oracle
import quantised_gemm_gb300 as q
import synth_inputs as si
from helpers import dev_f32_bits, f32_bits, to_dev_bf16

pytestmark = pytest.mark.gpu

E4M3, E5M2 = oracle.E4M3, oracle.E5M2
SHAPES = [(16, 16), (128, 128), (144, 272), (272, 144), (48, 4096), (4096, 48), (1040, 1552)]


@pytest.fixture(scope="module")
def ws():
    return q.Workspace()


def _tensor(shape, seed, outliers=True):
    x = si.normal_bf16(shape, 1.0, seed, 1)
    if outliers:
        x = si.add_outliers(x, 1e-3, 50.0, seed)
    return x


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("algo", [q.AMAX_ATOMIC, q.AMAX_REDUCTION])
def test_amax_bit_exact(shape, algo, ws):
    x = _tensor(shape, seed=shape[0] * 7 + shape[1])
    out = torch.full((1,), -1.0, device="cuda")
    q.amax(to_dev_bf16(x), out, algo, ws)
    assert dev_f32_bits(out) == f32_bits(oracle.amax(x))


@pytest.mark.parametrize("kind", si.EDGE_KINDS)
def test_amax_edge_tensors(kind, ws):
    x = si.edge_tensor(kind, 256, 4096, seed=3)
    ref = f32_bits(oracle.amax(x))
    for algo in (q.AMAX_ATOMIC, q.AMAX_REDUCTION):
        out = torch.full((1,), -1.0, device="cuda")
        q.amax(to_dev_bf16(x), out, algo, ws)
        assert dev_f32_bits(out) == ref, (kind, algo)


def test_amax_strided_and_empty(ws):
    full = _tensor((64, 512), seed=5)
    full[:, 256:] = si.f32_to_bf16_bits(np.full((64, 256), 1e6, dtype=np.float32))
    d = to_dev_bf16(full)[:, :256]                 # row stride 512, 256 columns
    out = torch.zeros(1, device="cuda")
    q.amax(d, out, q.AMAX_ATOMIC, ws)
    assert dev_f32_bits(out) == f32_bits(oracle.amax(full[:, :256]))
    out.fill_(7.0)
    q.amax(torch.empty((0, 64), dtype=torch.bfloat16, device="cuda"), out, q.AMAX_ATOMIC, ws)
    assert out.item() == 0.0


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_scale_dynamic_bit_exact(fmt):
    g = np.random.default_rng(17)
    amaxes = np.concatenate([[0.0, 1e-30, 0.5, 1.0, 3.0e38],
                             np.exp2(g.uniform(-30, 30, 40))]).astype(np.float32)
    st = q.ScalingState(fmt, q.DYNAMIC)
    for a in amaxes:
        st.amax.fill_(float(a))
        q.scale(st)
        s, inv = oracle.scale_dynamic(float(a), fmt)
        assert dev_f32_bits(st.scale) == f32_bits(s), a
        assert dev_f32_bits(st.inv_scale) == f32_bits(inv), a


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_scale_delayed_ring_matches_oracle(fmt):
    g = np.random.default_rng(23)
    amaxes = np.exp2(g.uniform(-6, 6, 25)).astype(np.float32)
    H = 16
    st = q.ScalingState(fmt, q.DELAYED, history_len=H)
    ref = oracle.DelayedState(H, fmt)
    for a in amaxes:
        st.amax.fill_(float(a))
        q.scale(st)
        ref.update(float(a))
        assert dev_f32_bits(st.scale) == f32_bits(ref.scale)
        assert dev_f32_bits(st.inv_scale) == f32_bits(ref.inv_scale)
        assert int(st.head.item()) == ref.head
        assert np.array_equal(st.amax_history.cpu().numpy().view(np.uint32),
                              ref.ring.view(np.uint32))


def test_scale_many_matches_the_oracle_state_by_state():
    """fp8lin_scale_many: eight states in one launch -- delayed ones with
    rings of 1, 3, 16 and 7 (e4m3 and e5m2) and dynamic ones -- each updated
    exactly as one fp8lin_scale would, over 20 steps."""
    g = np.random.default_rng(29)
    specs = [(E4M3, q.DELAYED, 16), (E5M2, q.DELAYED, 16), (E4M3, q.DELAYED, 1),
             (E5M2, q.DELAYED, 3), (E4M3, q.DYNAMIC, 1), (E5M2, q.DYNAMIC, 1),
             (E4M3, q.DELAYED, 7), (E5M2, q.DYNAMIC, 1)]
    sts = [q.ScalingState(f, k, history_len=h) for f, k, h in specs]
    refs = [oracle.DelayedState(h, f) if k == q.DELAYED else None for f, k, h in specs]
    for step in range(20):
        amaxes = np.exp2(g.uniform(-6, 6, len(specs))).astype(np.float32)
        amaxes[step % len(specs)] = 0.0                    # an all-zero tensor now and then
        for st, a in zip(sts, amaxes):
            st.amax.fill_(float(a))
        q.scale_many(sts)
        for (f, k, h), st, ref, a in zip(specs, sts, refs, amaxes):
            if ref is not None:
                ref.update(float(a))
                s, inv = ref.scale, ref.inv_scale
                assert int(st.head.item()) == ref.head
                assert np.array_equal(st.amax_history.cpu().numpy().view(np.uint32),
                                      ref.ring.view(np.uint32))
            else:
                s, inv = oracle.scale_dynamic(float(a), f)
            assert dev_f32_bits(st.scale) == f32_bits(s), (step, f, k, h)
            assert dev_f32_bits(st.inv_scale) == f32_bits(inv), (step, f, k, h)


def test_scale_many_states_may_share_an_amax():
    """Two states reading one amax (the update only reads it) are accepted
    and each gets its own format's scale; a state given twice is refused
    before anything is enqueued."""
    a, b = q.ScalingState(E4M3, q.DYNAMIC), q.ScalingState(E5M2, q.DELAYED, history_len=4)
    b.amax = a.amax
    a.amax.fill_(3.0)
    q.scale_many([a, b])
    for st, fmt in ((a, E4M3), (b, E5M2)):
        s, inv = oracle.scale_dynamic(3.0, fmt)   # (a delayed ring of one amax: the same)
        assert dev_f32_bits(st.scale) == f32_bits(s)
        assert dev_f32_bits(st.inv_scale) == f32_bits(inv)
    before = a.scale.clone()
    with pytest.raises(RuntimeError):
        q.scale_many([a, a])
    torch.cuda.synchronize()
    assert torch.equal(a.scale, before)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("trans", [False, True])
@pytest.mark.parametrize("shape", SHAPES)
def test_cast_bit_exact(fmt, trans, shape):
    x = _tensor(shape, seed=11 + shape[0])
    s, _ = oracle.scale_dynamic(oracle.amax(x), fmt)
    qr, qtr, a = oracle.cast(x, s, fmt, transpose=True)
    rows, cols = shape
    out = torch.full((rows, cols), 0xAA, dtype=torch.uint8, device="cuda")
    out_t = torch.full((cols, rows), 0xAA, dtype=torch.uint8, device="cuda") if trans else None
    amax_out = torch.zeros(1, device="cuda")
    q.cast(to_dev_bf16(x), fmt, torch.tensor([s], device="cuda"), out, out_t, amax_out)
    assert np.array_equal(out.cpu().numpy(), qr)
    if trans:
        assert np.array_equal(out_t.cpu().numpy(), qtr)
    assert dev_f32_bits(amax_out) == f32_bits(a)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_cast_every_bf16_pattern(fmt):
    """All 65536 bf16 patterns except NaN (infinities included) under a set
    of scales: exercises ties, subnormals, saturation and signed zero."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = si.bf16_bits_to_f32(pats)
    pats = np.where(np.isnan(f), np.uint16(0), pats).reshape(256, 256)
    dx = to_dev_bf16(pats)
    scales = [1.0, 448.0, 1.0 / 448, 2.0 ** -20, 2.0 ** 20, 3.7e-3, 12345.678, 0.999999, 57344.0]
    for sv in scales:
        s32 = np.float32(sv)
        qr, qtr, _ = oracle.cast(pats, s32, fmt, transpose=True)
        out = torch.empty((256, 256), dtype=torch.uint8, device="cuda")
        out_t = torch.empty((256, 256), dtype=torch.uint8, device="cuda")
        q.cast(dx, fmt, torch.tensor([s32], device="cuda"), out, out_t)
        got = out.cpu().numpy()
        assert np.array_equal(got, qr), (sv, np.argwhere(got != qr)[:4].tolist())
        assert np.array_equal(out_t.cpu().numpy(), qtr), sv


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("algo", [q.AMAX_ATOMIC, q.AMAX_REDUCTION, q.AMAX_SINGLE_PASS, q.AMAX_AUTO])
@pytest.mark.parametrize("shape", [(144, 272), (1024, 4096), (4096, 1024), (4096, 4096)])
def test_cast_dynamic_all_algorithms(fmt, algo, shape, ws):
    x = _tensor(shape, seed=29)
    a = oracle.amax(x)
    s, inv = oracle.scale_dynamic(a, fmt)
    qr, qtr, _ = oracle.cast(x, s, fmt, transpose=True)
    st = q.ScalingState(fmt, q.DYNAMIC, amax_algo=algo)
    out = torch.empty(shape, dtype=torch.uint8, device="cuda")
    out_t = torch.empty(shape[::-1], dtype=torch.uint8, device="cuda")
    q.cast_dynamic(to_dev_bf16(x), st, out, out_t, ws)
    q.check(ws)
    assert dev_f32_bits(st.amax) == f32_bits(a)
    assert dev_f32_bits(st.scale) == f32_bits(s)
    assert dev_f32_bits(st.inv_scale) == f32_bits(inv)
    assert np.array_equal(out.cpu().numpy(), qr)
    assert np.array_equal(out_t.cpu().numpy(), qtr)


def _random_cast_shapes(n, seed=61):
    """Seeded [rows, cols], multiples of 16 up to 8192 each, within the single
    pass's capacity (at most 152 x 7 tiles of 128 x 128): small ones go to the
    one-cluster kernel, the rest to the cooperative one; mostly ragged."""
    g = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        hi = 33 if len(out) % 2 == 0 else 513   # every other shape at most 512 x 512
        r, c = (int(v) * 16 for v in g.integers(1, hi, 2))
        if -(-r // 128) * -(-c // 128) <= 152 * 7:
            out.append((r, c))
    return out


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("algo", [q.AMAX_ATOMIC, q.AMAX_REDUCTION, q.AMAX_SINGLE_PASS, q.AMAX_AUTO])
@pytest.mark.parametrize("shape", _random_cast_shapes(6))
def test_cast_dynamic_random_shapes(fmt, algo, shape, ws):
    """Every amax algorithm of the dynamic cast on random ragged shapes: amax,
    scale, inverse and every byte of q and q^T as the oracle has them."""
    x = _tensor(shape, seed=shape[0] + 3 * shape[1])
    a = oracle.amax(x)
    s, inv = oracle.scale_dynamic(a, fmt)
    qr, qtr, _ = oracle.cast(x, s, fmt, transpose=True)
    st = q.ScalingState(fmt, q.DYNAMIC, amax_algo=algo)
    out = torch.empty(shape, dtype=torch.uint8, device="cuda")
    out_t = torch.empty(shape[::-1], dtype=torch.uint8, device="cuda")
    q.cast_dynamic(to_dev_bf16(x), st, out, out_t, ws)
    q.check(ws)
    assert dev_f32_bits(st.amax) == f32_bits(a)
    assert dev_f32_bits(st.scale) == f32_bits(s)
    assert dev_f32_bits(st.inv_scale) == f32_bits(inv)
    assert np.array_equal(out.cpu().numpy(), qr)
    assert np.array_equal(out_t.cpu().numpy(), qtr)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("shape", _random_cast_shapes(6, seed=67))
def test_cast_delayed_random_shapes(fmt, shape, ws):
    """Delayed scaling's one-read cast on random ragged shapes: the first call
    takes its scale from its own amax (amax init), the second keeps the stored
    scale; every byte of q and q^T and the recorded amax as the oracle has
    them."""
    x0 = _tensor(shape, seed=shape[0] + shape[1])
    x1 = si.normal_bf16(shape, 3.0, shape[0] * 7 + shape[1], 1)   # a larger spread: saturates
    st = q.ScalingState(fmt, q.DELAYED, history_len=4)
    out = torch.empty(shape, dtype=torch.uint8, device="cuda")
    out_t = torch.empty(shape[::-1], dtype=torch.uint8, device="cuda")
    s0, _ = oracle.scale_dynamic(oracle.amax(x0), fmt)
    for xh in (x0, x1):
        q.cast_delayed(to_dev_bf16(xh), st, out, out_t, ws)
        q.check(ws)
        assert st.needs_init == 0
        assert dev_f32_bits(st.scale) == f32_bits(s0)
        assert dev_f32_bits(st.amax) == f32_bits(oracle.amax(xh))
        qr, qtr, _ = oracle.cast(xh, s0, fmt, transpose=True)
        assert np.array_equal(out.cpu().numpy(), qr)
        assert np.array_equal(out_t.cpu().numpy(), qtr)


def test_single_pass_capacity_and_refusal(ws):
    cap = q.single_pass_max_elems()
    assert cap >= 4096 * 4096, cap             # holds a 4096 x 4096 weight
    rows = ((cap // 4096) // 128 + 8) * 128     # just above capacity
    x = torch.zeros((rows, 4096), dtype=torch.bfloat16, device="cuda")
    st = q.ScalingState(E4M3, q.DYNAMIC, amax_algo=q.AMAX_SINGLE_PASS)
    out = torch.empty((rows, 4096), dtype=torch.uint8, device="cuda")
    with pytest.raises(q.Fp8linError) as ei:
        q.cast_dynamic(x, st, out, None, ws)
    assert ei.value.status == 2     # FP8LIN_EUNSUPPORTED, nothing enqueued


@pytest.mark.parametrize("algo", [q.AMAX_ATOMIC, q.AMAX_SINGLE_PASS, q.AMAX_AUTO])
def test_workspace_counters_clean_themselves(algo, ws):
    """Consecutive calls share the workspace's counters with no memset in
    between: a large maximum, then a smaller one, then the large one again
    must each come out exactly."""
    big = _tensor((1024, 4096), seed=31)                       # outliers: amax ~ 200
    small = si.normal_bf16((272, 1552), 0.5, 32, 1)            # amax ~ 2.5
    for host in (big, small, big, small):
        st = q.ScalingState(E4M3, q.DYNAMIC, amax_algo=algo)
        rows, cols = host.shape
        out = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
        out_t = torch.empty((cols, rows), dtype=torch.uint8, device="cuda")
        q.cast_dynamic(to_dev_bf16(host), st, out, out_t, ws)
        a = oracle.amax(host)
        s, _ = oracle.scale_dynamic(a, E4M3)
        assert dev_f32_bits(st.amax) == f32_bits(a)
        qr, qtr, _ = oracle.cast(host, s, E4M3, transpose=True)
        assert np.array_equal(out.cpu().numpy(), qr)
        assert np.array_equal(out_t.cpu().numpy(), qtr)
    q.check(ws)
    out = torch.full((1,), -1.0, device="cuda")
    for host in (big, small):                                  # ticketed fp8lin_amax
        q.amax(to_dev_bf16(host), out, q.AMAX_ATOMIC, ws)
        assert dev_f32_bits(out) == f32_bits(oracle.amax(host))


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("shape", [(144, 272), (1040, 1552), (4096, 4096)])
def test_cast_dynamic_precomputed_amax(fmt, shape, ws):
    """AMAX_PRECOMPUTED takes the amax already in the state (as a producing
    GEMM's epilogue leaves it) and runs scale + cast only: same scale, same
    bytes as the oracle; the amax is left as given."""
    x = _tensor(shape, seed=41)
    a = oracle.amax(x)
    s, inv = oracle.scale_dynamic(a, fmt)
    qr, qtr, _ = oracle.cast(x, s, fmt, transpose=True)
    st = q.ScalingState(fmt, q.DYNAMIC, amax_algo=q.AMAX_PRECOMPUTED)
    st.amax.fill_(a)                              # a bf16 magnitude: exact in fp32
    out = torch.empty(shape, dtype=torch.uint8, device="cuda")
    out_t = torch.empty(shape[::-1], dtype=torch.uint8, device="cuda")
    q.cast_dynamic(to_dev_bf16(x), st, out, out_t, ws)
    q.check(ws)
    assert dev_f32_bits(st.amax) == f32_bits(a)
    assert dev_f32_bits(st.scale) == f32_bits(s)
    assert dev_f32_bits(st.inv_scale) == f32_bits(inv)
    assert np.array_equal(out.cpu().numpy(), qr)
    assert np.array_equal(out_t.cpu().numpy(), qtr)


# Shapes that the one-cluster single pass takes (up to 16 tiles of 16384
# elements: 16-row tiles for 16 rows, ... 128-row tiles above 64 rows), and
# one just past it that goes to the cooperative single pass.
CLUSTER_SHAPES = [(16, 16), (16, 4096), (16, 16384), (32, 1552), (48, 4096), (64, 4096),
                  (80, 2048), (128, 2048)]


@pytest.mark.parametrize("trans", [False, True])
@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("shape", CLUSTER_SHAPES + [(128, 2176)])
def test_small_tensor_single_pass(shape, fmt, trans, ws):
    x = _tensor(shape, seed=53 + shape[0])
    a = oracle.amax(x)
    s, inv = oracle.scale_dynamic(a, fmt)
    qr, qtr, _ = oracle.cast(x, s, fmt, transpose=True)
    for algo in (q.AMAX_SINGLE_PASS, q.AMAX_AUTO):
        st = q.ScalingState(fmt, q.DYNAMIC, amax_algo=algo)
        out = torch.full(shape, 0xAA, dtype=torch.uint8, device="cuda")
        out_t = torch.full(shape[::-1], 0xAA, dtype=torch.uint8, device="cuda") if trans else None
        q.cast_dynamic(to_dev_bf16(x), st, out, out_t, ws)
        q.check(ws)
        assert dev_f32_bits(st.amax) == f32_bits(a)
        assert dev_f32_bits(st.scale) == f32_bits(s)
        assert dev_f32_bits(st.inv_scale) == f32_bits(inv)
        assert np.array_equal(out.cpu().numpy(), qr)
        if trans:
            assert np.array_equal(out_t.cpu().numpy(), qtr)


@pytest.mark.parametrize("kind", si.EDGE_KINDS)
def test_small_tensor_single_pass_edge_tensors(kind, ws):
    x = si.edge_tensor(kind, 64, 4096, seed=6)
    for fmt in (E4M3, E5M2):
        a = oracle.amax(x)
        s, inv = oracle.scale_dynamic(a, fmt)
        qr, qtr, _ = oracle.cast(x, s, fmt, transpose=True)
        st = q.ScalingState(fmt, q.DYNAMIC, amax_algo=q.AMAX_AUTO)
        out = torch.empty((64, 4096), dtype=torch.uint8, device="cuda")
        out_t = torch.empty((4096, 64), dtype=torch.uint8, device="cuda")
        q.cast_dynamic(to_dev_bf16(x), st, out, out_t, ws)
        assert dev_f32_bits(st.amax) == f32_bits(a), kind
        assert dev_f32_bits(st.scale) == f32_bits(s), kind
        assert np.array_equal(out.cpu().numpy(), qr), kind
        assert np.array_equal(out_t.cpu().numpy(), qtr), kind


@pytest.mark.parametrize("shape,kernel", [((16, 4096), "cast_cluster_kernel"),
                                          ((128, 2048), "cast_cluster_kernel"),
                                          ((128, 2176), "cast_single_pass_kernel")])
def test_small_tensor_single_pass_kernel_choice(shape, kernel, ws):
    """Up to 16 tiles the single pass runs in one cluster; above, cooperatively."""
    from torch.profiler import ProfilerActivity, profile
    x = to_dev_bf16(_tensor(shape, seed=3))
    out = torch.empty(shape, dtype=torch.uint8, device="cuda")
    st = q.ScalingState(E4M3, q.DYNAMIC, amax_algo=q.AMAX_AUTO)
    names = []
    for _ in range(2):      # the first profiling session of a process may miss kernels
        torch.cuda.synchronize()
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            q.cast_dynamic(x, st, out, None, ws)
            torch.cuda.synchronize()
        names = [e.name for e in prof.events() if "cast" in e.name]
        if names:
            break
    if not names:
        pytest.skip("the profiler recorded no kernels (no CUPTI activity on this host)")
    assert len(names) == 1 and kernel in names[0], names


@pytest.mark.parametrize("algo", [q.AMAX_ATOMIC, q.AMAX_REDUCTION])
@pytest.mark.parametrize("shape", [(1040, 1552), (4096, 4096), (272, 144)])
def test_cast_dynamic_transpose_only(algo, shape, ws):
    """A dynamic cast that asks only for the transposed copy (no q): the
    streaming kernel stages q on chip for the transpose and stores q^T alone."""
    x = _tensor(shape, seed=61)
    a = oracle.amax(x)
    s, inv = oracle.scale_dynamic(a, E5M2)
    _, qtr, _ = oracle.cast(x, s, E5M2, transpose=True)
    st = q.ScalingState(E5M2, q.DYNAMIC, amax_algo=algo)
    out_t = torch.full(shape[::-1], 0xAA, dtype=torch.uint8, device="cuda")
    q.cast_dynamic(to_dev_bf16(x), st, None, out_t, ws)
    q.check(ws)
    assert dev_f32_bits(st.scale) == f32_bits(s)
    assert np.array_equal(out_t.cpu().numpy(), qtr)
