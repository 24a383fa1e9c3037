"""The torch.nn front end (Float8Linear, convert_to_float8_training,
sync_float8_amax_and_scale_history) against the oracle: forward output and
both gradients through autograd meet the GEMM bound, casts bit-exact."""
import numpy as np
import pytest
import torch
from torch import nn

import oracle
import quantised_gemm_gb300 as q
import synth_inputs as si
from helpers import assert_within_bound, bf16_to_f64, to_dev_bf16

pytestmark = pytest.mark.gpu

E4M3, E5M2 = oracle.E4M3, oracle.E5M2


def test_float8_linear_autograd_matches_oracle():
    B, T, K, N = 2, 72, 272, 208                   # M = 144 tokens
    x_h, w_h, dy_h = si.linear_inputs(B * T, K, N, w_init="kaiming", seed=13)
    lin = q.Float8Linear(K, N)
    with torch.no_grad():
        lin.weight.copy_(to_dev_bf16(w_h))
    x = to_dev_bf16(x_h).reshape(B, T, K).requires_grad_(True)
    y = lin(x)
    assert y.shape == (B, T, N) and y.dtype == torch.bfloat16
    y.backward(to_dev_bf16(dy_h).reshape(B, T, N))
    sx = oracle.scale_dynamic(oracle.amax(x_h), E4M3)[0]
    sw = oracle.scale_dynamic(oracle.amax(w_h), E4M3)[0]
    sd = oracle.scale_dynamic(oracle.amax(dy_h), E5M2)[0]
    ref = oracle.linear_fwd_bwd(x_h, w_h, dy_h, sx, sw, sd)
    assert_within_bound(bf16_to_f64(y.reshape(B * T, N)), ref["y"], ref["sy"], "y")
    assert_within_bound(bf16_to_f64(x.grad.reshape(B * T, K)), ref["dx"], ref["sdx"], "dx")
    assert_within_bound(bf16_to_f64(lin.weight.grad), ref["dw"], ref["sdw"], "dw")


def test_two_forwards_before_backward_keep_their_scales():
    """Each backward uses the inverse scales of its own forward."""
    K, N, M = 256, 128, 64
    lin = q.Float8Linear(K, N)
    x1_h = si.normal_bf16((M, K), 1.0, 1, 1)
    x2_h = si.normal_bf16((M, K), 8.0, 2, 1)       # different amax -> different scale
    dy_h = si.normal_bf16((M, N), 1e-3, 3, 3)
    w_h = lin.weight.detach().float().cpu()
    w_bits = si.f32_to_bf16_bits(w_h.numpy())
    x1 = to_dev_bf16(x1_h).requires_grad_(True)
    x2 = to_dev_bf16(x2_h).requires_grad_(True)
    y1 = lin(x1)
    y2 = lin(x2)                                   # overwrites the module's live scales
    y1.backward(to_dev_bf16(dy_h))
    sx1 = oracle.scale_dynamic(oracle.amax(x1_h), E4M3)[0]
    sw = oracle.scale_dynamic(oracle.amax(w_bits), E4M3)[0]
    sd = oracle.scale_dynamic(oracle.amax(dy_h), E5M2)[0]
    ref = oracle.linear_fwd_bwd(x1_h, w_bits, dy_h, sx1, sw, sd)
    assert_within_bound(bf16_to_f64(x1.grad), ref["dx"], ref["sdx"], "dx of the first forward")
    del y2


def test_convert_swaps_linears_and_trains():
    torch.manual_seed(0)
    model = nn.Sequential(nn.Linear(256, 512), nn.GELU(), nn.Linear(512, 256)).cuda().to(
        torch.bfloat16)
    q.convert_to_float8_training(model)
    assert isinstance(model[0], q.Float8Linear) and isinstance(model[2], q.Float8Linear)
    x = torch.randn(128, 256, device="cuda", dtype=torch.bfloat16)
    out = model(x)
    loss = out.float().pow(2).mean()
    loss.backward()
    for p in model.parameters():
        assert p.grad is not None and torch.isfinite(p.grad.float()).all()


def test_delayed_config_and_sync():
    cfg = q.Float8LinearConfig(
        cast_config_input=q.CastConfig("delayed", history_len=4),
        cast_config_weight=q.CastConfig("delayed", history_len=4),
        cast_config_grad_output=q.CastConfig("delayed", history_len=4))
    model = nn.Sequential(nn.Linear(128, 128, bias=False)).cuda().to(torch.bfloat16)
    q.convert_to_float8_training(model, cfg)
    lin = model[0]
    for step in range(3):
        x = torch.randn(64, 128, device="cuda", dtype=torch.bfloat16) * (step + 1)
        model(x).float().sum().backward()
        q.sync_float8_amax_and_scale_history(model)
    hist = lin.sx.amax_history.cpu().numpy()
    assert np.count_nonzero(hist) == 3 and int(lin.sx.head.item()) == 3
    F = 448.0
    assert lin.sx.scale.item() == pytest.approx(F / hist.max(), rel=1e-6)


def test_rejects_non_bf16():
    lin = q.Float8Linear(64, 64)
    with pytest.raises(TypeError):
        lin(torch.randn(16, 64, device="cuda"))


def test_float8_linears_share_one_workspace_per_stream():
    """Every Float8Linear on a stream uses the same workspace (scratch only);
    another stream gets its own, so calls that may overlap never share one."""
    a, b = q.Float8Linear(64, 32), q.Float8Linear(32, 16)
    dev = torch.device("cuda")
    assert a._workspace(dev) is b._workspace(dev)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        other = a._workspace(dev)
        assert other is b._workspace(dev)
    assert other is not a._workspace(dev)
