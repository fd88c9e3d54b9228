"""The autograd Function / nn.Module level on the GPU: same kernels as the
op level, parity with the fp64 oracle, and the destructive-backward guard."""
import numpy as np
import pytest
import torch

import oracle
from backward_tcgen05_tma_gb300 import api, build, synthetic
from backward_tcgen05_tma_gb300.module import SwiGLUMLP, SwiGLUMLPFunction, swiglu_mlp

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "f16": 1e-2, "f32": 1e-5}
ODT = {"bf16": oracle.BF16, "f16": oracle.F16, "f32": oracle.F32}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    api.lib()


def f64(t):
    return t.detach().cpu().double().numpy()


def _module(t):
    return SwiGLUMLP.from_weights(t["Wg"], t["Wu"], t["Wd"])


@pytest.mark.parametrize("dtn", ["bf16", "f16", "f32"])
def test_module_matches_oracle(dtn):
    # [B=3, S=111, D=320] input (ragged tiles), H=392
    B, S, D, H = 3, 111, 320, 392
    if dtn == "f32":
        B, S, D, H = 2, 16, 64, 176
    t = synthetic.make_inputs(B * S, D, H, dtn, seed=21, device="cuda")
    m = _module(t)
    x = t["X"].reshape(B, S, D).clone().requires_grad_(True)
    y = m(x)
    assert y.shape == (B, S, D)
    y.backward(t["dY"].reshape(B, S, D))
    torch.cuda.synchronize()
    c = {k: v.cpu() for k, v in t.items()}
    f = oracle.forward(c["X"], c["Wg"], c["Wu"], c["Wd"], dt=ODT[dtn])
    b = oracle.backward(c["dY"], c["X"], c["Wg"], c["Wu"], c["Wd"], f, dt=ODT[dtn])
    got = {"Y": f64(y.reshape(B * S, D)), "dX": f64(x.grad.reshape(B * S, D)),
           "dWg": f64(m.gate_up_weight.grad[:H]), "dWu": f64(m.gate_up_weight.grad[H:]),
           "dWd": f64(m.down_weight.grad)}
    for k, v in got.items():
        e = oracle.rel_frob(v, b[k] if k in b else f[k])
        assert e <= TOL[dtn], (k, e)


def test_module_equals_op_level_bitwise():
    t = synthetic.make_inputs(300, 256, 392, "bf16", seed=22, device="cuda")
    m = _module(t)
    x = t["X"].clone().requires_grad_(True)
    y = m(x)
    y.backward(t["dY"])
    Y, saved = api.swiglu_mlp_fwd(t["X"], t["Wgu"], t["Wd"])
    dX, dWgu, dWd = api.swiglu_mlp_bwd(t["dY"], t["X"], t["Wgu"], t["Wd"], saved)
    torch.cuda.synchronize()
    assert torch.equal(y.detach(), Y)
    assert torch.equal(x.grad, dX)
    assert torch.equal(m.gate_up_weight.grad, dWgu)
    assert torch.equal(m.down_weight.grad, dWd)


def test_no_grad_uses_inference_path():
    t = synthetic.make_inputs(17, 256, 392, "bf16", seed=23, device="cuda")
    m = _module(t)
    with torch.no_grad():
        y = m(t["X"])
    assert not y.requires_grad and y.grad_fn is None
    Yn, _ = api.swiglu_mlp_fwd_nograd(t["X"], t["Wgu"], t["Wd"])
    torch.cuda.synchronize()
    assert torch.equal(y, Yn)


def test_packed_inference_copy_is_used_and_dropped_on_update():
    """pack_for_inference: no-grad calls of up to 64 tokens stream the packed
    copy (bitwise equal to the plain path, a single packed launch pair); an
    in-place weight update drops the copy, so the next call reads the new
    weights; calls with more tokens or with autograd take the usual paths."""
    t = synthetic.make_inputs(16, 256, 392, "bf16", seed=29, device="cuda")
    m = _module(t).pack_for_inference()
    x = t["X"]
    with torch.no_grad():
        y = m(x)
        y_ref, _ = api.swiglu_mlp_fwd_nograd(x, m.gate_up_weight, m.down_weight)
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref)
        assert m._packed_copy() is not None
        m.down_weight.mul_(0.5)  # an optimiser-style in-place update
        y2 = m(x)
        assert m._packed_copy() is None
        y2_ref, _ = api.swiglu_mlp_fwd_nograd(x, m.gate_up_weight, m.down_weight)
        torch.cuda.synchronize()
        assert torch.equal(y2, y2_ref) and not torch.equal(y2, y)
        m.pack_for_inference()
        x65 = torch.randn(65, 256, device="cuda").bfloat16()
        y65 = m(x65)  # beyond the few-token path: the row-major weights
        y65_ref, _ = api.swiglu_mlp_fwd_nograd(x65, m.gate_up_weight, m.down_weight)
        torch.cuda.synchronize()
        assert torch.equal(y65, y65_ref)
    xg = x.clone().requires_grad_(True)
    yg = m(xg)  # autograd: the training kernels, G/U saved
    assert yg.grad_fn is not None
    m.pack_for_inference(False)
    assert m._packed_copy() is None


def test_second_backward_is_refused():
    t = synthetic.make_inputs(64, 64, 176, "bf16", seed=24, device="cuda")
    m = _module(t)
    x = t["X"].clone().requires_grad_(True)
    y = m(x)
    loss = (y.float() * t["dY"].float()).sum()
    loss.backward(retain_graph=True)
    with pytest.raises(RuntimeError):
        loss.backward()
    torch.cuda.synchronize()


def test_double_backward_is_refused():
    t = synthetic.make_inputs(64, 64, 176, "bf16", seed=25, device="cuda")
    x = t["X"].clone().requires_grad_(True)
    Wgu = t["Wgu"].clone().requires_grad_(True)
    y = SwiGLUMLPFunction.apply(x, Wgu, t["Wd"])
    (gx,) = torch.autograd.grad(y, x, t["dY"], create_graph=True)
    with pytest.raises(RuntimeError):
        gx.sum().backward()
    torch.cuda.synchronize()


def test_training_loop_reduces_loss():
    """A few SGD steps through the module drive ||Y - T||^2 down (the
    gradients point downhill), all in the library's kernels."""
    D, H, M = 128, 256, 256
    t = synthetic.make_inputs(M, D, H, "bf16", seed=26, device="cuda")
    m = _module(t)
    target = (t["dY"].float() * 10).bfloat16()
    opt = torch.optim.SGD(m.parameters(), lr=0.5)
    losses = []
    for _ in range(5):
        opt.zero_grad()
        y = swiglu_mlp(t["X"], m.gate_up_weight, m.down_weight)
        diff = y.float() - target.float()
        loss = (diff * diff).mean()
        loss.backward()
        opt.step()
        losses.append(float(loss.detach()))
    assert all(np.isfinite(losses)) and losses[-1] < losses[0], losses
