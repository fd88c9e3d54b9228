"""Host-side checks of the autograd Function / nn.Module level (no GPU)."""
import pytest
import torch

from backward_tcgen05_tma_gb300.module import SwiGLUMLP, swiglu_mlp


class _Cfg:
    hidden_size = 64
    intermediate_size = 176
    hidden_act = "silu"
    mlp_bias = False


def test_config_and_size_constructors_agree():
    a = SwiGLUMLP(_Cfg(), dtype=torch.float32)
    b = SwiGLUMLP(64, 176, dtype=torch.float32)
    c = SwiGLUMLP(hidden_size=64, intermediate_size=176, dtype=torch.float32)
    for m in (a, b, c):
        assert m.gate_up_weight.shape == (352, 64)
        assert m.down_weight.shape == (64, 176)
        assert m.gate_weight.shape == m.up_weight.shape == (176, 64)
        # nn.Linear's default init bound 1/sqrt(fan_in)
        assert float(m.gate_up_weight.detach().abs().max()) <= 64 ** -0.5
        assert float(m.down_weight.detach().abs().max()) <= 176 ** -0.5


def test_gate_and_up_are_views_of_one_parameter():
    m = SwiGLUMLP(64, 176, dtype=torch.float32)
    with torch.no_grad():
        m.gate_weight.fill_(1.0)
        m.up_weight.fill_(2.0)
    assert torch.all(m.gate_up_weight[:176] == 1.0) and torch.all(m.gate_up_weight[176:] == 2.0)


def test_three_linear_state_dict_loads():
    g = torch.randn(176, 64)
    u = torch.randn(176, 64)
    d = torch.randn(64, 176)
    m = SwiGLUMLP(64, 176, dtype=torch.float32)
    m.load_state_dict({"gate_proj.weight": g, "up_proj.weight": u, "down_proj.weight": d})
    assert torch.equal(m.gate_weight, g) and torch.equal(m.up_weight, u)
    assert torch.equal(m.down_weight, d)
    # nested under a parent module's prefix
    parent = torch.nn.Module()
    parent.mlp = SwiGLUMLP(64, 176, dtype=torch.float32)
    parent.load_state_dict({"mlp.gate_proj.weight": g, "mlp.up_proj.weight": u,
                            "mlp.down_proj.weight": d})
    assert torch.equal(parent.mlp.up_weight, u)
    # and the module's own layout round-trips
    m2 = SwiGLUMLP(64, 176, dtype=torch.float32)
    m2.load_state_dict(m.state_dict())
    assert torch.equal(m2.gate_up_weight, m.gate_up_weight)


def test_from_weights():
    g, u, d = torch.randn(176, 64), torch.randn(176, 64), torch.randn(64, 176)
    m = SwiGLUMLP.from_weights(g, u, d)
    assert torch.equal(m.gate_up_weight, torch.cat([g, u])) and torch.equal(m.down_weight, d)


def test_rejects_bias_and_other_activations():
    class Biased(_Cfg):
        mlp_bias = True

    class Gelu(_Cfg):
        hidden_act = "gelu"

    with pytest.raises(ValueError):
        SwiGLUMLP(Biased())
    with pytest.raises(ValueError):
        SwiGLUMLP(Gelu())


def test_no_cpu_fallback():
    """The product path has no CPU implementation: host tensors are refused."""
    m = SwiGLUMLP(64, 176, dtype=torch.float32)
    x = torch.randn(4, 64)
    with pytest.raises(ValueError):
        m(x)
    with torch.no_grad(), pytest.raises(ValueError):
        swiglu_mlp(x, m.gate_up_weight, m.down_weight)
