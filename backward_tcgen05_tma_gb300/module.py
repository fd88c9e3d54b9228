"""autograd.Function and nn.Module levels over the C-ABI binding.

The three levels of API from the maintainer thread of "[RFC] Full-pipeline
SwiGLU MLP with forward/backward co-optimization" (Liger-Kernel #1347): the
op level (``api.swiglu_mlp_fwd`` / ``_nograd`` / ``_bwd``), an autograd
Function composing them, and a module usable in place of a transformer
block's SwiGLU MLP (``gate_proj``, ``up_proj``, ``down_proj`` without bias).

Backward writes dG and dU into the buffer that held G and U (the page's
Known limitations), so ``retain_graph=True`` followed by a second backward, and
double differentiation, are refused with an error instead of returning wrong
values.  Every computation runs in the library's CUDA kernels; the tensors
must be contiguous CUDA tensors of one dtype (bf16, fp16, or fp32 for the
IEEE mode).
"""
from __future__ import annotations

import math

import torch

from . import api


class SwiGLUMLPFunction(torch.autograd.Function):
    """Y = md (SiLU(mg X Wg^T) * (X Wu^T)) Wd^T with Wgu = [Wg; Wu] ([2H, D]);
    the gate/down multipliers mg, md are 1 for the standard MLP."""

    @staticmethod
    def forward(ctx, X, Wgu, Wd, gate_mul=1.0, down_mul=1.0):
        D = X.shape[-1]
        lead = X.shape[:-1]
        X2 = X.reshape(-1, D).contiguous()
        Y, saved = api.swiglu_mlp_fwd(X2, Wgu, Wd, gate_mul=gate_mul, down_mul=down_mul)
        ctx.save_for_backward(X2, Wgu, Wd, saved)
        ctx.lead = lead
        ctx.muls = (gate_mul, down_mul)
        ctx.consumed = False
        return Y.reshape(*lead, D)

    @staticmethod
    @torch.autograd.function.once_differentiable
    def backward(ctx, dY):
        if ctx.consumed:
            raise RuntimeError("SwiGLUMLPFunction: backward already ran; dG and dU now occupy "
                               "the buffer that held G and U, so a second backward is "
                               "impossible (retain_graph is not supported)")
        ctx.consumed = True
        X2, Wgu, Wd, saved = ctx.saved_tensors
        D = X2.shape[1]
        dY2 = dY.reshape(-1, D).to(X2.dtype).contiguous()
        dX, dWgu, dWd = api.swiglu_mlp_bwd(dY2, X2, Wgu, Wd, saved, gate_mul=ctx.muls[0],
                                           down_mul=ctx.muls[1])
        return dX.reshape(*ctx.lead, D), dWgu, dWd, None, None


def swiglu_mlp(X, Wgu, Wd, gate_mul: float = 1.0, down_mul: float = 1.0):
    """Functional form: autograd-aware when any input requires grad, otherwise
    the no-grad path (A and Y only, no G/U saved)."""
    if torch.is_grad_enabled() and (X.requires_grad or Wgu.requires_grad or Wd.requires_grad):
        return SwiGLUMLPFunction.apply(X, Wgu, Wd, float(gate_mul), float(down_mul))
    D = X.shape[-1]
    Y, _ = api.swiglu_mlp_fwd_nograd(X.reshape(-1, D).contiguous(), Wgu, Wd, gate_mul=gate_mul,
                                     down_mul=down_mul)
    return Y.reshape(*X.shape[:-1], D)


PACKED_MAX_TOKENS = 64  # the packed-weights entry point serves the few-token path


class SwiGLUMLP(torch.nn.Module):
    """SwiGLU MLP block: down(SiLU(gate(x)) * up(x)), no biases.

    The gate and up projection weights live in one parameter ``gate_up_weight``
    ([2H, D]: gate rows then up rows, as the kernels read them); ``gate_weight``
    and ``up_weight`` are views of it.  ``down_weight`` is [D, H].  Optional
    gate/down multipliers (the Falcon-H1 variant): down(SiLU(mg gate(x)) *
    up(x)) * md, taken from the arguments or from a config's
    ``mlp_multipliers`` pair.
    """

    def __init__(self, config=None, intermediate_size: int | None = None, *,
                 hidden_size: int | None = None, dtype=torch.bfloat16, device=None,
                 gate_multiplier: float | None = None, down_multiplier: float | None = None):
        super().__init__()
        mg, md = 1.0, 1.0
        if config is not None and not isinstance(config, int):
            mults = getattr(config, "mlp_multipliers", None)
            if mults is not None:
                mg, md = float(mults[0]), float(mults[1])
        self.gate_multiplier = float(mg if gate_multiplier is None else gate_multiplier)
        self.down_multiplier = float(md if down_multiplier is None else down_multiplier)
        # Either a transformers-style config (hidden_size, intermediate_size
        # attributes, as the xxxMLP classes take it) or the two sizes.
        if config is not None and not isinstance(config, int):
            D, H = int(config.hidden_size), int(config.intermediate_size)
            if getattr(config, "mlp_bias", False):
                raise ValueError("SwiGLUMLP has no bias terms")
            act = getattr(config, "hidden_act", "silu")
            if act not in ("silu", "swish"):
                raise ValueError("SwiGLUMLP computes SiLU gating, not %r" % (act,))
        else:
            D = int(hidden_size if config is None else config)
            H = int(intermediate_size)
        self.hidden_size, self.intermediate_size = D, H
        self.gate_up_weight = torch.nn.Parameter(torch.empty(2 * H, D, dtype=dtype, device=device))
        self.down_weight = torch.nn.Parameter(torch.empty(D, H, dtype=dtype, device=device))
        self.reset_parameters()
        self._register_load_state_dict_pre_hook(_split_linear_keys)

    def reset_parameters(self):
        # nn.Linear's default: U(-1/sqrt(fan_in), 1/sqrt(fan_in))
        with torch.no_grad():
            b = 1.0 / math.sqrt(self.hidden_size)
            self.gate_up_weight.uniform_(-b, b)
            b = 1.0 / math.sqrt(self.intermediate_size)
            self.down_weight.uniform_(-b, b)

    @property
    def gate_weight(self):
        return self.gate_up_weight[: self.intermediate_size]

    @property
    def up_weight(self):
        return self.gate_up_weight[self.intermediate_size:]

    @classmethod
    def from_weights(cls, gate_weight, up_weight, down_weight, **kwargs):
        """Builds the module from three nn.Linear-style weights ([H,D], [H,D], [D,H])."""
        H, D = gate_weight.shape
        m = cls(D, H, dtype=gate_weight.dtype, device=gate_weight.device, **kwargs)
        with torch.no_grad():
            m.gate_up_weight.copy_(torch.cat([gate_weight, up_weight], dim=0))
            m.down_weight.copy_(down_weight)
        return m

    def pack_for_inference(self, on: bool = True):
        """Keeps (or with ``on=False`` drops) a packed copy of the weights
        (``api.swiglu_mlp_pack_weights``) that no-grad calls of up to 64
        tokens then stream instead of the parameters: the same outputs, bit
        for bit, a few microseconds sooner per call, for a second copy of the
        weights in device memory.  The copy is dropped as soon as either
        parameter is modified in place (its version counter moves), so a
        stale copy is never read; call again after the update to re-pack."""
        self._packed = None
        if on:
            with torch.no_grad():
                pk = api.swiglu_mlp_pack_weights(self.gate_up_weight.detach(),
                                                 self.down_weight.detach())
            self._packed = (pk, self._weights_state())
        return self

    def _weights_state(self):
        w, d = self.gate_up_weight, self.down_weight
        return (w._version, d._version, w.data_ptr(), d.data_ptr(), w.device, w.dtype)

    def _packed_copy(self):
        pk = getattr(self, "_packed", None)
        if pk is None:
            return None
        if self._weights_state() != pk[1]:
            # updated in place, replaced, moved or cast since the copy was made
            self._packed = None
            return None
        return pk[0]

    def forward(self, x):
        packed = self._packed_copy()
        if packed is not None and not (torch.is_grad_enabled() and (
                x.requires_grad or self.gate_up_weight.requires_grad or
                self.down_weight.requires_grad)):
            D = x.shape[-1]
            X = x.reshape(-1, D).contiguous()
            if 0 < X.shape[0] <= PACKED_MAX_TOKENS:
                Y, _ = api.swiglu_mlp_fwd_nograd_packed(X, packed, self.intermediate_size,
                                                        gate_mul=self.gate_multiplier,
                                                        down_mul=self.down_multiplier)
                return Y.reshape(*x.shape[:-1], D)
        return swiglu_mlp(x, self.gate_up_weight, self.down_weight, self.gate_multiplier,
                          self.down_multiplier)

    def extra_repr(self):
        r = "hidden_size=%d, intermediate_size=%d" % (self.hidden_size, self.intermediate_size)
        if self.gate_multiplier != 1.0 or self.down_multiplier != 1.0:
            r += ", gate_multiplier=%g, down_multiplier=%g" % (self.gate_multiplier,
                                                               self.down_multiplier)
        return r


def _split_linear_keys(state_dict, prefix, *args, **kwargs):
    """Accepts the three-Linear layout (``gate_proj.weight``, ``up_proj.weight``,
    ``down_proj.weight``) of a transformers MLP and stacks it into this
    module's two parameters, so a checkpoint of that block loads unchanged."""
    g, u, d = (prefix + n + "_proj.weight" for n in ("gate", "up", "down"))
    if g in state_dict and u in state_dict:
        state_dict[prefix + "gate_up_weight"] = torch.cat([state_dict.pop(g), state_dict.pop(u)], 0)
    if d in state_dict:
        state_dict[prefix + "down_weight"] = state_dict.pop(d)
