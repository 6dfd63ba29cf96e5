"""Seeded synthetic inputs for the TTT layer forward.

This module draws random inputs only; it holds none of the layer's arithmetic, so
the CUDA path and the fp64 oracle can both be fed from it.  Everything is drawn on
the CPU from ``torch.Generator().manual_seed(seed)`` in a fixed order
(q, k, v, gate g, then the inner weights), so a (workload, seed) pair names one
input set.

Recipe (the workloads the pages describe, with their shapes; the pages' own data
sets -- Pile, Books3, ImageNet -- are not used):
  * q, k, v ~ N(0, 1) per element; q and k are L2-normalised per token in fp32,
    then rounded to the I/O dtype (bf16 or fp32).
  * inner learning rate: a constant eta, or a per-token, per-head eta_t =
    sigmoid(g_t) with g_t ~ N(0, 1) (the input-dependent learning rate of the
    "Learning to (Learn at Test Time)" walkthrough, section 2.2.3, with the gate's
    projection replaced by a random draw).
  * gate inputs (``gate_inputs``): layer input tokens x ~ N(0, 1) of the model
    width, bf16, and one gate vector per head ~ N(0, 1/width), bf16, so that the
    gate's argument theta . x is O(1) (the sigmoid's working range).
  * inner weights ~ N(0, 0.02^2), biases zero, one set per head shared over the
    batch (the learnable initial weights are shared across sequences, same
    walkthrough, section 2.2.2).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

# name -> (kind, B, H, T, d, m, b, causal, io dtype, eta (float) or "sigmoid", seed)
WORKLOADS = {
    # tiny fp32 TTT-Linear case
    "linear_tiny_f32": ("linear", 1, 2, 64, 16, 0, 16, True, torch.float32, 0.5, 0),
    # TTT-Linear at the 125M-model layer shape
    "linear_125m": ("linear", 8, 12, 2048, 64, 0, 16, True, torch.bfloat16, 1.0, 1),
    # its b = 1 (delta rule) check
    "linear_125m_b1": ("linear", 1, 12, 2048, 64, 0, 1, True, torch.bfloat16, 1.0, 2),
    # long context with input-dependent learning rate
    "linear_long_gated": ("linear", 2, 32, 32768, 64, 0, 16, True, torch.bfloat16, "sigmoid", 3),
    # TTT-MLP (SiLU, hidden 4d) at the 125M-model layer shape
    "mlp_125m": ("mlp", 8, 12, 2048, 64, 256, 16, True, torch.bfloat16, 0.1, 4),
    # full-batch non-causal vision variant (b = N = 196 tokens)
    "vision_linear": ("linear", 256, 6, 196, 64, 0, 196, False, torch.bfloat16, 1.0, 5),
    "vision_mlp": ("mlp", 256, 6, 196, 64, 256, 196, False, torch.bfloat16, 1.0, 6),
    # variants of the pages' other inner losses, epochs, activations and models
    "vision_linear_dot": ("linear", 256, 6, 196, 64, 0, 196, False, torch.bfloat16, 1.0, 8),
    "vision_linear_3ep": ("linear", 256, 6, 196, 64, 0, 196, False, torch.bfloat16, 1.0, 9),
    "mlp_125m_gelu": ("mlp", 8, 12, 2048, 64, 256, 16, True, torch.bfloat16, 0.1, 10),
    "vision_dwconv": ("dwconv", 256, 6, 196, 64, 0, 196, False, torch.bfloat16, 1.0, 7),
    "linear_125m_ln": ("linear", 8, 12, 2048, 64, 0, 16, True, torch.bfloat16, 1.0, 11),
    # the long gated context with the rate computed from the layer input (model width
    # H d = 2048) by the gate, every step
    "linear_long_gate_x": ("linear", 2, 32, 32768, 64, 0, 16, True, torch.bfloat16, 1.0, 12),
    # the rate gate alone at that shape (H heads of d: layer width H d = 2048; eta_base 1)
    "eta_gate_long": ("gate", 2, 32, 32768, 64, 0, 0, False, torch.bfloat16, 1.0, 13),
    # TTT-MLP with the inner norm and residual (the walkthrough's TTT-MLP) at the 125M shape
    "mlp_125m_ln": ("mlp", 8, 12, 2048, 64, 256, 16, True, torch.bfloat16, 0.1, 14),
    # the 125M TTT-MLP shape at eta = 0.01, whose plain inner GD stays finite
    "mlp_125m_eta001": ("mlp", 8, 12, 2048, 64, 256, 16, True, torch.bfloat16, 0.01, 15),
    # the full-batch vision TTT-MLP with the inner norm and residual
    "vision_mlp_ln": ("mlp", 256, 6, 196, 64, 256, 196, False, torch.bfloat16, 1.0, 16),
}

# options beyond the base layer: inner loss ("dot"), inner epochs, MLP activation,
# token grid of the convolution inner model
OPTIONS = {
    "vision_linear_dot": {"loss": "dot"},                   # the ViT3 block's inner loss
    "vision_linear_3ep": {"epochs": 3},                     # several full-batch epochs
    "mlp_125m_gelu": {"activation": "gelu"},                # the walkthrough's TTT-MLP
    "vision_dwconv": {"height": 14, "width": 14, "loss": "dot"},  # ViT3: depthwise conv, dot loss
    "linear_125m_ln": {"ln": True},                         # x + LN(x W): the walkthrough's TTT-Linear
    "linear_long_gate_x": {"gate": True},                   # eta = eta_base sigma(theta_lr . x)
    "mlp_125m_ln": {"ln": True},                            # x + LN(act(x W1 + c1) W2 + c2)
    "vision_mlp_ln": {"ln": True},
}


@dataclass
class Inputs:
    kind: str            # "linear", "mlp", "dwconv" or "gate"
    B: int
    H: int
    T: int
    d: int
    m: int               # hidden width of the MLP (0 for linear)
    b: int               # mini-batch size
    causal: bool
    q: torch.Tensor      # [B,H,T,d] io dtype, CPU
    k: torch.Tensor
    v: torch.Tensor
    eta: torch.Tensor | None   # [B,H,T] fp32 or None
    eta_scalar: float
    params: dict = field(default_factory=dict)   # fp32 CPU tensors: W0 | W1,c1,W2,c2
    options: dict = field(default_factory=dict)  # loss, epochs, activation, height, width
    gate_x: torch.Tensor | None = None      # [B,T,H d] bf16 layer input of the rate gate
    gate_theta: torch.Tensor | None = None  # [H,H d] bf16 gate vectors (eta_base = eta_scalar)

    @property
    def token_heads(self) -> int:
        return self.B * self.H * self.T


def _normal(shape, g, chunk_rows=1 << 22):
    """N(0,1) fp32 drawn in row chunks (bounded peak memory for large workloads)."""
    out = torch.empty(shape, dtype=torch.float32)
    flat = out.view(-1, shape[-1])
    for r0 in range(0, flat.shape[0], chunk_rows):
        r1 = min(r0 + chunk_rows, flat.shape[0])
        flat[r0:r1] = torch.randn((r1 - r0, shape[-1]), generator=g)
    return out


def _unit_rows(x):
    return x / x.norm(dim=-1, keepdim=True)


def make(kind, B, H, T, d, b, causal, dtype=torch.bfloat16, eta=1.0, seed=0, m=0, ln=False):
    """Draw one input set.  ``eta`` is a float (constant) or "sigmoid"; ``ln`` adds
    the inner layer norm's scale ~ 1 + N(0, 0.1^2) and shift ~ N(0, 0.1^2) per head
    (drawn after the weights, so the other draws do not change)."""
    if kind == "gate":  # the rate gate alone: q holds the layer input x [B,T,H d]
        x, theta = gate_inputs(B, T, H, H * d, seed)
        return Inputs(kind, B, H, T, d, 0, b, False, x, None, None, None, float(eta), {},
                      gate_theta=theta)
    g = torch.Generator().manual_seed(seed)
    shape = (B, H, T, d)
    q = _unit_rows(_normal(shape, g)).to(dtype)
    k = _unit_rows(_normal(shape, g)).to(dtype)
    v = _normal(shape, g).to(dtype)
    if eta == "sigmoid":
        eta_t = torch.sigmoid(torch.randn((B, H, T), generator=g)).float()
        eta_scalar = 0.0
    else:
        eta_t, eta_scalar = None, float(eta)
    if kind == "linear":
        params = {"W0": torch.randn((H, d, d), generator=g) * 0.02}
    elif kind == "dwconv":  # nine taps per channel of a depthwise 3x3 convolution
        params = {"W0": torch.randn((H, 9, d), generator=g) * 0.02}
    elif kind == "mlp":
        params = {"W1": torch.randn((H, d, m), generator=g) * 0.02,
                  "c1": torch.zeros((H, m)),
                  "W2": torch.randn((H, m, d), generator=g) * 0.02,
                  "c2": torch.zeros((H, d))}
    else:
        raise ValueError(kind)
    if ln:
        params["ln_gamma"] = 1.0 + 0.1 * torch.randn((H, d), generator=g)
        params["ln_beta"] = 0.1 * torch.randn((H, d), generator=g)
    return Inputs(kind, B, H, T, d, m, b, bool(causal), q, k, v, eta_t, eta_scalar, params)


def workload(name, **override):
    """Inputs of a named workload; keyword overrides (B, H, T, seed, ...) shrink it
    for tests while keeping its value distributions."""
    kind, B, H, T, d, m, b, causal, dtype, eta, seed = WORKLOADS[name]
    kw = dict(kind=kind, B=B, H=H, T=T, d=d, m=m, b=b, causal=causal, dtype=dtype,
              eta=eta, seed=seed)
    kw.update(override)
    kw.setdefault("ln", bool(OPTIONS.get(name, {}).get("ln", False)))
    inp = make(**kw)
    inp.options = dict(OPTIONS.get(name, {}))
    if inp.options.get("gate"):  # drawn after the layer's inputs, from a seed of its own
        inp.gate_x, inp.gate_theta = gate_inputs(inp.B, inp.T, inp.H, inp.H * inp.d, seed=kw["seed"] + 1000)
    return inp


def gate_inputs(B, T, H, dm, seed=0):
    """Layer input tokens x [B,T,dm] and per-head gate vectors theta [H,dm], both bf16
    on the CPU (x drawn first)."""
    g = torch.Generator().manual_seed(seed)
    x = _normal((B, T, dm), g).to(torch.bfloat16)
    theta = (torch.randn((H, dm), generator=g) / dm ** 0.5).to(torch.bfloat16)
    return x, theta
