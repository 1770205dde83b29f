"""Seeded synthetic inputs for the MoE layer forward.

This module only draws random tensors of fixed shapes and distributions; it holds none of the
layer's arithmetic (no routing, no dispatch, no expert math).  Both the CPU oracle and the CUDA
path receive the very same tensors from here (the oracle gets host copies widened to float64).

Workload shapes follow the model families the pages discuss: a Mixtral-8x7B-shaped layer and a
DeepSeek-V3-shaped layer ("Systems for Mixture-of-Experts Models" §1.2 and §5.2, "MoE 推理优化深入"
§1 table) and a DeepSeekMoE-16B-shaped layer ("MoE 路由数学" §1 table, §2.2).  No public dataset
or trained weights are involved: every tensor is i.i.d. random,

  x      ~ N(0, 1)                      [T, d]
  W_gate ~ N(0, 1/d)                    [E, d]   (row e = expert e's router vector)
  W1, W3 ~ N(0, 1/d), W2 ~ N(0, 1/F)    per expert, SwiGLU
  bias   ~ U(-0.1, 0.1)                 [E]      (selection-only bias, sigmoid scoring)
  d_topk_w ~ N(0, 1)                    [T, k]   (upstream gradient of the routing weights)

Each tensor is drawn from its own torch.Generator, seeded from (workload, tensor name, seed), so
the draws do not depend on the order in which tensors are made; every routed expert's W13 and W2
have generators of their own (tensor names "w13/e", "w2/e"), so any subset of experts can be
drawn alone (expert_weights).  Large weight sets may be drawn
on the GPU (device="cuda") with a CUDA generator; then the oracle receives host copies of them.

Layouts (row-major, contiguous):
  x      [T, d]
  w_gate [E, d]
  bias   [E] float32 (zeros unless the workload has a selection bias)
  w13    [E, 2F, d]  rows [0, F) = W1 (gate projection), rows [F, 2F) = W3 (up projection)
  w2     [E, d, F]
  ws13   [2 Fs, d]   the n_shared shared experts concatenated into one expert of width
                     Fs = n_shared * F_shared (gate rows first, then up rows)
  ws2    [d, Fs]
"""
from __future__ import annotations

import dataclasses
import hashlib
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int                 # tokens in one forward
    d: int                 # d_model
    E: int                 # routed experts
    k: int                 # experts per token (token choice) / T*k/E tokens per expert (expert choice)
    F: int                 # routed expert d_ff
    n_shared: int = 0      # shared (always-on) experts
    F_shared: int = 0      # d_ff of one shared expert
    score: str = "softmax"         # "softmax" | "sigmoid"
    routing: str = "token_choice"  # "token_choice" | "expert_choice"
    n_groups: int = 1
    topk_groups: int = 1
    renormalize: bool = True
    route_scale: float = 1.0
    capacity_factor: float = 0.0   # <= 0: no capacity limit
    dtype: str = "bf16"            # "bf16" (bf16 weights/activations) | "f32"
    bias_range: float = 0.0        # bias ~ U(-r, r) when > 0
    collapse_shift: float = 0.0    # added to expert 0's logit through a shift of x (see make_inputs)
    zero_router: bool = False      # W_gate = 0: forced-uniform routing

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def F_sh(self) -> int:
        return self.n_shared * self.F_shared


WORKLOADS = {
    # small case the oracle finishes in seconds (fp32 throughout)
    "tiny": Workload("tiny", T=256, d=64, E=8, k=2, F=128, capacity_factor=1.25, dtype="f32"),
    # k = E: softmax routing reduces to a dense gated mixture
    "tiny_dense": Workload("tiny_dense", T=256, d=64, E=4, k=4, F=128, dtype="f32"),
    # W_gate = 0: every probability is exactly 1/E
    "tiny_uniform": Workload("tiny_uniform", T=256, d=64, E=8, k=2, F=128, capacity_factor=1.25,
                             dtype="f32", zero_router=True),
    # Mixtral-8x7B-shaped layer
    "mixtral": Workload("mixtral", T=4096, d=4096, E=8, k=2, F=14336),
    "mixtral_collapsed": Workload("mixtral_collapsed", T=4096, d=4096, E=8, k=2, F=14336,
                                  collapse_shift=3.0),
    # DeepSeekMoE-16B-shaped layer: 64 routed (top-6) + 2 shared experts
    "dsmoe16b": Workload("dsmoe16b", T=8192, d=2048, E=64, k=6, F=1408, n_shared=2, F_shared=1408),
    "dsmoe16b_ec": Workload("dsmoe16b_ec", T=8192, d=2048, E=64, k=6, F=1408, n_shared=2,
                            F_shared=1408, routing="expert_choice"),
    # DeepSeek-V3-shaped layer: sigmoid + selection bias, 8 groups keep 4, top-8, scale 2.5
    "v3": Workload("v3", T=8192, d=7168, E=256, k=8, F=2048, n_shared=1, F_shared=2048,
                   score="sigmoid", n_groups=8, topk_groups=4, route_scale=2.5, bias_range=0.1),
}


def workload(name: str, **overrides) -> Workload:
    wl = WORKLOADS[name]
    return wl.replace(**overrides) if overrides else wl


def _seed(wl_name: str, tensor: str, seed: int) -> int:
    h = hashlib.sha256(f"{wl_name}/{tensor}/{seed}".encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(wl_name: str, tensor: str, seed: int, device: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed(wl_name, tensor, seed))
    return g


def _normal(shape, std, g, device, dtype) -> torch.Tensor:
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    t.mul_(std)
    return t.to(dtype)


def torch_dtype(wl: Workload) -> torch.dtype:
    return torch.bfloat16 if wl.dtype == "bf16" else torch.float32


def make_router_inputs(wl: Workload, seed: int = 0, device: str = "cpu", T: int | None = None):
    """x, w_gate and bias only (what routing, dispatch and the statistics read)."""
    T = wl.T if T is None else T
    dt = torch_dtype(wl)
    name = wl.name
    x = _normal((T, wl.d), 1.0, _gen(name, "x", seed, device), device, torch.float32)
    if wl.zero_router:
        w_gate = torch.zeros((wl.E, wl.d), dtype=torch.float32, device=device)
    else:
        w_gate = _normal((wl.E, wl.d), 1.0 / math.sqrt(wl.d), _gen(name, "w_gate", seed, device),
                         device, torch.float32)
    if wl.collapse_shift:
        # Raise expert 0's logit by about `collapse_shift` for every token while keeping the
        # router linear: x <- x + shift * w0 / |w0|^2, so that x.w0 grows by `shift`.
        w0 = w_gate[0].to(dt).to(torch.float64)
        x = (x.to(torch.float64) + wl.collapse_shift * w0 / (w0 @ w0)).to(torch.float32)
    if wl.bias_range > 0:
        g = _gen(name, "bias", seed, device)
        bias = (torch.rand((wl.E,), generator=g, device=device, dtype=torch.float32) * 2 - 1)
        bias.mul_(wl.bias_range)
    else:
        bias = torch.zeros((wl.E,), dtype=torch.float32, device=device)
    return {"x": x.to(dt).contiguous(), "w_gate": w_gate.to(dt).contiguous(), "bias": bias}


def expert_weights(wl: Workload, e: int, seed: int = 0, device: str = "cpu"):
    """Routed expert e alone: (w13_e [2F, d], w2_e [d, F]), the same values as row e of
    make_expert_weights."""
    dt = torch_dtype(wl)
    d, F = wl.d, wl.F
    return (_normal((2 * F, d), 1.0 / math.sqrt(d), _gen(wl.name, f"w13/{e}", seed, device),
                    device, dt),
            _normal((d, F), 1.0 / math.sqrt(F), _gen(wl.name, f"w2/{e}", seed, device), device,
                    dt))


def make_expert_weights(wl: Workload, seed: int = 0, device: str = "cpu"):
    """Routed expert weights w13 [E,2F,d], w2 [E,d,F] and the shared expert (ws13, ws2)."""
    dt = torch_dtype(wl)
    name = wl.name
    d, F, E = wl.d, wl.F, wl.E
    w13 = torch.empty((E, 2 * F, d), dtype=dt, device=device)
    w2 = torch.empty((E, d, F), dtype=dt, device=device)
    for e in range(E):
        a, b = expert_weights(wl, e, seed, device)
        w13[e].copy_(a)
        w2[e].copy_(b)
        del a, b
    out = {"w13": w13, "w2": w2, "ws13": None, "ws2": None}
    if wl.n_shared > 0:
        Fs = wl.F_shared
        gates, ups, downs = [], [], []
        for s in range(wl.n_shared):
            g13 = _normal((2 * Fs, d), 1.0 / math.sqrt(d), _gen(name, f"ws13_{s}", seed, device),
                          device, dt)
            gates.append(g13[:Fs])
            ups.append(g13[Fs:])
            downs.append(_normal((d, Fs), 1.0 / math.sqrt(Fs), _gen(name, f"ws2_{s}", seed, device),
                                 device, dt))
        out["ws13"] = torch.cat(gates + ups, dim=0).contiguous()
        out["ws2"] = torch.cat(downs, dim=1).contiguous()
    return out


def shared_weights(wl: Workload, seed: int = 0, device: str = "cpu"):
    """The shared experts alone, concatenated: (ws13 [2 Fs, d], ws2 [d, Fs]) or (None, None)."""
    if wl.n_shared == 0:
        return None, None
    w = make_expert_weights(wl.replace(E=0), seed, device)
    return w["ws13"], w["ws2"]


def make_inputs(wl: Workload, seed: int = 0, device: str = "cpu", T: int | None = None):
    d = make_router_inputs(wl, seed, device, T)
    d.update(make_expert_weights(wl, seed, device))
    return d


def make_grad_inputs(wl: Workload, seed: int = 0, device: str = "cpu", T: int | None = None):
    """Inputs of the router-side backward and the bias update: an upstream gradient of the
    routing weights d_topk_w ~ N(0, 1) [T, k] float32 and a bias state ~ U(-0.1, 0.1) [E]
    float32."""
    T = wl.T if T is None else T
    d_w = _normal((T, wl.k), 1.0, _gen(wl.name, "d_topk_w", seed, device), device, torch.float32)
    g = _gen(wl.name, "bias_state", seed, device)
    b = (torch.rand((wl.E,), generator=g, device=device, dtype=torch.float32) * 2 - 1) * 0.1
    return {"d_topk_w": d_w.contiguous(), "bias_state": b}


def to_f64(t: torch.Tensor | None):
    """Exact widening to a float64 numpy array (bf16 and fp32 values are representable)."""
    if t is None:
        return None
    return t.detach().to("cpu").to(torch.float64).numpy()
