"""Seeded synthetic layer inputs.

This module only draws numbers: it holds none of the layer's arithmetic, and
both the CUDA path's callers and the tests feed its tensors to the kernels and
to the CPU oracle alike.

Recipe (per workload, one torch.Generator seeded with the workload's seed,
tensors drawn in this order, float32 normals scaled then cast to the storage
dtype with round-to-nearest-even):
  W_g ~ N(0, 1/d_model) * router_scale            [N, d]
  b_g ~ N(0, 0.01^2)  or  2 ln(1/(e+1)) (Zipf)    [N]
  per expert e: W1[e] ~ N(0, 1/d_model) [d_ff, d], b1[e] ~ N(0, 0.01^2) [d_ff],
                W2[e] ~ N(0, 1/d_ff)    [d, d_ff], b2[e] ~ N(0, 0.01^2) [d]
  shared expert (if any): same recipe
  x ~ N(0, 1)                                      [T, d]
Weights are nn.Linear-shaped ([out, in]).  Draws happen on ``device``; the
same seed on another device type gives other (equally distributed) values.
"""

from __future__ import annotations

import math

import torch

from .workloads import DT_F32, Workload


def _dtype(wl: Workload):
    return torch.float32 if wl.dtype == DT_F32 else torch.bfloat16


def _normal(gen, shape, std, dtype, device):
    v = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    return (v * std).to(dtype)


def make_layer(wl: Workload, device="cpu", seed: int | None = None,
               with_x: bool = True) -> dict:
    """Draw the weights (and the tokens x) of ``wl``.  Returns a dict of
    tensors: W_g, b_g, W1, b1, W2, b2, (W1s, b1s, W2s, b2s), x."""
    seed = wl.seed if seed is None else seed
    dt = _dtype(wl)
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    N, d, f = wl.n_experts, wl.d_model, wl.d_ff
    out = {}
    out["W_g"] = _normal(gen, (N, d), wl.router_scale / math.sqrt(d), dt, dev)
    if wl.zipf_router_bias:
        e = torch.arange(N, dtype=torch.float64)
        out["b_g"] = (2.0 * torch.log(1.0 / (e + 1.0))).to(dt).to(dev)
    else:
        out["b_g"] = _normal(gen, (N,), 0.01, dt, dev)
    W1 = torch.empty((N, f, d), dtype=dt, device=dev)
    b1 = torch.empty((N, f), dtype=dt, device=dev)
    W2 = torch.empty((N, d, f), dtype=dt, device=dev)
    b2 = torch.empty((N, d), dtype=dt, device=dev)
    for i in range(N):
        W1[i] = _normal(gen, (f, d), 1.0 / math.sqrt(d), dt, dev)
        b1[i] = _normal(gen, (f,), 0.01, dt, dev)
        W2[i] = _normal(gen, (d, f), 1.0 / math.sqrt(f), dt, dev)
        b2[i] = _normal(gen, (d,), 0.01, dt, dev)
    out.update(W1=W1, b1=b1, W2=W2, b2=b2)
    if wl.d_ff_shared:
        fs = wl.d_ff_shared
        out["W1s"] = _normal(gen, (fs, d), 1.0 / math.sqrt(d), dt, dev)
        out["b1s"] = _normal(gen, (fs,), 0.01, dt, dev)
        out["W2s"] = _normal(gen, (d, fs), 1.0 / math.sqrt(fs), dt, dev)
        out["b2s"] = _normal(gen, (d,), 0.01, dt, dev)
    if with_x:
        out["x"] = _normal(gen, (wl.T, d), 1.0, dt, dev)
    return out


def make_tokens(wl: Workload, T: int, device="cpu", seed: int = 0) -> torch.Tensor:
    """Fresh tokens x ~ N(0, 1) of shape [T, d_model] from their own stream."""
    gen = torch.Generator(device=torch.device(device))
    gen.manual_seed(seed)
    return _normal(gen, (T, wl.d_model), 1.0, _dtype(wl), torch.device(device))
