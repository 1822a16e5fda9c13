"""The seeded input generator: shapes, dtypes, determinism, distributions."""

import math

import torch

from sparse_mixture_experts_68_b300 import synth
from sparse_mixture_experts_68_b300.workloads import WORKLOADS, Workload, DT_F32


def test_shapes_dtypes_and_determinism():
    wl = Workload("t", T=33, d_model=64, d_ff=128, n_experts=4, top_k=2, dtype=DT_F32,
                  d_ff_shared=128, seed=5)
    a = synth.make_layer(wl)
    b = synth.make_layer(wl)
    assert a["x"].shape == (33, 64) and a["W_g"].shape == (4, 64)
    assert a["W1"].shape == (4, 128, 64) and a["W2"].shape == (4, 64, 128)
    assert a["W1s"].shape == (128, 64) and a["b2s"].shape == (64,)
    for key in a:
        assert a[key].dtype == torch.float32
        assert torch.equal(a[key], b[key])
    c = synth.make_layer(wl, seed=6)
    assert not torch.equal(a["x"], c["x"])


def test_distributions_and_special_biases():
    wl = Workload("z", T=64, d_model=256, d_ff=512, n_experts=16, top_k=1,
                  zipf_router_bias=True, seed=2)
    t = synth.make_layer(wl)
    assert t["x"].dtype == torch.bfloat16
    e = torch.arange(wl.n_experts, dtype=torch.float64)
    zipf = (2.0 * torch.log(1.0 / (e + 1.0))).to(torch.bfloat16)
    assert torch.equal(t["b_g"], zipf)
    std = t["W1"].float().std().item()
    assert abs(std - 1 / math.sqrt(wl.d_model)) < 0.05 / math.sqrt(wl.d_model)
    assert abs(t["W2"].float().std().item() - 1 / math.sqrt(wl.d_ff)) < 0.05 / math.sqrt(wl.d_ff)
    assert abs(t["b1"].float().std().item() - 0.01) < 0.002


def test_capacity_of_switch_workload():
    assert WORKLOADS["c2_switch_top1"].capacity == 160
    assert WORKLOADS["c1_page1_bf16"].capacity == 0
