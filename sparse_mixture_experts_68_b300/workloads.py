"""The layer shapes this library is exercised on.

Each workload is one MoE FFN layer: router Linear(d_model -> N) with bias,
softmax over N, top-k, renormalised gates, N expert FFNs
Linear(d_model -> d_ff) -> activation -> Linear(d_ff -> d_model) with bias,
gate-weighted combine; optional capacity and shared expert.

The shapes come from the pages' examples: the 768-wide, 8-expert, top-2
module of botmartz.com "Mixture of Experts (MoE) and Mixtral", section
"Expert Routing" (run at batch 4 x seq 512 in its "Output" note); Switch-style
top-1 routing with a capacity (roadtointelligence.com "Keeping the experts
busy"; matteuscruz.github.io "Load balancing"); a Mixtral-8x7B-sized layer
(matteuscruz.github.io "Mixtral 8x7B: practical MoE"); and a DeepSeek-V3-sized
layer with 256 routed experts, top-8 and one shared expert
(roadtointelligence.com "Total versus active parameters").
"""

from __future__ import annotations

import math
from dataclasses import dataclass, replace

ACT_GELU_ERF = 0
ACT_RELU = 1
DT_F32 = 0
DT_BF16 = 1


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d_model: int
    d_ff: int
    n_experts: int
    top_k: int
    act: int = ACT_GELU_ERF
    dtype: int = DT_BF16
    capacity_factor: float = 0.0     # 0: no capacity limit
    d_ff_shared: int = 0             # 0: no shared expert
    renormalize: int = 1
    zipf_router_bias: bool = False   # b_g[e] = 2 ln(1 / (e + 1))
    router_scale: float = 1.0        # multiplies W_g
    expert_choice: bool = False      # each expert takes its capacity in tokens; top_k unused
    seed: int = 0
    description: str = ""

    @property
    def capacity(self) -> int:
        """Per-expert capacity, ceil(factor * T / N); 0 means unlimited."""
        if self.capacity_factor <= 0:
            return 0
        return int(math.ceil(self.capacity_factor * self.T / self.n_experts))

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == DT_F32 else 2

    def with_tokens(self, T: int) -> "Workload":
        return replace(self, T=T)


WORKLOADS = {
    "c0_pr1_fp32": Workload(
        "c0_pr1_fp32", T=512, d_model=768, d_ff=3072, n_experts=8, top_k=2,
        act=ACT_GELU_ERF, dtype=DT_F32, seed=0,
        description="T=512 (1x512), d=768, d_ff=3072, N=8, top-2, GELU, fp32"),
    "c1_page1_bf16": Workload(
        "c1_page1_bf16", T=2048, d_model=768, d_ff=3072, n_experts=8, top_k=2,
        act=ACT_GELU_ERF, dtype=DT_BF16, seed=1,
        description="T=2048 (4x512), d=768, d_ff=3072, N=8, top-2, GELU, bf16"),
    "c2_switch_top1": Workload(
        "c2_switch_top1", T=8192, d_model=1024, d_ff=4096, n_experts=64, top_k=1,
        act=ACT_RELU, dtype=DT_BF16, capacity_factor=1.25, zipf_router_bias=True,
        seed=2,
        description="T=8192, d=1024, d_ff=4096, N=64, top-1, ReLU, capacity "
                    "ceil(1.25 T/N)=160, Zipf-skewed router bias, bf16"),
    # the same layer with the raw softmax probability as the gate, no
    # renormalisation (codingnowai.in "Mixture of Experts", section "Code")
    "c2_switch_top1_raw": Workload(
        "c2_switch_top1_raw", T=8192, d_model=1024, d_ff=4096, n_experts=64, top_k=1,
        act=ACT_RELU, dtype=DT_BF16, capacity_factor=1.25, zipf_router_bias=True,
        renormalize=0, seed=2,
        description="T=8192, d=1024, d_ff=4096, N=64, top-1, ReLU, capacity "
                    "ceil(1.25 T/N)=160, Zipf-skewed router bias, raw-probability "
                    "gates (no renormalisation), bf16"),
    "c3_mixtral_prefill": Workload(
        "c3_mixtral_prefill", T=4096, d_model=4096, d_ff=14336, n_experts=8,
        top_k=2, act=ACT_GELU_ERF, dtype=DT_BF16, seed=3,
        description="T=4096, d=4096, d_ff=14336, N=8, top-2, GELU, bf16"),
    "c3_mixtral_decode": Workload(
        "c3_mixtral_decode", T=16, d_model=4096, d_ff=14336, n_experts=8,
        top_k=2, act=ACT_GELU_ERF, dtype=DT_BF16, seed=3,
        description="T=16, d=4096, d_ff=14336, N=8, top-2, GELU, bf16"),
    "c4_deepseek_v3": Workload(
        "c4_deepseek_v3", T=4096, d_model=7168, d_ff=2048, n_experts=256,
        top_k=8, act=ACT_GELU_ERF, dtype=DT_BF16, d_ff_shared=2048,
        router_scale=3.0, seed=4,
        description="T=4096, d=7168, 256 routed experts d_ff=2048 + 1 shared, "
                    "top-8, GELU, router weights x3, bf16"),
    # the DeepSeek-V3-sized layer at a quarter of its experts and tokens (same
    # d, d_ff, top-8 and ~128-row groups; 3.7 GB of weights): a case small
    # enough for an ncu capture of many passes, its DRAM traffic scaled by the
    # experts to the full layer
    "c4_deepseek_v3_quarter": Workload(
        "c4_deepseek_v3_quarter", T=1024, d_model=7168, d_ff=2048, n_experts=64,
        top_k=8, act=ACT_GELU_ERF, dtype=DT_BF16, d_ff_shared=2048, router_scale=3.0,
        seed=4,
        description="T=1024, d=7168, 64 routed experts d_ff=2048 + 1 shared, top-8, "
                    "GELU, router weights x3, bf16"),
    # expert-choice routing (matteuscruz.github.io "Load balancing": every
    # expert picks its top tokens) at the same expert work as top-k routing:
    # C = ceil(k * T / N) tokens per expert
    "c3_mixtral_prefill_ec": Workload(
        "c3_mixtral_prefill_ec", T=4096, d_model=4096, d_ff=14336, n_experts=8,
        top_k=2, act=ACT_GELU_ERF, dtype=DT_BF16, capacity_factor=2.0, expert_choice=True,
        seed=3,
        description="expert choice: T=4096, d=4096, d_ff=14336, N=8, C=ceil(2T/N)=1024 "
                    "tokens per expert, GELU, bf16"),
    "c4_deepseek_v3_ec": Workload(
        "c4_deepseek_v3_ec", T=4096, d_model=7168, d_ff=2048, n_experts=256,
        top_k=8, act=ACT_GELU_ERF, dtype=DT_BF16, d_ff_shared=2048, capacity_factor=8.0,
        expert_choice=True, router_scale=3.0, seed=4,
        description="expert choice: T=4096, d=7168, 256 routed experts d_ff=2048 + 1 "
                    "shared, C=ceil(8T/N)=128 tokens per expert, GELU, router weights x3, "
                    "bf16"),
}


def routed_rows(wl: Workload) -> int:
    """Expert rows of one call without capacity drops: T*k, or N*C for expert
    choice."""
    if wl.expert_choice:
        C = wl.T if wl.capacity <= 0 else min(wl.capacity, wl.T)
        return wl.n_experts * C
    return wl.T * wl.top_k


def flops(wl: Workload, kept_rows: int | None = None) -> float:
    """Algorithmic FLOPs of one layer call: router 2*T*d*N, routed experts
    4*d*d_ff per kept (token, slot) -- or per (expert, picked token) --, shared
    expert 4*d*d_ff_s per token."""
    rows = routed_rows(wl) if kept_rows is None else kept_rows
    return (2.0 * wl.T * wl.d_model * wl.n_experts
            + 4.0 * wl.d_model * wl.d_ff * rows
            + 4.0 * wl.d_model * wl.d_ff_shared * wl.T)
