"""Expert-choice routing on the GPU (through the C ABI) against the CPU oracle:
the selection step alone, bit for bit on fp32 scores with many exact ties;
whole layers on small shapes in full; the two expert-choice workloads at full
size with the output compared on tokens that visit every 128-row m-tile of
every expert's group; edge cases."""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_mixture_experts_68_b300 import binding as B
from sparse_mixture_experts_68_b300 import synth
from sparse_mixture_experts_68_b300.workloads import (ACT_GELU_ERF, ACT_RELU, DT_BF16, DT_F32,
                                                      WORKLOADS, Workload)

from parity import check_ec_layer, check_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    B.lib()
    yield
    torch.cuda.synchronize()
    assert B.get_device_status() == B.MOE_OK


def run_ec(wl, T=None, capacity=None, seed=None):
    t = synth.make_layer(wl if T is None else wl.with_tokens(T), device="cuda", seed=seed)
    layer = B.MoeEcLayer(wl, t, T=T, capacity=capacity)
    out = layer.forward(t["x"], with_logits=True)
    torch.cuda.synchronize()
    return t, layer, out


def sample(T, n, seed):
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(T, size=min(n, T), replace=False).tolist()) | {0, T - 1}
    return np.array(sorted(pick))


@pytest.mark.parametrize("T,N,C,shared", [(5000, 5, 1234, False), (300, 3, 300, True),
                                          (4100, 2, 4099, False), (77, 7, 1, True)])
def test_select_exact_on_tied_scores(T, N, C, shared):
    """moe_ec_select on fp32 scores drawn from 16 levels (so most comparisons
    are ties) equals the oracle's selection on the same values exactly, and
    lays the groups out as documented."""
    wl = Workload("ec_sel", T=T, d_model=64, d_ff=64, n_experts=N, top_k=1,
                  dtype=DT_BF16, capacity_factor=0.0, d_ff_shared=64 if shared else 0,
                  expert_choice=True)
    cfg = B.make_config(wl, capacity=C)
    assert B.ec_tokens_per_expert(cfg) == C
    g = torch.Generator(device="cpu").manual_seed(T + N)
    p = (torch.randint(0, 16, (N, T), generator=g).float() / 16.0).cuda()
    rows = B.ec_rows_max(cfg)
    Cpad = -(-C // 128) * 128
    assert rows == N * Cpad + (-(-T // 128) * 128 if shared else 0)
    dev = "cuda"
    ec_token = torch.full((N, C), -7, dtype=torch.int32, device=dev)
    ec_gate = torch.empty((N, C), dtype=torch.float32, device=dev)
    offsets = torch.empty(N + 2, dtype=torch.int32, device=dev)
    counts = torch.empty(N, dtype=torch.int32, device=dev)
    row_token = torch.full((rows,), -7, dtype=torch.int32, device=dev)
    token_row = torch.empty((T, N), dtype=torch.int32, device=dev)
    token_w = torch.empty((T, N), dtype=torch.float32, device=dev)
    picks = torch.zeros(T, dtype=torch.int32, device=dev)
    B.ec_select(cfg, p, ec_token, ec_gate, offsets, counts, row_token, token_row, token_w,
                picks)
    torch.cuda.synchronize()
    pn = p.cpu().numpy().astype(np.float64)
    sel = O.expert_choice_select(pn.T, C)
    et = ec_token.cpu().numpy()
    for e in range(N):
        np.testing.assert_array_equal(et[e], sel[e])
        np.testing.assert_array_equal(ec_gate[e].cpu().numpy(), pn[e, sel[e]])
    off = offsets.cpu().numpy()
    assert off[:N + 1].tolist() == [e * Cpad for e in range(N + 1)]
    assert off[N + 1] == rows
    assert counts.cpu().tolist() == [C] * N
    rt = row_token.cpu().numpy()
    tr = token_row.cpu().numpy()
    tw = token_w.cpu().numpy()
    want_picks = np.zeros(T, dtype=np.int64)
    for e in range(N):
        np.testing.assert_array_equal(rt[e * Cpad: e * Cpad + C], sel[e])
        assert np.all(rt[e * Cpad + C: (e + 1) * Cpad] == -1)
        inset = np.zeros(T, dtype=bool)
        inset[sel[e]] = True
        np.testing.assert_array_equal(tr[inset, e], e * Cpad + np.arange(C))
        assert np.all(tr[~inset, e] == -1)
        np.testing.assert_array_equal(tw[inset, e], pn[e, inset])
        assert np.all(tw[~inset, e] == 0.0)
        want_picks += inset
    np.testing.assert_array_equal(picks.cpu().numpy(), want_picks)
    if shared:
        np.testing.assert_array_equal(rt[N * Cpad: N * Cpad + T], np.arange(T))
        assert np.all(rt[N * Cpad + T: rows] == -1)


SMALL = [
    # C = ceil(capacity_factor * T / N) tokens per expert
    Workload("ec_bf16_multi_mtile", T=1000, d_model=256, d_ff=512, n_experts=8, top_k=2,
             act=ACT_GELU_ERF, dtype=DT_BF16, capacity_factor=2.0, expert_choice=True,
             seed=61),
    Workload("ec_bf16_shared_relu", T=1000, d_model=128, d_ff=256, n_experts=16, top_k=1,
             act=ACT_RELU, dtype=DT_BF16, capacity_factor=1.0, d_ff_shared=256,
             expert_choice=True, seed=62),
    Workload("ec_f32", T=300, d_model=128, d_ff=256, n_experts=4, top_k=1,
             act=ACT_GELU_ERF, dtype=DT_F32, capacity_factor=1.5, expert_choice=True,
             seed=63),
    # N % 64 == 0: the scores come from the tensor-core router GEMM
    Workload("ec_bf16_tc_router", T=700, d_model=128, d_ff=128, n_experts=64, top_k=1,
             act=ACT_GELU_ERF, dtype=DT_BF16, capacity_factor=4.0, expert_choice=True,
             seed=64),
    # every expert takes every token (capacity <= 0)
    Workload("ec_bf16_all_tokens", T=200, d_model=64, d_ff=128, n_experts=4, top_k=1,
             act=ACT_RELU, dtype=DT_BF16, capacity_factor=0.0, expert_choice=True, seed=65),
    # C >= 256: CTA-pair tiles; few experts
    Workload("ec_bf16_pair", T=1200, d_model=128, d_ff=256, n_experts=2, top_k=1,
             act=ACT_GELU_ERF, dtype=DT_BF16, capacity_factor=0.6, d_ff_shared=256,
             expert_choice=True, seed=66),
    # C < 24: decode tiles (weights as the 128-row operand)
    Workload("ec_bf16_decode", T=40, d_model=256, d_ff=384, n_experts=8, top_k=1,
             act=ACT_GELU_ERF, dtype=DT_BF16, capacity_factor=2.0, expert_choice=True,
             seed=67),
    Workload("ec_bf16_single_expert", T=150, d_model=64, d_ff=128, n_experts=1, top_k=1,
             act=ACT_RELU, dtype=DT_BF16, capacity_factor=0.5, expert_choice=True, seed=68),
]


@pytest.mark.parametrize("wl", SMALL, ids=[w.name for w in SMALL])
def test_small_layers_full_parity(wl):
    t, layer, out = run_ec(wl)
    C = B.ec_tokens_per_expert(layer.cfg)
    assert C == O.expert_choice_tokens(wl.T, wl.capacity)
    report, ref = check_ec_layer(wl, layer.cfg, t, out)
    print("parity", wl.name, report, "unpicked", ref.unpicked)
    # perfect balance by construction
    assert ref.token_picks.sum() == wl.n_experts * C


def test_all_tokens_equals_topk_with_k_equal_N():
    """C = T: each expert takes every token, so the layer is top-k routing with
    k = N (renormalised gates over all N are p) -- both GPU paths agree."""
    wl = Workload("ec_eq", T=256, d_model=128, d_ff=128, n_experts=4, top_k=4,
                  act=ACT_GELU_ERF, dtype=DT_F32, capacity_factor=0.0, expert_choice=True,
                  seed=69)
    t, layer, out = run_ec(wl)
    assert int(out.unpicked.cpu().item()) == 0
    assert torch.all(out.token_picks == 4)
    tk = B.MoeLayer(wl, t)
    out_k = tk.forward(t["x"], with_logits=True)
    torch.cuda.synchronize()
    check_layer(wl, tk.cfg, t, out_k)
    yk, ye = out_k.y.double(), out.y.double()
    assert float((yk - ye).norm() / yk.norm()) < 1e-5


def test_edge_tokens_0_and_1():
    wl = Workload("ec_edge", T=1, d_model=64, d_ff=64, n_experts=4, top_k=1, dtype=DT_BF16,
                  capacity_factor=3.0, expert_choice=True, seed=70)
    t, layer, out = run_ec(wl)
    assert B.ec_tokens_per_expert(layer.cfg) == 1
    check_ec_layer(wl, layer.cfg, t, out)
    assert int(out.token_picks.cpu().item()) == 4
    t0, layer0, out0 = run_ec(wl, T=0)
    assert B.ec_tokens_per_expert(layer0.cfg) == 0
    assert B.ec_forward_launch_count(layer0.cfg) == 2
    assert out0.unpicked.cpu().item() == 0
    assert out0.balance.cpu().item() == 0.0


def test_profiled_matches_forward_and_is_deterministic():
    wl = Workload("ec_prof", T=900, d_model=128, d_ff=256, n_experts=8, top_k=1,
                  act=ACT_GELU_ERF, dtype=DT_BF16, capacity_factor=1.5, d_ff_shared=256,
                  expert_choice=True, seed=71)
    t, layer, out = run_ec(wl)
    events = [torch.cuda.Event(enable_timing=True) for _ in range(7)]
    for ev in events:                   # torch creates the CUDA event on first record
        ev.record()
    out2 = B.alloc_ec_outputs(layer.cfg, "cuda", with_logits=True)
    B.ec_forward_profiled(layer.cfg, t["x"], layer.weights, out2, layer.workspace, events)
    out3 = layer.forward(t["x"], with_logits=True)
    torch.cuda.synchronize()
    for name in ("y", "ec_token", "ec_gate", "token_picks", "unpicked", "mean_prob", "balance",
                 "logits"):
        assert torch.equal(getattr(out, name), getattr(out2, name)), name
        assert torch.equal(getattr(out, name), getattr(out3, name)), name
    times = [events[i].elapsed_time(events[i + 1]) for i in range(6)]
    assert all(v > 0 for v in times)
    # fused router, selection, row copy, two grouped Linears, combine, statistics
    assert B.ec_forward_launch_count(layer.cfg) == 7


def tile_tokens(sel, T, seed):
    """One picked token at a random row of every 128-row m-tile of every
    expert's group (the GPU's selection; check_ec_layer checks it against the
    oracle's), plus the first and last token."""
    rng = np.random.default_rng(seed)
    toks = {0, T - 1}
    for s_ in sel:
        for s0 in range(0, len(s_), 128):
            toks.add(int(s_[int(rng.integers(s0, min(len(s_), s0 + 128)))]))
    return np.array(sorted(toks), dtype=np.int64)


def test_workload_c3_mixtral_prefill_ec_every_tile():
    wl = WORKLOADS["c3_mixtral_prefill_ec"]
    t, layer, out = run_ec(wl)
    assert B.ec_tokens_per_expert(layer.cfg) == 1024
    sel = out.ec_token.cpu().numpy().reshape(wl.n_experts, 1024)
    report, ref = check_ec_layer(wl, layer.cfg, t, out, tokens=tile_tokens(sel, wl.T, 6))
    print("parity", wl.name, report, "unpicked", ref.unpicked)


def test_workload_c4_deepseek_v3_ec_every_tile():
    wl = WORKLOADS["c4_deepseek_v3_ec"]
    t, layer, out = run_ec(wl)
    assert B.ec_tokens_per_expert(layer.cfg) == 128
    sel = out.ec_token.cpu().numpy().reshape(wl.n_experts, 128)
    report, ref = check_ec_layer(wl, layer.cfg, t, out, tokens=tile_tokens(sel, wl.T, 7))
    print("parity", wl.name, report, "unpicked", ref.unpicked)
    del t, layer, out
    torch.cuda.empty_cache()
