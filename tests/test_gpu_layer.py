"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Small shapes run in full and span several tiles with ragged tails.  The
layer workloads run at their full sizes with every token routed and grouped;
the output rows are compared on all tokens (the page-1, PR1 and Switch
layers), and on the two largest layers (Mixtral- and DeepSeek-V3-sized) the
grouped hidden rows and expert outputs are compared at rows that visit every
128-row m-tile of every expert group (first, last and one random live row per
tile) and every row of the shared group, with the layer output on a sample of
tokens that visits every m-tile."""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_mixture_experts_68_b300 import binding as B
from sparse_mixture_experts_68_b300 import synth
from sparse_mixture_experts_68_b300.workloads import (ACT_GELU_ERF, ACT_RELU, DT_BF16, DT_F32,
                                                      WORKLOADS, Workload)

from parity import (check_grouped_rows, check_grouping, check_layer, host_tensors, oracle_layer,
                    tile_cover)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    B.lib()
    yield
    torch.cuda.synchronize()
    assert B.get_device_status() == B.MOE_OK


def run_layer(wl, T=None, capacity=None, with_logits=True, seed=None):
    t = synth.make_layer(wl if T is None else wl.with_tokens(T), device="cuda", seed=seed)
    layer = B.MoeLayer(wl, t, T=T, capacity=capacity)
    out = layer.forward(t["x"], with_logits=with_logits)
    torch.cuda.synchronize()
    return t, layer, out


SMALL = [
    # name, T, d, f, N, k, act, dtype, cap, shared
    Workload("bf16_multi_mtile", T=1000, d_model=256, d_ff=512, n_experts=4, top_k=2,
             act=ACT_GELU_ERF, dtype=DT_BF16, seed=11),
    Workload("bf16_relu_cap_bn64", T=333, d_model=128, d_ff=192, n_experts=8, top_k=1,
             act=ACT_RELU, dtype=DT_BF16, capacity_factor=0.7, seed=12),
    Workload("bf16_shared_k4", T=200, d_model=64, d_ff=128, n_experts=16, top_k=4,
             act=ACT_GELU_ERF, dtype=DT_BF16, d_ff_shared=128, seed=13),
    Workload("bf16_bn128_N3", T=257, d_model=192, d_ff=384, n_experts=3, top_k=3,
             act=ACT_GELU_ERF, dtype=DT_BF16, seed=14),
    Workload("bf16_single_expert", T=130, d_model=64, d_ff=256, n_experts=1, top_k=1,
             act=ACT_RELU, dtype=DT_BF16, seed=15),
    Workload("bf16_many_experts", T=300, d_model=128, d_ff=128, n_experts=300, top_k=6,
             act=ACT_GELU_ERF, dtype=DT_BF16, d_ff_shared=128, seed=16),
    Workload("f32_small", T=190, d_model=72, d_ff=136, n_experts=5, top_k=2,
             act=ACT_GELU_ERF, dtype=DT_F32, seed=17),
    Workload("f32_cap_shared", T=150, d_model=64, d_ff=96, n_experts=6, top_k=2,
             act=ACT_RELU, dtype=DT_F32, capacity_factor=1.0, d_ff_shared=96, seed=18),
    Workload("bf16_noreorm", T=400, d_model=128, d_ff=256, n_experts=8, top_k=2,
             act=ACT_GELU_ERF, dtype=DT_BF16, renormalize=0, seed=19),
    # router paths: tensor-core scores (N % 64 == 0, ragged T), fused kernel
    # with two experts per lane (32 < N <= 64), CUDA-core GEMM (large fp32 W_g)
    Workload("bf16_tc_router", T=333, d_model=128, d_ff=128, n_experts=128, top_k=3,
             act=ACT_GELU_ERF, dtype=DT_BF16, seed=20),
    # 64 experts in bf16: the router GEMM with the softmax, top-k and gates in
    # its epilogue (ragged last 128-row tile; raw gates; k = 8 with capacity
    # drops and a shared expert)
    Workload("bf16_router64_k4_raw", T=333, d_model=128, d_ff=128, n_experts=64, top_k=4,
             act=ACT_GELU_ERF, dtype=DT_BF16, renormalize=0, seed=44),
    Workload("bf16_router64_k8_cap_shared", T=700, d_model=256, d_ff=128, n_experts=64,
             top_k=8, act=ACT_RELU, dtype=DT_BF16, capacity_factor=6.0, d_ff_shared=128,
             seed=45),
    Workload("f32_fused_router_npl2", T=97, d_model=96, d_ff=64, n_experts=48, top_k=5,
             act=ACT_RELU, dtype=DT_F32, seed=22),
    Workload("f32_simt_router", T=70, d_model=1024, d_ff=64, n_experts=64, top_k=2,
             act=ACT_GELU_ERF, dtype=DT_F32, seed=23),
    # groups of >= 256 rows and K >= 2048: the CTA-pair 256 x 256 tiles for both
    # Linears, with a shared expert and ragged groups
    Workload("bf16_pair_shared", T=700, d_model=2048, d_ff=2048, n_experts=2, top_k=2,
             act=ACT_GELU_ERF, dtype=DT_BF16, d_ff_shared=2048, seed=27),
    # few tokens per expert: weights as the MMA's 128-row operand (decode)
    Workload("bf16_decode_nb16", T=9, d_model=256, d_ff=384, n_experts=8, top_k=2,
             act=ACT_RELU, dtype=DT_BF16, seed=28),
    Workload("bf16_decode_nb32_cap", T=60, d_model=128, d_ff=256, n_experts=12, top_k=3,
             act=ACT_GELU_ERF, dtype=DT_BF16, capacity_factor=1.5, seed=29),
    # capacity-capped groups: skewed routing leaves some experts empty and
    # fills others to the cap; a capacity of 240 with two slots per token
    Workload("bf16_cap_zipf", T=1000, d_model=256, d_ff=512, n_experts=16, top_k=1,
             act=ACT_RELU, dtype=DT_BF16, capacity_factor=1.4, zipf_router_bias=True,
             seed=38),
    Workload("bf16_cap240_k2", T=1200, d_model=384, d_ff=256, n_experts=12, top_k=2,
             act=ACT_GELU_ERF, dtype=DT_BF16, capacity_factor=2.4, seed=39),
    # a few tokens: router, sort and statistics in the two front-end kernels
    # (a ragged last slice of d; 64 experts x 32 tokens with capacity drops;
    # 40 experts with a shared expert and raw gates)
    Workload("f32_front_ragged_d", T=5, d_model=72, d_ff=64, n_experts=6, top_k=3,
             act=ACT_GELU_ERF, dtype=DT_F32, seed=41),
    Workload("bf16_front_n64_k8_cap", T=32, d_model=256, d_ff=256, n_experts=64, top_k=8,
             act=ACT_RELU, dtype=DT_BF16, capacity_factor=4.0, seed=42),
    Workload("bf16_front_n40_shared_raw", T=20, d_model=128, d_ff=128, n_experts=40,
             top_k=2, act=ACT_GELU_ERF, dtype=DT_BF16, d_ff_shared=128, renormalize=0,
             seed=43),
    # more than 32 slots per token: gates written in blocks of 32 lanes
    Workload("f32_k40_fused", T=50, d_model=64, d_ff=64, n_experts=64, top_k=40,
             act=ACT_RELU, dtype=DT_F32, seed=25),
    Workload("bf16_k33_tc_router", T=70, d_model=64, d_ff=64, n_experts=128, top_k=33,
             act=ACT_GELU_ERF, dtype=DT_BF16, seed=26),
    # 2048..16384 assignments: the two-launch sort (three blocks of 1024
    # assignments, the last one ragged) with 300 experts, capacity drops and a
    # shared expert; the statistics from the scatter launch's extra block
    Workload("bf16_mid_sort_n300_cap_shared", T=333, d_model=128, d_ff=128, n_experts=300,
             top_k=8, act=ACT_RELU, dtype=DT_BF16, capacity_factor=6.0, d_ff_shared=128,
             seed=48),
    # the two-launch sort at its limits: 64 blocks of 1024 assignments; 384
    # experts (the tensor-core router scores) with capacity drops
    Workload("bf16_mid_sort_64_blocks", T=32768, d_model=64, d_ff=64, n_experts=8, top_k=2,
             act=ACT_RELU, dtype=DT_BF16, seed=49),
    Workload("bf16_mid_sort_n384_cap", T=2048, d_model=64, d_ff=64, n_experts=384, top_k=8,
             act=ACT_GELU_ERF, dtype=DT_BF16, capacity_factor=1.5, seed=50),
    # exactly 2048 assignments, one expert, half of them past the capacity
    Workload("bf16_mid_sort_one_expert_cap", T=2048, d_model=64, d_ff=128, n_experts=1,
             top_k=1, act=ACT_RELU, dtype=DT_BF16, capacity_factor=0.5, seed=51),
    # T*k too large for the one-block counting sort: histogram/scan/rank blocks
    Workload("bf16_multiblock_permute", T=40000, d_model=64, d_ff=64, n_experts=12,
             top_k=3, act=ACT_RELU, dtype=DT_BF16, capacity_factor=1.05, seed=24),
    # 256-wide tiles in both Linears: with a shared expert and GELU; with ReLU,
    # capacity drops and ragged groups
    Workload("bf16_bn256_shared", T=1000, d_model=256, d_ff=512, n_experts=8, top_k=2,
             act=ACT_GELU_ERF, dtype=DT_BF16, d_ff_shared=512, seed=25),
    Workload("bf16_bn256_relu_cap", T=777, d_model=512, d_ff=256, n_experts=6, top_k=2,
             act=ACT_RELU, dtype=DT_BF16, capacity_factor=2.0, seed=26),
    # the same layer with a capacity of 117 (half the assignments dropped)
    Workload("bf16_cap117_relu", T=777, d_model=512, d_ff=256, n_experts=6, top_k=2,
             act=ACT_RELU, dtype=DT_BF16, capacity_factor=0.9, seed=26),
    # fp32 CUDA-core GEMMs on each tile size: the first Linear (d_ff = 1024 columns
    # over ~4500 grouped rows) on 128 x 64 tiles, the second on 64 x 64
    Workload("f32_tile128x64", T=2000, d_model=64, d_ff=1024, n_experts=4, top_k=2,
             act=ACT_GELU_ERF, dtype=DT_F32, seed=27),
]


@pytest.mark.parametrize("wl", SMALL, ids=[w.name for w in SMALL])
def test_small_layers_full_parity(wl):
    t, layer, out = run_layer(wl)
    report, ref = check_layer(wl, layer.cfg, t, out)
    assert report["max_row_rel_l2"] <= (1e-4 if wl.dtype == DT_F32 else 2e-2)


def run_staged(cfg, t, dev="cuda"):
    """The layer's steps called one by one through the ABI: router + top-k,
    permute, grouped FFN (hidden rows H and expert outputs Yp kept), combine,
    statistics.  Returns every buffer."""
    T, k, N = cfg.T, cfg.top_k, cfg.n_experts
    rows = B.rows_max(cfg)
    dt = torch.float32 if cfg.dtype == B.MOE_F32 else torch.bfloat16
    f32, i32 = torch.float32, torch.int32
    b = dict(logits=torch.empty((T, N), dtype=f32, device=dev),
             idx=torch.empty((T, k), dtype=i32, device=dev),
             w=torch.empty((T, k), dtype=f32, device=dev),
             pp=torch.empty((B.router_blocks(cfg), N), dtype=f32, device=dev),
             counts=torch.empty(N, dtype=i32, device=dev),
             kept=torch.empty(N, dtype=i32, device=dev),
             offsets=torch.empty(N + 2, dtype=i32, device=dev),
             row_token=torch.empty(rows, dtype=i32, device=dev),
             token_row=torch.empty((T, k), dtype=i32, device=dev),
             Xp=torch.empty((rows, cfg.d_model), dtype=dt, device=dev),
             scratch=torch.empty(B.permute_scratch_size(cfg), dtype=torch.uint8, device=dev),
             H=torch.empty((rows, cfg.d_ff), dtype=dt, device=dev),
             Yp=torch.empty((rows, cfg.d_model), dtype=dt, device=dev),
             y=torch.empty((T, cfg.d_model), dtype=dt, device=dev),
             mean_prob=torch.empty(N, dtype=f32, device=dev),
             balance=torch.empty(1, dtype=f32, device=dev),
             dropped=torch.empty(1, dtype=i32, device=dev),
             cv2=torch.empty(1, dtype=f32, device=dev))
    B.router_topk(cfg, t["x"], t["W_g"], t["b_g"], b["logits"], b["idx"], b["w"], b["pp"])
    B.permute(cfg, t["x"], b["idx"], b["counts"], b["kept"], b["offsets"], b["row_token"],
              b["token_row"], b["Xp"], b["scratch"])
    B.grouped_ffn(cfg, b["Xp"], b["offsets"], b["kept"], B.make_weights(t), b["H"], b["Yp"])
    B.combine(cfg, b["Yp"], b["token_row"], b["w"], b["offsets"], b["y"])
    B.load_stats(cfg, b["pp"], b["counts"], b["kept"], b["mean_prob"], b["balance"],
                 b["dropped"], b["cv2"])
    torch.cuda.synchronize()
    b["out"] = B.Outputs(b["y"], b["idx"], b["w"], b["counts"], b["kept"], b["dropped"],
                         b["mean_prob"], b["balance"], b["logits"], b["cv2"])
    return b


def test_stages_through_the_abi():
    """Each step called on its own: router, permute (layout checked), grouped
    FFN (hidden rows and expert outputs of every group checked), combine, stats."""
    wl = Workload("stages", T=700, d_model=128, d_ff=256, n_experts=6, top_k=2,
                  act=ACT_GELU_ERF, dtype=DT_BF16, capacity_factor=1.1, d_ff_shared=256,
                  seed=21)
    t = synth.make_layer(wl, device="cuda")
    cfg = B.make_config(wl)
    st = run_staged(cfg, t)
    th = host_tensors(t)
    L = oracle_layer(cfg, th)
    report, ref = check_layer(wl, cfg, t, st["out"], th=th, L=L)
    assert ref.grouping.dropped > 0                   # the capacity bites
    check_grouping(cfg, t["x"], st["offsets"], st["row_token"], st["token_row"], st["Xp"],
                   ref.grouping, wl.T)
    rep = check_grouped_rows(cfg, L, ref.grouping, st["offsets"], st["H"], st["Yp"], seed=21,
                             all_shared=True)
    assert rep["grouped_rows_compared"] >= wl.T


def test_edge_cases_tokens_0_and_1():
    wl = Workload("edge", T=1, d_model=64, d_ff=64, n_experts=4, top_k=2, dtype=DT_BF16,
                  seed=31)
    t, layer, out = run_layer(wl)
    check_layer(wl, layer.cfg, t, out)
    t0, layer0, out0 = run_layer(wl, T=0)
    assert out0.counts.cpu().sum().item() == 0
    assert out0.dropped.cpu().item() == 0
    assert out0.balance.cpu().item() == 0.0
    assert out0.cv_squared.cpu().item() == 0.0


def test_capacity_one_and_all_tokens_to_one_expert():
    wl = Workload("collapse", T=260, d_model=64, d_ff=128, n_experts=4, top_k=1,
                  dtype=DT_BF16, seed=32)
    t = synth.make_layer(wl, device="cuda")
    t["W_g"].zero_()
    t["b_g"].copy_(torch.tensor([3.0, 0.0, -1.0, -2.0], device="cuda").to(torch.bfloat16))
    for cap in (1, 3, 0):
        layer = B.MoeLayer(wl, t, capacity=cap)
        out = layer.forward(t["x"], with_logits=True)
        torch.cuda.synchronize()
        report, ref = check_layer(wl, layer.cfg, t, out, capacity=cap)
        kept0 = ref.grouping.kept[0]
        assert kept0 == (cap if cap > 0 else 260)
        # balance of a collapsed router: every token puts the same p on expert 0
        assert ref.grouping.counts.tolist() == [260, 0, 0, 0]
        # all assignments on one of N experts: cv^2 = N exactly
        assert out.cv_squared.cpu().item() == 4.0


def test_deterministic_bitwise():
    wl = Workload("det", T=513, d_model=256, d_ff=512, n_experts=8, top_k=2,
                  dtype=DT_BF16, capacity_factor=1.2, seed=33)
    t, layer, out1 = run_layer(wl)
    out2 = layer.forward(t["x"], with_logits=True)
    torch.cuda.synchronize()
    for a, b in [(out1.y, out2.y), (out1.topk_idx, out2.topk_idx), (out1.topk_w, out2.topk_w),
                 (out1.mean_prob, out2.mean_prob), (out1.balance, out2.balance),
                 (out1.cv_squared, out2.cv_squared)]:
        assert torch.equal(a, b)


def test_forward_host_matches_device_path():
    wl = Workload("host", T=300, d_model=128, d_ff=256, n_experts=8, top_k=2,
                  dtype=DT_BF16, seed=34)
    t, layer, out = run_layer(wl)
    cfg = layer.cfg
    ws = torch.empty(B.host_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    xh = t["x"].cpu().pin_memory()
    oh = B.alloc_outputs(cfg, "cpu", with_logits=True, pin_memory=True)
    B.forward_host(cfg, xh, layer.weights, oh, ws)
    assert torch.equal(oh.y, out.y.cpu())
    assert torch.equal(oh.topk_idx, out.topk_idx.cpu())
    assert torch.equal(oh.counts, out.counts.cpu())
    assert torch.equal(oh.logits, out.logits.cpu())


@pytest.mark.parametrize("wl", [
    Workload("host_chunks", T=2048, d_model=256, d_ff=512, n_experts=8, top_k=2,
             dtype=DT_BF16, seed=46),
    # an odd token count (halves of 1024 and 1027 tokens) with a shared expert
    Workload("host_chunks_shared", T=2051, d_model=128, d_ff=256, n_experts=4, top_k=2,
             act=ACT_RELU, dtype=DT_BF16, d_ff_shared=256, seed=47),
], ids=lambda w: w.name)
def test_forward_host_in_two_chunks_matches_device_path(wl):
    """moe_forward_host runs these layers as two token chunks, the copies
    overlapping the layer on a second stream: per-token results and the counts
    are those of moe_forward bit for bit, the statistics (summed over both
    chunks' partial sums) equal up to fp32 rounding; two calls agree."""
    t, layer, out = run_layer(wl)
    cfg = layer.cfg
    assert B.forward_host_chunks(cfg) == 2
    ws = torch.empty(B.host_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    xh = t["x"].cpu().pin_memory()
    for _ in range(2):
        oh = B.alloc_outputs(cfg, "cpu", with_logits=True, pin_memory=True)
        B.forward_host(cfg, xh, layer.weights, oh, ws)
        for name in ("y", "topk_idx", "topk_w", "counts", "kept", "dropped", "logits"):
            assert torch.equal(getattr(oh, name), getattr(out, name).cpu()), name
        for name in ("mean_prob", "balance", "cv_squared"):
            np.testing.assert_allclose(getattr(oh, name).numpy(),
                                       getattr(out, name).cpu().numpy(), rtol=1e-5, atol=1e-7,
                                       err_msg=name)
    assert B.get_device_status() == B.MOE_OK


def test_bounded_wait_reports_timeout_and_context_survives():
    B.selftest_bounded_wait(2_000_000)            # 2 ms; nothing ever arrives
    assert B.get_device_status() == B.MOE_ERR_TIMEOUT
    assert B.get_device_status() == B.MOE_OK      # read clears it
    wl = Workload("after", T=64, d_model=64, d_ff=64, n_experts=4, top_k=2, seed=35)
    t, layer, out = run_layer(wl)
    check_layer(wl, layer.cfg, t, out)


# ---- the five layer workloads at full size ----------------------------------------

def sample_tokens(T, n, seed, must=()):
    rng = np.random.default_rng(seed)
    pick = set(must) | {0, T - 1}
    pick |= set(rng.choice(T, size=min(n, T), replace=False).tolist())
    return np.array(sorted(pick))


def test_workload_c0_pr1_fp32_full():
    wl = WORKLOADS["c0_pr1_fp32"]
    t, layer, out = run_layer(wl)
    report, _ = check_layer(wl, layer.cfg, t, out)
    print("parity", wl.name, report)
    assert report["max_row_rel_l2"] <= 1e-4


def test_workload_c1_page1_bf16_full():
    wl = WORKLOADS["c1_page1_bf16"]
    t, layer, out = run_layer(wl)
    report, _ = check_layer(wl, layer.cfg, t, out)
    print("parity", wl.name, report)


def test_workload_c2_switch_top1_capacity():
    wl = WORKLOADS["c2_switch_top1"]
    assert O.expert_capacity(wl.capacity_factor, wl.T, wl.n_experts) == wl.capacity == 160
    t, layer, out = run_layer(wl)
    kept = out.kept.cpu().numpy()
    grp = O.group_by_expert(out.topk_idx.cpu().numpy(), wl.n_experts, 160)
    assert (~grp.keep[:, 0]).sum() > 0
    report, ref = check_layer(wl, layer.cfg, t, out)
    print("parity", wl.name, report, "dropped", ref.grouping.dropped)
    assert ref.grouping.dropped > 0 and kept.max() == 160
    assert report["fully_dropped_checked"] > 0


def test_workload_c2_raw_gates_variant():
    wl = WORKLOADS["c2_switch_top1"]
    from dataclasses import replace
    wl = replace(wl, renormalize=0)
    t, layer, out = run_layer(wl, T=2048)
    check_layer(wl, layer.cfg, t, out, tokens=sample_tokens(2048, 128, 3))


def test_workload_c3_mixtral_decode_full():
    wl = WORKLOADS["c3_mixtral_decode"]
    t, layer, out = run_layer(wl)
    report, _ = check_layer(wl, layer.cfg, t, out)
    print("parity", wl.name, report)


def tile_tokens(grouping, T, seed, shared=False, extra=0):
    """One token at a random live row of every 128-row m-tile of every group
    (and of the shared group), plus `extra` seeded tokens."""
    rng = np.random.default_rng(seed)
    toks = set()
    for grp in grouping.groups:
        for s0 in range(0, len(grp), 128):
            toks.add(grp[int(rng.integers(s0, min(len(grp), s0 + 128)))][0])
    if shared:
        toks |= {int(rng.integers(s0, min(T, s0 + 128))) for s0 in range(0, T, 128)}
    if extra:
        toks |= set(rng.choice(T, size=min(extra, T), replace=False).tolist())
    return np.array(sorted(toks | {0, T - 1}), dtype=np.int64)


def check_large_layer(wl, seed, y_extra=0, y_tile_tokens=True):
    """A large layer at full size: the staged calls (keeping H and Yp) and
    moe_forward give the same results; the grouped rows are compared at every
    m-tile of every group and every shared row; y on tokens that visit every
    m-tile (plus a seeded sample)."""
    t = synth.make_layer(wl, device="cuda")
    cfg = B.make_config(wl)
    st = run_staged(cfg, t)
    layer = B.MoeLayer(wl, t)
    out = layer.forward(t["x"], with_logits=True)
    torch.cuda.synchronize()
    # the same kernels on the same inputs: the same bits
    for name in ("y", "topk_idx", "topk_w", "counts", "kept", "logits"):
        assert torch.equal(getattr(out, name), getattr(st["out"], name)), name
    th = host_tensors(t)
    L = oracle_layer(cfg, th)
    grp = O.group_by_expert(out.topk_idx.cpu().numpy(), cfg.n_experts, cfg.capacity)
    if y_tile_tokens:
        toks = tile_tokens(grp, wl.T, seed, shared=bool(cfg.d_ff_shared), extra=y_extra)
    else:
        toks = sample_tokens(wl.T, y_extra, seed)
    report, ref = check_layer(wl, cfg, t, out, tokens=toks, th=th, L=L)
    check_grouping(cfg, t["x"], st["offsets"], st["row_token"], st["token_row"], st["Xp"],
                   ref.grouping, wl.T)
    report.update(check_grouped_rows(cfg, L, ref.grouping, st["offsets"], st["H"], st["Yp"],
                                     seed, all_shared=True))
    print("parity", wl.name, report)
    del t, layer, out, st
    torch.cuda.empty_cache()
    return report


def test_workload_c3_mixtral_prefill_every_tile():
    report = check_large_layer(WORKLOADS["c3_mixtral_prefill"], 4)
    # 8 groups of ~1024 rows: ~8 m-tiles each, three rows per tile
    assert report["grouped_rows_compared"] >= 8 * 8 * 2


def test_workload_c4_deepseek_v3_every_tile():
    wl = WORKLOADS["c4_deepseek_v3"]
    report = check_large_layer(wl, 5, y_extra=64, y_tile_tokens=False)
    # 256 groups of ~128 rows (one or two m-tiles each) and all 4096 shared rows
    assert report["grouped_rows_compared"] >= 256 * 2 + wl.T


def test_forward_profiled_and_graph_replay_match_forward():
    """moe_forward_profiled (events at the kernel boundaries), eagerly and
    captured into a CUDA graph and replayed, gives moe_forward's results bit
    for bit, and its events time every step."""
    wl = Workload("graph", T=600, d_model=128, d_ff=256, n_experts=16, top_k=2,
                  dtype=DT_BF16, capacity_factor=1.3, d_ff_shared=256, seed=36)
    t, layer, ref = run_layer(wl)
    cfg = layer.cfg
    # fused router, one-block sort (with the statistics) + row copy, two
    # grouped Linears, combine
    assert B.forward_launch_count(cfg) == 6
    stream = torch.cuda.Stream()
    events = [torch.cuda.Event(enable_timing=True) for _ in range(7)]
    out = B.alloc_outputs(cfg, "cuda", with_logits=True)
    with torch.cuda.stream(stream):
        for ev in events:
            ev.record(stream)
        B.forward_profiled(cfg, t["x"], layer.weights, out, layer.workspace, events, stream)
    stream.synchronize()
    for name in ("y", "topk_idx", "topk_w", "counts", "kept", "mean_prob", "balance", "logits"):
        assert torch.equal(getattr(out, name), getattr(ref, name)), name
    times = [events[i].elapsed_time(events[i + 1]) for i in range(6)]
    assert all(v > 0 for v in times[:5]) and times[5] >= 0   # statistics fused into permute
    graph = torch.cuda.CUDAGraph()
    out2 = B.alloc_outputs(cfg, "cuda", with_logits=True)
    with torch.cuda.graph(graph, stream=stream):
        B.forward_profiled(cfg, t["x"], layer.weights, out2, layer.workspace, events, stream)
    for _ in range(2):
        out2.y.zero_()
        with torch.cuda.stream(stream):
            graph.replay()
        stream.synchronize()
        assert torch.equal(out2.y, ref.y)
        assert torch.equal(out2.counts, ref.counts)
        assert events[0].elapsed_time(events[6]) > 0


def test_activation_matches_cuda_erf_gelu_and_relu():
    """The kernels' GELU (erf by Abramowitz & Stegun 7.1.26) against torch's
    exact GELU on the GPU (CUDA's erff) and the float64 definition."""
    x = torch.linspace(-12, 12, 200001, device="cuda", dtype=torch.float32)
    y = torch.empty_like(x)
    B.activation(B.MOE_ACT_GELU_ERF, x, y)
    ref = torch.nn.functional.gelu(x)                     # CUDA erff
    ref64 = O.activation(x.double().cpu().numpy(), O.ACT_GELU_ERF)
    torch.cuda.synchronize()
    err_cuda = (y - ref).abs().max().item()
    err_def = float(np.max(np.abs(y.double().cpu().numpy() - ref64)))
    # |GELU error| <= 0.5 |x| 1.5e-7 (formula bound) + fp32 rounding of the result
    assert err_def <= 0.5 * 12 * 1.5e-7 + 12 * 2.0 ** -23, err_def
    assert err_cuda <= 2e-6, err_cuda
    B.activation(B.MOE_ACT_RELU, x, y)
    torch.cuda.synchronize()
    assert torch.equal(y, torch.relu(x))


SK_LAYERS = [
    (Workload("decode_sk", T=24, d_model=512, d_ff=1024, n_experts=8, top_k=2,
              act=ACT_GELU_ERF, dtype=DT_BF16, seed=37), "x 16 tokens"),
    (Workload("decode_sk_nb32_cap", T=40, d_model=512, d_ff=1024, n_experts=4, top_k=2,
              act=ACT_RELU, dtype=DT_BF16, capacity_factor=0.9, seed=40), "x 32 tokens"),
]


@pytest.mark.parametrize("wl,tile", SK_LAYERS, ids=[w.name for w, _ in SK_LAYERS])
def test_decode_stream_k_deterministic_and_close_to_whole_tiles(wl, tile):
    """moe_forward runs the token-column tiles stream-K: every CTA streams an
    equal share of the k-blocks, and a tile split between CTAs is summed by
    the last of them, in k order.  Three calls give the same bits; the staged
    calls (moe_grouped_ffn, whole tiles per CTA) agree within bf16 rounding;
    both match the oracle.  Cases: a decode layer (16 token columns) and one
    with 32 token columns and capacity drops."""
    t, layer, out1 = run_layer(wl)
    for linear in (1, 2):
        name = B.ffn_kernel_name(layer.cfg, linear)
        assert "stream-K" in name and tile in name, name
    again = [layer.forward(t["x"], with_logits=True) for _ in range(2)]
    torch.cuda.synchronize()
    for o in again:
        assert torch.equal(o.y, out1.y)
    st = run_staged(layer.cfg, t)
    a = st["y"].double().cpu().numpy()
    b = out1.y.double().cpu().numpy()
    rel = np.linalg.norm(a - b, axis=1) / np.maximum(np.linalg.norm(b, axis=1), 1e-6)
    assert rel.max() <= 1e-2, rel.max()
    check_layer(wl, layer.cfg, t, out1)
    check_layer(wl, layer.cfg, t, st["out"])
