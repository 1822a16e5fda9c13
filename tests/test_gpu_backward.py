"""The backward pass on the GPU (through the C ABI) against the oracle's
backward (float64 chain rule, pinned to torch autograd and finite
differences): every gradient of total = <dy, y> + aux * balance.

Bars, for bf16 layers 2e-2 (1e-4 for fp32 layers, whose CUDA-core path keeps
every intermediate in fp32: a few 1e-7 of rounding per value), applied
  * per expert: the relative L2 error of each expert's dW1[e], db1[e],
    dW2[e] and db2[e] (and the shared expert's), maximised over experts;
  * per token row: the relative L2 error of dx[t] and dz[t], maximised over
    tokens, with each row's norm floored at a thousandth of the median row
    norm for dx (a row whose every slot was dropped carries only the tiny
    balance term), and for dz against the larger of its norm and its gate
    gradients' scale ||dy[t]|| sum_j w_j ||o[t, j]|| (a difference of gate
    gradients that can cancel; see dz_row_max_rel);
  * dW_g, db_g and dw as whole tensors.
The GPU stores five bf16 intermediates on the way (dO = w dy, the recomputed
pre-activation, dA, dXp and the expert outputs behind dw), each rounded to 8
significant bits (relative 2^-9 ~ 2e-3 per element, independent across
elements), so a row's or an expert's relative L2 error is a few 1e-3; the bar
leaves a 5-10x margin.  The oracle takes the GPU's top-k choice (the forward
parity checks that choice against the oracle's own).

The two largest layers (Mixtral- and DeepSeek-V3-sized) are compared in the
training configuration the benchmark times: dx, dz and dw of sampled tokens
(several from every expert group); for every expert (and the shared one), the
rows of dW1[e] and the columns of dW2[e] of one hidden unit in every 128-unit
block (so every output tile of both weight-gradient GEMMs is visited, at a
different lane in each block), db1[e] at those units and db2[e] in full; and
the router's weight gradients through the identities dW_g = dz^T x,
db_g = sum_t dz and sum_e dz[t, e] = 0, on the GPU's own dz (itself checked
on the sampled tokens)."""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_mixture_experts_68_b300 import binding as B
from sparse_mixture_experts_68_b300 import synth
from sparse_mixture_experts_68_b300.workloads import (ACT_GELU_ERF, ACT_RELU, DT_BF16, DT_F32,
                                                      WORKLOADS, Workload)

from parity import WORKERS, check_layer, check_routing, host_tensors, oracle_layer, to64

pytestmark = pytest.mark.gpu

GRAD_TOL = {DT_BF16: 2e-2, DT_F32: 1e-4}


def gate_grad_scale(L, r, dy, tokens):
    """S_t = ||dy[t]|| sum_j w[t, j] ||o[t, j]|| over the token's kept slots,
    o[t, j] the oracle's expert output.  By Cauchy-Schwarz it bounds
    sum_j w[t, j] |dw[t, j]|, the scale of the gate gradients whose rounding
    reaches the score gradient dz[t]."""
    from concurrent.futures import ThreadPoolExecutor
    tokens = np.asarray(tokens, dtype=np.int64)
    k = r.idx.shape[1]
    slots = {}
    for i, t in enumerate(tokens):
        for j in range(k):
            if r.keep[t, j]:
                slots.setdefault(int(r.idx[t, j]), []).append((i, j))

    def one(item):
        e, lst = item
        _, _, o = L.expert_rows(e, tokens[[i for i, _ in lst]], want=("o",))
        return lst, np.linalg.norm(o, axis=1)

    S = np.zeros(len(tokens))
    with ThreadPoolExecutor(max_workers=WORKERS) as ex:
        for lst, on in ex.map(one, slots.items()):
            for (i, j), n in zip(lst, on):
                S[i] += r.w[tokens[i], j] * n
    dyn = np.linalg.norm(np.asarray(dy, dtype=np.float64)[tokens], axis=1)
    return S * dyn


def dz_row_max_rel(gz, rz, scale):
    """Max over tokens of ||dz_gpu[t] - dz_ref[t]|| / max(||dz_ref[t]||, scale[t]).
    A token's renormalised score gradient is a difference of its gate
    gradients -- for k = 2, w0 w1 (dw0 - dw1) on its two experts -- which can
    cancel to almost nothing, while the rounding it inherits from dw (inner
    products of dy with bf16 expert outputs) stays at the gate gradients'
    scale: scale = gate_grad_scale."""
    gz, rz = np.asarray(gz, np.float64), np.asarray(rz, np.float64)
    if gz.shape[0] == 0:
        return 0.0
    den = np.maximum(np.maximum(np.linalg.norm(rz, axis=1), scale), 1e-30)
    return float(np.max(np.linalg.norm(gz - rz, axis=1) / den))


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    B.lib()
    yield
    torch.cuda.synchronize()
    assert B.get_device_status() == B.MOE_OK


def make_dy(wl, seed):
    g = torch.Generator(device="cpu").manual_seed(1000 + seed)
    dt = torch.float32 if wl.dtype == DT_F32 else torch.bfloat16
    return torch.randn((wl.T, wl.d_model), generator=g).to(dt).cuda()


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def row_max_rel(a, b, floor_frac=1e-3):
    """Max over rows of ||a_r - b_r|| / max(||b_r||, floor_frac median_r ||b_r||)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.shape[0] == 0:
        return 0.0
    nb = np.linalg.norm(b, axis=1)
    floor = max(floor_frac * float(np.median(nb)), 1e-30)
    return float(np.max(np.linalg.norm(a - b, axis=1) / np.maximum(nb, floor)))


def run_backward(wl, aux):
    t = synth.make_layer(wl, device="cuda")
    layer = B.MoeLayer(wl, t)
    out = layer.forward(t["x"], with_logits=True)
    torch.cuda.synchronize()
    check_layer(wl, layer.cfg, t, out)
    dy = make_dy(wl, wl.seed)
    grads = layer.backward(t["x"], out, dy, aux_weight=aux, with_scores=True)
    torch.cuda.synchronize()
    return t, layer, out, dy, grads


def check_backward(wl, layer, t, out, dy, aux, grads):
    """Every gradient of a whole layer against the oracle's backward (from
    its pieces, on several threads)."""
    cfg = layer.cfg
    th = host_tensors(t)
    L = oracle_layer(cfg, th)
    r = L.route(cfg.capacity, bool(cfg.renormalize), out.topk_idx.cpu().numpy(),
                workers=WORKERS)
    ref = L.backward(r, dy.cpu(), aux, renormalize=bool(cfg.renormalize), workers=WORKERS)
    report = {"dx_row": row_max_rel(to64(grads.dx), ref.dx),
              "dz_row": dz_row_max_rel(to64(grads.dz), ref.dz,
                                       gate_grad_scale(L, r, to64(dy), np.arange(cfg.T))),
              "dw": rel_l2(to64(grads.dw), ref.dw),
              "dW_g": rel_l2(to64(grads.dW_g), ref.dW_g),
              "db_g": rel_l2(to64(grads.db_g), ref.db_g)}
    for name in ("dW1", "db1", "dW2", "db2"):
        gpu = to64(getattr(grads, name))
        report[name + "_expert"] = max(rel_l2(gpu[e], getattr(ref, name)[e])
                                       for e in range(cfg.n_experts))
    if cfg.d_ff_shared:
        for name, rr in zip(("dW1s", "db1s", "dW2s", "db2s"), ref.shared):
            report[name] = rel_l2(to64(getattr(grads, name)), rr)
    bad = {n: v for n, v in report.items() if not v <= GRAD_TOL[wl.dtype]}
    assert not bad, f"gradients off: {bad} (all: {report})"
    # dropped slots pass no gradient to their gate; an expert with no rows
    # gets exact zeros
    dw = grads.dw.cpu().numpy()
    keep = r.keep.astype(bool)
    assert np.all(dw[~keep] == 0.0)
    for e in np.nonzero(r.kept == 0)[0]:
        assert torch.all(grads.dW1[int(e)] == 0) and torch.all(grads.dW2[int(e)] == 0)
    return report


SMALL = [
    Workload("bwd_gelu", T=300, d_model=128, d_ff=256, n_experts=4, top_k=2,
             act=ACT_GELU_ERF, dtype=DT_BF16, seed=81),
    # d = 192: dW2's rows (d) end inside a 128-row tile; d_ff = 320: 64-wide tiles;
    # capacity drops; shared expert; ReLU
    Workload("bwd_relu_cap_shared", T=500, d_model=192, d_ff=320, n_experts=8, top_k=2,
             act=ACT_RELU, dtype=DT_BF16, capacity_factor=0.8, d_ff_shared=320, seed=82),
    Workload("bwd_raw_gates", T=700, d_model=256, d_ff=256, n_experts=16, top_k=3,
             act=ACT_GELU_ERF, dtype=DT_BF16, renormalize=0, seed=83),
    # N % 64 == 0 (tensor-core router), shared expert
    Workload("bwd_many_experts", T=400, d_model=128, d_ff=128, n_experts=64, top_k=6,
             act=ACT_GELU_ERF, dtype=DT_BF16, d_ff_shared=128, seed=84),
    # groups of >= 256 rows and K = d = 2048: the dgrad dA = (dO W2) GELU'(A1) on
    # CTA-pair tiles (MN-major weights), with a shared expert and ragged groups
    Workload("bwd_pair_dgrad", T=600, d_model=2048, d_ff=512, n_experts=2, top_k=1,
             act=ACT_GELU_ERF, dtype=DT_BF16, d_ff_shared=512, seed=86),
    # fp32 layers: the GEMMs on CUDA cores; capacity, shared expert, raw gates
    Workload("bwd_f32", T=300, d_model=96, d_ff=160, n_experts=6, top_k=2,
             act=ACT_GELU_ERF, dtype=DT_F32, capacity_factor=0.9, d_ff_shared=160, seed=87),
    Workload("bwd_f32_relu_raw", T=257, d_model=64, d_ff=128, n_experts=4, top_k=3,
             act=ACT_RELU, dtype=DT_F32, renormalize=0, seed=88),
    # ~1000-row groups: several m-tiles per group in the dgrads, many K blocks in the wgrads
    Workload("bwd_big_groups", T=2000, d_model=256, d_ff=512, n_experts=2, top_k=1,
             act=ACT_GELU_ERF, dtype=DT_BF16, seed=85),
    # 32 < N, N % 64 != 0: router gradients by the split-K CUDA-core GEMMs
    Workload("bwd_router_splitk", T=700, d_model=128, d_ff=128, n_experts=40, top_k=4,
             act=ACT_GELU_ERF, dtype=DT_BF16, seed=89),
    # N = 32 (the widest few-expert router kernel), fp32, d = 2056 spans two column blocks
    Workload("bwd_f32_router32", T=150, d_model=2056, d_ff=64, n_experts=32, top_k=2,
             act=ACT_RELU, dtype=DT_F32, seed=90),
    # N = 1 and N = 12: the narrowest and a non-power-of-two few-expert router
    Workload("bwd_single_expert", T=100, d_model=64, d_ff=64, n_experts=1, top_k=1,
             act=ACT_GELU_ERF, dtype=DT_BF16, seed=91),
    Workload("bwd_twelve_experts", T=333, d_model=1088, d_ff=128, n_experts=12, top_k=3,
             act=ACT_GELU_ERF, dtype=DT_BF16, seed=92),
    # a few tokens: the forward routes with the small-batch front end and runs
    # the token-column tiles; bf16, and fp32 with capacity drops and a shared expert
    Workload("bwd_front_decode", T=24, d_model=256, d_ff=384, n_experts=8, top_k=2,
             act=ACT_GELU_ERF, dtype=DT_BF16, seed=94),
    Workload("bwd_front_f32_cap_shared", T=9, d_model=72, d_ff=64, n_experts=6, top_k=3,
             act=ACT_RELU, dtype=DT_F32, capacity_factor=1.5, d_ff_shared=64, seed=95),
]


@pytest.mark.parametrize("wl", SMALL, ids=[w.name for w in SMALL])
@pytest.mark.parametrize("aux", [0.01, 0.5])
def test_small_layers_backward(wl, aux):
    t, layer, out, dy, grads = run_backward(wl, aux)
    report = check_backward(wl, layer, t, out, dy, aux, grads)
    print("grad parity", wl.name, aux, report)


def test_workload_c0_pr1_fp32_backward():
    wl = WORKLOADS["c0_pr1_fp32"]
    t, layer, out, dy, grads = run_backward(wl, 0.01)
    report = check_backward(wl, layer, t, out, dy, 0.01, grads)
    print("grad parity", wl.name, report)


def test_workload_c1_page1_bf16_backward():
    wl = WORKLOADS["c1_page1_bf16"]
    t, layer, out, dy, grads = run_backward(wl, 0.01)
    report = check_backward(wl, layer, t, out, dy, 0.01, grads)
    print("grad parity", wl.name, report)


def test_backward_deterministic_and_launch_count():
    wl = SMALL[1]
    t, layer, out, dy, g1 = run_backward(wl, 0.01)
    g2 = layer.backward(t["x"], out, dy, aux_weight=0.01, with_scores=True)
    torch.cuda.synchronize()
    for n in ("dx", "dW_g", "db_g", "dW1", "db1", "dW2", "db2", "dW1s", "db1s", "dW2s", "db2s",
              "dz", "dw"):
        assert torch.equal(getattr(g1, n), getattr(g2, n)), n
    # N = 8: few-expert router gradients (dW_g with db_g, their reduction; the
    # router's part of dx inside the dx kernel)
    assert B.backward_launch_count(layer.cfg) == 11


def test_backward_no_tokens():
    wl = SMALL[0]
    t = synth.make_layer(wl.with_tokens(0), device="cuda")
    layer = B.MoeLayer(wl, t, T=0)
    out = layer.forward(t["x"], with_logits=True)
    dy = torch.empty((0, wl.d_model), dtype=torch.bfloat16, device="cuda")
    grads = B.alloc_grads(layer.cfg, "cuda")
    for n in ("dW_g", "db_g", "dW1", "db1", "dW2", "db2"):
        getattr(grads, n).fill_(1.0)
    layer.backward(t["x"], out, dy, grads=grads)
    torch.cuda.synchronize()
    # no tokens: every parameter gradient is zero
    for n in ("dW_g", "db_g", "dW1", "db1", "dW2", "db2"):
        assert torch.all(getattr(grads, n) == 0), n
    assert B.backward_launch_count(layer.cfg) == 6


def test_balance_term_alone():
    """dy = 0: only aux * balance has a gradient.  The expert weights get none;
    the router and, through it, x get the balance statistic's gradient."""
    wl = SMALL[3]
    t = synth.make_layer(wl, device="cuda")
    layer = B.MoeLayer(wl, t)
    out = layer.forward(t["x"], with_logits=True)
    dy = torch.zeros((wl.T, wl.d_model), dtype=torch.bfloat16, device="cuda")
    grads = layer.backward(t["x"], out, dy, aux_weight=1.0, with_scores=True)
    torch.cuda.synchronize()
    for n in ("dW1", "db1", "dW2", "db2", "dW1s", "db1s", "dW2s", "db2s", "dw"):
        assert torch.all(getattr(grads, n) == 0), n
    L = oracle_layer(layer.cfg, host_tensors(t))
    r = L.route(0, True, out.topk_idx.cpu().numpy(), workers=WORKERS)
    ref = L.backward(r, dy.cpu(), 1.0, workers=WORKERS)
    for name, g, rr in [("dz", grads.dz, ref.dz), ("dW_g", grads.dW_g, ref.dW_g),
                        ("db_g", grads.db_g, ref.db_g), ("dx", grads.dx, ref.dx)]:
        err = rel_l2(to64(g), rr)
        assert err <= GRAD_TOL[DT_BF16], (name, err)
    assert float(np.abs(ref.dz).max()) > 0.0


def test_training_step_graph_replay_matches_eager():
    """Forward + backward captured once in a CUDA graph and replayed give the
    eager call sequence's outputs and gradients bit for bit."""
    wl = SMALL[1]
    t, layer, out, dy, g_eager = run_backward(wl, 0.01)
    cfg = layer.cfg
    out2 = B.alloc_outputs(cfg, "cuda", with_logits=True)
    g2 = B.alloc_grads(cfg, "cuda", with_scores=True)
    bws = torch.empty(B.backward_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):          # warm: module loading, tensor maps
        B.forward(cfg, t["x"], layer.weights, out2, layer.workspace, stream)
        B.backward(cfg, t["x"], layer.weights, out2, layer.workspace, dy, 0.01, g2, bws, stream)
    stream.synchronize()
    for n in ("dx", "dW1", "dz"):
        getattr(g2, n).zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        B.forward(cfg, t["x"], layer.weights, out2, layer.workspace, stream)
        B.backward(cfg, t["x"], layer.weights, out2, layer.workspace, dy, 0.01, g2, bws, stream)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out2.y, out.y)
    for n in ("dx", "dW_g", "db_g", "dW1", "db1", "dW2", "db2", "dW1s", "db1s", "dW2s", "db2s",
              "dz", "dw"):
        assert torch.equal(getattr(g2, n), getattr(g_eager, n)), n


KEEP_PRE = [
    SMALL[0],                                    # 128 x 256 tiles: from the epilogue
    SMALL[1],                                    # 64-wide tiles, shared expert
    Workload("bwd_keep_decode", T=40, d_model=256, d_ff=384, n_experts=8, top_k=1,
             act=ACT_GELU_ERF, dtype=DT_BF16, seed=89),   # decode tiles: a second pass
    Workload("bwd_keep_f32", T=120, d_model=64, d_ff=96, n_experts=4, top_k=2,
             act=ACT_RELU, dtype=DT_F32, seed=90),        # CUDA cores: from the epilogue
    # 256-wide tiles, shared expert: the pre-activation from the first Linear's epilogue
    Workload("bwd_keep_bn256", T=600, d_model=256, d_ff=512, n_experts=4, top_k=2,
             act=ACT_GELU_ERF, dtype=DT_BF16, d_ff_shared=512, seed=93),
]


@pytest.mark.parametrize("wl", KEEP_PRE, ids=[w.name for w in KEEP_PRE])
def test_kept_pre_activation_gives_the_same_gradients(wl):
    """A forward that keeps the first Linear's pre-activation gives the same
    outputs, and the backward that uses it (no recompute) the same gradients,
    bit for bit, as the forward / backward without it."""
    t, layer, out, dy, g_plain = run_backward(wl, 0.01)
    out_k = layer.forward(t["x"], with_logits=True, with_pre_act=True)
    g_kept = layer.backward(t["x"], out_k, dy, aux_weight=0.01, with_scores=True)
    torch.cuda.synchronize()
    assert torch.equal(out_k.y, out.y)
    for n in ("dx", "dW_g", "db_g", "dW1", "db1", "dW2", "db2", "dz", "dw"):
        assert torch.equal(getattr(g_kept, n), getattr(g_plain, n)), n
    if wl.d_ff_shared:
        for n in ("dW1s", "db1s", "dW2s", "db2s"):
            assert torch.equal(getattr(g_kept, n), getattr(g_plain, n)), n


def unit_sample(f, salt):
    """One hidden unit in every 128-unit block, at a lane that moves from
    block to block (and from expert to expert)."""
    blocks = np.arange((f + 127) // 128)
    u = blocks * 128 + (blocks * 37 + 11 * salt + 5) % 128
    return np.minimum(u, f - 1)


def check_large_backward(wl, aux, tokens_per_group, seed):
    """The training configuration at full size (forward keeping the first
    Linear's pre-activation, backward with aux): sampled tokens' dx, dz, dw;
    every expert's weight gradients on one hidden unit per 128-unit block; the
    router's weight gradients through identities on the GPU's own dz."""
    t = synth.make_layer(wl, device="cuda")
    layer = B.MoeLayer(wl, t)
    out = layer.forward(t["x"], with_logits=True, with_pre_act=True)
    dy = make_dy(wl, wl.seed)
    g = layer.backward(t["x"], out, dy, aux_weight=aux, with_scores=True)
    torch.cuda.synchronize()
    assert B.get_device_status() == B.MOE_OK
    cfg = layer.cfg
    th = host_tensors(t)
    dyh = dy.cpu()
    L = oracle_layer(cfg, th)
    z = L.logits(WORKERS)
    rep = {}
    idx = check_routing(cfg.dtype, cfg, t, out, z, rep,
                        z_gpu=out.logits.cpu().numpy().astype(np.float64))
    r = L.route(cfg.capacity, bool(cfg.renormalize), idx, workers=WORKERS, z=z)
    grp = r.grouping()
    N, f = cfg.n_experts, cfg.d_ff
    rng = np.random.default_rng(seed)

    # tokens: several from every expert group, and the first and last
    toks = {0, wl.T - 1}
    for e in range(N):
        rows = grp.groups[e]
        if rows:
            for i in rng.choice(len(rows), size=min(tokens_per_group, len(rows)), replace=False):
                toks.add(rows[int(i)][0])
    toks = np.array(sorted(toks), dtype=np.int64)
    rdw, rdz, rdx = L.token_grads(r, dyh, aux, toks, bool(cfg.renormalize), WORKERS)
    report = {"tokens": len(toks),
              "dx_row": row_max_rel(to64(g.dx[torch.from_numpy(toks).cuda()]), rdx),
              "dz_row": dz_row_max_rel(to64(g.dz[torch.from_numpy(toks).cuda()]), rdz,
                                       gate_grad_scale(L, r, to64(dy), toks)),
              "dw": rel_l2(to64(g.dw[torch.from_numpy(toks).cuda()]), rdw)}

    # every expert (and the shared one): sampled hidden units
    from concurrent.futures import ThreadPoolExecutor
    jobs = list(range(N + (1 if cfg.d_ff_shared else 0)))

    def one(e):
        fe = cfg.d_ff_shared if e == N else f
        units = unit_sample(fe, e)
        if e == N:
            ts, gs = np.arange(wl.T), np.ones(wl.T)
        else:
            ts = np.array([tt for tt, _ in grp.groups[e]], dtype=np.int64)
            gs = np.array([r.w[tt, j] for tt, j in grp.groups[e]])
        return e, units, L.expert_weight_grads(e, ts, gs, dyh, units=units)

    with ThreadPoolExecutor(max_workers=WORKERS) as ex:
        res = list(ex.map(one, jobs))
    worst = {"dW1": 0.0, "db1": 0.0, "dW2": 0.0, "db2": 0.0}
    for e, units, (w1, b1_, w2, b2_) in res:
        u = torch.from_numpy(units).cuda()
        if e == N:
            gw1, gb1, gw2, gb2 = g.dW1s[u], g.db1s[u], g.dW2s[:, u], g.db2s
        else:
            gw1, gb1, gw2, gb2 = g.dW1[e][u], g.db1[e][u], g.dW2[e][:, u], g.db2[e]
        for name, a, b in (("dW1", gw1, w1), ("db1", gb1, b1_), ("dW2", gw2, w2),
                           ("db2", gb2, b2_)):
            worst[name] = max(worst[name], rel_l2(to64(a), b))
    report.update({k + "_expert_units": v for k, v in worst.items()})
    report["units_per_expert"] = len(unit_sample(f, 0))

    # router weights: identities on the GPU's own dz (dz itself checked above)
    dzg = to64(g.dz)
    x64 = to64(t["x"])
    dzTx = dzg.T @ x64
    dWg = to64(g.dW_g)
    report["dW_g_vs_dzTx"] = max(rel_l2(dWg[e], dzTx[e]) for e in range(N))
    report["db_g_vs_sum_dz"] = rel_l2(to64(g.db_g), dzg.sum(axis=0))
    report["sum_e_dz"] = float(np.abs(dzg.sum(axis=1)).max() /
                               max(np.abs(dzg).max(), 1e-30))
    print("grad parity", wl.name, report)
    bad = {n: v for n, v in report.items()
           if n not in ("tokens", "units_per_expert", "sum_e_dz") and not v <= GRAD_TOL[DT_BF16]}
    assert not bad, f"gradients off: {bad} (all: {report})"
    assert report["sum_e_dz"] <= 1e-3
    del t, layer, out, g
    torch.cuda.empty_cache()
    return report


def test_workload_c3_mixtral_prefill_grads_every_expert():
    """Mixtral-sized layer (T = 4096, d = 4096, d_ff = 14336, 8 experts, top-2)."""
    check_large_backward(WORKLOADS["c3_mixtral_prefill"], 0.01, tokens_per_group=4, seed=11)


def test_workload_c4_deepseek_v3_grads_every_expert():
    """DeepSeek-V3-sized layer (T = 4096, d = 7168, 256 routed experts of d_ff =
    2048 and a shared one, top-8): ~128-row groups, K = 7168, and the router's
    gradients on the tensor cores (N % 64 == 0)."""
    check_large_backward(WORKLOADS["c4_deepseek_v3"], 0.01, tokens_per_group=1, seed=12)
