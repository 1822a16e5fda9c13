"""The backward pass on the GPU (through the C ABI) against the oracle's
backward (float64 chain rule, pinned to torch autograd and finite
differences): every gradient of total = <dy, y> + aux * balance.

Bar: each gradient tensor within 2e-2 relative L2 of the oracle for bf16
layers (1e-4 for fp32 layers, whose CUDA-core path keeps every intermediate in
fp32: a few 1e-7 of rounding per value).  The GPU
stores five bf16 intermediates on the way (dO = w dy, the recomputed
pre-activation, dA, dXp and the expert outputs behind dw), each rounded to 8
significant bits (relative 2^-9 ~ 2e-3 per element, independent across
elements), so a tensor's relative L2 error is a few 1e-3; the bar leaves a
5-10x margin.  The oracle takes the GPU's top-k choice (the forward parity
checks that choice against the oracle's own)."""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_mixture_experts_68_b300 import binding as B
from sparse_mixture_experts_68_b300 import synth
from sparse_mixture_experts_68_b300.workloads import (ACT_GELU_ERF, ACT_RELU, DT_BF16, DT_F32,
                                                      WORKLOADS, Workload)

from parity import Experts, check_layer, to64

pytestmark = pytest.mark.gpu

GRAD_TOL = {DT_BF16: 2e-2, DT_F32: 1e-4}   # per gradient tensor, relative L2


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
    cfg = layer.cfg
    shared = None
    if cfg.d_ff_shared:
        shared = tuple(to64(t[n]) for n in ("W1s", "b1s", "W2s", "b2s"))
    ref = O.moe_backward(to64(t["x"]), to64(t["W_g"]), to64(t["b_g"]), Experts(t["W1"]),
                         Experts(t["b1"]), Experts(t["W2"]), Experts(t["b2"]), to64(dy),
                         k=cfg.top_k, act=cfg.act, capacity=cfg.capacity,
                         renormalize=bool(cfg.renormalize), shared=shared, aux_weight=aux,
                         round_hidden_bf16=(wl.dtype == DT_BF16),
                         idx_override=out.topk_idx.cpu().numpy().astype(np.int64))
    pairs = [("dx", grads.dx, ref.dx), ("dW_g", grads.dW_g, ref.dW_g),
             ("db_g", grads.db_g, ref.db_g), ("dW1", grads.dW1, ref.dW1),
             ("db1", grads.db1, ref.db1), ("dW2", grads.dW2, ref.dW2),
             ("db2", grads.db2, ref.db2), ("dz", grads.dz, ref.dz), ("dw", grads.dw, ref.dw)]
    if shared is not None:
        pairs += [(n, getattr(grads, n), r) for n, r in zip(("dW1s", "db1s", "dW2s", "db2s"),
                                                            ref.shared)]
    report = {}
    for name, g, r in pairs:
        report[name] = rel_l2(to64(g), r)
    bad = {n: v for n, v in report.items() if not v <= GRAD_TOL[wl.dtype]}
    assert not bad, f"gradients off: {bad} (all: {report})"
    # dropped slots pass no gradient to their gate
    dw = grads.dw.cpu().numpy()
    keep = O.group_by_expert(out.topk_idx.cpu().numpy(), cfg.n_experts, cfg.capacity).keep
    assert np.all(dw[~keep] == 0.0)
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
    ref = O.moe_backward(to64(t["x"]), to64(t["W_g"]), to64(t["b_g"]), Experts(t["W1"]),
                         Experts(t["b1"]), Experts(t["W2"]), Experts(t["b2"]), to64(dy),
                         k=wl.top_k, act=wl.act, shared=tuple(to64(t[n]) for n in
                                                              ("W1s", "b1s", "W2s", "b2s")),
                         aux_weight=1.0, round_hidden_bf16=True,
                         idx_override=out.topk_idx.cpu().numpy().astype(np.int64))
    for name, g, r in [("dz", grads.dz, ref.dz), ("dW_g", grads.dW_g, ref.dW_g),
                       ("db_g", grads.db_g, ref.db_g), ("dx", grads.dx, ref.dx)]:
        err = rel_l2(to64(g), r)
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


def sampled_token_grads(x, dy, W_g, idx, w, p, keep, experts, act, aux, tokens):
    """Oracle dx, dz and dw of the given tokens only, by the chain rule of
    moe_backward restricted to their rows: each kept slot's expert FFN
    forward and backward on that one row, the gates' softmax backward, the
    balance term (through all tokens' mean probabilities) and the router."""
    W1, b1, W2, b2 = experts
    T, N = p.shape
    k = idx.shape[1]
    m = p.mean(axis=0)
    dm = aux * 2.0 * (m - 1.0 / N) / (N - 1)
    dx = np.zeros((len(tokens), x.shape[1]))
    dz = np.zeros((len(tokens), N))
    dw = np.zeros((len(tokens), k))
    for e in range(N):
        slots = [(i, j) for i, t in enumerate(tokens) for j in range(k)
                 if idx[t, j] == e and keep[t, j]]
        if not slots:
            continue
        W1e, W2e = W1[e], W2[e]
        for i, j in slots:
            t = tokens[i]
            a = x[t] @ W1e.T + b1[e]
            h = O.round_to_bf16(O.activation(a, act))
            o = h @ W2e.T + b2[e]
            dw[i, j] = float(dy[t] @ o)
            dh = (w[t, j] * dy[t]) @ W2e
            dx[i] += (dh * O.activation_grad(a, act)) @ W1e
    for i, t in enumerate(tokens):
        dsel = w[t] * (dw[i] - np.sum(w[t] * dw[i]))
        dz[i, idx[t]] = dsel
        dz[i] += O.softmax_backward(p[t], dm / T)
        dx[i] += dz[i] @ W_g
    return dx, dz, dw


def test_workload_c3_mixtral_prefill_sampled_grads():
    """The Mixtral-sized layer (T = 4096, d = 4096, d_ff = 14336, 8 experts,
    top-2, GELU) in the training configuration the bench times: the forward
    keeps the pre-activation, the backward takes aux = 0.01.  Expert 0's
    weight and bias gradients in full, and dx / dz / dw of sampled tokens,
    against the oracle's chain rule on those rows (the full oracle backward
    would take minutes of float64 GEMMs)."""
    wl = WORKLOADS["c3_mixtral_prefill"]
    aux = 0.01
    t = synth.make_layer(wl, device="cuda")
    layer = B.MoeLayer(wl, t)
    out = layer.forward(t["x"], with_logits=True, with_pre_act=True)
    dy = make_dy(wl, wl.seed)
    g = layer.backward(t["x"], out, dy, aux_weight=aux, with_scores=True)
    torch.cuda.synchronize()
    assert B.get_device_status() == B.MOE_OK
    cfg = layer.cfg
    x, dy64 = to64(t["x"]), to64(dy)
    idx = out.topk_idx.cpu().numpy().astype(np.int64)
    z = O.router_logits(x, to64(t["W_g"]), to64(t["b_g"]))
    p = O.softmax(z)
    assert cfg.renormalize
    w = O.gates_softmax_of_topk(z, idx)
    grouping = O.group_by_expert(idx, cfg.n_experts, cfg.capacity)
    experts = (Experts(t["W1"]), Experts(t["b1"]), Experts(t["W2"]), Experts(t["b2"]))

    # expert 0: every weight and bias gradient
    rows = grouping.groups[0]
    ts = np.array([r for r, _ in rows])
    js = np.array([j for _, j in rows])
    dO = w[ts, js][:, None] * dy64[ts]
    _, gW1, gb1, gW2, gb2 = O.expert_ffn_backward(
        x[ts], experts[0][0], experts[1][0], experts[2][0], experts[3][0], cfg.act, dO,
        round_hidden_bf16=True)
    report = {"dW1[0]": rel_l2(to64(g.dW1[0]), gW1), "db1[0]": rel_l2(to64(g.db1[0]), gb1),
              "dW2[0]": rel_l2(to64(g.dW2[0]), gW2), "db2[0]": rel_l2(to64(g.db2[0]), gb2)}

    # sampled tokens: dx, dz, dw
    rng = np.random.default_rng(11)
    tokens = sorted(set(rng.choice(wl.T, size=12, replace=False).tolist()) | {0, wl.T - 1})
    rdx, rdz, rdw = sampled_token_grads(x, dy64, to64(t["W_g"]), idx, w, p, grouping.keep,
                                        experts, cfg.act, aux, tokens)
    report["dx"] = rel_l2(to64(g.dx[tokens]), rdx)
    report["dz"] = rel_l2(to64(g.dz[tokens]), rdz)
    report["dw"] = rel_l2(to64(g.dw[tokens]), rdw)
    print("grad parity c3_mixtral_prefill (sampled)", report)
    bad = {n: v for n, v in report.items() if not v <= GRAD_TOL[DT_BF16]}
    assert not bad, f"gradients off: {bad} (all: {report})"
    del t, layer, out, g
    torch.cuda.empty_cache()
