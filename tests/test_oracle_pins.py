"""Pins for the CPU oracle: facts fixed by the pages or by mathematics, not by
the oracle itself.  Each test is chosen so that a plausible slip in the oracle
(a dropped term, a wrong sign or index, a transposed operand) fails it."""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _layer(rng, T, d, f, N, fs=0):
    W_g = rng.normal(0, 1 / math.sqrt(d), (N, d))
    b_g = rng.normal(0, 0.1, N)
    W1 = rng.normal(0, 1 / math.sqrt(d), (N, f, d))
    b1 = rng.normal(0, 0.1, (N, f))
    W2 = rng.normal(0, 1 / math.sqrt(f), (N, d, f))
    b2 = rng.normal(0, 0.1, (N, d))
    x = rng.normal(0, 1, (T, d))
    shared = None
    if fs:
        shared = (rng.normal(0, 1 / math.sqrt(d), (fs, d)), rng.normal(0, 0.1, fs),
                  rng.normal(0, 1 / math.sqrt(fs), (d, fs)), rng.normal(0, 0.1, d))
    return x, W_g, b_g, W1, b1, W2, b2, shared


# --- router ---------------------------------------------------------------

def test_worked_example_page3():
    """Scores [1.2,-0.3,2.0,0.1,0.4,-1.0,1.9,0.0], top-2: experts 3 and 7
    (1-based) with gates 0.52 / 0.48 as printed on the page."""
    g = json.load(open(os.path.join(GOLDEN, "worked_example_router.json")))
    z = np.array([g["scores"]])
    idx = O.topk_indices(z, g["top_k"])
    assert [int(i) + 1 for i in idx[0]] == g["selected_experts_1based"]
    w = O.gates_softmax_of_topk(z, idx)[0]
    assert [round(float(v), g["printed_decimals"]) for v in w] == g["gates_printed"]
    # closed form of a two-way softmax: 1 / (1 + e^{-(2.0 - 1.9)})
    assert w[0] == pytest.approx(1.0 / (1.0 + math.exp(-0.1)), rel=1e-14)
    assert w[1] == pytest.approx(1.0 / (1.0 + math.exp(0.1)), rel=1e-14)
    runs = ["runs" if e in idx[0] else "idle" for e in range(8)]
    assert runs == g["widget_state"]


def test_renormalised_probs_equal_softmax_of_topk():
    """softmax -> top-k -> renormalise (botmartz.com, matteuscruz.github.io)
    equals Softmax(TopK(z)) (roadtointelligence.com)."""
    rng = _rng(1)
    for N, k in [(8, 2), (64, 1), (256, 8), (5, 5), (3, 2)]:
        z = rng.normal(0, 3, (200, N))
        idx = O.topk_indices(z, k)
        a = O.gates_softmax_of_topk(z, idx)
        b = O.gates_renormalised_probs(O.softmax(z), idx)
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(a.sum(-1), 1.0, rtol=1e-13)


def test_topk_properties_and_ties():
    rng = _rng(2)
    z = rng.normal(0, 1, (100, 16))
    idx = O.topk_indices(z, 4)
    for t in range(100):
        kept = z[t, idx[t]]
        rest = np.delete(z[t], idx[t])
        assert np.all(np.diff(kept) <= 0)           # slot 0 = largest
        assert kept.min() >= rest.max()
    # equal scores: the lower expert index wins
    zt = np.array([[1.0, 2.0, 2.0, 0.0, 2.0]])
    assert O.topk_indices(zt, 1).tolist() == [[1]]
    assert O.topk_indices(zt, 2).tolist() == [[1, 2]]
    assert O.topk_indices(zt, 3).tolist() == [[1, 2, 4]]


def test_softmax_against_library_and_edge_cases():
    rng = _rng(3)
    z = rng.normal(0, 4, (50, 9))
    ref = torch.softmax(torch.from_numpy(z), dim=-1).numpy()
    np.testing.assert_allclose(O.softmax(z), ref, rtol=1e-13, atol=1e-300)
    # k == N: the gates are the plain softmax
    idx = O.topk_indices(z, 9)
    np.testing.assert_allclose(np.take_along_axis(ref, idx, -1),
                               O.gates_softmax_of_topk(z, idx), rtol=1e-12)
    # one expert: gate 1; k = 1 renormalised: gate exactly 1
    assert O.gates_softmax_of_topk(np.array([[0.3]]), np.array([[0]]))[0, 0] == 1.0
    i1 = O.topk_indices(z, 1)
    assert np.all(O.gates_softmax_of_topk(z, i1) == 1.0)
    # raw gates without renormalisation are the kept probabilities
    np.testing.assert_allclose(O.gates_raw_probs(ref, i1)[:, 0], ref.max(-1), rtol=1e-13)
    # no renormalisation: gates of a top-2 sum to less than 1
    i2 = O.topk_indices(z, 2)
    assert np.all(O.gates_raw_probs(ref, i2).sum(-1) < 1.0)


def test_router_linear_matches_torch_linear():
    """The router is nn.Linear(d_model, N): weight [N, d], bias [N]."""
    rng = _rng(4)
    x = rng.normal(0, 1, (7, 12))
    lin = torch.nn.Linear(12, 5, dtype=torch.float64)
    with torch.no_grad():
        ref = lin(torch.from_numpy(x)).numpy()
    z = O.router_logits(x, lin.weight.detach().numpy(), lin.bias.detach().numpy())
    np.testing.assert_allclose(z, ref, rtol=1e-13, atol=1e-13)


def test_topk_gap():
    z = np.array([[3.0, 1.0, 2.0, 2.0 - 5e-5], [0.0, 1.0, 2.0, 3.0]])
    g = O.topk_gap(z, 2)
    assert g[0] == pytest.approx(5e-5, rel=1e-9)
    assert g[1] == pytest.approx(1.0)
    assert np.isinf(O.topk_gap(z, 4)).all()


# --- grouping and capacity ---------------------------------------------------

def test_capacity_formula_switch_case():
    # capacity factor 1.25, 8192 tokens, 64 experts -> 160 per expert
    assert O.expert_capacity(1.25, 8192, 64) == 160
    assert O.expert_capacity(1.0, 10, 3) == 4          # rounded up
    assert O.expert_capacity(2.0, 9, 3) == 6


def test_grouping_hand_case_all_to_one_expert():
    idx = np.zeros((6, 1), dtype=np.int64)
    g = O.group_by_expert(idx, 4, capacity=3)
    assert g.groups[0] == [(0, 0), (1, 0), (2, 0)]
    assert g.counts.tolist() == [6, 0, 0, 0]
    assert g.kept.tolist() == [3, 0, 0, 0]
    assert g.keep[:, 0].tolist() == [True, True, True, False, False, False]
    assert g.dropped == 3


def test_grouping_invariants():
    rng = _rng(5)
    T, N, k, C = 300, 7, 3, 40
    z = rng.normal(0, 1, (T, N)) + np.linspace(2, 0, N)   # skewed toward low experts
    idx = O.topk_indices(z, k)
    g = O.group_by_expert(idx, N, C)
    assert g.counts.sum() == T * k
    assert np.array_equal(g.kept, np.minimum(g.counts, C))
    assert g.dropped == int((g.counts - g.kept).sum()) > 0
    for e in range(N):
        ts = [t for t, _ in g.groups[e]]
        assert ts == sorted(ts)
        for r, (t, j) in enumerate(g.groups[e]):
            assert idx[t, j] == e and g.rank[t, j] == r
    # brute-force rank: number of earlier (token-major) assignments to e
    flat = idx.reshape(-1)
    for a in range(0, T * k, 17):
        assert g.rank.reshape(-1)[a] == np.count_nonzero(flat[:a] == flat[a])


# --- experts and the layer -------------------------------------------------

def test_dense_special_case_matches_torch_modules():
    """N = 1, k = 1: the layer is Linear -> GELU/ReLU -> Linear."""
    torch.manual_seed(0)
    for act, mod in [(O.ACT_GELU_ERF, torch.nn.GELU()), (O.ACT_RELU, torch.nn.ReLU())]:
        l1 = torch.nn.Linear(6, 10, dtype=torch.float64)
        l2 = torch.nn.Linear(10, 6, dtype=torch.float64)
        x = torch.randn(9, 6, dtype=torch.float64)
        with torch.no_grad():
            ref = l2(mod(l1(x))).numpy()
        W = lambda m: m.weight.detach().numpy()   # noqa: E731
        B = lambda m: m.bias.detach().numpy()     # noqa: E731
        out = O.moe_forward(x.numpy(), np.ones((1, 6)), np.zeros(1), [W(l1)], [B(l1)],
                            [W(l2)], [B(l2)], k=1, act=act)
        np.testing.assert_allclose(out.y, ref, rtol=1e-12, atol=1e-12)


def test_gelu_against_library():
    h = np.linspace(-6, 6, 97)
    ref = torch.nn.functional.gelu(torch.from_numpy(h)).numpy()
    np.testing.assert_allclose(O.activation(h, O.ACT_GELU_ERF), ref, rtol=1e-12, atol=1e-15)
    assert O.activation(np.array([0.0]), O.ACT_GELU_ERF)[0] == 0.0


@pytest.mark.parametrize("N,k,C,fs,act,renorm", [
    (4, 2, 0, 0, O.ACT_GELU_ERF, True),
    (5, 1, 3, 0, O.ACT_RELU, True),
    (6, 3, 4, 8, O.ACT_GELU_ERF, True),
    (3, 2, 0, 0, O.ACT_RELU, False),
    (1, 1, 0, 0, O.ACT_GELU_ERF, True),
])
def test_grouped_forward_equals_bruteforce(N, k, C, fs, act, renorm):
    rng = _rng(10 + N)
    x, W_g, b_g, W1, b1, W2, b2, shared = _layer(rng, 13, 8, 16, N, fs)
    W_g = W_g + 0.5 * np.arange(N)[:, None] / N          # uneven routing
    out = O.moe_forward(x, W_g, b_g, W1, b1, W2, b2, k=k, act=act, capacity=C,
                        renormalize=renorm, shared=shared)
    ref = O.moe_bruteforce(x, W_g, b_g, W1, b1, W2, b2, k=k, act=act, capacity=C,
                           renormalize=renorm, shared=shared)
    np.testing.assert_allclose(out.y, ref, rtol=1e-12, atol=1e-12)
    assert out.y.shape == x.shape
    # a subset of tokens gives the same rows
    sub = np.array([12, 0, 5])
    part = O.moe_forward(x, W_g, b_g, W1, b1, W2, b2, k=k, act=act, capacity=C,
                         renormalize=renorm, shared=shared, tokens=sub)
    np.testing.assert_allclose(part.y, out.y[sub], rtol=1e-13, atol=1e-14)


def test_fully_dropped_token_outputs_zero():
    rng = _rng(7)
    x, W_g, b_g, W1, b1, W2, b2, _ = _layer(rng, 8, 4, 8, 3)
    W_g = np.zeros_like(W_g)
    b_g = np.array([5.0, 0.0, -5.0])                    # every token picks expert 0
    out = O.moe_forward(x, W_g, b_g, W1, b1, W2, b2, k=1, act=O.ACT_RELU, capacity=2)
    assert out.grouping.kept.tolist() == [2, 0, 0]
    assert np.all(out.y[2:] == 0.0)
    assert np.any(out.y[:2] != 0.0)


def test_zero_expert_weights_give_bias_path():
    """With zero weights the expert output is act(b1) . W2 + b2 = b2, and the
    renormalised gates sum to one, so y = b2 for every token (one expert)."""
    rng = _rng(8)
    x, W_g, b_g, W1, b1, W2, b2, _ = _layer(rng, 5, 4, 6, 2)
    W1 = np.zeros_like(W1)
    W2 = np.zeros_like(W2)
    b2[:] = b2[0]
    out = O.moe_forward(x, W_g, b_g, W1, b1, W2, b2, k=2, act=O.ACT_GELU_ERF)
    np.testing.assert_allclose(out.y, np.broadcast_to(b2[0], out.y.shape), rtol=1e-13)


# --- balance statistic -----------------------------------------------------

def test_balance_closed_forms():
    N = 8
    uniform = np.full((10, N), 1.0 / N)
    m, b = O.balance_statistic(uniform)
    assert b == pytest.approx(0.0, abs=1e-30)
    collapse = np.zeros((10, N))
    collapse[:, 3] = 1.0
    m, b = O.balance_statistic(collapse)
    assert b == pytest.approx(1.0 / N, rel=1e-14)      # unbiased std: exactly 1/N
    rng = _rng(9)
    p = O.softmax(rng.normal(0, 2, (40, N)))
    m, b = O.balance_statistic(p)
    assert m.mean() == pytest.approx(1.0 / N, rel=1e-13)
    assert b == pytest.approx(float(torch.std(torch.from_numpy(m)) ** 2), rel=1e-12)
    assert O.balance_statistic(np.ones((3, 1)))[1] == 0.0


# --- number format -----------------------------------------------------------

def test_cv_squared_closed_forms():
    """Uniform counts give 0; all of S assignments on one of N experts give
    exactly N (var = S^2/N, mean^2 = S^2/N^2); two experts with counts (a, b)
    give 2(a-b)^2/(a+b)^2; one expert or nothing routed gives 0."""
    assert O.cv_squared([5, 5, 5, 5]) == 0.0
    for N in (2, 3, 8, 64):
        c = np.zeros(N, dtype=np.int64)
        c[N // 2] = 1000
        assert O.cv_squared(c) == pytest.approx(float(N), rel=1e-14)
    for a, b in [(3, 1), (10, 0), (7, 9)]:
        assert O.cv_squared([a, b]) == pytest.approx(2 * (a - b) ** 2 / (a + b) ** 2, rel=1e-14)
    assert O.cv_squared([17]) == 0.0
    assert O.cv_squared([0, 0, 0]) == 0.0
    # the forward reports it for the routed counts (before capacity)
    x, W_g, b_g, W1, b1, W2, b2, _ = _layer(_rng(11), 40, 8, 16, 4)
    out = O.moe_forward(x, W_g, b_g, W1, b1, W2, b2, k=2, act=O.ACT_RELU, capacity=5)
    c = out.grouping.counts
    assert c.sum() == 80 and out.grouping.kept.max() <= 5
    mean = 80 / 4
    assert out.cv_squared == pytest.approx(sum((ci - mean) ** 2 for ci in c) / 3 / mean ** 2,
                                           rel=1e-12)


def test_round_to_bf16_matches_torch():
    rng = _rng(11)
    v = np.concatenate([rng.normal(0, 1, 5000), rng.normal(0, 1e-3, 500),
                        rng.normal(0, 1e4, 500)]).astype(np.float32)
    ties = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 0.0], np.float32)
    v = np.concatenate([v, ties])
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.round_to_bf16(v.astype(np.float64)), ref)


# --- expert-choice routing ------------------------------------------------

def _bruteforce_pick(col, C):
    """The C-subset of tokens with the largest total score; among equal totals
    the lexicographically smallest ascending index tuple.  With distinct scores
    that is the top C; with ties at the cut it keeps the lower token indices."""
    import itertools
    best, best_key = None, None
    for sub in itertools.combinations(range(len(col)), C):
        key = (-sum(col[list(sub)]), sub)
        if best_key is None or key < best_key:
            best, best_key = sub, key
    return np.array(best, dtype=np.int64)


def test_expert_choice_select_against_subset_bruteforce():
    rng = _rng(41)
    for trial in range(30):
        T = int(rng.integers(1, 8))
        N = int(rng.integers(1, 5))
        # a few distinct levels (dyadic, so the subset sums are exact), many ties
        p = rng.integers(0, 4, (T, N)) / 8.0
        for C in range(0, T + 1):
            sel = O.expert_choice_select(p, C)
            for e in range(N):
                np.testing.assert_array_equal(sel[e], _bruteforce_pick(p[:, e], C))


def test_expert_choice_hand_case_and_balance():
    p = np.array([[0.9, 0.1], [0.2, 0.8], [0.6, 0.4], [0.6, 0.4]])
    sel = O.expert_choice_select(p, 2)
    assert sel[0].tolist() == [0, 2]          # 0.9, then the tie 0.6 / 0.6 -> token 2
    assert sel[1].tolist() == [1, 2]          # 0.8, then the tie 0.4 / 0.4 -> token 2
    gaps = O.expert_choice_gap(p, 2)
    assert gaps.tolist() == [0.0, 0.0]
    assert O.expert_choice_gap(p, 1).tolist() == pytest.approx([0.3, 0.4])
    assert np.isinf(O.expert_choice_gap(p, 4)).all()
    assert O.expert_choice_tokens(100, 0) == 100
    assert O.expert_choice_tokens(100, 250) == 100
    assert O.expert_choice_tokens(100, 25) == 25
    # perfect balance by construction: every expert takes exactly C tokens
    x, W_g, b_g, W1, b1, W2, b2, _ = _layer(_rng(42), 37, 8, 16, 5)
    out = O.expert_choice_forward(x, W_g, b_g, W1, b1, W2, b2, capacity=9, act=O.ACT_RELU)
    assert [len(s) for s in out.sel] == [9] * 5
    assert out.token_picks.sum() == 45
    assert out.unpicked == int((out.token_picks == 0).sum())
    assert O.cv_squared([len(s) for s in out.sel]) == 0.0
    for e in range(5):
        assert np.all(np.diff(out.sel[e]) > 0)
        # every picked score is at least every unpicked one
        rest = np.setdiff1d(np.arange(37), out.sel[e])
        assert out.p[out.sel[e], e].min() >= out.p[rest, e].max()


def test_expert_choice_all_tokens_equals_soft_mixture():
    """C = T: every expert takes every token, so y = sum_e p[t, e] expert_e(x):
    top-k routing with k = N (gates renormalised over all N are p)."""
    x, W_g, b_g, W1, b1, W2, b2, shared = _layer(_rng(43), 12, 8, 16, 4, fs=16)
    for cap in (0, 12, 50):
        ec = O.expert_choice_forward(x, W_g, b_g, W1, b1, W2, b2, capacity=cap,
                                     act=O.ACT_GELU_ERF, shared=shared)
        ref = O.moe_bruteforce(x, W_g, b_g, W1, b1, W2, b2, k=4, act=O.ACT_GELU_ERF,
                               shared=shared)
        np.testing.assert_allclose(ec.y, ref, rtol=1e-12, atol=1e-12)
        assert ec.unpicked == 0


def test_expert_choice_single_expert_is_dense_ffn():
    d, f = 8, 16
    x, W_g, b_g, W1, b1, W2, b2, _ = _layer(_rng(44), 10, d, f, 1)
    out = O.expert_choice_forward(x, W_g, b_g, W1, b1, W2, b2, capacity=0, act=O.ACT_GELU_ERF)
    lin1 = torch.nn.Linear(d, f, dtype=torch.float64)
    lin2 = torch.nn.Linear(f, d, dtype=torch.float64)
    with torch.no_grad():
        lin1.weight.copy_(torch.from_numpy(W1[0])); lin1.bias.copy_(torch.from_numpy(b1[0]))
        lin2.weight.copy_(torch.from_numpy(W2[0])); lin2.bias.copy_(torch.from_numpy(b2[0]))
        dense = lin2(torch.nn.GELU()(lin1(torch.from_numpy(x)))).numpy()
    np.testing.assert_allclose(out.y, dense, rtol=1e-12, atol=1e-12)


def test_expert_choice_forward_equals_masked_bruteforce():
    """Every expert on every token, then the pick mask (chosen by the subset
    brute force) and the p gates; unpicked tokens get only the shared expert."""
    for seed, (T, N, C, fs) in enumerate([(7, 3, 2, 0), (6, 4, 1, 16), (8, 2, 5, 0)]):
        x, W_g, b_g, W1, b1, W2, b2, shared = _layer(_rng(50 + seed), T, 8, 16, N, fs=fs)
        out = O.expert_choice_forward(x, W_g, b_g, W1, b1, W2, b2, capacity=C,
                                      act=O.ACT_RELU, shared=shared)
        p = torch.softmax(torch.from_numpy(x @ W_g.T + b_g), dim=1).numpy()
        y = np.zeros_like(x)
        for e in range(N):
            mask = np.zeros(T, dtype=bool)
            mask[_bruteforce_pick(p[:, e], C)] = True
            h = np.maximum(x @ W1[e].T + b1[e], 0.0)
            y[mask] += p[mask, e][:, None] * (h @ W2[e].T + b2[e])[mask]
        if shared is not None:
            y += np.maximum(x @ shared[0].T + shared[1], 0.0) @ shared[2].T + shared[3]
        np.testing.assert_allclose(out.y, y, rtol=1e-12, atol=1e-12)
        if shared is None:
            for t in np.nonzero(out.token_picks == 0)[0]:
                assert np.all(out.y[t] == 0.0)
