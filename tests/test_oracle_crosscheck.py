"""The C++ oracle against a second, independent statement of the same
definitions in float64 numpy (oracle/moe_oracle_np.py), and the oracle's
pieces against its own whole.

The two statements were written separately (library matmuls and sorts on one
side, scalar loops on the other), so a slip in either -- an index, a
transposed operand, a dropped term -- shows up as a disagreement.  The pieces
the large-layer GPU tests use (per-token gradients, per-hidden-unit weight
gradients, threaded row splits, bf16 inputs read as raw bits) must equal the
whole-layer calls, which the pins tie to the pages and to torch."""

import math

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from oracle import moe_oracle_np as NP


def _layer(seed, T, d, f, N, fs=0):
    rng = np.random.default_rng(seed)
    W_g = rng.normal(0, 1 / math.sqrt(d), (N, d))
    b_g = rng.normal(0, 0.3, N) + np.linspace(0.5, -0.5, N)
    W1 = rng.normal(0, 1 / math.sqrt(d), (N, f, d))
    b1 = rng.normal(0, 0.1, (N, f))
    W2 = rng.normal(0, 1 / math.sqrt(f), (N, d, f))
    b2 = rng.normal(0, 0.1, (N, d))
    x = rng.normal(0, 1, (T, d))
    dy = rng.normal(0, 1, (T, d))
    shared = None
    if fs:
        shared = (rng.normal(0, 1 / math.sqrt(d), (fs, d)), rng.normal(0, 0.1, fs),
                  rng.normal(0, 1 / math.sqrt(fs), (d, fs)), rng.normal(0, 0.1, d))
    return x, W_g, b_g, W1, b1, W2, b2, shared, dy


CASES = [
    # T, d, f, N, k, act, capacity, renorm, fs, round_bf16
    (40, 16, 24, 6, 2, O.ACT_GELU_ERF, 0, True, 0, False),
    (64, 8, 12, 5, 3, O.ACT_RELU, 9, True, 12, True),
    (33, 12, 16, 4, 1, O.ACT_GELU_ERF, 5, False, 0, True),
    (20, 8, 8, 7, 7, O.ACT_RELU, 0, False, 8, False),
    (50, 10, 20, 1, 1, O.ACT_GELU_ERF, 30, True, 0, False),
]


@pytest.mark.parametrize("case", CASES)
def test_forward_and_backward_agree_with_numpy_statement(case):
    T, d, f, N, k, act, cap, renorm, fs, rb = case
    x, W_g, b_g, W1, b1, W2, b2, shared, dy = _layer(200 + T + N, T, d, f, N, fs)
    kw = dict(k=k, act=act, capacity=cap, renormalize=renorm, shared=shared,
              round_hidden_bf16=rb)
    a = O.moe_forward(x, W_g, b_g, W1, b1, W2, b2, **kw)
    b = NP.moe_forward(x, W_g, b_g, W1, b1, W2, b2, **kw)
    np.testing.assert_allclose(a.z, b.z, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(a.p, b.p, rtol=1e-12, atol=1e-15)
    np.testing.assert_array_equal(a.idx, b.idx)
    np.testing.assert_allclose(a.w, b.w, rtol=1e-12)
    np.testing.assert_array_equal(a.grouping.counts, b.grouping.counts)
    np.testing.assert_array_equal(a.grouping.kept, b.grouping.kept)
    np.testing.assert_array_equal(a.grouping.rank, b.grouping.rank)
    np.testing.assert_array_equal(a.grouping.keep, b.grouping.keep)
    assert a.grouping.groups == b.grouping.groups
    assert a.grouping.dropped == b.grouping.dropped
    np.testing.assert_allclose(a.y, b.y, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(a.mean_prob, b.mean_prob, rtol=1e-13)
    assert a.balance == pytest.approx(b.balance, rel=1e-10, abs=1e-18)
    assert a.cv_squared == pytest.approx(b.cv_squared, rel=1e-12, abs=1e-15)
    ga = O.moe_backward(x, W_g, b_g, W1, b1, W2, b2, dy, aux_weight=0.3, **kw)
    gb = NP.moe_backward(x, W_g, b_g, W1, b1, W2, b2, dy, aux_weight=0.3, **kw)
    for name in ("dx", "dW_g", "db_g", "dW1", "db1", "dW2", "db2", "dz", "dw"):
        np.testing.assert_allclose(getattr(ga, name), getattr(gb, name), rtol=1e-10,
                                   atol=1e-12, err_msg=name)
    if shared is not None:
        for u, v in zip(ga.shared, gb.shared):
            np.testing.assert_allclose(u, v, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("C", [0, 3, 11, 40])
def test_expert_choice_agrees_with_numpy_statement(C):
    x, W_g, b_g, W1, b1, W2, b2, shared, _ = _layer(300 + C, 29, 8, 12, 5, fs=12)
    kw = dict(capacity=C, act=O.ACT_GELU_ERF, shared=shared, round_hidden_bf16=True)
    a = O.expert_choice_forward(x, W_g, b_g, W1, b1, W2, b2, **kw)
    b = NP.expert_choice_forward(x, W_g, b_g, W1, b1, W2, b2, **kw)
    for u, v in zip(a.sel, b.sel):
        np.testing.assert_array_equal(u, v)
    np.testing.assert_array_equal(a.token_picks, b.token_picks)
    assert a.unpicked == b.unpicked
    np.testing.assert_allclose(a.y, b.y, rtol=1e-11, atol=1e-12)
    Cn = O.expert_choice_tokens(29, C)
    np.testing.assert_allclose(O.expert_choice_gap(a.p, Cn), NP.expert_choice_gap(b.p, Cn),
                               rtol=1e-9, atol=1e-15)


def test_small_helpers_agree_with_numpy_statement():
    rng = np.random.default_rng(7)
    z = rng.normal(0, 2, (30, 9))
    z[3, 4] = z[3, 1]                                   # a tie
    for k in (1, 2, 5, 9):
        np.testing.assert_array_equal(O.topk_indices(z, k), NP.topk_indices(z, k))
        np.testing.assert_array_equal(O.topk_gap(z, k), NP.topk_gap(z, k))
    v = rng.normal(0, 3, 1000)
    np.testing.assert_array_equal(O.round_to_bf16(v), NP.round_to_bf16(v))
    for act in (O.ACT_GELU_ERF, O.ACT_RELU):
        np.testing.assert_allclose(O.activation(v, act), NP.activation(v, act), rtol=1e-13,
                                   atol=1e-15)
        np.testing.assert_allclose(O.activation_grad(v, act), NP.activation_grad(v, act),
                                   rtol=1e-12, atol=1e-15)
    for cf, T, N in [(1.25, 8192, 64), (1.0, 10, 3), (0.7, 333, 8)]:
        assert O.expert_capacity(cf, T, N) == NP.expert_capacity(cf, T, N)


# ---- the oracle's pieces against its whole -------------------------------------------

def test_threaded_rows_and_token_subsets_equal_one_call():
    x, W_g, b_g, W1, b1, W2, b2, shared, _ = _layer(11, 57, 12, 20, 6, fs=20)
    kw = dict(k=2, act=O.ACT_GELU_ERF, capacity=15, shared=shared, round_hidden_bf16=True)
    one = O.moe_forward(x, W_g, b_g, W1, b1, W2, b2, **kw)
    many = O.moe_forward(x, W_g, b_g, W1, b1, W2, b2, workers=5, **kw)
    assert np.array_equal(one.y, many.y) and np.array_equal(one.z, many.z)
    sub = np.array([56, 3, 17, 0])
    part = O.moe_forward(x, W_g, b_g, W1, b1, W2, b2, tokens=sub, workers=3, **kw)
    assert np.array_equal(part.y, one.y[sub])


def test_bf16_inputs_are_read_as_their_values():
    """bf16 tensors passed as raw bits give the results of their float64 values."""
    x, W_g, b_g, W1, b1, W2, b2, shared, dy = _layer(12, 30, 16, 16, 4, fs=16)
    bf = lambda a: torch.from_numpy(np.asarray(a)).to(torch.bfloat16)       # noqa: E731
    up = lambda a: bf(a).to(torch.float64).numpy()                          # noqa: E731
    kw = dict(k=2, act=O.ACT_RELU, round_hidden_bf16=True)
    a = O.moe_forward(*(bf(v) for v in (x, W_g, b_g, W1, b1, W2, b2)),
                      shared=tuple(bf(v) for v in shared), **kw)
    b = O.moe_forward(*(up(v) for v in (x, W_g, b_g, W1, b1, W2, b2)),
                      shared=tuple(up(v) for v in shared), **kw)
    assert np.array_equal(a.y, b.y) and np.array_equal(a.w, b.w)
    f32 = lambda a: np.asarray(a, dtype=np.float32)                        # noqa: E731
    c = O.moe_forward(*(f32(v) for v in (x, W_g, b_g, W1, b1, W2, b2)),
                      shared=tuple(f32(v) for v in shared), **kw)
    d = O.moe_forward(*(f32(v).astype(np.float64) for v in (x, W_g, b_g, W1, b1, W2, b2)),
                      shared=tuple(f32(v).astype(np.float64) for v in shared), **kw)
    assert np.array_equal(c.y, d.y)


@pytest.mark.parametrize("renorm,cap", [(True, 0), (False, 7), (True, 5)])
def test_token_and_unit_gradients_equal_the_whole_backward(renorm, cap):
    x, W_g, b_g, W1, b1, W2, b2, shared, dy = _layer(21, 41, 10, 24, 5, fs=16)
    kw = dict(k=2, act=O.ACT_GELU_ERF, shared=shared, round_hidden_bf16=True)
    aux = 0.2
    g = O.moe_backward(x, W_g, b_g, W1, b1, W2, b2, dy, capacity=cap, renormalize=renorm,
                       aux_weight=aux, **kw)
    L = O.Layer(x, W_g, b_g, W1, b1, W2, b2, **kw)
    r = L.route(cap, renorm)
    toks = np.array([0, 7, 40, 13])
    dw, dz, dx = L.token_grads(r, dy, aux, toks, renormalize=renorm, workers=2)
    np.testing.assert_allclose(dw, g.dw[toks], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dz, g.dz[toks], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(dx, g.dx[toks], rtol=1e-11, atol=1e-12)
    grp = r.grouping()
    for e in range(5):
        ts = np.array([t for t, _ in grp.groups[e]], dtype=np.int64)
        gates = np.array([r.w[t, j] for t, j in grp.groups[e]])
        units = np.array([23, 0, 5])
        a1, c1, a2, c2 = L.expert_weight_grads(e, ts, gates, dy, units=units)
        np.testing.assert_allclose(a1, g.dW1[e][units], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(c1, g.db1[e][units], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(a2, g.dW2[e][:, units], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(c2, g.db2[e], rtol=1e-11, atol=1e-13)
        f1, fb1, f2, fb2 = L.expert_weight_grads(e, ts, gates, dy)
        np.testing.assert_allclose(f1, g.dW1[e], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(f2, g.dW2[e], rtol=1e-11, atol=1e-13)
    s1, sb1, s2, sb2 = L.expert_weight_grads(5, np.arange(41), np.ones(41), dy,
                                             units=np.array([1, 15]))
    np.testing.assert_allclose(s1, g.shared[0][[1, 15]], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(s2, g.shared[2][:, [1, 15]], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(sb2, g.shared[3], rtol=1e-11, atol=1e-13)


def test_expert_rows_hidden_and_output():
    x, W_g, b_g, W1, b1, W2, b2, shared, _ = _layer(31, 9, 8, 12, 3, fs=12)
    L = O.Layer(x, W_g, b_g, W1, b1, W2, b2, act=O.ACT_GELU_ERF, shared=shared)
    pre, h, o = L.expert_rows(1, [4, 2], want=("pre", "h", "o"))
    np.testing.assert_allclose(pre, x[[4, 2]] @ W1[1].T + b1[1], rtol=1e-13)
    np.testing.assert_allclose(h, NP.activation(pre, NP.ACT_GELU_ERF), rtol=1e-13)
    np.testing.assert_allclose(o, h @ W2[1].T + b2[1], rtol=1e-12)
    _, _, os_ = L.expert_rows(3, [0], want=("o",))             # e == N: the shared expert
    np.testing.assert_allclose(os_[0], NP.expert_ffn(x[[0]], *shared, NP.ACT_GELU_ERF)[0],
                               rtol=1e-12)


@pytest.mark.parametrize("renorm,cap", [(True, 0), (False, 6)])
def test_backward_from_pieces_equals_the_whole_backward(renorm, cap):
    x, W_g, b_g, W1, b1, W2, b2, shared, dy = _layer(22, 37, 12, 16, 6, fs=8)
    kw = dict(k=3, act=O.ACT_RELU, shared=shared, round_hidden_bf16=True)
    g = O.moe_backward(x, W_g, b_g, W1, b1, W2, b2, dy, capacity=cap, renormalize=renorm,
                       aux_weight=0.05, **kw)
    L = O.Layer(x, W_g, b_g, W1, b1, W2, b2, **kw)
    p = L.backward(L.route(cap, renorm), dy, 0.05, renormalize=renorm, workers=3)
    for name in ("dx", "dW_g", "db_g", "dW1", "db1", "dW2", "db2", "dz", "dw"):
        np.testing.assert_allclose(getattr(p, name), getattr(g, name), rtol=1e-11,
                                   atol=1e-13, err_msg=name)
    for u, v in zip(p.shared, g.shared):
        np.testing.assert_allclose(u, v, rtol=1e-11, atol=1e-13)
