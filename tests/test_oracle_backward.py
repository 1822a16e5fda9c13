"""Pins for the oracle's backward pass.  Its gradients are checked against
(a) torch.autograd through an independently written torch forward (every
expert on every token, then masked -- a different structure from the oracle's
grouped loop), and (b) central finite differences of the oracle's own forward
loss along random directions.  Plus the softmax invariant sum_e dz[t, e] = 0."""

import math

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O


def _layer(seed, T, d, f, N, fs=0, gap=True):
    rng = np.random.default_rng(seed)
    W_g = rng.normal(0, 1 / math.sqrt(d), (N, d))
    b_g = rng.normal(0, 0.1, N)
    if gap:   # well-separated scores, so the top-k set is stable under small steps
        b_g = np.linspace(1.5, -1.5, N) + rng.normal(0, 0.01, N)
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


def _torch_loss(x, W_g, b_g, W1, b1, W2, b2, shared, dy, k, act, capacity, renorm, aux):
    """The layer and the loss in torch, every expert on every token and a mask."""
    T, d = x.shape
    N = W_g.shape[0]
    z = x @ W_g.T + b_g
    p = torch.softmax(z, dim=1)
    idx = torch.argsort(-z.detach(), dim=1, stable=True)[:, :k]
    if renorm:
        w = torch.softmax(torch.gather(z, 1, idx), dim=1)
    else:
        w = torch.gather(p, 1, idx)
    count = [0] * N
    keep = torch.zeros((T, k), dtype=torch.bool)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            keep[t, j] = capacity <= 0 or count[e] < capacity
            count[e] += 1
    gelu = torch.nn.GELU()
    actf = (lambda a: gelu(a)) if act == O.ACT_GELU_ERF else torch.relu
    y = torch.zeros_like(x)
    for e in range(N):
        out = actf(x @ W1[e].T + b1[e]) @ W2[e].T + b2[e]
        for j in range(k):
            m = ((idx[:, j] == e) & keep[:, j]).to(x.dtype)
            y = y + (m * w[:, j])[:, None] * out
    if shared is not None:
        W1s, b1s, W2s, b2s = shared
        y = y + actf(x @ W1s.T + b1s) @ W2s.T + b2s
    m = p.mean(dim=0)
    bal = ((m - 1.0 / N) ** 2).sum() / (N - 1) if N > 1 else torch.zeros((), dtype=x.dtype)
    return (dy * y).sum() + aux * bal


CASES = [
    # T, d, f, N, k, act, capacity, renorm, shared, aux
    (9, 6, 10, 4, 2, O.ACT_GELU_ERF, 0, True, 0, 0.01),
    (12, 8, 12, 5, 3, O.ACT_RELU, 4, True, 12, 0.5),
    (10, 6, 8, 3, 1, O.ACT_GELU_ERF, 3, False, 0, 0.3),
    (7, 5, 9, 1, 1, O.ACT_GELU_ERF, 0, True, 0, 0.0),
    (11, 6, 8, 6, 6, O.ACT_RELU, 0, False, 8, 1.0),
]


@pytest.mark.parametrize("case", CASES)
def test_backward_equals_torch_autograd(case):
    T, d, f, N, k, act, cap, renorm, fs, aux = case
    x, W_g, b_g, W1, b1, W2, b2, shared, dy = _layer(7 + T + N, T, d, f, N, fs, gap=False)
    g = O.moe_backward(x, W_g, b_g, W1, b1, W2, b2, dy, k=k, act=act, capacity=cap,
                       renormalize=renorm, shared=shared, aux_weight=aux)
    tt = lambda a: torch.tensor(a, dtype=torch.float64, requires_grad=True)  # noqa: E731
    params = [tt(v) for v in (x, W_g, b_g, W1, b1, W2, b2)]
    sh = tuple(tt(v) for v in shared) if shared is not None else None
    loss = _torch_loss(*params, sh, torch.tensor(dy), k, act, cap, renorm, aux)
    loss.backward()
    ours = [g.dx, g.dW_g, g.db_g, g.dW1, g.db1, g.dW2, g.db2]
    for name, a, b in zip(("dx", "dW_g", "db_g", "dW1", "db1", "dW2", "db2"), ours, params):
        np.testing.assert_allclose(a, b.grad.numpy(), rtol=1e-10, atol=1e-12, err_msg=name)
    if shared is not None:
        for a, b in zip(g.shared, sh):
            np.testing.assert_allclose(a, b.grad.numpy(), rtol=1e-10, atol=1e-12)
    # softmax invariant: each token's score gradient sums to zero
    np.testing.assert_allclose(g.dz.sum(axis=1), 0.0, atol=1e-12)


def _oracle_loss(x, W_g, b_g, W1, b1, W2, b2, shared, dy, k, act, cap, renorm, aux):
    out = O.moe_forward(x, W_g, b_g, W1, b1, W2, b2, k=k, act=act, capacity=cap,
                        renormalize=renorm, shared=shared)
    return float(np.sum(dy * out.y) + aux * out.balance)


@pytest.mark.parametrize("case", CASES[:3])
def test_backward_matches_finite_differences(case):
    T, d, f, N, k, act, cap, renorm, fs, aux = case
    x, W_g, b_g, W1, b1, W2, b2, shared, dy = _layer(100 + T, T, d, f, N, fs, gap=True)
    g = O.moe_backward(x, W_g, b_g, W1, b1, W2, b2, dy, k=k, act=act, capacity=cap,
                       renormalize=renorm, shared=shared, aux_weight=aux)
    rng = np.random.default_rng(5)
    base = [x, W_g, b_g, W1, b1, W2, b2]
    grads = [g.dx, g.dW_g, g.db_g, g.dW1, g.db1, g.dW2, g.db2]
    eps = 1e-6
    for i in range(len(base)):
        v = rng.normal(0, 1, base[i].shape)
        plus = [b if j != i else b + eps * v for j, b in enumerate(base)]
        minus = [b if j != i else b - eps * v for j, b in enumerate(base)]
        fd = (_oracle_loss(*plus, shared, dy, k, act, cap, renorm, aux) -
              _oracle_loss(*minus, shared, dy, k, act, cap, renorm, aux)) / (2 * eps)
        an = float(np.sum(grads[i] * v))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (i, fd, an)


def test_zero_upstream_and_zero_aux_give_zero_gradients():
    x, W_g, b_g, W1, b1, W2, b2, shared, dy = _layer(3, 8, 6, 8, 4, 8)
    g = O.moe_backward(x, W_g, b_g, W1, b1, W2, b2, np.zeros_like(dy), k=2,
                       act=O.ACT_GELU_ERF, shared=shared, aux_weight=0.0)
    for a in (g.dx, g.dW_g, g.db_g, g.dW1, g.db1, g.dW2, g.db2, *g.shared):
        assert np.all(a == 0.0)
    # the balance term alone moves only the router and, through it, x
    g = O.moe_backward(x, W_g, b_g, W1, b1, W2, b2, np.zeros_like(dy), k=2,
                       act=O.ACT_GELU_ERF, shared=shared, aux_weight=0.01)
    assert np.all(g.dW1 == 0.0) and np.all(g.dW2 == 0.0)
    assert np.abs(g.dW_g).max() > 0.0


def test_activation_grad_against_torch():
    a = np.linspace(-6, 6, 1201)
    ta = torch.tensor(a, requires_grad=True)
    torch.nn.GELU()(ta).sum().backward()
    np.testing.assert_allclose(O.activation_grad(a, O.ACT_GELU_ERF), ta.grad.numpy(),
                               rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(O.activation_grad(a, O.ACT_RELU), (a > 0).astype(float))
