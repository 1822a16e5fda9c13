"""Float64 numpy statement of the CPU oracle, kept as a cross-check of the
C++ oracle (moe_oracle.cpp), which is the oracle the tests and the benchmark use.

TEST INFRASTRUCTURE ONLY.  Nothing in the library path imports this module:
only the tests, the smoke check in ``__graft_entry__`` and the CPU-baseline leg
of ``bench.py`` may call it.  It shares no code with the CUDA path.

Everything here is the plain definition of what the layer computes, in
float64 numpy, with no blocking, fusion or reordering beyond the definition:

* router scores ``z = x . W_g^T + b_g`` -- botmartz.com "Mixture of Experts (MoE)
  and Mixtral: Scaling Without Dense Computation", section "Expert Routing"
  (the router is an ``nn.Linear(d_model, num_experts)``); roadtointelligence.com
  "Mixture of Experts (MoE)", the router formula G(x) = Softmax(TopK(x . W_g)).
* softmax over all N experts, then the top-k, then renormalisation of the kept
  k probabilities -- botmartz.com "Expert Routing"; matteuscruz.github.io
  "What is a Mixture of Experts?", section "Architecture: router + experts".
* the same gates written as a softmax over only the kept top-k logits --
  roadtointelligence.com, router formula and the "Tiny example".
* gates without renormalisation (the raw softmax probability of each kept
  expert) -- codingnowai.in "Mixture of Experts", section "Code".
* expert FFN Linear -> GELU -> Linear (botmartz.com "Expert Routing") or
  Linear -> ReLU -> Linear (codingnowai.in "Code"), each with bias.
* output y = sum over kept experts of gate * expert(x) -- roadtointelligence.com
  output equation; matteuscruz.github.io "Architecture: router + experts".
* expert capacity = capacity factor x batch / num_experts, tokens over capacity
  dropped (layer output 0, the token passes on through the residual) --
  matteuscruz.github.io "Load balancing: the core training challenge";
  roadtointelligence.com "Keeping the experts busy".
* one shared expert applied to every token with weight 1 --
  roadtointelligence.com "Total versus active parameters" (DeepSeek-V3).
* balance statistic std(mean_t router_probs)^2 with torch's default
  (unbiased) std -- botmartz.com "Load Balancing: The Hidden Challenge".
* expert-choice routing: each expert takes the tokens it scores highest
  instead of each token taking its top-k experts, so every expert gets the same
  load -- matteuscruz.github.io "Load balancing: the core training challenge"
  (Zhou et al., 2022, as the page describes it).  Readings: the score is the
  router probability p[t, e]; an expert takes C tokens (C = the capacity,
  clamped to T; C <= 0 means all T); ties go to the lower token index; a picked
  token's gate is p[t, e]; a token no expert picked outputs 0.
* the backward pass of the layer for the training loss
  total = task + alpha * balance (botmartz.com "Load Balancing: The Hidden
  Challenge": total_loss = task_loss + 0.01 * balance_loss; roadtointelligence.com
  "Keeping the experts busy": coefficient 0.01).  The task loss enters as its
  gradient dy = d task / d y; every other derivative is the chain rule through
  the forward above, written out step by step (no automatic differentiation).
  The top-k choice and the capacity drops are piecewise constant: they pass
  no gradient.
* squared coefficient of variation of the expert counts, the quantity the
  auxiliary loss penalises -- matteuscruz.github.io "Load balancing: the core
  training challenge"; named cv_squared(expert_counts) in invest-in.ai
  "MoE - Mixture of Experts", "Common Usage Examples".  The pages give no
  formula; read as var/mean^2 with the unbiased variance over the N counts.

Readings taken where the pages are silent (each also listed in the design
notes): top-k ties go to the lower expert index; slot 0 holds the largest
score; capacity priority is token-major (token, then slot); the capacity is
ceil(capacity_factor * T / N); a dropped (token, slot) contributes exactly 0;
the shared expert uses the routed experts' FFN form and activation.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

try:                                    # library erf; math.erf elementwise otherwise
    from scipy.special import erf as _erf
except ImportError:                     # pragma: no cover
    _erf = np.vectorize(math.erf, otypes=[np.float64])

ACT_GELU_ERF = 0
ACT_RELU = 1


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def round_to_bf16(v):
    """Round float64 values to the nearest bfloat16 value (ties to even).

    bfloat16 keeps 8 significant bits and float32's exponent range, so for the
    normal numbers this layer produces, rounding to 8 significant bits with
    round-half-to-even is the whole definition.  Zeros, infinities and NaNs
    pass through unchanged.
    """
    v = np.asarray(v, dtype=np.float64)
    mant, expo = np.frexp(v)                      # v = mant * 2**expo, |mant| in [0.5, 1)
    q = np.round(mant * 256.0)                    # numpy rounds half to even
    out = np.ldexp(q / 256.0, expo)
    return np.where(np.isfinite(v), out, v)


# ---------------------------------------------------------------------------
# router: scores, softmax, top-k, gates
# ---------------------------------------------------------------------------

def router_logits(x, W_g, b_g):
    """z[t, e] = sum_i x[t, i] * W_g[e, i] + b_g[e]   (nn.Linear(d_model, N))."""
    x = np.asarray(x, dtype=np.float64)
    W_g = np.asarray(W_g, dtype=np.float64)
    b_g = np.asarray(b_g, dtype=np.float64)
    return x @ W_g.T + b_g


def softmax(z):
    """Softmax over the last axis (over all N experts), max-subtracted."""
    z = np.asarray(z, dtype=np.float64)
    m = np.max(z, axis=-1, keepdims=True)
    e = np.exp(z - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def topk_indices(z, k):
    """Indices of the k largest scores per row, largest first.

    Equal scores are ordered by the lower expert index (a stable sort of -z).
    Selecting on the logits is the same as selecting on the softmax
    probabilities, since the softmax is strictly increasing in each logit.
    """
    z = np.asarray(z, dtype=np.float64)
    order = np.argsort(-z, axis=-1, kind="stable")
    return order[..., :k]


def gates_softmax_of_topk(z, idx):
    """Gates as Softmax(TopK(z)): the scores outside the top-k are set to
    minus infinity and a softmax is taken, so only the kept k are non-zero
    (roadtointelligence.com router formula and "Tiny example")."""
    z = np.asarray(z, dtype=np.float64)
    masked = np.full_like(z, -np.inf)
    np.put_along_axis(masked, idx, np.take_along_axis(z, idx, axis=-1), axis=-1)
    g = softmax(masked)
    return np.take_along_axis(g, idx, axis=-1)


def gates_renormalised_probs(p, idx):
    """Gates as top-k probabilities divided by their sum
    (botmartz.com "Expert Routing"; matteuscruz.github.io "Architecture")."""
    kept = np.take_along_axis(np.asarray(p, dtype=np.float64), idx, axis=-1)
    return kept / np.sum(kept, axis=-1, keepdims=True)


def gates_raw_probs(p, idx):
    """Gates as the raw softmax probability of each kept expert, no
    renormalisation (codingnowai.in "Mixture of Experts", section "Code")."""
    return np.take_along_axis(np.asarray(p, dtype=np.float64), idx, axis=-1)


def route(x, W_g, b_g, k, renormalize=True):
    """Router + softmax + top-k (+ renormalise).  Returns (z, p, idx, w)."""
    z = router_logits(x, W_g, b_g)
    p = softmax(z)
    idx = topk_indices(z, k)
    w = gates_softmax_of_topk(z, idx) if renormalize else gates_raw_probs(p, idx)
    return z, p, idx, w


def topk_gap(z, k):
    """Score gap between the k-th and (k+1)-th largest score of each token
    (infinite when k == N).  Tokens with a gap below a threshold are near-ties
    whose top-k set may legitimately differ under another summation order."""
    z = np.asarray(z, dtype=np.float64)
    N = z.shape[-1]
    if k >= N:
        return np.full(z.shape[:-1], np.inf)
    s = -np.sort(-z, axis=-1)
    return s[..., k - 1] - s[..., k]


# ---------------------------------------------------------------------------
# capacity and the per-expert grouping of (token, slot) assignments
# ---------------------------------------------------------------------------

def expert_capacity(capacity_factor, T, N):
    """capacity factor x batch size / number of experts, rounded up."""
    return int(math.ceil(capacity_factor * T / N))


@dataclass
class Grouping:
    """Assignments grouped by expert.

    groups[e]  : list of (t, j) kept for expert e, in token-major order
    counts[e]  : assignments routed to e before capacity
    kept[e]    : assignments kept (min(counts[e], capacity))
    rank[t, j] : position of (t, j) among the assignments to its expert
    keep[t, j] : True when the assignment is within capacity
    """
    groups: list
    counts: np.ndarray
    kept: np.ndarray
    rank: np.ndarray
    keep: np.ndarray
    dropped: int = field(default=0)


def group_by_expert(idx, N, capacity=0):
    """Walk the assignments (t, j) in ascending token, then ascending slot;
    an assignment's rank is how many earlier assignments chose the same
    expert; it is kept when capacity <= 0 (unlimited) or rank < capacity."""
    idx = np.asarray(idx)
    T, k = idx.shape
    counts = np.zeros(N, dtype=np.int64)
    rank = np.zeros((T, k), dtype=np.int64)
    keep = np.zeros((T, k), dtype=bool)
    groups = [[] for _ in range(N)]
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            r = int(counts[e])
            counts[e] += 1
            rank[t, j] = r
            if capacity <= 0 or r < capacity:
                keep[t, j] = True
                groups[e].append((t, j))
    kept = np.array([len(g) for g in groups], dtype=np.int64)
    return Grouping(groups, counts, kept, rank, keep, int(counts.sum() - kept.sum()))


# ---------------------------------------------------------------------------
# experts and the layer
# ---------------------------------------------------------------------------

def activation(h, act):
    h = np.asarray(h, dtype=np.float64)
    if act == ACT_GELU_ERF:
        # nn.GELU() default: 0.5 * h * (1 + erf(h / sqrt(2)))
        return 0.5 * h * (1.0 + _erf(h / math.sqrt(2.0)))
    if act == ACT_RELU:
        return np.maximum(h, 0.0)
    raise ValueError(f"unknown activation {act}")


def expert_ffn(xr, W1, b1, W2, b2, act, round_hidden_bf16=False):
    """Linear(d, d_ff) -> activation -> Linear(d_ff, d) on the rows xr.

    With round_hidden_bf16 the hidden activation is rounded to bfloat16
    before the second Linear, the storage format of the hidden layer in the
    bf16 layer; everything else stays float64.
    """
    xr = np.asarray(xr, dtype=np.float64)
    h = xr @ np.asarray(W1, dtype=np.float64).T + np.asarray(b1, dtype=np.float64)
    h = activation(h, act)
    if round_hidden_bf16:
        h = round_to_bf16(h)
    return h @ np.asarray(W2, dtype=np.float64).T + np.asarray(b2, dtype=np.float64)


@dataclass
class LayerOutput:
    y: np.ndarray            # [len(tokens), d] float64 layer output
    tokens: np.ndarray       # token ids the rows of y belong to
    z: np.ndarray            # [T, N] router scores
    p: np.ndarray            # [T, N] router probabilities
    idx: np.ndarray          # [T, k] selected experts, largest first
    w: np.ndarray            # [T, k] gates
    grouping: Grouping
    mean_prob: np.ndarray    # [N]
    balance: float
    cv_squared: float = 0.0  # of the routed counts


def balance_statistic(p):
    """std(mean over tokens of the router probabilities)^2, torch.std's default
    unbiased estimator (botmartz.com "Load Balancing: The Hidden Challenge").
    Returns (mean_prob, balance); balance is 0 for a single expert."""
    m = np.mean(np.asarray(p, dtype=np.float64), axis=0)
    if m.shape[0] < 2:
        return m, 0.0
    return m, float(np.std(m, ddof=1) ** 2)


def cv_squared(counts):
    """Squared coefficient of variation of the per-expert counts: the unbiased
    variance over the N experts divided by the squared mean (matteuscruz.github.io
    "Load balancing: the core training challenge" names the coefficient of
    variation of the expert load; invest-in.ai "MoE - Mixture of Experts",
    "Common Usage Examples", names cv_squared(expert_counts); the variance
    estimator is torch's default, as in the balance statistic).  0 for a single
    expert or when nothing was routed."""
    c = np.asarray(counts, dtype=np.float64)
    if c.shape[0] < 2:
        return 0.0
    m = float(np.mean(c))
    if m == 0.0:
        return 0.0
    return float(np.var(c, ddof=1) / (m * m))


def moe_forward(x, W_g, b_g, W1, b1, W2, b2, *, k, act, capacity=0,
                renormalize=True, shared=None, round_hidden_bf16=False,
                tokens=None, idx_override=None):
    """The whole layer for the tokens listed in ``tokens`` (default: all).

    Routing, grouping and the statistics always cover all T tokens, because a
    token's capacity rank depends on every earlier token.  ``W1`` etc. may be
    any indexable of per-expert arrays (W1[e] is [d_ff, d]); experts are read
    one at a time.  ``shared`` is None or (W1s, b1s, W2s, b2s).
    ``idx_override`` replaces the top-k choice (used only for tokens whose
    k-th score gap is a near-tie); the gates are then taken for those experts.
    """
    x = np.asarray(x, dtype=np.float64)
    T = x.shape[0]
    N = np.asarray(b_g).shape[0]
    z = router_logits(x, W_g, b_g)
    p = softmax(z)
    idx = topk_indices(z, k) if idx_override is None else np.asarray(idx_override, dtype=np.int64)
    w = gates_softmax_of_topk(z, idx) if renormalize else gates_raw_probs(p, idx)
    grouping = group_by_expert(idx, N, capacity)
    mean_prob, balance = balance_statistic(p)

    tokens = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    pos = {int(t): i for i, t in enumerate(tokens)}
    y = np.zeros((len(tokens), x.shape[1]), dtype=np.float64)
    for e in range(N):
        rows = [(t, j) for (t, j) in grouping.groups[e] if t in pos]
        if not rows:
            continue
        ts = np.array([t for t, _ in rows])
        js = np.array([j for _, j in rows])
        o = expert_ffn(x[ts], W1[e], b1[e], W2[e], b2[e], act, round_hidden_bf16)
        for r, (t, j) in enumerate(zip(ts, js)):
            y[pos[int(t)]] += w[t, j] * o[r]
    if shared is not None:
        W1s, b1s, W2s, b2s = shared
        y += expert_ffn(x[tokens], W1s, b1s, W2s, b2s, act, round_hidden_bf16)
    return LayerOutput(y, tokens, z, p, idx, w, grouping, mean_prob, balance,
                       cv_squared(grouping.counts))


def moe_bruteforce(x, W_g, b_g, W1, b1, W2, b2, *, k, act, capacity=0,
                   renormalize=True, shared=None):
    """Every expert on every token, then mask and weight: the per-slot,
    per-expert loop of botmartz.com "Expert Routing" and codingnowai.in "Code"
    (output[mask] += weight[mask] * expert(x)[mask]), with the capacity mask
    applied on top.  For tiny inputs only."""
    x = np.asarray(x, dtype=np.float64)
    T, d = x.shape
    N = np.asarray(b_g).shape[0]
    z = router_logits(x, W_g, b_g)
    p = softmax(z)
    idx = topk_indices(z, k)
    if renormalize:
        w = gates_renormalised_probs(p, idx)
    else:
        w = gates_raw_probs(p, idx)
    keep = group_by_expert(idx, N, capacity).keep
    all_out = np.stack([expert_ffn(x, W1[e], b1[e], W2[e], b2[e], act) for e in range(N)])
    y = np.zeros((T, d))
    for j in range(k):
        for e in range(N):
            mask = (idx[:, j] == e) & keep[:, j]
            y[mask] += w[mask, j][:, None] * all_out[e][mask]
    if shared is not None:
        y += expert_ffn(x, *shared, act)
    return y


# ---------------------------------------------------------------------------
# expert-choice routing
# ---------------------------------------------------------------------------

def expert_choice_tokens(T, capacity):
    """Tokens each expert takes: the capacity, clamped to T; <= 0 means T."""
    return T if capacity <= 0 else min(int(capacity), T)


def expert_choice_select(p, C):
    """For every expert e, the C tokens with the largest p[t, e], the lower
    token index first among equal scores (matteuscruz.github.io "Load balancing:
    the core training challenge": each expert selects its top tokens).  Returns
    a list of N int arrays, each in ascending token order."""
    p = np.asarray(p, dtype=np.float64)
    T, N = p.shape
    sel = []
    for e in range(N):
        order = np.lexsort((np.arange(T), -p[:, e]))   # by score descending, then token
        sel.append(np.sort(order[:C]).astype(np.int64))
    return sel


def expert_choice_gap(p, C):
    """Per expert, the score gap between its C-th and (C+1)-th largest token
    (inf when C = T or C = 0)."""
    p = np.asarray(p, dtype=np.float64)
    T, N = p.shape
    gaps = np.full(N, np.inf)
    if 0 < C < T:
        srt = -np.sort(-p, axis=0)
        gaps = srt[C - 1] - srt[C]
    return gaps


@dataclass
class ExpertChoiceOutput:
    y: np.ndarray            # [len(tokens), d]
    tokens: np.ndarray
    z: np.ndarray            # [T, N]
    p: np.ndarray            # [T, N]
    sel: list                # N arrays of picked tokens, ascending
    gate: list               # N arrays: p[sel[e], e]
    token_picks: np.ndarray  # [T] experts that picked each token
    unpicked: int            # tokens no expert picked
    mean_prob: np.ndarray
    balance: float


def expert_choice_forward(x, W_g, b_g, W1, b1, W2, b2, *, capacity, act, shared=None,
                          round_hidden_bf16=False, tokens=None, sel_override=None):
    """The layer with expert-choice routing: router scores and softmax as in
    top-k routing, then every expert e runs its FFN on its C picked tokens and
    y[t] = sum over the experts that picked t of p[t, e] * expert_e(x[t])
    (+ the shared expert with weight 1).  ``sel_override`` replaces the
    selection (used only for experts whose C-th score gap is a near-tie)."""
    x = np.asarray(x, dtype=np.float64)
    T = x.shape[0]
    N = np.asarray(b_g).shape[0]
    z = router_logits(x, W_g, b_g)
    p = softmax(z)
    C = expert_choice_tokens(T, capacity)
    sel = expert_choice_select(p, C) if sel_override is None else \
        [np.asarray(s_, dtype=np.int64) for s_ in sel_override]
    gate = [p[s_, e] for e, s_ in enumerate(sel)]
    picks = np.zeros(T, dtype=np.int64)
    for s_ in sel:
        picks[s_] += 1
    mean_prob, balance = balance_statistic(p)
    tokens = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    pos = {int(t): i for i, t in enumerate(tokens)}
    y = np.zeros((len(tokens), x.shape[1]), dtype=np.float64)
    for e in range(N):
        ts = np.array([t for t in sel[e] if int(t) in pos], dtype=np.int64)
        if ts.size == 0:
            continue
        o = expert_ffn(x[ts], W1[e], b1[e], W2[e], b2[e], act, round_hidden_bf16)
        for r, t in enumerate(ts):
            y[pos[int(t)]] += p[t, e] * o[r]
    if shared is not None:
        W1s, b1s, W2s, b2s = shared
        y += expert_ffn(x[tokens], W1s, b1s, W2s, b2s, act, round_hidden_bf16)
    return ExpertChoiceOutput(y, tokens, z, p, sel, gate, picks, int((picks == 0).sum()),
                              mean_prob, balance)


# ---------------------------------------------------------------------------
# backward pass
# ---------------------------------------------------------------------------

def activation_grad(a, act):
    """d act / d a.  GELU(a) = a Phi(a), so GELU'(a) = Phi(a) + a phi(a) with
    Phi the normal CDF 0.5 (1 + erf(a / sqrt 2)) and phi its density."""
    a = np.asarray(a, dtype=np.float64)
    if act == ACT_GELU_ERF:
        cdf = 0.5 * (1.0 + _erf(a / math.sqrt(2.0)))
        pdf = np.exp(-0.5 * a * a) / math.sqrt(2.0 * math.pi)
        return cdf + a * pdf
    if act == ACT_RELU:
        return (a > 0.0).astype(np.float64)
    raise ValueError(f"unknown activation {act}")


def softmax_backward(p, dp):
    """Gradient through p = softmax(z) along the last axis: p (dp - <p, dp>)."""
    p = np.asarray(p, dtype=np.float64)
    dp = np.asarray(dp, dtype=np.float64)
    return p * (dp - np.sum(p * dp, axis=-1, keepdims=True))


@dataclass
class LayerGrads:
    dx: np.ndarray           # [T, d]
    dW_g: np.ndarray         # [N, d]
    db_g: np.ndarray         # [N]
    dW1: np.ndarray          # [N, d_ff, d]
    db1: np.ndarray          # [N, d_ff]
    dW2: np.ndarray          # [N, d, d_ff]
    db2: np.ndarray          # [N, d]
    dz: np.ndarray           # [T, N] gradient of the router scores
    dw: np.ndarray           # [T, k] gradient of the gates
    shared: tuple | None     # (dW1s, db1s, dW2s, db2s) or None


def expert_ffn_backward(xr, W1, b1, W2, b2, act, dO, round_hidden_bf16=False):
    """One expert's FFN backward on its rows xr given dO = d loss / d output:
    returns (dxr, dW1, db1, dW2, db2).  The hidden activation h that multiplies
    dO in dW2 is the one the forward fed to the second Linear (bf16-rounded
    with round_hidden_bf16)."""
    xr = np.asarray(xr, dtype=np.float64)
    W1 = np.asarray(W1, dtype=np.float64)
    W2 = np.asarray(W2, dtype=np.float64)
    a = xr @ W1.T + np.asarray(b1, dtype=np.float64)      # pre-activation
    h = activation(a, act)
    if round_hidden_bf16:
        h = round_to_bf16(h)
    dW2 = dO.T @ h                                        # [d, d_ff]
    db2 = dO.sum(axis=0)
    dh = dO @ W2                                          # [rows, d_ff]
    da = dh * activation_grad(a, act)
    dW1 = da.T @ xr                                       # [d_ff, d]
    db1 = da.sum(axis=0)
    dxr = da @ W1                                         # [rows, d]
    return dxr, dW1, db1, dW2, db2


def moe_backward(x, W_g, b_g, W1, b1, W2, b2, dy, *, k, act, capacity=0, renormalize=True,
                 shared=None, aux_weight=0.0, round_hidden_bf16=False, idx_override=None):
    """Gradients of total = <dy, y> + aux_weight * balance with respect to x
    and every parameter (botmartz.com "Load Balancing": total_loss = task_loss
    + 0.01 * balance_loss, with dy standing for d task_loss / d y).

    Steps, each the chain rule through the matching forward step:
      1. combine y[t] = sum_kept w[t,j] o[t,j] (+ shared): d o[t,j] = w[t,j] dy[t],
         d w[t,j] = <dy[t], o[t,j]> for kept (t, j), 0 for dropped ones;
      2. each expert's FFN on its kept rows (expert_ffn_backward);
      3. gates: renormalised, w = softmax over the k selected scores, so
         dz[selected] = w (dw - <w, dw>); raw, w = p[selected], so
         dp[selected] = dw and dz = p (dp - <p, dp>);
      4. balance = sum_e (m_e - 1/N)^2 / (N - 1), m_e = mean_t p[t,e]:
         d m_e = 2 (m_e - 1/N) / (N - 1), d p[t,e] = d m_e / T, through the softmax;
      5. router scores z = x W_g^T + b_g: dW_g = dz^T x, db_g = sum_t dz, dx += dz W_g.
    """
    x = np.asarray(x, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    W_g = np.asarray(W_g, dtype=np.float64)
    T, d = x.shape
    N = W_g.shape[0]
    z = router_logits(x, W_g, b_g)
    p = softmax(z)
    idx = topk_indices(z, k) if idx_override is None else np.asarray(idx_override, dtype=np.int64)
    w = gates_softmax_of_topk(z, idx) if renormalize else gates_raw_probs(p, idx)
    grouping = group_by_expert(idx, N, capacity)

    dx = np.zeros_like(x)
    dw = np.zeros((T, k))
    dW1, db1, dW2, db2 = [], [], [], []
    for e in range(N):
        rows = grouping.groups[e]
        W1e, W2e = np.asarray(W1[e], dtype=np.float64), np.asarray(W2[e], dtype=np.float64)
        if not rows:
            dW1.append(np.zeros_like(W1e)); db1.append(np.zeros(W1e.shape[0]))
            dW2.append(np.zeros_like(W2e)); db2.append(np.zeros(W2e.shape[0]))
            continue
        ts = np.array([t for t, _ in rows])
        js = np.array([j for _, j in rows])
        o = expert_ffn(x[ts], W1e, b1[e], W2e, b2[e], act, round_hidden_bf16)
        dw[ts, js] = np.sum(dy[ts] * o, axis=1)                       # step 1
        dO = w[ts, js][:, None] * dy[ts]
        dxr, gW1, gb1, gW2, gb2 = expert_ffn_backward(x[ts], W1e, b1[e], W2e, b2[e], act, dO,
                                                      round_hidden_bf16)   # step 2
        np.add.at(dx, ts, dxr)
        dW1.append(gW1); db1.append(gb1); dW2.append(gW2); db2.append(gb2)
    shared_grads = None
    if shared is not None:
        dxs, gW1, gb1, gW2, gb2 = expert_ffn_backward(x, *shared, act, dy, round_hidden_bf16)
        dx += dxs
        shared_grads = (gW1, gb1, gW2, gb2)

    dz = np.zeros((T, N))                                             # step 3
    if renormalize:
        dz_sel = w * (dw - np.sum(w * dw, axis=1, keepdims=True))
        np.put_along_axis(dz, idx, dz_sel, axis=1)
    else:
        dp = np.zeros((T, N))
        np.put_along_axis(dp, idx, dw, axis=1)
        dz += softmax_backward(p, dp)
    if aux_weight != 0.0 and N > 1 and T > 0:                         # step 4
        m = p.mean(axis=0)
        dm = aux_weight * 2.0 * (m - 1.0 / N) / (N - 1)
        dz += softmax_backward(p, np.broadcast_to(dm / T, p.shape))
    dW_g = dz.T @ x                                                   # step 5
    db_g = dz.sum(axis=0)
    dx += dz @ W_g
    return LayerGrads(dx, dW_g, db_g, np.stack(dW1), np.stack(db1), np.stack(dW2),
                      np.stack(db2), dz, dw, shared_grads)
