"""Comparison of the CUDA path with the CPU oracle on the same seeded inputs.

Bars (per-token row error e_t = ||y_gpu[t] - y_ref[t]||_2 / max(||y_ref[t]||_2, 1e-6)):
  fp32 layer: max_t e_t <= 1e-4;  bf16 layer: max_t e_t <= 2e-2.
Top-k sets, counts, kept counts, group order and the dropped set are compared
exactly.  A token whose oracle score gap between the k-th and (k+1)-th expert
is below 1e-4 may pick another set; a token with a gap below 1e-4 inside its
kept k may order them differently.  For the rest of the comparison the oracle
is re-run with the GPU's choice for every token (the same choice as the
oracle's own wherever it is not a near-tie).
"""

from __future__ import annotations

import os

import numpy as np
import torch

from oracle import moe_oracle as O

# threads that each run the single-threaded oracle on their own token rows
WORKERS = max(1, min(48, os.cpu_count() or 1))

TIE_EPS = 1e-4
TOL = {0: 1e-4, 1: 2e-2}          # by dtype code: fp32, bf16
GATE_RTOL = 1e-5
MEAN_PROB_RTOL = 1e-5
BALANCE_RTOL = 1e-4
CV_RTOL = 1e-7             # one fp32 rounding of an almost exact fp64 value


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def host_tensors(tensors: dict) -> dict:
    """Host copies of a layer's tensors in their storage dtype (the oracle reads
    bf16 values as they are stored)."""
    return {n: v.detach().cpu() for n, v in tensors.items()}


def oracle_layer(cfg, th: dict, k=None) -> O.Layer:
    shared = tuple(th[n] for n in ("W1s", "b1s", "W2s", "b2s")) if cfg.d_ff_shared else None
    return O.Layer(th["x"], th["W_g"], th["b_g"], th["W1"], th["b1"], th["W2"], th["b2"],
                   k=cfg.top_k if k is None else k, act=cfg.act, shared=shared,
                   round_hidden_bf16=(cfg.dtype == 1))


def near_tie_sets(z: np.ndarray, k: int):
    """(set_tie, order_tie) boolean masks over tokens."""
    N = z.shape[1]
    s = -np.sort(-z, axis=1)
    set_tie = np.zeros(z.shape[0], dtype=bool)
    if k < N:
        set_tie = (s[:, k - 1] - s[:, k]) < TIE_EPS
    order_tie = np.zeros(z.shape[0], dtype=bool)
    if k > 1:
        order_tie = np.any(np.diff(-s[:, :k], axis=1) < TIE_EPS, axis=1)
    return set_tie, order_tie


def row_errors(y_gpu: np.ndarray, y_ref: np.ndarray) -> np.ndarray:
    num = np.linalg.norm(y_gpu - y_ref, axis=1)
    den = np.maximum(np.linalg.norm(y_ref, axis=1), 1e-6)
    return num / den


def check_routing(wl_dtype, cfg, tensors, out, z_ref, report, z_gpu=None):
    """Top-k, gates: exact / near-tie rules above.  Returns the GPU top-k."""
    k = cfg.top_k
    idx_gpu = out.topk_idx.cpu().numpy().astype(np.int64)
    w_gpu = out.topk_w.cpu().numpy().astype(np.float64)
    idx_ref = O.topk_indices(z_ref, k)
    set_tie, order_tie = near_tie_sets(z_ref, k)
    same_set = np.all(np.sort(idx_gpu, 1) == np.sort(idx_ref, 1), axis=1)
    bad_set = ~same_set & ~set_tie
    assert not bad_set.any(), f"top-k set differs for tokens {np.nonzero(bad_set)[0][:10]}"
    same_order = np.all(idx_gpu == idx_ref, axis=1)
    bad_order = same_set & ~same_order & ~order_tie & ~set_tie
    assert not bad_order.any(), f"top-k order differs for tokens {np.nonzero(bad_order)[0][:10]}"
    # gates for the GPU's choice.  (a) From the GPU's own scores, in float64:
    # checks the softmax / renormalisation arithmetic to fp32 rounding.
    # (b) From the oracle's scores: a softmax moves each gate by at most a
    # relative 2 max|dz| when its scores move by dz, so the bar is the
    # measured score error times two (plus fp32 rounding).
    def gates(z):
        if cfg.renormalize:
            return O.gates_softmax_of_topk(z, idx_gpu)
        return O.gates_raw_probs(O.softmax(z), idx_gpu)

    if z_gpu is not None:
        np.testing.assert_allclose(w_gpu, gates(z_gpu), rtol=GATE_RTOL, atol=1e-7)
        dz = float(np.abs(z_gpu - z_ref).max())
    else:
        dz = 0.0
    report["gate_rtol_from_scores"] = 2.0 * dz + GATE_RTOL
    np.testing.assert_allclose(w_gpu, gates(z_ref), rtol=2.0 * dz + GATE_RTOL, atol=1e-7)
    report["near_tie_tokens"] = int(set_tie.sum())
    report["order_tie_tokens"] = int(order_tie.sum())
    return idx_gpu


def check_layer(wl, cfg, tensors, out, tokens=None, capacity=None, check_logits=True,
                th=None, L=None):
    """Full comparison of one moe_forward against the oracle.  Returns
    (report, oracle LayerOutput for `tokens`)."""
    report = {}
    th = host_tensors(tensors) if th is None else th
    L = oracle_layer(cfg, th) if L is None else L
    z_ref = L.logits(WORKERS)
    zg = None
    if check_logits and out.logits is not None:
        # fp32 sums of d products: the statistical rounding error is about
        # sqrt(d) * 2^-24 * |partial sums|, ~1e-6 of the largest score here;
        # the bar leaves a 10x margin.
        zg = out.logits.cpu().numpy().astype(np.float64)
        err = np.abs(zg - z_ref).max() / max(np.abs(z_ref).max(), 1e-30) if zg.size else 0.0
        report["logit_max_rel"] = float(err)
        assert err < 1e-5, f"router scores differ: {err}"
    idx_gpu = check_routing(cfg.dtype, cfg, tensors, out, z_ref, report, z_gpu=zg)

    cap = cfg.capacity if capacity is None else capacity
    r = L.route(cap, bool(cfg.renormalize), idx_gpu, workers=WORKERS, z=z_ref)
    g = r.grouping()
    # counts and drops: exact
    np.testing.assert_array_equal(out.counts.cpu().numpy(), g.counts)
    np.testing.assert_array_equal(out.kept.cpu().numpy(), g.kept)
    assert int(out.dropped.cpu().item()) == g.dropped
    # statistics
    np.testing.assert_allclose(out.mean_prob.cpu().numpy(), r.mean_prob,
                               rtol=MEAN_PROB_RTOL, atol=1e-8)
    bal = float(out.balance.cpu().item())
    assert abs(bal - r.balance) <= BALANCE_RTOL * abs(r.balance) + 1e-9, \
        f"balance {bal} vs {r.balance}"
    if out.cv_squared is not None:
        # exact integer sums, then one fp64 quotient rounded to fp32
        cv = float(out.cv_squared.cpu().item())
        assert abs(cv - r.cv_squared) <= CV_RTOL * abs(r.cv_squared), \
            f"cv_squared {cv} vs {r.cv_squared}"
    # output rows
    rows = np.arange(cfg.T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    y_ref = L.combine_rows(r, rows, WORKERS)
    ref = O.LayerOutput(y_ref, rows, r.z, r.p, r.idx, r.w, g, r.mean_prob, r.balance,
                        r.cv_squared)
    y_gpu = out.y.float().cpu().numpy().astype(np.float64)
    e = row_errors(y_gpu[rows], y_ref)
    report["rows_compared"] = int(len(rows))
    report["max_row_rel_l2"] = float(e.max()) if e.size else 0.0
    report["tensor_rel_l2"] = float(np.linalg.norm(y_gpu[rows] - y_ref) /
                                    max(np.linalg.norm(y_ref), 1e-30)) if e.size else 0.0
    tol = TOL[cfg.dtype]
    assert report["max_row_rel_l2"] <= tol, \
        f"max row rel L2 {report['max_row_rel_l2']} > {tol} (token {rows[int(np.argmax(e))]})"
    # fully dropped tokens without a shared expert: exactly zero
    if not cfg.d_ff_shared:
        dropped_all = ~g.keep.any(axis=1)
        for t in rows[dropped_all[rows]]:
            assert np.all(y_gpu[t] == 0.0), f"dropped token {t} is not zero"
        report["fully_dropped_checked"] = int(dropped_all[rows].sum())
    return report, ref


def tile_cover(live: int, rng, tile=128):
    """Positions in a group of `live` rows that visit every `tile`-row m-tile:
    each tile's first and last live row and one at random in between."""
    pos = set()
    for s0 in range(0, live, tile):
        s1 = min(live, s0 + tile) - 1
        pos |= {s0, s1, int(rng.integers(s0, s1 + 1))}
    return sorted(pos)


def tile_cover_tokens(grouping, T, seed, shared=False):
    """Tokens whose grouped rows visit every 128-row m-tile of every expert
    group (and of the shared group: every token is a row of it)."""
    rng = np.random.default_rng(seed)
    toks = set()
    for e, grp in enumerate(grouping.groups):
        for i in tile_cover(len(grp), rng):
            toks.add(grp[i][0])
    if shared:
        toks |= set(tile_cover(T, rng))
    return np.array(sorted(toks), dtype=np.int64)


def check_grouped_rows(cfg, L, grouping, offsets, H, Yp, seed, all_shared=False):
    """Grouped hidden rows H and expert outputs Yp against the oracle's expert
    FFN on the same token, at positions that visit every 128-row m-tile of
    every group (the first and last live row of each tile and one more), and
    every row of the shared group when all_shared.  Per-row relative L2 within
    the layer's bar.  Returns a report."""
    rng = np.random.default_rng(seed)
    off = offsets.cpu().numpy().astype(np.int64)
    N, T = cfg.n_experts, cfg.T
    jobs = []                                   # (group, positions, tokens)
    for e in range(N):
        grp = grouping.groups[e]
        pos = tile_cover(len(grp), rng)
        if pos:
            jobs.append((e, np.array(pos), np.array([grp[i][0] for i in pos], np.int64)))
    if cfg.d_ff_shared and T:
        pos = np.arange(T) if all_shared else np.array(tile_cover(T, rng))
        # the shared group holds token t at row offsets[N] + t
        for lo in range(0, len(pos), 256):
            jobs.append((N, pos[lo:lo + 256], pos[lo:lo + 256].astype(np.int64)))
    from concurrent.futures import ThreadPoolExecutor

    def run(job):
        e, pos, toks = job
        _, h, o = L.expert_rows(e, toks, want=("h", "o"))
        rows = off[e] + pos
        hg = H[torch.from_numpy(rows)].float().cpu().numpy().astype(np.float64)
        og = Yp[torch.from_numpy(rows)].float().cpu().numpy().astype(np.float64)
        return e, row_errors(hg, h), row_errors(og, o)

    with ThreadPoolExecutor(max_workers=WORKERS) as ex:
        res = list(ex.map(run, jobs))
    tol = TOL[cfg.dtype]
    worst_h = max((float(eh.max()) for _, eh, _ in res), default=0.0)
    worst_o = max((float(eo.max()) for _, _, eo in res), default=0.0)
    n_rows = sum(len(eo) for _, _, eo in res)
    for e, eh, eo in res:
        assert eh.max() <= tol, f"group {e}: hidden row error {eh.max()}"
        assert eo.max() <= tol, f"group {e}: expert output row error {eo.max()}"
    return {"grouped_rows_compared": n_rows, "max_hidden_row_rel_l2": worst_h,
            "max_expert_row_rel_l2": worst_o}


def check_grouping(cfg, tensors_x, offsets, row_token, token_row, Xp, ref_grouping, T):
    """Permutation layout: offsets padded per group, rows in token order, the
    copied rows equal x, dropped slots -1."""
    N, k = cfg.n_experts, cfg.top_k
    off = offsets.cpu().numpy().astype(np.int64)
    rt = row_token.cpu().numpy().astype(np.int64)
    tr = token_row.cpu().numpy().astype(np.int64).reshape(T, k)
    kept = ref_grouping.kept
    for e in range(N):
        assert off[e + 1] - off[e] == -(-kept[e] // 128) * 128
        want = [t for t, _ in ref_grouping.groups[e]]
        got = rt[off[e]: off[e] + kept[e]].tolist()
        assert got == want, f"expert {e}: group order differs"
        assert np.all(rt[off[e] + kept[e]: off[e + 1]] == -1)
        for r, (t, j) in enumerate(ref_grouping.groups[e]):
            assert tr[t, j] == off[e] + r
    assert np.all(tr[~ref_grouping.keep] == -1)
    shared_rows = -(-T // 128) * 128 if cfg.d_ff_shared else 0
    assert off[N + 1] == off[N] + shared_rows
    # copied rows: sample up to 64 kept rows and every shared row
    x = tensors_x
    xs = Xp[: off[N + 1]]
    rows = [r for r in range(off[N]) if rt[r] >= 0]
    rng = np.random.default_rng(0)
    for r in rng.choice(rows, size=min(64, len(rows)), replace=False) if rows else []:
        assert torch.equal(xs[int(r)], x[int(rt[r])])
    if cfg.d_ff_shared:
        assert torch.equal(xs[off[N]: off[N] + T], x)


# ---- expert-choice routing -----------------------------------------------------------

EC_GATE_RTOL = 1e-5


def check_ec_layer(wl, cfg, tensors, out, tokens=None, th=None, L=None):
    """Full comparison of one moe_ec_forward against the oracle.

    The selection is exact for every expert whose oracle gap between its C-th
    and (C+1)-th score exceeds what the GPU's fp32 scores can move p by
    (4 max|dz| max_t p + 1e-7: a softmax moves p by at most 2 p max|dz|, on
    both sides of the cut); for the others the GPU's set must still take every
    token clearly above the cut and none clearly below.  The oracle then runs
    on the GPU's selection."""
    report = {}
    th = host_tensors(tensors) if th is None else th
    L = oracle_layer(cfg, th, k=1) if L is None else L
    z_ref = L.logits(WORKERS)
    p_ref = O.softmax(z_ref)
    T, N = z_ref.shape
    C = O.expert_choice_tokens(T, cfg.capacity)
    dz = 0.0
    if out.logits is not None:
        zg = out.logits.cpu().numpy().astype(np.float64)
        dz = float(np.abs(zg - z_ref).max()) if T else 0.0
        err = dz / max(np.abs(z_ref).max(), 1e-30) if T else 0.0
        report["logit_max_rel"] = float(err)
        assert err < 1e-5, f"router scores differ: {err}"
    sel_gpu = out.ec_token.cpu().numpy().astype(np.int64).reshape(N, C)
    gate_gpu = out.ec_gate.cpu().numpy().astype(np.float64).reshape(N, C)
    sel_ref = O.expert_choice_select(p_ref, C)
    gaps = O.expert_choice_gap(p_ref, C)
    eps = 4.0 * dz * (p_ref.max(axis=0) if T else np.zeros(N)) + 1e-7
    near = gaps < eps
    sel_use = []
    for e in range(N):
        g = sel_gpu[e]
        assert np.all((g >= 0) & (g < T)) and np.all(np.diff(g) > 0), f"expert {e}: bad picks"
        if not near[e]:
            np.testing.assert_array_equal(g, sel_ref[e], err_msg=f"expert {e} picks differ")
        else:
            col = p_ref[:, e]
            thr = -np.sort(-col)[C - 1]
            inset = np.zeros(T, dtype=bool)
            inset[g] = True
            assert np.all(inset[col > thr + eps[e]]), f"expert {e}: misses a clear pick"
            assert not np.any(inset[col < thr - eps[e]]), f"expert {e}: takes a clear reject"
        sel_use.append(g)
        if C:
            np.testing.assert_allclose(gate_gpu[e], p_ref[g, e], rtol=2.0 * dz + EC_GATE_RTOL,
                                       atol=1e-7, err_msg=f"expert {e} gates")
    report["near_tie_experts"] = int(near.sum())
    sel = np.stack(sel_use) if N else np.empty((0, C), np.int64)
    picks, unpicked = O.expert_choice_picks(T, sel)
    np.testing.assert_array_equal(out.token_picks.cpu().numpy(), picks)
    assert int(out.unpicked.cpu().item()) == unpicked
    mean_prob, balance = O.balance_statistic(p_ref)
    np.testing.assert_allclose(out.mean_prob.cpu().numpy(), mean_prob,
                               rtol=MEAN_PROB_RTOL, atol=1e-8)
    bal = float(out.balance.cpu().item())
    assert abs(bal - balance) <= BALANCE_RTOL * abs(balance) + 1e-9, \
        f"balance {bal} vs {balance}"
    rows = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    y_ref = L.ec_combine_rows(C, sel, p_ref, rows, WORKERS)
    ref = O.ExpertChoiceOutput(y_ref, rows, z_ref, p_ref, sel_use,
                               [p_ref[s_, e] for e, s_ in enumerate(sel_use)], picks,
                               unpicked, mean_prob, balance)
    y_gpu = out.y.float().cpu().numpy().astype(np.float64)
    e = row_errors(y_gpu[rows], y_ref)
    report["rows_compared"] = int(len(rows))
    report["max_row_rel_l2"] = float(e.max()) if e.size else 0.0
    tol = TOL[cfg.dtype]
    assert report["max_row_rel_l2"] <= tol, \
        f"max row rel L2 {report['max_row_rel_l2']} > {tol} (token {rows[int(np.argmax(e))]})"
    if not cfg.d_ff_shared:
        lonely = ref.token_picks[rows] == 0
        for t in rows[lonely]:
            assert np.all(y_gpu[t] == 0.0), f"unpicked token {t} is not zero"
        report["unpicked_checked"] = int(lonely.sum())
    return report, ref
