"""The work splits the kernels use, restated on the host and checked against
the plain definitions in the oracle (CPU only).  They pin the reasoning behind
a split, not the CUDA code, which the GPU parity tests compare with the oracle:

- the 64-expert router epilogue selects each part's k best of 16 scores and
  merges the four lists by (score descending, expert ascending): the same
  experts, in the same order, as one scan over all 64 scores;
- the two-launch counting sort ranks an assignment within its warp (earlier
  equal experts among the warp's 32), adds its warp's base inside the block
  (a scan over the block's warps) and its block's base (a sum over earlier
  blocks): the stable rank of the assignment among its expert's assignments in
  token-major order, which with the capacity decides what is kept."""

import numpy as np
import pytest

from oracle import moe_oracle as O


def split_topk(z, k, parts=4):
    """Per row: each part's k best (larger score first, then lower expert),
    then k rounds over the list heads with the same order."""
    T, N = z.shape
    w = N // parts
    out = np.empty((T, k), np.int64)
    for t in range(T):
        lists = []
        for p in range(parts):
            cols = list(range(p * w, (p + 1) * w))
            cols.sort(key=lambda e: (-z[t, e], e))
            lists.append(cols[:k])
        heads = [0] * parts
        for j in range(k):
            best = None
            for p in range(parts):
                if heads[p] >= len(lists[p]):
                    continue
                e = lists[p][heads[p]]
                if best is None or (z[t, e], -e) > (z[t, best[1]], -best[1]):
                    best = (p, e)
            heads[best[0]] += 1
            out[t, j] = best[1]
    return out


@pytest.mark.parametrize("k", [1, 2, 4, 8])
def test_router_split_topk_equals_one_scan(k):
    rng = np.random.default_rng(100 + k)
    z = rng.normal(0, 1, (300, 64))
    # ties inside and across the parts, and -inf scores
    z[:100] = np.round(z[:100] * 2) / 2
    z[100:120, 5::7] = -np.inf
    z[120:140] = 0.25
    np.testing.assert_array_equal(split_topk(z, k), O.topk_indices(z, k))


def two_level_ranks(idx, N, block=1024, warp=32):
    """Rank of each assignment as the two-launch sort forms it."""
    a_all = np.asarray(idx).reshape(-1)
    A = a_all.size
    nblk = (A + block - 1) // block
    counts = np.zeros((nblk, N), np.int64)
    local = np.empty(A, np.int64)
    for b in range(nblk):
        a0, a1 = b * block, min(A, (b + 1) * block)
        nw = (a1 - a0 + warp - 1) // warp
        wc = np.zeros((nw, N), np.int64)
        within = np.empty(a1 - a0, np.int64)
        for w in range(nw):
            ids = a_all[a0 + w * warp: min(a1, a0 + (w + 1) * warp)]
            for lane, e in enumerate(ids):
                within[w * warp + lane] = np.count_nonzero(ids[:lane] == e)
                wc[w, e] += 1
        wbase = np.cumsum(wc, axis=0) - wc           # exclusive scan over warps
        for i in range(a1 - a0):
            local[a0 + i] = wbase[i // warp, a_all[a0 + i]] + within[i]
        counts[b] = wc.sum(axis=0)
    bbase = np.cumsum(counts, axis=0) - counts       # exclusive sum over blocks
    ranks = np.array([bbase[a // block, a_all[a]] + local[a] for a in range(A)])
    return ranks.reshape(np.asarray(idx).shape), counts.sum(axis=0)


@pytest.mark.parametrize("T,k,N,cap", [(1500, 2, 8, 0), (700, 4, 40, 60), (333, 8, 300, 7),
                                       (2500, 1, 16, 100)])
def test_two_level_ranks_equal_the_stable_order(T, k, N, cap):
    rng = np.random.default_rng(T + N)
    # skewed routing, so that experts fill up and the capacity bites
    p = rng.dirichlet(np.full(N, 0.3))
    idx = np.stack([rng.choice(N, size=k, replace=False, p=p) for _ in range(T)])
    ranks, totals = two_level_ranks(idx, N)
    g = O.group_by_expert(idx, N, cap)
    np.testing.assert_array_equal(ranks, g.rank)
    np.testing.assert_array_equal(totals, g.counts)
    keep = (ranks < cap) if cap > 0 else np.ones_like(ranks, bool)
    np.testing.assert_array_equal(keep, g.keep.astype(bool))
