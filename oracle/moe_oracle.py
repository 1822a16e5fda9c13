"""CPU oracle for the sparse Mixture-of-Experts FFN layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the library path imports this module:
only the tests, the smoke check in ``__graft_entry__`` and the CPU-baseline leg
of ``bench.py`` may call it.  It shares no code with the CUDA path.

The arithmetic is in ``moe_oracle.cpp``: plain single-threaded C++ in float64,
each function the plain definition of one step of the layer, citing the page
passage it follows (router scores, softmax, top-k, gates, grouping with a
capacity, expert FFNs, combine, balance statistic and cv^2, expert-choice
routing, and the backward pass of task + alpha * balance).  This module only
marshals arrays to it through ctypes and arranges the results in the shapes the
tests use.  Inputs may be numpy arrays or CPU torch tensors in float32,
bfloat16 or float64: the C++ side reads each element in its own format and
upcasts it exactly.

``workers`` (where offered) splits independent token rows over that many
threads, each running the single-threaded oracle on its own rows; the results
are those of one call.
"""

from __future__ import annotations

import ctypes as C
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

ACT_GELU_ERF = 0
ACT_RELU = 1
_F32, _BF16, _F64 = 0, 1, 2

_HERE = os.path.dirname(os.path.abspath(__file__))


def threads() -> int:
    """Host threads one oracle call uses."""
    return 1


def describe() -> str:
    return "plain single-threaded C++ oracle, float64"


# ---------------------------------------------------------------------------
# the shared library

class _Tensor(C.Structure):
    _fields_ = [("data", C.c_void_p), ("dtype", C.c_int32), ("reserved", C.c_int32)]


_TENSORS = ("x", "W_g", "b_g", "W1", "b1", "W2", "b2", "W1s", "b1s", "W2s", "b2s")


class _Layer(C.Structure):
    _fields_ = ([(n, C.c_int64) for n in ("T", "d", "f", "N", "k", "f_shared")] +
                [("act", C.c_int32), ("round_hidden_bf16", C.c_int32)] +
                [(n, _Tensor) for n in _TENSORS])


_lib = None


def lib() -> C.CDLL:
    global _lib
    if _lib is None:
        from . import build
        L = C.CDLL(build.build())
        P, I64, I32, D = C.c_void_p, C.c_int64, C.c_int32, C.c_double
        LP = C.POINTER(_Layer)
        sig = {
            "orc_round_bf16_array": (None, [P, P, I64]),
            "orc_activation": (I32, [I32, P, P, I64]),
            "orc_activation_grad": (I32, [I32, P, P, I64]),
            "orc_router_logits": (I32, [LP, I64, I64, P]),
            "orc_softmax_rows": (I32, [I64, I64, P, P]),
            "orc_topk": (I32, [I64, I64, I64, P, P]),
            "orc_topk_gap": (I32, [I64, I64, I64, P, P]),
            "orc_gates_softmax_of_topk": (I32, [I64, I64, I64, P, P, P]),
            "orc_gates_renormalised_probs": (I32, [I64, I64, I64, P, P, P]),
            "orc_gates_raw_probs": (I32, [I64, I64, I64, P, P, P]),
            "orc_capacity": (I64, [D, I64, I64]),
            "orc_group": (I64, [I64, I64, I64, I64, P, P, P, P, P, P, P]),
            "orc_balance": (I32, [I64, I64, P, P, P]),
            "orc_cv_squared": (D, [I64, P]),
            "orc_route": (I32, [LP, I64, I32, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P,
                                P]),
            "orc_expert_rows": (I32, [LP, I64, P, I64, P, P, P]),
            "orc_combine_rows": (I32, [LP, P, P, P, P, I64, P]),
            "orc_bruteforce": (I32, [LP, I64, I32, P]),
            "orc_ec_tokens": (I64, [I64, I64]),
            "orc_ec_select": (I32, [I64, I64, I64, P, P]),
            "orc_ec_gap": (I32, [I64, I64, I64, P, P]),
            "orc_ec_picks": (I64, [I64, I64, I64, P, P]),
            "orc_ec_combine_rows": (I32, [LP, I64, P, P, P, I64, P]),
            "orc_backward": (I32, [LP, I64, I32, P, _Tensor, D] + [P] * 13),
            "orc_expert_weight_grads": (I32, [LP, I64, P, P, I64, _Tensor, P, I64, P, P, P,
                                              P]),
            "orc_token_grads": (I32, [LP, I32, P, P, P, P, _Tensor, D, P, I64, P, P, P]),
            "orc_router_weight_grads": (I32, [LP, P, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ok(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid argument")


# ---------------------------------------------------------------------------
# marshalling

def _host(a):
    """(C-contiguous host array, format code) of a in its own number format:
    float32, bfloat16 (its raw 16-bit patterns) or float64; anything else as
    float64."""
    try:
        import torch
    except ImportError:                                     # pragma: no cover
        torch = None
    if torch is not None and isinstance(a, torch.Tensor):
        t = a.detach()
        if t.device.type != "cpu":
            t = t.cpu()
        t = t.contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16), _BF16
        if t.dtype == torch.float32:
            return t.numpy(), _F32
        return t.to(torch.float64).numpy(), _F64
    if isinstance(a, (list, tuple)):          # per-expert pieces: stacked as float64
        a = np.stack([_values(v) for v in a])
    a = np.asarray(a)
    if a.dtype == np.float32:
        return np.ascontiguousarray(a), _F32
    return np.ascontiguousarray(a, dtype=np.float64), _F64


def _values(a):
    """The values of a as a float64 array (bfloat16 is the upper half of a float32)."""
    arr, code = _host(a)
    if code == _BF16:
        return (arr.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return arr.astype(np.float64)


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


def _p(a):
    return None if a is None else a.ctypes.data


def _shape(a):
    return tuple(a.shape) if a is not None else None


def _chunks(n, parts):
    parts = max(1, min(parts, n))
    bounds = np.linspace(0, n, parts + 1).astype(np.int64)
    return [(int(bounds[i]), int(bounds[i + 1])) for i in range(parts) if bounds[i] < bounds[i + 1]]


def _parallel(fn, n, workers):
    """fn(lo, hi) over row ranges covering [0, n), on up to `workers` threads
    (ctypes drops the GIL for the duration of each oracle call)."""
    ranges = _chunks(n, workers)
    if len(ranges) <= 1:
        for lo, hi in ranges:
            fn(lo, hi)
        return
    with ThreadPoolExecutor(max_workers=len(ranges)) as ex:
        for fut in [ex.submit(fn, lo, hi) for lo, hi in ranges]:
            fut.result()


class Layer:
    """One layer's tensors marshalled once for the C++ oracle.

    x [T, d]; W_g [N, d]; b_g [N]; W1 [N, f, d]; b1 [N, f]; W2 [N, d, f];
    b2 [N, d]; shared = (W1s [fs, d], b1s, W2s [d, fs], b2s) or None.  Any of the
    router or expert tensors may be None for calls that do not read them."""

    def __init__(self, x, W_g=None, b_g=None, W1=None, b1=None, W2=None, b2=None, *, k=1,
                 act=ACT_GELU_ERF, shared=None, round_hidden_bf16=False):
        self._keep = []
        ts = {}
        for name, a in zip(_TENSORS, (x, W_g, b_g, W1, b1, W2, b2) +
                           (tuple(shared) if shared is not None else (None,) * 4)):
            if a is None:
                ts[name] = _Tensor(None, _F64, 0)
                continue
            arr, code = _host(a)
            self._keep.append(arr)
            ts[name] = _Tensor(arr.ctypes.data, code, 0)
        T, d = _shape(x)
        if b_g is not None:
            N = _shape(b_g)[0]
        elif W1 is not None:
            N = len(W1) if isinstance(W1, (list, tuple)) else _shape(W1)[0]
        else:
            N = 1
        f = 1
        if W1 is not None:
            f = _host(W1[0])[0].shape[0] if isinstance(W1, (list, tuple)) else _shape(W1)[-2]
        fs = _shape(shared[0])[0] if shared is not None else 0
        self.T, self.d, self.f, self.N, self.k, self.fs = int(T), int(d), int(f), int(N), \
            int(k), int(fs)
        self.act = int(act)
        self.c = _Layer(self.T, self.d, self.f, self.N, self.k, self.fs, self.act,
                        int(bool(round_hidden_bf16)), *[ts[n] for n in _TENSORS])

    def ref(self):
        return C.byref(self.c)

    # ---- router and routing
    def logits(self, workers=1):
        z = np.empty((self.T, self.N))

        def run(lo, hi):
            _ok(lib().orc_router_logits(self.ref(), lo, hi, _p(z[lo:hi])), "router")
        _parallel(run, self.T, workers)
        return z

    def route(self, capacity=0, renormalize=True, idx_override=None, workers=1, z=None):
        """Returns a Routing of all T tokens (z: the scores, when already computed)."""
        T, N, k = self.T, self.N, self.k
        z = self.logits(workers) if z is None else _f64(z)
        r = Routing(z=np.empty((T, N)), p=np.empty((T, N)), idx=np.empty((T, k), np.int64),
                    w=np.empty((T, k)), counts=np.empty(N, np.int64),
                    kept=np.empty(N, np.int64), rank=np.empty((T, k), np.int64),
                    keep=np.empty((T, k), np.uint8), order=np.empty(T * k, np.int64),
                    group_start=np.empty(N + 1, np.int64), mean_prob=np.empty(N))
        dropped = C.c_int64()
        bal = C.c_double()
        cv = C.c_double()
        ov = _i64(idx_override) if idx_override is not None else None
        _ok(lib().orc_route(self.ref(), int(capacity), int(bool(renormalize)), _p(ov), _p(z),
                            _p(r.z), _p(r.p), _p(r.idx), _p(r.w), _p(r.counts), _p(r.kept),
                            _p(r.rank), _p(r.keep), _p(r.order), _p(r.group_start),
                            C.byref(dropped), _p(r.mean_prob), C.byref(bal), C.byref(cv)),
            "route")
        r.dropped, r.balance, r.cv_squared = int(dropped.value), float(bal.value), \
            float(cv.value)
        return r

    # ---- experts and the layer
    def expert_rows(self, e, tokens, want=("o",)):
        """(pre, h, o) of expert e (e == N: shared) on x[tokens]; only the
        requested ones are computed, the others are None."""
        tok = _i64(tokens)
        fe = self.fs if e == self.N else self.f
        pre = np.empty((len(tok), fe)) if "pre" in want else None
        h = np.empty((len(tok), fe)) if "h" in want else None
        o = np.empty((len(tok), self.d)) if "o" in want else None
        _ok(lib().orc_expert_rows(self.ref(), int(e), _p(tok), len(tok), _p(pre), _p(h), _p(o)),
            "expert_rows")
        return pre, h, o

    def combine_rows(self, routing, tokens, workers=1):
        tok = _i64(tokens)
        y = np.empty((len(tok), self.d))

        def run(lo, hi):
            _ok(lib().orc_combine_rows(self.ref(), _p(routing.idx), _p(routing.w),
                                       _p(routing.keep), _p(tok[lo:hi]), hi - lo, _p(y[lo:hi])),
                "combine_rows")
        _parallel(run, len(tok), workers)
        return y

    def ec_combine_rows(self, C_, sel, p, tokens, workers=1):
        tok = _i64(tokens)
        sel = _i64(sel)
        p = _f64(p)
        y = np.empty((len(tok), self.d))

        def run(lo, hi):
            _ok(lib().orc_ec_combine_rows(self.ref(), int(C_), _p(sel), _p(p), _p(tok[lo:hi]),
                                          hi - lo, _p(y[lo:hi])), "ec_combine_rows")
        _parallel(run, len(tok), workers)
        return y

    # ---- backward pieces
    def token_grads(self, routing, dy, aux_weight, tokens, renormalize=True, workers=1):
        """(dw [n, k], dz [n, N], dx [n, d]) of the listed tokens."""
        tok = _i64(tokens)
        dyh, code = _host(dy)
        dyt = _Tensor(dyh.ctypes.data, code, 0)
        n = len(tok)
        dw, dz, dx = np.empty((n, self.k)), np.empty((n, self.N)), np.empty((n, self.d))

        def run(lo, hi):
            _ok(lib().orc_token_grads(self.ref(), int(bool(renormalize)), _p(routing.p),
                                      _p(routing.idx), _p(routing.w), _p(routing.keep), dyt,
                                      float(aux_weight), _p(tok[lo:hi]), hi - lo,
                                      _p(dw[lo:hi]), _p(dz[lo:hi]), _p(dx[lo:hi])),
                "token_grads")
        _parallel(run, n, workers)
        return dw, dz, dx

    def router_weight_grads(self, dz):
        """(dW_g [N, d], db_g [N]) from the score gradients dz [T, N]."""
        dz = _f64(dz)
        dW_g, db_g = np.empty((self.N, self.d)), np.empty(self.N)
        _ok(lib().orc_router_weight_grads(self.ref(), _p(dz), _p(dW_g), _p(db_g)),
            "router_weight_grads")
        return dW_g, db_g

    def backward(self, routing, dy, aux_weight, renormalize=True, workers=1):
        """The whole backward pass from its pieces: every token's dw, dz and dx
        (token rows split over `workers` threads), every expert's weight
        gradients (experts spread over the threads), the router's.  Equal to
        moe_backward up to the order of floating-point sums."""
        T, N, k = self.T, self.N, self.k
        dw, dz, dx = self.token_grads(routing, dy, aux_weight, np.arange(T), renormalize,
                                      workers)
        grp = routing.grouping()
        jobs = list(range(N + (1 if self.fs else 0)))

        def one(e):
            if e == N:
                return self.expert_weight_grads(e, np.arange(T), np.ones(T), dy)
            rows = grp.groups[e]
            ts = np.array([t for t, _ in rows], dtype=np.int64)
            gs = np.array([routing.w[t, j] for t, j in rows])
            return self.expert_weight_grads(e, ts, gs, dy)

        with ThreadPoolExecutor(max_workers=max(1, workers)) as ex:
            res = list(ex.map(one, jobs))
        dW_g, db_g = self.router_weight_grads(dz)
        g = LayerGrads(dx, dW_g, db_g, np.stack([r[0] for r in res[:N]]),
                       np.stack([r[1] for r in res[:N]]), np.stack([r[2] for r in res[:N]]),
                       np.stack([r[3] for r in res[:N]]), dz, dw, None)
        if self.fs:
            g.shared = res[N]
        return g

    def expert_weight_grads(self, e, tokens, gates, dy, units=None):
        """(dW1 rows [u, d], db1 [u], dW2 columns [d, u], db2 [d]) of expert e
        (e == N: shared) over rows tokens with gates; units=None: all."""
        tok = _i64(tokens)
        g = _f64(gates)
        dyh, code = _host(dy)
        fe = self.fs if e == self.N else self.f
        un = _i64(units) if units is not None else None
        u = fe if un is None else len(un)
        dW1, db1, dW2, db2 = np.empty((u, self.d)), np.empty(u), np.empty((self.d, u)), \
            np.empty(self.d)
        _ok(lib().orc_expert_weight_grads(self.ref(), int(e), _p(tok), _p(g), len(tok),
                                          _Tensor(dyh.ctypes.data, code, 0), _p(un), u,
                                          _p(dW1), _p(db1), _p(dW2), _p(db2)),
            "expert_weight_grads")
        return dW1, db1, dW2, db2


@dataclass
class Routing:
    z: np.ndarray
    p: np.ndarray
    idx: np.ndarray
    w: np.ndarray
    counts: np.ndarray
    kept: np.ndarray
    rank: np.ndarray
    keep: np.ndarray
    order: np.ndarray
    group_start: np.ndarray
    mean_prob: np.ndarray
    dropped: int = 0
    balance: float = 0.0
    cv_squared: float = 0.0

    def grouping(self) -> "Grouping":
        k = self.idx.shape[1]
        gs = self.group_start
        groups = [[(int(a) // k, int(a) % k) for a in self.order[gs[e]:gs[e + 1]]]
                  for e in range(len(self.counts))]
        return Grouping(groups, self.counts.copy(), self.kept.copy(), self.rank.copy(),
                        self.keep.astype(bool), self.dropped)


# ---------------------------------------------------------------------------
# number formats and elementwise definitions

def round_to_bf16(v):
    """Nearest bfloat16 value (8 significant bits, ties to even)."""
    v = _f64(v)
    out = np.empty_like(v)
    lib().orc_round_bf16_array(_p(v), _p(out), v.size)
    return out


def activation(h, act):
    h = _f64(h)
    out = np.empty_like(h)
    _ok(lib().orc_activation(int(act), _p(h), _p(out), h.size), "activation")
    return out


def activation_grad(a, act):
    a = _f64(a)
    out = np.empty_like(a)
    _ok(lib().orc_activation_grad(int(act), _p(a), _p(out), a.size), "activation_grad")
    return out


# ---------------------------------------------------------------------------
# router: scores, softmax, top-k, gates

def router_logits(x, W_g, b_g):
    """z[t, e] = sum_i x[t, i] W_g[e, i] + b_g[e]  (nn.Linear(d_model, N))."""
    return Layer(x, W_g, b_g).logits()


def softmax(z):
    """Softmax over the last axis, max-subtracted."""
    z = _f64(z)
    flat = z.reshape(-1, z.shape[-1])
    p = np.empty_like(flat)
    _ok(lib().orc_softmax_rows(flat.shape[0], flat.shape[1], _p(flat), _p(p)), "softmax")
    return p.reshape(z.shape)


def topk_indices(z, k):
    """Indices of the k largest scores per row, largest first; equal scores
    in ascending index order."""
    z = _f64(z)
    idx = np.empty((z.shape[0], k), np.int64)
    _ok(lib().orc_topk(z.shape[0], z.shape[1], int(k), _p(z), _p(idx)), "topk")
    return idx


def topk_gap(z, k):
    z = _f64(z)
    g = np.empty(z.shape[0])
    _ok(lib().orc_topk_gap(z.shape[0], z.shape[1], int(k), _p(z), _p(g)), "topk_gap")
    return g


def _gates(fn, a, idx, what):
    a = _f64(a)
    idx = _i64(idx)
    w = np.empty(idx.shape)
    _ok(fn(a.shape[0], a.shape[1], idx.shape[1], _p(a), _p(idx), _p(w)), what)
    return w


def gates_softmax_of_topk(z, idx):
    """Softmax(TopK(z)) at the kept experts."""
    return _gates(lib().orc_gates_softmax_of_topk, z, idx, "gates_softmax_of_topk")


def gates_renormalised_probs(p, idx):
    return _gates(lib().orc_gates_renormalised_probs, p, idx, "gates_renormalised_probs")


def gates_raw_probs(p, idx):
    return _gates(lib().orc_gates_raw_probs, p, idx, "gates_raw_probs")


def route(x, W_g, b_g, k, renormalize=True):
    """Router + softmax + top-k (+ renormalise).  Returns (z, p, idx, w)."""
    r = Layer(x, W_g, b_g, k=k).route(renormalize=renormalize)
    return r.z, r.p, r.idx, r.w


# ---------------------------------------------------------------------------
# capacity, grouping, statistics

def expert_capacity(capacity_factor, T, N):
    """ceil(capacity factor x batch / number of experts)."""
    return int(lib().orc_capacity(float(capacity_factor), int(T), int(N)))


@dataclass
class Grouping:
    """groups[e]: kept (t, j) of expert e in token-major order; counts / kept
    per expert; rank[t, j]; keep[t, j]; dropped total."""
    groups: list
    counts: np.ndarray
    kept: np.ndarray
    rank: np.ndarray
    keep: np.ndarray
    dropped: int = field(default=0)


def group_by_expert(idx, N, capacity=0):
    idx = _i64(idx)
    T, k = idx.shape
    r = Routing(z=None, p=None, idx=idx, w=None, counts=np.empty(N, np.int64),
                kept=np.empty(N, np.int64), rank=np.empty((T, k), np.int64),
                keep=np.empty((T, k), np.uint8), order=np.empty(T * k, np.int64),
                group_start=np.empty(N + 1, np.int64), mean_prob=None)
    dropped = lib().orc_group(T, k, int(N), int(capacity), _p(idx), _p(r.counts), _p(r.kept),
                              _p(r.rank), _p(r.keep), _p(r.order), _p(r.group_start))
    if dropped < 0:
        raise ValueError("oracle group: invalid argument")
    r.dropped = int(dropped)
    return r.grouping()


def balance_statistic(p):
    """(mean_prob, std_unbiased(mean_prob)^2)."""
    p = _f64(p)
    T, N = p.shape
    m = np.empty(N)
    b = C.c_double()
    _ok(lib().orc_balance(T, N, _p(p), _p(m), C.byref(b)), "balance")
    return m, float(b.value)


def cv_squared(counts):
    c = _i64(counts)
    return float(lib().orc_cv_squared(c.shape[0], _p(c)))


# ---------------------------------------------------------------------------
# experts and the layer

def expert_ffn(xr, W1, b1, W2, b2, act, round_hidden_bf16=False):
    """Linear -> activation -> Linear of one expert (W1 [f, d], W2 [d, f]) on the rows xr."""
    L = Layer(xr, None, None, [W1], [b1], [W2], [b2], act=act,
              round_hidden_bf16=round_hidden_bf16)
    return L.expert_rows(0, np.arange(L.T))[2]


@dataclass
class LayerOutput:
    y: np.ndarray            # [len(tokens), d]
    tokens: np.ndarray
    z: np.ndarray            # [T, N]
    p: np.ndarray            # [T, N]
    idx: np.ndarray          # [T, k]
    w: np.ndarray            # [T, k]
    grouping: Grouping
    mean_prob: np.ndarray    # [N]
    balance: float
    cv_squared: float = 0.0


def moe_forward(x, W_g, b_g, W1, b1, W2, b2, *, k, act, capacity=0, renormalize=True,
                shared=None, round_hidden_bf16=False, tokens=None, idx_override=None,
                workers=1):
    """The whole layer; y for the tokens listed in ``tokens`` (default all).
    Routing, grouping and statistics always cover all T tokens.
    ``idx_override`` replaces the top-k choice (near-tie tokens)."""
    L = Layer(x, W_g, b_g, W1, b1, W2, b2, k=k, act=act, shared=shared,
              round_hidden_bf16=round_hidden_bf16)
    r = L.route(capacity, renormalize, idx_override, workers)
    tok = np.arange(L.T) if tokens is None else _i64(tokens)
    y = L.combine_rows(r, tok, workers)
    return LayerOutput(y, tok, r.z, r.p, r.idx, r.w, r.grouping(), r.mean_prob, r.balance,
                       r.cv_squared)


def moe_bruteforce(x, W_g, b_g, W1, b1, W2, b2, *, k, act, capacity=0, renormalize=True,
                   shared=None):
    """Every expert on every token, then masks and weights (tiny inputs only)."""
    L = Layer(x, W_g, b_g, W1, b1, W2, b2, k=k, act=act, shared=shared)
    y = np.empty((L.T, L.d))
    _ok(lib().orc_bruteforce(L.ref(), int(capacity), int(bool(renormalize)), _p(y)),
        "bruteforce")
    return y


# ---------------------------------------------------------------------------
# expert-choice routing

def expert_choice_tokens(T, capacity):
    return int(lib().orc_ec_tokens(int(T), int(capacity)))


def expert_choice_select(p, C_):
    p = _f64(p)
    T, N = p.shape
    sel = np.empty((N, C_), np.int64)
    _ok(lib().orc_ec_select(T, N, int(C_), _p(p), _p(sel)), "ec_select")
    return [sel[e].copy() for e in range(N)]


def expert_choice_gap(p, C_):
    p = _f64(p)
    T, N = p.shape
    g = np.empty(N)
    _ok(lib().orc_ec_gap(T, N, int(C_), _p(p), _p(g)), "ec_gap")
    return g


def expert_choice_picks(T, sel):
    """(picks [T]: experts that picked each token, number of tokens no expert picked)."""
    sel = _i64(sel)
    N, C_ = sel.shape if sel.ndim == 2 else (0, 0)
    picks = np.empty(T, np.int64)
    unpicked = int(lib().orc_ec_picks(int(T), max(N, 1) if N else 1, C_ if N else 0,
                                      _p(sel), _p(picks)))
    if unpicked < 0:
        raise ValueError("oracle ec_picks: invalid argument")
    return picks, unpicked


@dataclass
class ExpertChoiceOutput:
    y: np.ndarray
    tokens: np.ndarray
    z: np.ndarray
    p: np.ndarray
    sel: list                # N arrays of picked tokens, ascending
    gate: list               # N arrays: p[sel[e], e]
    token_picks: np.ndarray  # [T]
    unpicked: int
    mean_prob: np.ndarray
    balance: float


def expert_choice_forward(x, W_g, b_g, W1, b1, W2, b2, *, capacity, act, shared=None,
                          round_hidden_bf16=False, tokens=None, sel_override=None, workers=1):
    """Expert-choice layer; ``sel_override`` replaces the selection (near-tie experts)."""
    L = Layer(x, W_g, b_g, W1, b1, W2, b2, k=1, act=act, shared=shared,
              round_hidden_bf16=round_hidden_bf16)
    z = L.logits(workers)
    p = softmax(z)
    T, N = p.shape
    C_ = expert_choice_tokens(T, capacity)
    if sel_override is None:
        sel = np.empty((N, C_), np.int64)
        _ok(lib().orc_ec_select(T, N, C_, _p(p), _p(sel)), "ec_select")
    else:
        sel = _i64(np.stack([np.asarray(s, np.int64) for s in sel_override])
                   if N else np.empty((0, C_), np.int64)).reshape(N, C_)
    picks = np.empty(T, np.int64)
    unpicked = int(lib().orc_ec_picks(T, N, C_, _p(sel), _p(picks)))
    if unpicked < 0:
        raise ValueError("oracle ec_picks: invalid argument")
    m, bal = balance_statistic(p)
    tok = np.arange(T) if tokens is None else _i64(tokens)
    y = L.ec_combine_rows(C_, sel, p, tok, workers)
    return ExpertChoiceOutput(y, tok, z, p, [sel[e].copy() for e in range(N)],
                              [p[sel[e], e] for e in range(N)], picks, unpicked, m, bal)


# ---------------------------------------------------------------------------
# backward pass

@dataclass
class LayerGrads:
    dx: np.ndarray
    dW_g: np.ndarray
    db_g: np.ndarray
    dW1: np.ndarray
    db1: np.ndarray
    dW2: np.ndarray
    db2: np.ndarray
    dz: np.ndarray
    dw: np.ndarray
    shared: tuple | None


def moe_backward(x, W_g, b_g, W1, b1, W2, b2, dy, *, k, act, capacity=0, renormalize=True,
                 shared=None, aux_weight=0.0, round_hidden_bf16=False, idx_override=None):
    """Gradients of total = <dy, y> + aux_weight * balance w.r.t. x and every parameter."""
    L = Layer(x, W_g, b_g, W1, b1, W2, b2, k=k, act=act, shared=shared,
              round_hidden_bf16=round_hidden_bf16)
    T, d, f, N, fs = L.T, L.d, L.f, L.N, L.fs
    dyh, code = _host(dy)
    g = LayerGrads(np.empty((T, d)), np.empty((N, d)), np.empty(N), np.empty((N, f, d)),
                   np.empty((N, f)), np.empty((N, d, f)), np.empty((N, d)), np.empty((T, N)),
                   np.empty((T, k)), None)
    sh = (np.empty((fs, d)), np.empty(fs), np.empty((d, fs)), np.empty(d)) if fs else \
        (None,) * 4
    ov = _i64(idx_override) if idx_override is not None else None
    _ok(lib().orc_backward(L.ref(), int(capacity), int(bool(renormalize)), _p(ov),
                           _Tensor(dyh.ctypes.data, code, 0), float(aux_weight), _p(g.dx),
                           _p(g.dW_g), _p(g.db_g), _p(g.dW1), _p(g.db1), _p(g.dW2), _p(g.db2),
                           *[_p(a) for a in sh], _p(g.dz), _p(g.dw)), "backward")
    if fs:
        g.shared = sh
    return g
