"""ctypes binding of libmoe.so (the C ABI in include/moe.h).

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels.  torch supplies device memory and streams.  If the library has
not been built, loading it raises -- there is no fallback.
"""

from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

import torch

from .workloads import DT_F32, Workload

_HERE = os.path.dirname(os.path.abspath(__file__))
# MOE_LIBRARY=checks loads the build with device index checks and workspace
# guards (libmoe_checks.so, same ABI); the default is libmoe.so.
LIB_PATH = os.path.join(_HERE, "libmoe_checks.so" if os.environ.get("MOE_LIBRARY") == "checks"
                        else "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, \
    MOE_ERR_TIMEOUT = range(6)
MOE_F32, MOE_BF16 = 0, 1
MOE_ACT_GELU_ERF, MOE_ACT_RELU = 0, 1

# Every symbol include/moe.h declares.
EXPORTS = [
    "moe_rows_max", "moe_router_blocks", "moe_permute_scratch_size", "moe_workspace_size",
    "moe_router_topk", "moe_permute", "moe_grouped_ffn", "moe_combine", "moe_load_stats",
    "moe_forward", "moe_host_workspace_size", "moe_forward_host", "moe_forward_host_chunks",
    "moe_get_device_status",
    "moe_set_wait_limit_ns", "moe_get_wait_limit_ns", "moe_selftest_bounded_wait",
    "moe_status_string", "moe_version", "moe_permute_noalloc", "moe_forward_profiled",
    "moe_forward_launch_count", "moe_activation",
    "moe_ec_tokens_per_expert", "moe_ec_rows_max", "moe_ec_workspace_size",
    "moe_ec_forward_launch_count", "moe_ec_router", "moe_ec_select", "moe_ec_forward",
    "moe_ec_forward_profiled", "moe_backward", "moe_backward_workspace_size",
    "moe_backward_launch_count", "moe_backward_profiled", "moe_ffn_kernel_name",
    "moe_build_flags", "moe_workspace_guards", "moe_checks_read",
]
MOE_BUILD_CHECKS = 1
GUARD_BYTES = 256
PERMUTE_STATIC_SCRATCH_INTS = 1 << 18


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class MoeConfig(C.Structure):
    _fields_ = [("T", C.c_int64), ("d_model", C.c_int64), ("d_ff", C.c_int64),
                ("n_experts", C.c_int64), ("top_k", C.c_int64), ("capacity", C.c_int64),
                ("d_ff_shared", C.c_int64), ("renormalize", C.c_int32), ("act", C.c_int32),
                ("dtype", C.c_int32), ("reserved", C.c_int32)]


class MoeWeights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in
                ("W_g", "b_g", "W1", "b1", "W2", "b2", "W1s", "b1s", "W2s", "b2s")]


class MoeOutputs(C.Structure):
    _fields_ = [("y", C.c_void_p), ("topk_idx", C.c_void_p), ("topk_w", C.c_void_p),
                ("counts", C.c_void_p), ("kept", C.c_void_p), ("dropped", C.c_void_p),
                ("mean_prob", C.c_void_p), ("balance", C.c_void_p), ("logits", C.c_void_p),
                ("cv_squared", C.c_void_p), ("pre_act", C.c_void_p)]


class MoeGrads(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in
                ("dx", "dW_g", "db_g", "dW1", "db1", "dW2", "db2", "dW1s", "db1s", "dW2s",
                 "db2s", "dz", "dw")]


class MoeEcOutputs(C.Structure):
    _fields_ = [("y", C.c_void_p), ("ec_token", C.c_void_p), ("ec_gate", C.c_void_p),
                ("token_picks", C.c_void_p), ("unpicked", C.c_void_p),
                ("mean_prob", C.c_void_p), ("balance", C.c_void_p), ("logits", C.c_void_p)]


_lib = None
_LAYERS = []        # checks build: layers whose workspace guards tests inspect


def lib() -> C.CDLL:
    """Load libmoe.so (once).  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built: run "
                           "`python -m sparse_mixture_experts_68_b300.build`")
    L = C.CDLL(LIB_PATH)
    P = C.c_void_p
    CP = C.POINTER(MoeConfig)
    sig = {
        "moe_rows_max": (C.c_int64, [CP]),
        "moe_router_blocks": (C.c_int64, [CP]),
        "moe_permute_scratch_size": (C.c_size_t, [CP]),
        "moe_workspace_size": (C.c_size_t, [CP]),
        "moe_forward_launch_count": (C.c_int32, [CP]),
        "moe_ffn_kernel_name": (C.c_char_p, [CP, C.c_int32]),
        "moe_build_flags": (C.c_int32, []),
        "moe_workspace_guards": (C.c_int32, [CP, P, C.c_int32]),
        "moe_checks_read": (C.c_int32, [P, P, P, C.c_int32]),
        "moe_host_workspace_size": (C.c_size_t, [CP]),
        "moe_forward_host_chunks": (C.c_int32, [CP]),
        "moe_router_topk": (C.c_int32, [CP, P, P, P, P, P, P, P, P]),
        "moe_permute": (C.c_int32, [CP, P, P, P, P, P, P, P, P, P, C.c_size_t, P]),
        "moe_permute_noalloc": (C.c_int32, [CP, P, P, P, P, P, P, P, P, P]),
        "moe_grouped_ffn": (C.c_int32, [CP, P, P, P, C.POINTER(MoeWeights), P, P, P]),
        "moe_combine": (C.c_int32, [CP, P, P, P, P, P, P]),
        "moe_load_stats": (C.c_int32, [CP, P, P, P, P, P, P, P, P]),
        "moe_forward": (C.c_int32, [CP, P, C.POINTER(MoeWeights), C.POINTER(MoeOutputs), P,
                                    C.c_size_t, P]),
        "moe_forward_profiled": (C.c_int32, [CP, P, C.POINTER(MoeWeights),
                                             C.POINTER(MoeOutputs), P, C.c_size_t,
                                             C.POINTER(C.c_void_p), P]),
        "moe_forward_host": (C.c_int32, [CP, P, C.POINTER(MoeWeights),
                                         C.POINTER(MoeOutputs), P, C.c_size_t, P]),
        "moe_get_device_status": (C.c_int32, [P]),
        "moe_set_wait_limit_ns": (None, [C.c_uint64]),
        "moe_get_wait_limit_ns": (C.c_uint64, []),
        "moe_selftest_bounded_wait": (C.c_int32, [C.c_uint64, P]),
        "moe_activation": (C.c_int32, [C.c_int32, P, P, C.c_int64, P]),
        "moe_ec_tokens_per_expert": (C.c_int64, [CP]),
        "moe_ec_rows_max": (C.c_int64, [CP]),
        "moe_ec_workspace_size": (C.c_size_t, [CP]),
        "moe_ec_forward_launch_count": (C.c_int32, [CP]),
        "moe_ec_router": (C.c_int32, [CP, P, P, P, P, P, P, P, P]),
        "moe_ec_select": (C.c_int32, [CP, P, P, P, P, P, P, P, P, P, P]),
        "moe_ec_forward": (C.c_int32, [CP, P, C.POINTER(MoeWeights), C.POINTER(MoeEcOutputs),
                                       P, C.c_size_t, P]),
        "moe_ec_forward_profiled": (C.c_int32, [CP, P, C.POINTER(MoeWeights),
                                                C.POINTER(MoeEcOutputs), P, C.c_size_t,
                                                C.POINTER(C.c_void_p), P]),
        "moe_backward_workspace_size": (C.c_size_t, [CP]),
        "moe_backward_launch_count": (C.c_int32, [CP]),
        "moe_backward": (C.c_int32, [CP, P, C.POINTER(MoeWeights), C.POINTER(MoeOutputs), P,
                                     C.c_size_t, P, C.c_float, C.POINTER(MoeGrads), P,
                                     C.c_size_t, P]),
        "moe_backward_profiled": (C.c_int32, [CP, P, C.POINTER(MoeWeights),
                                              C.POINTER(MoeOutputs), P, C.c_size_t, P,
                                              C.c_float, C.POINTER(MoeGrads), P, C.c_size_t,
                                              C.POINTER(C.c_void_p), P]),
        "moe_status_string": (C.c_char_p, [C.c_int32]),
        "moe_version": (C.c_int32, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def take_checked_layers() -> list:
    """Checks build: the MoeLayers made since the last call (their guards can
    be inspected), forgetting them."""
    out = list(_LAYERS)
    _LAYERS.clear()
    return out


def status_string(s: int) -> str:
    return lib().moe_status_string(s).decode()


def _check(status: int, what: str):
    if status != MOE_OK:
        raise MoeError(status, what)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream=None) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def make_config(wl: Workload, T: int | None = None, capacity: int | None = None) -> MoeConfig:
    return MoeConfig(T=wl.T if T is None else T, d_model=wl.d_model, d_ff=wl.d_ff,
                     n_experts=wl.n_experts, top_k=wl.top_k,
                     capacity=wl.capacity if capacity is None else capacity,
                     d_ff_shared=wl.d_ff_shared, renormalize=wl.renormalize, act=wl.act,
                     dtype=MOE_F32 if wl.dtype == DT_F32 else MOE_BF16, reserved=0)


def make_weights(t: dict) -> MoeWeights:
    return MoeWeights(*[_ptr(t.get(n)) for n in
                        ("W_g", "b_g", "W1", "b1", "W2", "b2", "W1s", "b1s", "W2s", "b2s")])


def rows_max(cfg: MoeConfig) -> int:
    return int(lib().moe_rows_max(C.byref(cfg)))


def router_blocks(cfg: MoeConfig) -> int:
    return int(lib().moe_router_blocks(C.byref(cfg)))


def workspace_size(cfg: MoeConfig) -> int:
    return int(lib().moe_workspace_size(C.byref(cfg)))


def forward_launch_count(cfg: MoeConfig) -> int:
    return int(lib().moe_forward_launch_count(C.byref(cfg)))


def is_checks_build() -> bool:
    return (int(lib().moe_build_flags()) & MOE_BUILD_CHECKS) != 0


def workspace_guards(cfg: MoeConfig) -> list:
    """Byte offsets of the guard gaps in moe_forward's workspace (checks build)."""
    n = int(lib().moe_workspace_guards(C.byref(cfg), None, 0))
    if n <= 0:
        return []
    buf = (C.c_int64 * n)()
    lib().moe_workspace_guards(C.byref(cfg), buf, n)
    return list(buf)


def checks_read(clear: bool = True):
    """(failed checks since the last clear, site of the first, its source line)."""
    f, s_, l_ = C.c_int32(), C.c_int32(), C.c_int32()
    _check(lib().moe_checks_read(C.byref(f), C.byref(s_), C.byref(l_), int(clear)),
           "moe_checks_read")
    return int(f.value), int(s_.value), int(l_.value)


def ffn_kernel_name(cfg: MoeConfig, linear: int) -> str | None:
    """Kernel and tile that moe_forward launches for grouped Linear 1 or 2."""
    r = lib().moe_ffn_kernel_name(C.byref(cfg), int(linear))
    return None if r is None else r.decode()


def host_workspace_size(cfg: MoeConfig) -> int:
    return int(lib().moe_host_workspace_size(C.byref(cfg)))


def forward_host_chunks(cfg: MoeConfig) -> int:
    return int(lib().moe_forward_host_chunks(C.byref(cfg)))


def permute_scratch_size(cfg: MoeConfig) -> int:
    return int(lib().moe_permute_scratch_size(C.byref(cfg)))


# ---- one call per step -------------------------------------------------------------

def router_topk(cfg, x, W_g, b_g, logits, topk_idx, topk_w, prob_partials, stream=None):
    _check(lib().moe_router_topk(C.byref(cfg), _ptr(x), _ptr(W_g), _ptr(b_g), _ptr(logits),
                                 _ptr(topk_idx), _ptr(topk_w), _ptr(prob_partials),
                                 _stream(stream)), "moe_router_topk")


def permute(cfg, x, topk_idx, counts, kept, offsets, row_token, token_row, Xp, scratch,
            stream=None):
    _check(lib().moe_permute(C.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(counts), _ptr(kept),
                             _ptr(offsets), _ptr(row_token), _ptr(token_row), _ptr(Xp),
                             _ptr(scratch), scratch.numel() * scratch.element_size(),
                             _stream(stream)), "moe_permute")


def permute_noalloc(cfg, x, topk_idx, counts, kept, offsets, row_token, token_row, Xp,
                    stream=None):
    """moe_permute with the library's fixed scratch array (no scratch argument)."""
    _check(lib().moe_permute_noalloc(C.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(counts),
                                     _ptr(kept), _ptr(offsets), _ptr(row_token),
                                     _ptr(token_row), _ptr(Xp), _stream(stream)),
           "moe_permute_noalloc")


def grouped_ffn(cfg, Xp, offsets, kept, weights: MoeWeights, H, Yp, stream=None):
    _check(lib().moe_grouped_ffn(C.byref(cfg), _ptr(Xp), _ptr(offsets), _ptr(kept),
                                 C.byref(weights), _ptr(H), _ptr(Yp), _stream(stream)),
           "moe_grouped_ffn")


def combine(cfg, Yp, token_row, topk_w, offsets, y, stream=None):
    _check(lib().moe_combine(C.byref(cfg), _ptr(Yp), _ptr(token_row), _ptr(topk_w),
                             _ptr(offsets), _ptr(y), _stream(stream)), "moe_combine")


def load_stats(cfg, prob_partials, counts, kept, mean_prob, balance, dropped, cv_squared=None,
               stream=None):
    _check(lib().moe_load_stats(C.byref(cfg), _ptr(prob_partials), _ptr(counts), _ptr(kept),
                                _ptr(mean_prob), _ptr(balance), _ptr(dropped), _ptr(cv_squared),
                                _stream(stream)), "moe_load_stats")


def get_device_status(stream=None) -> int:
    return int(lib().moe_get_device_status(_stream(stream)))


def set_wait_limit_ns(ns: int):
    lib().moe_set_wait_limit_ns(int(ns))


def get_wait_limit_ns() -> int:
    return int(lib().moe_get_wait_limit_ns())


def activation(act: int, x, y, stream=None):
    """The FFN kernels' activation applied elementwise (fp32 device tensors)."""
    _check(lib().moe_activation(int(act), _ptr(x), _ptr(y), x.numel(), _stream(stream)),
           "moe_activation")


def selftest_bounded_wait(limit_ns: int, stream=None):
    _check(lib().moe_selftest_bounded_wait(int(limit_ns), _stream(stream)),
           "moe_selftest_bounded_wait")


# ---- the whole layer --------------------------------------------------------------

@dataclass
class Outputs:
    y: torch.Tensor
    topk_idx: torch.Tensor
    topk_w: torch.Tensor
    counts: torch.Tensor
    kept: torch.Tensor
    dropped: torch.Tensor
    mean_prob: torch.Tensor
    balance: torch.Tensor
    logits: torch.Tensor | None = None
    cv_squared: torch.Tensor | None = None
    pre_act: torch.Tensor | None = None      # kept for moe_backward (grouped rows)

    def struct(self) -> MoeOutputs:
        return MoeOutputs(_ptr(self.y), _ptr(self.topk_idx), _ptr(self.topk_w),
                          _ptr(self.counts), _ptr(self.kept), _ptr(self.dropped),
                          _ptr(self.mean_prob), _ptr(self.balance), _ptr(self.logits),
                          _ptr(self.cv_squared), _ptr(self.pre_act))


def alloc_outputs(cfg: MoeConfig, device, with_logits=False, pin_memory=False,
                  with_pre_act=False) -> Outputs:
    T, k, N, d = cfg.T, cfg.top_k, cfg.n_experts, cfg.d_model
    dt = torch.float32 if cfg.dtype == MOE_F32 else torch.bfloat16
    kw = dict(device=device, pin_memory=pin_memory) if pin_memory else dict(device=device)
    return Outputs(
        y=torch.empty((T, d), dtype=dt, **kw),
        topk_idx=torch.empty((T, k), dtype=torch.int32, **kw),
        topk_w=torch.empty((T, k), dtype=torch.float32, **kw),
        counts=torch.empty((N,), dtype=torch.int32, **kw),
        kept=torch.empty((N,), dtype=torch.int32, **kw),
        dropped=torch.empty((1,), dtype=torch.int32, **kw),
        mean_prob=torch.empty((N,), dtype=torch.float32, **kw),
        balance=torch.empty((1,), dtype=torch.float32, **kw),
        logits=torch.empty((T, N), dtype=torch.float32, **kw) if with_logits else None,
        cv_squared=torch.empty((1,), dtype=torch.float32, **kw),
        pre_act=torch.empty((rows_max(cfg), cfg.d_ff), dtype=dt, **kw) if with_pre_act else None)


def forward(cfg: MoeConfig, x, weights: MoeWeights, out: Outputs, workspace, stream=None):
    _check(lib().moe_forward(C.byref(cfg), _ptr(x), C.byref(weights), C.byref(out.struct()),
                             _ptr(workspace), workspace.numel() * workspace.element_size(),
                             _stream(stream)), "moe_forward")


def forward_profiled(cfg: MoeConfig, x, weights: MoeWeights, out: Outputs, workspace,
                     events, stream=None):
    """moe_forward recording seven torch.cuda.Event (timing enabled) at the step
    boundaries: before the router, after router / permute / first Linear /
    second Linear / combine / statistics."""
    assert len(events) == 7
    handles = (C.c_void_p * 7)(*[ev.cuda_event if ev is not None else None for ev in events])
    _check(lib().moe_forward_profiled(C.byref(cfg), _ptr(x), C.byref(weights),
                                      C.byref(out.struct()), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), handles,
                                      _stream(stream)), "moe_forward_profiled")


def forward_host(cfg: MoeConfig, x_host, weights: MoeWeights, out_host: Outputs, workspace,
                 stream=None):
    _check(lib().moe_forward_host(C.byref(cfg), _ptr(x_host), C.byref(weights),
                                  C.byref(out_host.struct()), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(),
                                  _stream(stream)), "moe_forward_host")


# ---- backward pass -----------------------------------------------------------------

def backward_workspace_size(cfg: MoeConfig) -> int:
    return int(lib().moe_backward_workspace_size(C.byref(cfg)))


def backward_launch_count(cfg: MoeConfig) -> int:
    return int(lib().moe_backward_launch_count(C.byref(cfg)))


@dataclass
class Grads:
    dx: torch.Tensor
    dW_g: torch.Tensor
    db_g: torch.Tensor
    dW1: torch.Tensor
    db1: torch.Tensor
    dW2: torch.Tensor
    db2: torch.Tensor
    dW1s: torch.Tensor | None = None
    db1s: torch.Tensor | None = None
    dW2s: torch.Tensor | None = None
    db2s: torch.Tensor | None = None
    dz: torch.Tensor | None = None
    dw: torch.Tensor | None = None

    def struct(self) -> MoeGrads:
        return MoeGrads(*[_ptr(getattr(self, n)) for n in
                          ("dx", "dW_g", "db_g", "dW1", "db1", "dW2", "db2", "dW1s", "db1s",
                           "dW2s", "db2s", "dz", "dw")])


def alloc_grads(cfg: MoeConfig, device, with_scores=False) -> Grads:
    T, d, f, N, k = cfg.T, cfg.d_model, cfg.d_ff, cfg.n_experts, cfg.top_k
    dt = torch.float32 if cfg.dtype == MOE_F32 else torch.bfloat16
    e = lambda *shape: torch.empty(shape, dtype=dt, device=device)  # noqa: E731
    sh = cfg.d_ff_shared > 0
    return Grads(
        dx=e(T, d), dW_g=e(N, d), db_g=e(N), dW1=e(N, f, d), db1=e(N, f), dW2=e(N, d, f),
        db2=e(N, d), dW1s=e(f, d) if sh else None, db1s=e(f) if sh else None,
        dW2s=e(d, f) if sh else None, db2s=e(d) if sh else None,
        dz=torch.empty((T, N), dtype=torch.float32, device=device) if with_scores else None,
        dw=torch.empty((T, k), dtype=torch.float32, device=device) if with_scores else None)


def backward(cfg: MoeConfig, x, weights: MoeWeights, fwd: Outputs, fwd_workspace, dy,
             aux_weight: float, grads: Grads, workspace, stream=None):
    _check(lib().moe_backward(C.byref(cfg), _ptr(x), C.byref(weights), C.byref(fwd.struct()),
                              _ptr(fwd_workspace),
                              fwd_workspace.numel() * fwd_workspace.element_size(), _ptr(dy),
                              float(aux_weight), C.byref(grads.struct()), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream)),
           "moe_backward")


def backward_profiled(cfg: MoeConfig, x, weights: MoeWeights, fwd: Outputs, fwd_workspace, dy,
                      aux_weight: float, grads: Grads, workspace, events, stream=None):
    """moe_backward recording eight torch.cuda.Event at its step boundaries."""
    assert len(events) == 8
    handles = (C.c_void_p * 8)(*[ev.cuda_event if ev is not None else None for ev in events])
    _check(lib().moe_backward_profiled(C.byref(cfg), _ptr(x), C.byref(weights),
                                       C.byref(fwd.struct()), _ptr(fwd_workspace),
                                       fwd_workspace.numel() * fwd_workspace.element_size(),
                                       _ptr(dy), float(aux_weight), C.byref(grads.struct()),
                                       _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), handles,
                                       _stream(stream)), "moe_backward_profiled")


class MoeLayer:
    """Device-resident weights + workspace of one layer; ``forward`` runs it."""

    def __init__(self, wl: Workload, tensors: dict, device="cuda", T: int | None = None,
                 capacity: int | None = None):
        self.wl = wl
        self.t = tensors
        self.device = torch.device(device)
        self.cfg = make_config(wl, T=T, capacity=capacity)
        self.weights = make_weights(tensors)
        self.workspace = torch.empty(max(workspace_size(self.cfg), 256), dtype=torch.uint8,
                                     device=self.device)
        self._fill_guards()

    GUARD_PATTERN = 0xA5

    def _fill_guards(self):
        """Checks build: the guard gaps hold a fixed pattern (see guards_intact)."""
        if self.device.type == "cuda" and is_checks_build():
            self.workspace.fill_(self.GUARD_PATTERN)
            _LAYERS.append(self)

    def guards_intact(self) -> bool:
        """Whether every guard gap of the workspace still holds the pattern."""
        for off in workspace_guards(self.cfg):
            gap = self.workspace[off: off + GUARD_BYTES]
            if not bool(torch.all(gap == self.GUARD_PATTERN)):
                return False
        return True

    def set_tokens(self, T: int):
        self.cfg = make_config(self.wl, T=T, capacity=self.cfg.capacity)
        need = workspace_size(self.cfg)
        if need > self.workspace.numel():
            self.workspace = torch.empty(need, dtype=torch.uint8, device=self.device)
        self._fill_guards()

    def forward(self, x, out: Outputs | None = None, with_logits=False, with_pre_act=False,
                stream=None) -> Outputs:
        """with_pre_act keeps the first Linear's pre-activation for ``backward``."""
        if out is None:
            out = alloc_outputs(self.cfg, self.device, with_logits=with_logits,
                                with_pre_act=with_pre_act)
        forward(self.cfg, x, self.weights, out, self.workspace, stream)
        return out

    def backward(self, x, out: Outputs, dy, aux_weight=0.01, grads: Grads | None = None,
                 with_scores=False, stream=None) -> Grads:
        """Gradients of total = task + aux_weight * balance given dy = d task / d y,
        for the last ``forward`` (its outputs ``out`` and this layer's workspace)."""
        if grads is None:
            grads = alloc_grads(self.cfg, self.device, with_scores=with_scores)
        need = backward_workspace_size(self.cfg)
        if getattr(self, "bwd_workspace", None) is None or self.bwd_workspace.numel() < need:
            self.bwd_workspace = torch.empty(max(need, 256), dtype=torch.uint8,
                                             device=self.device)
        backward(self.cfg, x, self.weights, out, self.workspace, dy, aux_weight, grads,
                 self.bwd_workspace, stream)
        return grads


# ---- expert-choice routing ---------------------------------------------------------

def ec_tokens_per_expert(cfg: MoeConfig) -> int:
    return int(lib().moe_ec_tokens_per_expert(C.byref(cfg)))


def ec_rows_max(cfg: MoeConfig) -> int:
    return int(lib().moe_ec_rows_max(C.byref(cfg)))


def ec_workspace_size(cfg: MoeConfig) -> int:
    return int(lib().moe_ec_workspace_size(C.byref(cfg)))


def ec_forward_launch_count(cfg: MoeConfig) -> int:
    return int(lib().moe_ec_forward_launch_count(C.byref(cfg)))


def ec_router(cfg, x, W_g, b_g, logits, probT, token_picks, prob_partials, stream=None):
    _check(lib().moe_ec_router(C.byref(cfg), _ptr(x), _ptr(W_g), _ptr(b_g), _ptr(logits),
                               _ptr(probT), _ptr(token_picks), _ptr(prob_partials),
                               _stream(stream)), "moe_ec_router")


def ec_select(cfg, probT, ec_token, ec_gate, offsets, counts, row_token, token_row, token_w,
              token_picks, stream=None):
    _check(lib().moe_ec_select(C.byref(cfg), _ptr(probT), _ptr(ec_token), _ptr(ec_gate),
                               _ptr(offsets), _ptr(counts), _ptr(row_token), _ptr(token_row),
                               _ptr(token_w), _ptr(token_picks), _stream(stream)),
           "moe_ec_select")


@dataclass
class EcOutputs:
    y: torch.Tensor
    ec_token: torch.Tensor
    ec_gate: torch.Tensor
    token_picks: torch.Tensor
    unpicked: torch.Tensor
    mean_prob: torch.Tensor
    balance: torch.Tensor
    logits: torch.Tensor | None = None

    def struct(self) -> MoeEcOutputs:
        return MoeEcOutputs(_ptr(self.y), _ptr(self.ec_token), _ptr(self.ec_gate),
                            _ptr(self.token_picks), _ptr(self.unpicked), _ptr(self.mean_prob),
                            _ptr(self.balance), _ptr(self.logits))


def alloc_ec_outputs(cfg: MoeConfig, device, with_logits=False) -> EcOutputs:
    T, N, d = cfg.T, cfg.n_experts, cfg.d_model
    Cn = ec_tokens_per_expert(cfg)
    dt = torch.float32 if cfg.dtype == MOE_F32 else torch.bfloat16
    kw = dict(device=device)
    return EcOutputs(
        y=torch.empty((T, d), dtype=dt, **kw),
        ec_token=torch.empty((N, Cn), dtype=torch.int32, **kw),
        ec_gate=torch.empty((N, Cn), dtype=torch.float32, **kw),
        token_picks=torch.empty((T,), dtype=torch.int32, **kw),
        unpicked=torch.empty((1,), dtype=torch.int32, **kw),
        mean_prob=torch.empty((N,), dtype=torch.float32, **kw),
        balance=torch.empty((1,), dtype=torch.float32, **kw),
        logits=torch.empty((T, N), dtype=torch.float32, **kw) if with_logits else None)


def ec_forward(cfg: MoeConfig, x, weights: MoeWeights, out: EcOutputs, workspace, stream=None):
    _check(lib().moe_ec_forward(C.byref(cfg), _ptr(x), C.byref(weights), C.byref(out.struct()),
                                _ptr(workspace), workspace.numel() * workspace.element_size(),
                                _stream(stream)), "moe_ec_forward")


def ec_forward_profiled(cfg: MoeConfig, x, weights: MoeWeights, out: EcOutputs, workspace,
                        events, stream=None):
    assert len(events) == 7
    handles = (C.c_void_p * 7)(*[ev.cuda_event if ev is not None else None for ev in events])
    _check(lib().moe_ec_forward_profiled(C.byref(cfg), _ptr(x), C.byref(weights),
                                         C.byref(out.struct()), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), handles,
                                         _stream(stream)), "moe_ec_forward_profiled")


class MoeEcLayer:
    """A layer with expert-choice routing: weights, workspace, ``forward``."""

    def __init__(self, wl: Workload, tensors: dict, device="cuda", T: int | None = None,
                 capacity: int | None = None):
        self.wl = wl
        self.t = tensors
        self.device = torch.device(device)
        self.cfg = make_config(wl, T=T, capacity=capacity)
        self.weights = make_weights(tensors)
        self.workspace = torch.empty(max(ec_workspace_size(self.cfg), 256), dtype=torch.uint8,
                                     device=self.device)

    def forward(self, x, out: EcOutputs | None = None, with_logits=False,
                stream=None) -> EcOutputs:
        if out is None:
            out = alloc_ec_outputs(self.cfg, self.device, with_logits=with_logits)
        ec_forward(self.cfg, x, self.weights, out, self.workspace, stream)
        return out
