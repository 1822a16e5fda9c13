"""moe_permute_noalloc: the permute step for callers that cannot allocate
device memory (a host framework that owns all device memory and forbids
allocation while it runs the layer, or a latency-bound loop that cannot
afford the device-wide synchronisation of a cudaMalloc).  Its scratch is a
fixed array inside the library, so the caller passes only inputs and outputs.

Checked against moe_permute (caller-provided scratch) and against the CPU
oracle's grouping of the same top-k choice, on two calls in a row with
different layers, so stale contents of the shared array from the first call
cannot leak into the second.  Integer and row-copy results: bit-exact.  This
file is collected last on purpose."""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O

from sparse_mixture_experts_68_b300 import binding as B
from sparse_mixture_experts_68_b300 import synth
from sparse_mixture_experts_68_b300.workloads import DT_BF16, Workload

pytestmark = pytest.mark.gpu


def _buffers(cfg, dev):
    T, k, N = cfg.T, cfg.top_k, cfg.n_experts
    rows = B.rows_max(cfg)
    dt = torch.bfloat16
    return dict(counts=torch.empty(N, dtype=torch.int32, device=dev),
                kept=torch.empty(N, dtype=torch.int32, device=dev),
                offsets=torch.empty(N + 2, dtype=torch.int32, device=dev),
                row_token=torch.full((rows,), -7, dtype=torch.int32, device=dev),
                token_row=torch.empty((T, k), dtype=torch.int32, device=dev),
                Xp=torch.zeros((rows, cfg.d_model), dtype=dt, device=dev))


def _route(cfg, t, dev):
    T, k, N = cfg.T, cfg.top_k, cfg.n_experts
    logits = torch.empty((T, N), dtype=torch.float32, device=dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    pp = torch.empty((B.router_blocks(cfg), N), dtype=torch.float32, device=dev)
    B.router_topk(cfg, t["x"], t["W_g"], t["b_g"], logits, idx, w, pp)
    return idx


def _same(ref, got, cfg):
    for key in ("counts", "kept", "offsets", "token_row"):
        assert torch.equal(ref[key], got[key]), key
    off = ref["offsets"].cpu().numpy()
    N = cfg.n_experts
    routed_end, end = int(off[N]), int(off[N + 1])
    assert torch.equal(ref["row_token"][:routed_end], got["row_token"][:routed_end])
    live = torch.zeros(end, dtype=torch.bool, device=ref["Xp"].device)
    live[:routed_end] = ref["row_token"][:routed_end] >= 0
    if end > routed_end:
        live[routed_end: routed_end + cfg.T] = True
    assert torch.equal(ref["Xp"][:end][live], got["Xp"][:end][live])


def _matches_oracle(got, idx, cfg):
    """counts, kept, group order and each assignment's row: the oracle's
    grouping of the same top-k choice."""
    g = O.group_by_expert(idx.cpu().numpy(), cfg.n_experts, cfg.capacity)
    np.testing.assert_array_equal(got["counts"].cpu().numpy(), g.counts)
    np.testing.assert_array_equal(got["kept"].cpu().numpy(), g.kept)
    off = got["offsets"].cpu().numpy().astype(np.int64)
    rt = got["row_token"].cpu().numpy()
    tr = got["token_row"].cpu().numpy().reshape(cfg.T, cfg.top_k)
    for e in range(cfg.n_experts):
        assert off[e + 1] - off[e] == -(-int(g.kept[e]) // 128) * 128
        toks = np.array([t for t, _ in g.groups[e]], dtype=np.int64)
        np.testing.assert_array_equal(rt[off[e]: off[e] + len(toks)], toks)
        for r, (t, j) in enumerate(g.groups[e]):
            assert tr[t, j] == off[e] + r
    assert np.all(tr[~g.keep] == -1)


# The first layer is large enough that the permute step runs as several
# blocks and uses the scratch array; the second is small enough for the
# one-block sort.  Both calls go through moe_permute_noalloc.
LAYERS = [
    Workload("noalloc_a", T=40000, d_model=64, d_ff=64, n_experts=40, top_k=3,
             dtype=DT_BF16, capacity_factor=1.1, seed=41),
    Workload("noalloc_b", T=700, d_model=64, d_ff=128, n_experts=40, top_k=4,
             dtype=DT_BF16, d_ff_shared=128, seed=42),
]


def test_noalloc_permute_matches_permute_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    dev = "cuda"
    for wl in LAYERS:
        t = synth.make_layer(wl, device=dev)
        cfg = B.make_config(wl)
        idx = _route(cfg, t, dev)
        ref = _buffers(cfg, dev)
        scratch = torch.empty(B.permute_scratch_size(cfg), dtype=torch.uint8, device=dev)
        B.permute(cfg, t["x"], idx, ref["counts"], ref["kept"], ref["offsets"],
                  ref["row_token"], ref["token_row"], ref["Xp"], scratch)
        got = _buffers(cfg, dev)
        B.permute_noalloc(cfg, t["x"], idx, got["counts"], got["kept"], got["offsets"],
                          got["row_token"], got["token_row"], got["Xp"])
        torch.cuda.synchronize()
        _same(ref, got, cfg)
        assert int(ref["counts"].sum().item()) == wl.T * wl.top_k
        _matches_oracle(got, idx, cfg)
    assert B.get_device_status() == B.MOE_OK


def test_noalloc_permute_rejects_layers_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    wl = Workload("too_big", T=128 * 200, d_model=64, d_ff=64, n_experts=1024, top_k=1,
                  dtype=DT_BF16)
    cfg = B.make_config(wl)
    assert B.permute_scratch_size(cfg) > B.PERMUTE_STATIC_SCRATCH_INTS * 4
    fake = torch.empty(16, dtype=torch.int32, device="cuda")   # never touched
    with pytest.raises(B.MoeError) as err:
        B.permute_noalloc(cfg, fake, fake, fake, fake, fake, fake, fake, fake)
    assert err.value.status == B.MOE_ERR_WORKSPACE
