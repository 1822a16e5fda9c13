"""The C-ABI library loads, exports every symbol include/moe.h declares, and
rejects bad arguments on the host before touching a GPU (no compute calls)."""

import ctypes as C
import dataclasses
import os
import re

import pytest

from sparse_mixture_experts_68_b300 import binding as B
from sparse_mixture_experts_68_b300.workloads import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(moe_[a-z_]+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(B.LIB_PATH):
        from sparse_mixture_experts_68_b300 import build
        build.build()
    return B.lib()


def test_exports_every_declared_symbol(lib):
    declared = header_functions()
    assert len(declared) >= 15
    assert sorted(B.EXPORTS) == declared
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    assert lib.moe_version() == 1
    assert B.status_string(B.MOE_OK) == "ok"
    assert B.status_string(B.MOE_ERR_TIMEOUT) == "device wait timed out"
    assert B.status_string(99) == "unknown status"


def test_sizes(lib):
    wl = WORKLOADS["c4_deepseek_v3"]
    cfg = B.make_config(wl)
    assert B.rows_max(cfg) == 4096 * 8 + 256 * 127 + 4096
    assert B.router_blocks(cfg) == min(4096 // 8, 296)   # 8-token groups, at most 296 blocks
    assert B.workspace_size(cfg) > B.rows_max(cfg) * (2 * 7168 + 2048) * 2
    assert B.host_workspace_size(cfg) > B.workspace_size(cfg)
    c1 = B.make_config(WORKLOADS["c1_page1_bf16"])
    assert B.rows_max(c1) == 2048 * 2 + 8 * 127
    # the host path's extra room: x and y, topk_idx and topk_w, counts, kept and
    # mean_prob, dropped, balance and cv_squared, logits; each 256-byte rounded.
    # This layer runs as two chunks of 1024 tokens, which adds both chunks'
    # probability partial-sum rows (128 router blocks each), their counts and
    # kept counts, and unused per-chunk statistics.
    r = lambda n: (n + 255) // 256 * 256
    T, d, k, N = 2048, 768, 2, 8
    extra = 2 * r(T * d * 2) + 2 * r(T * k * 4) + 3 * r(N * 4) + 3 * r(4) + r(T * N * 4)
    assert B.forward_host_chunks(c1) == 2
    extra += r(256 * N * 4) + 5 * r(N * 4) + 3 * r(4)
    assert B.host_workspace_size(c1) - B.workspace_size(c1) == extra
    # capacity, few tokens, or a half with less FFN work than the ridge and
    # weights that do not fit in L2: one pass
    for name in ("c2_switch_top1", "c3_mixtral_decode", "c4_deepseek_v3", "c0_pr1_fp32"):
        assert B.forward_host_chunks(B.make_config(WORKLOADS[name])) == 1, name
    assert B.forward_host_chunks(B.make_config(WORKLOADS["c3_mixtral_prefill"])) == 2


@pytest.mark.parametrize("field,value,status", [
    ("top_k", 0, B.MOE_ERR_INVALID_ARG),
    ("top_k", 9, B.MOE_ERR_INVALID_ARG),          # k > N
    ("T", -1, B.MOE_ERR_INVALID_ARG),
    ("dtype", 7, B.MOE_ERR_INVALID_ARG),
    ("act", 5, B.MOE_ERR_INVALID_ARG),
    ("reserved", 1, B.MOE_ERR_INVALID_ARG),
    ("n_experts", 2048, B.MOE_ERR_UNSUPPORTED),
    ("d_model", 100, B.MOE_ERR_UNSUPPORTED),       # bf16 needs d % 64 == 0
    ("d_ff_shared", 64, B.MOE_ERR_UNSUPPORTED),    # shared width must equal d_ff
])
def test_invalid_configs_rejected_on_host(lib, field, value, status):
    cfg = B.make_config(WORKLOADS["c1_page1_bf16"])
    setattr(cfg, field, value)
    if field == "n_experts":
        cfg.top_k = 2
    assert B.workspace_size(cfg) == 0
    assert B.rows_max(cfg) == -1
    w = B.MoeWeights()
    o = B.MoeOutputs()
    st = lib.moe_forward(C.byref(cfg), None, C.byref(w), C.byref(o), None, 0, None)
    assert st == status


def test_null_and_misaligned_pointers_rejected(lib):
    cfg = B.make_config(WORKLOADS["c1_page1_bf16"])
    w = B.MoeWeights()
    o = B.MoeOutputs()
    assert lib.moe_forward(C.byref(cfg), None, C.byref(w), C.byref(o), None, 0, None) == \
        B.MOE_ERR_INVALID_ARG
    # misaligned (never dereferenced: validation fails first)
    fake = 0x1000
    w = B.MoeWeights(*([fake] * 6 + [None] * 4))
    w.W1 = fake + 2
    assert lib.moe_grouped_ffn(C.byref(cfg), fake, fake, fake, C.byref(w), fake, fake, None) \
        == B.MOE_ERR_INVALID_ARG
    assert lib.moe_permute(C.byref(cfg), fake, fake, fake, fake, fake, fake, fake, fake, fake,
                           0, None) == B.MOE_ERR_WORKSPACE
    assert lib.moe_router_topk(C.byref(cfg), fake, fake, fake + 4, fake, fake, fake, fake,
                               None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(None, fake, fake, fake, fake, fake, None) == B.MOE_ERR_INVALID_ARG


def test_workspace_too_small_rejected(lib):
    cfg = B.make_config(WORKLOADS["c1_page1_bf16"])
    fake = 0x10000
    w = B.MoeWeights(*([fake] * 6 + [None] * 4))
    o = B.MoeOutputs(*([fake] * 8 + [None]))
    st = lib.moe_forward(C.byref(cfg), fake, C.byref(w), C.byref(o), fake, 1024, None)
    assert st == B.MOE_ERR_WORKSPACE


def test_wait_limit_setting(lib):
    old = B.get_wait_limit_ns()
    B.set_wait_limit_ns(12345)
    assert B.get_wait_limit_ns() == 12345
    B.set_wait_limit_ns(old)


def test_expert_choice_sizes_and_validation(lib):
    wl = WORKLOADS["c3_mixtral_prefill_ec"]
    cfg = B.make_config(wl)
    assert B.ec_tokens_per_expert(cfg) == 1024                  # ceil(2 * 4096 / 8)
    assert B.ec_rows_max(cfg) == 8 * 1024
    assert B.ec_workspace_size(cfg) > B.ec_rows_max(cfg) * (2 * 4096 + 14336) * 2
    c4 = B.make_config(WORKLOADS["c4_deepseek_v3_ec"])
    assert B.ec_tokens_per_expert(c4) == 128
    assert B.ec_rows_max(c4) == 256 * 128 + 4096               # + the shared group
    # capacity clamps to T; <= 0 means every token
    for cap, want in [(0, 4096), (-3, 4096), (5000, 4096), (100, 100)]:
        cfg.capacity = cap
        assert B.ec_tokens_per_expert(cfg) == want
        assert B.ec_rows_max(cfg) == 8 * (-(-want // 128) * 128)
    # top_k and renormalize are not read
    cfg.capacity = 100
    cfg.top_k, cfg.renormalize = 0, 7
    assert B.ec_workspace_size(cfg) > 0
    cfg.top_k, cfg.renormalize = 2, 1
    for field, value in [("n_experts", 2048), ("d_model", 100), ("dtype", 5), ("T", -1),
                         ("reserved", 1)]:
        bad = B.make_config(wl)
        setattr(bad, field, value)
        assert B.ec_workspace_size(bad) == 0
        assert B.ec_tokens_per_expert(bad) == -1
        assert B.ec_forward_launch_count(bad) == -1
    o = B.MoeEcOutputs()
    w = B.MoeWeights()
    assert lib.moe_ec_forward(C.byref(cfg), None, C.byref(w), C.byref(o), None, 0, None) == \
        B.MOE_ERR_INVALID_ARG
    fake = 0x10000
    w = B.MoeWeights(*([fake] * 6 + [None] * 4))
    o = B.MoeEcOutputs(*([fake] * 7 + [None]))
    assert lib.moe_ec_forward(C.byref(cfg), fake, C.byref(w), C.byref(o), fake, 1024, None) \
        == B.MOE_ERR_WORKSPACE


def test_backward_sizes_and_validation(lib):
    cfg = B.make_config(WORKLOADS["c1_page1_bf16"])
    assert B.backward_workspace_size(cfg) > B.rows_max(cfg) * (2 * 768 + 2 * 3072) * 2
    assert B.backward_launch_count(cfg) == 11          # N = 8: few-expert router kernels
    c4 = B.make_config(WORKLOADS["c4_deepseek_v3"])
    assert B.backward_launch_count(c4) == 12           # N % 64 == 0: on the tensor cores
    f32 = B.make_config(WORKLOADS["c0_pr1_fp32"])
    assert B.backward_workspace_size(f32) > B.rows_max(f32) * (2 * 768 + 2 * 3072) * 4
    assert B.backward_launch_count(f32) == 11           # GEMMs on CUDA cores
    n40 = B.make_config(dataclasses.replace(WORKLOADS["c1_page1_bf16"], n_experts=40))
    assert B.backward_launch_count(n40) == 13          # split-K CUDA-core router GEMMs
    t0 = B.make_config(WORKLOADS["c1_page1_bf16"], T=0)
    assert B.backward_launch_count(t0) == 6             # zero parameter gradients
    w = B.MoeWeights()
    o = B.MoeOutputs()
    g = B.MoeGrads()
    st = lib.moe_backward(C.byref(cfg), None, C.byref(w), C.byref(o), None, 0, None, 0.01,
                          C.byref(g), None, 0, None)
    assert st == B.MOE_ERR_INVALID_ARG
    fake = 0x10000
    w = B.MoeWeights(*([fake] * 6 + [None] * 4))
    o = B.MoeOutputs(*([fake] * 8 + [None, None]))
    g = B.MoeGrads(*([fake] * 7 + [None] * 6))
    st = lib.moe_backward(C.byref(cfg), fake, C.byref(w), C.byref(o), fake, 1 << 40, fake,
                          0.01, C.byref(g), fake, 1024, None)
    assert st == B.MOE_ERR_WORKSPACE
    st = lib.moe_backward(C.byref(cfg), fake, C.byref(w), C.byref(o), fake, 1 << 40, fake,
                          float("nan"), C.byref(g), fake, 1 << 40, None)
    assert st == B.MOE_ERR_INVALID_ARG


def test_permute_path_follows_the_assignment_count():
    """The permutation path (host only: launch counts and scratch sizes) follows
    T*k and N: the one-block sort below 2048 assignments (statistics fused), the
    two-launch sort from 2048 up to 64 blocks of 1024 assignments with at most
    384 experts (statistics fused; scratch [blocks][N] counts, then T*k ranks),
    the histogram/scan/rank path beyond (statistics as their own launch;
    scratch two [ceil(T/128)][N] arrays)."""
    from sparse_mixture_experts_68_b300.workloads import ACT_RELU, DT_BF16, Workload
    r64 = lambda n: (n + 63) // 64 * 64                                        # noqa: E731

    def cfg(T, k, N):
        return B.make_config(Workload("p", T=T, d_model=64, d_ff=64, n_experts=N, top_k=k,
                                      act=ACT_RELU, dtype=DT_BF16, seed=1))

    def hist_ints(T, N):
        return 2 * r64((T + 127) // 128 * N)

    # N = 8: router (1), sort launches, row copy, two Linears, combine
    for T, k, sort_launches, stats in [(1023, 2, 1, 0), (1024, 2, 2, 0), (32768, 2, 2, 0),
                                       (32769, 2, 3, 1)]:
        c = cfg(T, k, 8)
        assert B.forward_launch_count(c) == 1 + sort_launches + 1 + 3 + stats, (T, k)
        ints = hist_ints(T, 8)
        if sort_launches == 2:
            mb = (T * k + 1023) // 1024
            ints = r64(mb * 8) + T * k
        assert B.permute_scratch_size(c) == 4 * ints, (T, k)
    # the two-launch sort's scratch fits the allocation-free entry's fixed array
    # even where the histogram path's would not (65536 tokens, 384 experts)
    big = cfg(65536, 1, 384)
    assert B.permute_scratch_size(big) == 4 * (r64(64 * 384) + 65536)
    assert hist_ints(65536, 384) > (1 << 18)
    # 384 experts take the two-launch sort, 385 the one-block sort (16384
    # assignments); past 16384 assignments with 385 experts, the histogram path.
    # Router: scores on the tensor cores (N % 64 == 0) or CUDA cores, then top-k.
    assert B.forward_launch_count(cfg(2048, 8, 384)) == 2 + 2 + 1 + 3
    assert B.forward_launch_count(cfg(2048, 8, 385)) == 2 + 1 + 1 + 3
    assert B.forward_launch_count(cfg(10000, 2, 385)) == 2 + 3 + 1 + 3 + 1


def test_ffn_kernel_names_follow_the_layer_shape():
    """moe_ffn_kernel_name (host only) names the tile family each grouped
    Linear launches for the benchmark's layers."""
    from sparse_mixture_experts_68_b300.workloads import WORKLOADS
    name = lambda w, i: B.ffn_kernel_name(B.make_config(WORKLOADS[w]), i)   # noqa: E731
    assert "tc2_grouped_gemm_kernel" in name("c3_mixtral_prefill", 1)
    assert "tc2_grouped_gemm_kernel" in name("c3_mixtral_prefill", 2)
    assert "tc_swap_gemm_kernel" in name("c3_mixtral_decode", 1)
    assert "tc_swap_gemm_kernel" in name("c3_mixtral_decode", 2)
    assert name("c1_page1_bf16", 1).startswith("tc_grouped_gemm_kernel")
    assert "tc2_grouped_gemm_kernel" in name("c1_page1_bf16", 2)
    assert "simt_gemm_kernel" in name("c0_pr1_fp32", 1)
    cfg = B.make_config(WORKLOADS["c1_page1_bf16"])
    assert B.lib().moe_ffn_kernel_name(C.byref(cfg), 3) is None


def test_checks_build_flags_and_workspace_guards():
    """The ordinary build reports no checks and no guard gaps; the checks
    build (when built) reports both, with the gaps inside the workspace."""
    from sparse_mixture_experts_68_b300.workloads import WORKLOADS
    lib = B.lib()
    assert lib.moe_build_flags() == 0 or os.environ.get("MOE_LIBRARY") == "checks"
    path = os.path.join(os.path.dirname(B.LIB_PATH), "libmoe_checks.so")
    if not os.path.exists(path):
        pytest.skip("libmoe_checks.so not built")
    chk = C.CDLL(path)
    chk.moe_build_flags.restype = C.c_int32
    chk.moe_workspace_guards.restype = C.c_int32
    chk.moe_workspace_guards.argtypes = [C.POINTER(B.MoeConfig), C.c_void_p, C.c_int32]
    chk.moe_workspace_size.restype = C.c_size_t
    chk.moe_workspace_size.argtypes = [C.POINTER(B.MoeConfig)]
    assert chk.moe_build_flags() == B.MOE_BUILD_CHECKS
    cfg = B.make_config(WORKLOADS["c1_page1_bf16"])
    n = chk.moe_workspace_guards(C.byref(cfg), None, 0)
    assert n >= 8
    buf = (C.c_int64 * n)()
    chk.moe_workspace_guards(C.byref(cfg), buf, n)
    size = chk.moe_workspace_size(C.byref(cfg))
    offs = list(buf)
    assert offs == sorted(offs) and offs[-1] + B.GUARD_BYTES <= size
    assert lib.moe_workspace_guards(C.byref(cfg), None, 0) == 0
