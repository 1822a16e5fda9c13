"""Benchmark of the sparse-MoE FFN layer forward pass on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

One step = one pass of the whole layer (router + softmax + top-k, permute,
grouped expert FFN, combine, load statistics) over one batch of T synthetic
tokens, through the library's C ABI.  Prints one JSON line (rank 0).

Timing: W untimed warm-up steps, then K timed steps between a barrier and a
device synchronise on both sides; each step is bracketed by CUDA events on the
launching stream, with L2 flushed before every step, outside the events: a
512 MiB buffer is written, then a separate 384 MiB buffer is read, so that the
flush's own dirty lines are written back before the step starts.  Multi-GPU
(torchrun): every rank runs its own replica of the layer on its own GPU (data
parallel, no exchange); the time is the max over ranks and the value counts
every rank's tokens.

The headline line times the Mixtral-sized prefill layer (T=4096, d=4096,
d_ff=14336, 8 experts, top-2).  The same run adds ``per_workload``: full
sub-lines (value, ms_per_step, roofline, e2e, cpu_baseline, clocks) for the
Mixtral-sized decode (T=16), the DeepSeek-V3-sized layer, the page-1 layer and
the Switch layer with renormalised and with raw-probability gates.

--impl reference times the CPU oracle (plain single-threaded C++, float64) on
one host core, on a bounded sample of the same workload per step.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "c3_mixtral_prefill"
SUB_WORKLOADS = ("c3_mixtral_decode", "c4_deepseek_v3", "c1_page1_bf16", "c2_switch_top1",
                 "c2_switch_top1_raw")
# the B300's nominal HBM3e bandwidth, beside the measured copy rate
NOMINAL_HBM_GBS = 8000.0
METRIC = "MoE-layer tokens/s on 1 B300; % of bf16 tensor peak / % of HBM BW"
TRAIN_METRIC = ("MoE-layer training tokens/s (forward + backward of task + 0.01 balance) "
                "on 1 B300")
AUX_WEIGHT = 0.01
L2_FLUSH_BYTES = 512 << 20
L2_FLUSH_READ_BYTES = 384 << 20


class L2Flush:
    """Evicts the layer's data from L2 between steps, outside the timed events:
    a write of L2_FLUSH_BYTES, then a read of L2_FLUSH_READ_BYTES from another
    buffer.  The write alone would leave L2 full of the flush's dirty lines,
    whose write-back to HBM would then fall inside the next timed step."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        self.r = torch.ones(L2_FLUSH_READ_BYTES // 4, dtype=torch.int32, device=dev)
        self.acc = torch.empty((), dtype=torch.int64, device=dev)

    def __call__(self, i, stream):
        import torch
        with torch.cuda.stream(stream):
            self.w.fill_(i)
            torch.sum(self.r, dim=0, dtype=torch.int64, out=self.acc)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--sub-workloads", default=",".join(SUB_WORKLOADS),
                    help="comma list of workloads timed as per_workload sub-lines; 'none'")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--mode", default="forward", choices=["forward", "train"],
                    help="train: one step = moe_forward + moe_backward (bf16 top-k layers)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


# fp32 layers run their GEMMs on the CUDA cores (FFMA): 148 SMs x 128 fp32 lanes x
# 2 flop per FFMA x the 2032 MHz maximum SM clock
F32_ALU_TFLOPS = 148 * 128 * 2 * 2032e6 / 1e12
F32_ALU_SOURCE = "derived: 148 SMs x 128 fp32 lanes x 2 flop (FFMA) x 2032 MHz"


# ---------------------------------------------------------------------------------------
# DRAM traffic of the dominant kernel, from the committed ncu summary

KERNEL_SOURCES = ("sparse_mixture_experts_68_b300/csrc/grouped_ffn_sm103.cu",
                  "sparse_mixture_experts_68_b300/csrc/common.cuh",
                  "sparse_mixture_experts_68_b300/csrc/tc_common.cuh")


def kernel_sources_sha256():
    import hashlib
    return hashlib.sha256(b"".join(open(os.path.join(ROOT, f), "rb").read()
                                   for f in KERNEL_SOURCES)).hexdigest()


def profiled_traffic(workload):
    """(DRAM bytes per launch of the grouped FFN, source) from the machine-readable
    ncu summary profiles/ffn_<workload>.json, when the kernel sources still hash
    to its source_sha256; else (None, why)."""
    path = os.path.join(ROOT, "profiles", f"ffn_{workload}.json")
    if not os.path.exists(path):
        return None, "no ncu summary for this workload"
    rec = json.load(open(path))
    if rec.get("source_sha256") != kernel_sources_sha256():
        return None, f"profiles/ffn_{workload}.json predates the current kernel sources"
    return float(rec["traffic_bytes_per_launch"]), f"profiles/ffn_{workload}.json"


# ---------------------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    """Polls the GPU's SM clock and clock-event reasons (read-only NVML queries,
    the same counters nvidia-smi prints) every ~2 ms on a thread; keeps only the
    samples taken between mark_start() and mark_end()."""

    def __init__(self, gpu_index: int):
        import threading
        self.gpu = gpu_index
        self.samples = []
        self.window = [None, None]
        self.stop_evt = threading.Event()
        self.thread = None
        self.err = None

    # clock-event reason bits of NVML's nvmlClocksEventReason* constants
    MASKS = {"hw_slowdown": 0x8, "hw_thermal_slowdown": 0x40, "sw_thermal_slowdown": 0x20,
             "sw_power_cap": 0x4}

    def _run(self):
        # the driver's NVML library through ctypes: read-only queries
        import ctypes as C
        try:
            nv = C.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit_v2 failed")
            h = C.c_void_p()
            if nv.nvmlDeviceGetHandleByIndex_v2(C.c_uint(self.gpu), C.byref(h)) != 0:
                raise RuntimeError("nvmlDeviceGetHandleByIndex_v2 failed")
            v = C.c_uint()
            nv.nvmlDeviceGetMaxClockInfo(h, C.c_int(1), C.byref(v))   # 1: SM clock
            self.max_mhz = int(v.value)
            reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            r = C.c_ulonglong()
            while not self.stop_evt.is_set():
                t = time.time()
                nv.nvmlDeviceGetClockInfo(h, C.c_int(1), C.byref(v))
                reasons_fn(h, C.byref(r))
                self.samples.append((t, int(v.value),
                                     [k for k, m in self.MASKS.items() if r.value & m]))
                time.sleep(0.002)
            nv.nvmlShutdown()
        except Exception as e:  # no NVML: report it, do not fail the run
            self.err = repr(e)

    def start(self):
        import threading
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def mark_start(self):
        self.window[0] = time.time()

    def mark_end(self):
        self.window[1] = time.time()

    def stop(self):
        self.stop_evt.set()
        if self.thread:
            self.thread.join(timeout=5)
        if self.err:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [f"nvml: {self.err}"]}
        t0, t1 = self.window
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        if not inside and self.samples:   # window shorter than one poll: nearest sample
            mid = 0.5 * (t0 + t1)
            inside = [min(self.samples, key=lambda s: abs(s[0] - mid))]
        reasons = sorted({r for s in inside for r in s[2]})
        return {"sm_mhz": statistics.median(s[1] for s in inside) if inside else None,
                "sm_max_mhz": getattr(self, "max_mhz", None), "reasons": reasons,
                "samples": len(inside), "source": "NVML, polled every ~2 ms"}


# ---------------------------------------------------------------------------------------
# the CPU oracle as a timed baseline (plain single-threaded C++, one host core)

def host_copy(tensors):
    """Host copies of a layer's tensors in their storage dtype; the oracle
    upcasts each value to float64 as it reads it."""
    return {n: v.detach().to("cpu") for n, v in tensors.items()}


def oracle_step(host, wl, S, train=False):
    """One oracle pass over the first S tokens of the batch, run as a layer of
    S tokens (its capacity recomputed for S tokens); with train=True, the
    forward and the backward of task + 0.01 balance."""
    import torch

    from oracle import moe_oracle as O
    x = host["x"][:S]
    shared = tuple(host[n] for n in ("W1s", "b1s", "W2s", "b2s")) if wl.d_ff_shared else None
    cap = O.expert_capacity(wl.capacity_factor, S, wl.n_experts) \
        if wl.capacity_factor > 0 else 0
    W = [host[n] for n in ("W_g", "b_g", "W1", "b1", "W2", "b2")]
    bf16 = wl.dtype == 1
    dy = torch.randn(x.shape, generator=torch.Generator().manual_seed(7)).to(x.dtype) \
        if train else None

    def run():
        if wl.expert_choice:
            return O.expert_choice_forward(x, *W, capacity=cap, act=wl.act, shared=shared,
                                           round_hidden_bf16=bf16)
        if train:
            return O.moe_backward(x, *W, dy, k=wl.top_k, act=wl.act, capacity=cap,
                                  renormalize=bool(wl.renormalize), shared=shared,
                                  aux_weight=AUX_WEIGHT, round_hidden_bf16=bf16)
        return O.moe_forward(x, *W, k=wl.top_k, act=wl.act, capacity=cap,
                             renormalize=bool(wl.renormalize), shared=shared,
                             round_hidden_bf16=bf16)
    return run


def oracle_sample_size(host, wl, budget_s, train=False):
    """Tokens per oracle pass so that one pass takes about budget_s: the time
    of a 2-token pass, scaled."""
    t0 = time.perf_counter()
    oracle_step(host, wl, min(2, wl.T), train)()
    per_token = (time.perf_counter() - t0) / min(2, wl.T)
    return int(max(1, min(wl.T, budget_s / max(per_token, 1e-9))))


def cpu_baseline(wl, host, budget_s, train=False):
    """The oracle, as it stands, on one host core over a bounded sample."""
    from oracle import moe_oracle as O
    S = oracle_sample_size(host, wl, budget_s / 2, train)
    step = oracle_step(host, wl, S, train)
    t0 = time.perf_counter()
    n = 0
    while n < 2 or (time.perf_counter() - t0 < budget_s / 2 and n < 3):
        step()
        n += 1
    dt = time.perf_counter() - t0
    return {"value": S * n / dt, "unit": "tokens/s", "cores": O.threads(), "kind": "oracle",
            "sample": f"{n} pass(es) over the first {S} of {wl.T} tokens, each run as a "
                      f"layer of {S} tokens ({O.describe()}"
                      + (", forward and backward)" if train else ")")}


def run_reference(args, wl, rank, world):
    from oracle import moe_oracle as O
    from sparse_mixture_experts_68_b300 import synth
    if rank != 0:
        return None
    train = args.mode == "train"
    host = host_copy(synth.make_layer(wl, device="cpu"))
    # each step a bounded sample, so that the K + W steps end in a few minutes
    S = oracle_sample_size(host, wl, min(3.0, 120.0 / max(1, args.steps + args.warmup)),
                           train)
    step = oracle_step(host, wl, S, train)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = S * args.steps / dt
    return {
        "metric": TRAIN_METRIC if train else METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": run_config(wl, world, train),
        "sample_tokens_per_step": S,
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": O.threads(),
                         "kind": "oracle",
                         "sample": f"first {S} of {wl.T} tokens per step, each run as a layer "
                                   f"of {S} tokens ({O.describe()})"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_config(wl, world, train=False):
    """The `config` object of a line: the same for both arms."""
    cfg = {"workload": wl.name, "description": wl.description, "T": wl.T,
           "parallelism": f"replicas{world}" if world > 1 else "single",
           "l2": f"flushed before every step ({L2_FLUSH_BYTES >> 20} MiB written, then "
                 f"{L2_FLUSH_READ_BYTES >> 20} MiB of another buffer read)"}
    if train:
        cfg["aux_weight"] = AUX_WEIGHT
    return cfg


# ---------------------------------------------------------------------------------------
# the CUDA path

STAGES = ("router_topk", "permute", "ffn_linear1", "ffn_linear2", "combine", "load_stats")
EC_STAGES = ("router_probs", "select_and_copy", "ffn_linear1", "ffn_linear2", "combine",
             "load_stats")


class LayerCalls:
    """The library calls one bench step makes: top-k routing (moe_forward) or
    expert-choice routing (moe_ec_forward)."""

    def __init__(self, wl, tensors, dev):
        from sparse_mixture_experts_68_b300 import binding as B
        self.B = B
        self.ec = wl.expert_choice
        if self.ec:
            self.layer = B.MoeEcLayer(wl, tensors, device=dev)
            self.out = B.alloc_ec_outputs(self.layer.cfg, dev)
            self.stages = EC_STAGES
            self.entry = "moe_ec_forward"
        else:
            self.layer = B.MoeLayer(wl, tensors, device=dev)
            self.out = B.alloc_outputs(self.layer.cfg, dev)
            self.stages = STAGES
            self.entry = "moe_forward"
        self.cfg = self.layer.cfg

    def forward(self, x, stream):
        B, L = self.B, self.layer
        if self.ec:
            B.ec_forward(L.cfg, x, L.weights, self.out, L.workspace, stream)
        else:
            B.forward(L.cfg, x, L.weights, self.out, L.workspace, stream)

    def forward_profiled(self, x, events, stream):
        B, L = self.B, self.layer
        if self.ec:
            B.ec_forward_profiled(L.cfg, x, L.weights, self.out, L.workspace, events, stream)
        else:
            B.forward_profiled(L.cfg, x, L.weights, self.out, L.workspace, events, stream)

    def launch_count(self):
        if self.ec:
            return self.B.ec_forward_launch_count(self.cfg)
        return self.B.forward_launch_count(self.cfg)

    def kept(self):
        """(routed rows the experts processed, experts with at least one row)"""
        if self.ec:
            C = self.B.ec_tokens_per_expert(self.cfg)
            return self.cfg.n_experts * C, (self.cfg.n_experts if C > 0 else 0)
        return int(self.out.kept.sum().item()), int((self.out.kept > 0).sum().item())


def job_time_ms(local_ms: float, world: int, device=None) -> float:
    """The job's time for the timed steps: the max over ranks (each rank runs
    its own replica of the layer on its own GPU)."""
    if world <= 1:
        return local_ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([local_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_step: int, steps: int, world: int, job_ms: float) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return tokens_per_step * steps * world / (job_ms * 1e-3)


def run_ours(args, wl, rank, world, local_rank, cpu_budget_s=None):
    import torch
    import torch.distributed as dist

    from sparse_mixture_experts_68_b300 import binding as B
    from sparse_mixture_experts_68_b300 import synth
    from sparse_mixture_experts_68_b300.workloads import flops

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    tensors = synth.make_layer(wl, device=dev)
    calls = LayerCalls(wl, tensors, dev)
    layer = calls.layer
    x = tensors["x"]
    flush = L2Flush(dev)
    # The inputs and buffers come from torch's current stream, the layer runs on
    # its own stream: let every producer finish (torch may hand out memory that
    # a still-running kernel of the current stream is writing) before the first call.
    torch.cuda.synchronize(dev)

    # the layer as a CUDA graph of moe_forward (kernels overlap their
    # neighbours through programmatic dependent launch); per-kernel times come
    # from direct calls of moe_forward_profiled (seven events between kernels)
    stream = torch.cuda.Stream(dev)
    events = [torch.cuda.Event(enable_timing=True) for _ in range(7)]
    with torch.cuda.stream(stream):
        for ev in events:
            ev.record(stream)               # creates the underlying CUDA events
        for _ in range(3):                  # warm: module loading, tensor-map setup
            calls.forward_profiled(x, events, stream)
            calls.forward(x, stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        calls.forward(x, stream)
    torch.cuda.synchronize(dev)

    def flush_l2(i):
        flush(i, stream)                    # L2 flush, outside the timed events

    for i in range(max(args.warmup, 3)):
        flush_l2(i)
        with torch.cuda.stream(stream):
            graph.replay()
    torch.cuda.synchronize(dev)
    assert B.get_device_status() == B.MOE_OK

    K = args.steps
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.05)
    for i in range(3):
        flush_l2(i)
        with torch.cuda.stream(stream):
            graph.replay()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks.mark_start()
    # timed region: K steps of the layer
    marks = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(K)]
    for i in range(K):
        flush_l2(i)
        with torch.cuda.stream(stream):
            marks[i][0].record(stream)
            graph.replay()
            marks[i][1].record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark_end()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in marks]
    total_ms = job_time_ms(sum(step_ms), world, dev)
    # per-kernel times: K steps of moe_forward_profiled, launched directly (its
    # events recorded between the kernels on the stream)
    stage_ms, prof_step_ms = [], []
    for i in range(K):
        flush_l2(i)
        with torch.cuda.stream(stream):
            calls.forward_profiled(x, events, stream)
        stream.synchronize()                # read this step's events before the next
        stage_ms.append([events[s].elapsed_time(events[s + 1]) for s in range(6)])
        prof_step_ms.append(events[0].elapsed_time(events[6]))
    assert B.get_device_status() == B.MOE_OK

    kept_rows, n_kept_experts = calls.kept()
    T = layer.cfg.T
    value = job_tokens_per_s(T, K, world, total_ms)
    mean_stage = {n: statistics.mean(s[i] for s in stage_ms)
                  for i, n in enumerate(calls.stages)}

    # roofline of the dominant kernel: the tcgen05 grouped GEMM, launched once
    # per Linear (two launches per step)
    pk = peaks()
    es = wl.elem_bytes
    rows_sh = T if wl.d_ff_shared else 0
    f1 = 2.0 * wl.d_model * wl.d_ff * (kept_rows + rows_sh)        # per Linear
    wbytes = (n_kept_experts + (1 if wl.d_ff_shared else 0)) * wl.d_model * wl.d_ff * es
    b1 = wbytes + (kept_rows + rows_sh) * (wl.d_model + wl.d_ff) * es   # Linear 1 bytes
    b2 = wbytes + (kept_rows + rows_sh) * (wl.d_ff + wl.d_model) * es   # Linear 2 bytes
    ffn_ms = mean_stage["ffn_linear1"] + mean_stage["ffn_linear2"]
    launches = 2
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    if wl.dtype != 1:                   # fp32: FFMA on the CUDA cores
        achieved = 2 * f1 / launches / (ffn_ms / launches * 1e-3) / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": F32_ALU_TFLOPS,
                "unit": "TFLOP/s"}
    elif (2 * f1) / (b1 + b2) >= ridge:  # the two Linears are tensor-bound
        achieved = 2 * f1 / launches / (ffn_ms / launches * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s"}
    else:
        achieved = (b1 + b2) / launches / (ffn_ms / launches * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"], roof["traffic_source"] = profiled_traffic(wl.name)
    roof["algorithmic_bytes_per_launch"] = (b1 + b2) / launches
    names = [B.ffn_kernel_name(layer.cfg, i) for i in (1, 2)]
    roof["kernel"] = f"Linear 1: {names[0]}; Linear 2: {names[1]}"
    roof["peak_source"] = F32_ALU_SOURCE if wl.dtype != 1 else pk["source"] + " (burst)"
    if roof["bound"] == "hbm":
        roof["frac_of_nominal_8tbs"] = roof["achieved"] / NOMINAL_HBM_GBS
    roof["per_launch"] = {
        "linear1": {"ms": mean_stage["ffn_linear1"], "flop": f1, "bytes": b1,
                    "tflops": f1 / (mean_stage["ffn_linear1"] * 1e-3) / 1e12,
                    "gbs": b1 / (mean_stage["ffn_linear1"] * 1e-3) / 1e9},
        "linear2": {"ms": mean_stage["ffn_linear2"], "flop": f1, "bytes": b2,
                    "tflops": f1 / (mean_stage["ffn_linear2"] * 1e-3) / 1e12,
                    "gbs": b2 / (mean_stage["ffn_linear2"] * 1e-3) / 1e9}}

    # whole-layer roofline time against the same peaks: both weight matrices of
    # every expert with a kept row, the router weight, x read and y written
    layer_flop = flops(wl, kept_rows)
    layer_bytes = (2 * wbytes + wl.n_experts * wl.d_model * es + 2 * T * wl.d_model * es)
    floor_ms = max(layer_flop / (pk["bf16_tflops"] * 1e12),
                   layer_bytes / (pk["hbm_gbs"] * 1e9)) * 1e3
    step_s = total_ms / K * 1e-3
    lfig = {"flop": layer_flop, "bytes": layer_bytes,
            "tflops": layer_flop / step_s / 1e12, "gbs": layer_bytes / step_s / 1e9}
    lfig["frac_of_tensor_peak"] = lfig["tflops"] / pk["bf16_tflops"]
    lfig["frac_of_hbm_measured"] = lfig["gbs"] / pk["hbm_gbs"]
    lfig["frac_of_nominal_8tbs"] = lfig["gbs"] / NOMINAL_HBM_GBS

    res = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if wl.dtype == 1 else "f32", "data": "synthetic",
        "config": run_config(wl, world),
        "launch": f"{calls.entry} captured once as a CUDA graph, replayed; per-kernel "
                  f"times from direct {calls.entry}_profiled calls",
        "tflops": layer_flop / (total_ms / K * 1e-3) / 1e12,
        "layer_roofline_floor_ms": floor_ms,
        "layer_roofline_frac": floor_ms / (total_ms / K),
        "layer": lfig,
        "stage_ms": mean_stage,
        "profiled_ms_per_step": statistics.mean(prof_step_ms),
        "roofline": roof,
        "gpu_launches": calls.launch_count() * K,
        "clocks": clk,
    }

    if not args.no_e2e:
        res["e2e"] = measure_e2e_ec(args, calls, wl, dev) if calls.ec else \
            measure_e2e(args, calls.layer, wl, dev)
    if rank == 0 and cpu_budget_s:
        host = host_copy(tensors)
        del tensors, calls, x
        res["cpu_baseline"] = cpu_baseline(wl, host, cpu_budget_s)
    return res


def run_train(args, wl, rank, world, local_rank, cpu_budget_s=None):
    """One step = moe_forward + moe_backward of total = task + 0.01 balance with
    a fixed synthetic dy, captured once as a CUDA graph and replayed."""
    import torch
    import torch.distributed as dist

    from sparse_mixture_experts_68_b300 import binding as B
    from sparse_mixture_experts_68_b300 import synth
    from sparse_mixture_experts_68_b300.workloads import flops

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    tensors = synth.make_layer(wl, device=dev)
    layer = B.MoeLayer(wl, tensors, device=dev)
    cfg = layer.cfg
    # the forward keeps the first Linear's pre-activation for the backward
    out = B.alloc_outputs(cfg, dev, with_pre_act=True)
    grads = B.alloc_grads(cfg, dev)
    bws = torch.empty(B.backward_workspace_size(cfg), dtype=torch.uint8, device=dev)
    g = torch.Generator(device="cpu").manual_seed(7)
    dy = torch.randn((wl.T, wl.d_model), generator=g).to(torch.bfloat16).to(dev)
    x = tensors["x"]
    flush = L2Flush(dev)
    torch.cuda.synchronize(dev)          # see run_ours: the layer runs on its own stream
    stream = torch.cuda.Stream(dev)
    fev = [torch.cuda.Event(enable_timing=True) for _ in range(7)]
    bev = [torch.cuda.Event(enable_timing=True) for _ in range(8)]

    def step():
        B.forward(cfg, x, layer.weights, out, layer.workspace, stream)
        B.backward(cfg, x, layer.weights, out, layer.workspace, dy, AUX_WEIGHT, grads, bws,
                   stream)

    def step_profiled():
        B.forward_profiled(cfg, x, layer.weights, out, layer.workspace, fev, stream)
        B.backward_profiled(cfg, x, layer.weights, out, layer.workspace, dy, AUX_WEIGHT, grads,
                            bws, bev, stream)

    with torch.cuda.stream(stream):
        for ev in fev + bev:
            ev.record(stream)
        for _ in range(3):
            step_profiled()
            step()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    torch.cuda.synchronize(dev)

    def flush_l2(i):
        flush(i, stream)

    for i in range(max(args.warmup, 3)):
        flush_l2(i)
        with torch.cuda.stream(stream):
            graph.replay()
    torch.cuda.synchronize(dev)
    assert B.get_device_status() == B.MOE_OK
    K = args.steps
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.05)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks.mark_start()
    marks = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(K)]
    for i in range(K):
        flush_l2(i)
        with torch.cuda.stream(stream):
            marks[i][0].record(stream)
            graph.replay()
            marks[i][1].record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark_end()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    total_ms = job_time_ms(sum(a.elapsed_time(b) for a, b in marks), world, dev)
    fwd_stage, bwd_stage = [], []
    for i in range(K):
        flush_l2(i)
        with torch.cuda.stream(stream):
            step_profiled()
        stream.synchronize()
        fwd_stage.append([fev[j].elapsed_time(fev[j + 1]) for j in range(6)])
        bwd_stage.append([bev[j].elapsed_time(bev[j + 1]) for j in range(7)])
    assert B.get_device_status() == B.MOE_OK
    fnames = STAGES
    bnames = ("gate", "recompute_A1", "dgrad_dA", "dgrad_dXp", "wgrad_dW2",
              "wgrad_dW1", "bias_router_dx")        # recompute_A1: ~0, the forward kept A1
    fmean = {n: statistics.mean(s[i] for s in fwd_stage) for i, n in enumerate(fnames)}
    bmean = {n: statistics.mean(s[i] for s in bwd_stage) for i, n in enumerate(bnames)}

    kept_rows = int(out.kept.sum().item())
    n_kept = int((out.kept > 0).sum().item())
    T = cfg.T
    rows = kept_rows + (T if wl.d_ff_shared else 0)
    es = wl.elem_bytes
    pk = peaks()
    gemm_flop = 2.0 * wl.d_model * wl.d_ff * rows           # one grouped GEMM launch
    wbytes = (n_kept + (1 if wl.d_ff_shared else 0)) * wl.d_model * wl.d_ff * es
    act = rows * (wl.d_model + wl.d_ff) * es
    # the forward's first Linear also stores the pre-activation, so the
    # backward has no recompute: six grouped GEMM launches per step
    gemm_names = [("forward_linear1", fmean["ffn_linear1"]), ("forward_linear2",
                                                               fmean["ffn_linear2"])] + \
        [(n, bmean[n]) for n in ("dgrad_dA", "dgrad_dXp", "wgrad_dW2", "wgrad_dW1")]
    gemm_ms = sum(ms for _, ms in gemm_names)
    launches = len(gemm_names)
    gemm_bytes = launches * (wbytes + act)
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    if wl.dtype != 1:                   # fp32: FFMA on the CUDA cores
        ach = gemm_flop * launches / (gemm_ms * 1e-3) / 1e12
        roof = {"bound": "alu", "achieved": ach, "peak": F32_ALU_TFLOPS, "unit": "TFLOP/s"}
    elif gemm_flop * launches / gemm_bytes >= ridge:
        ach = gemm_flop * launches / (gemm_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops"], "unit": "TFLOP/s"}
    else:
        ach = gemm_bytes / (gemm_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = None
    roof["traffic_source"] = "no ncu summary for the training step"
    if wl.dtype != 1:
        roof["kernel"] = ("CUDA-core GEMMs: simt_gemm_kernel (forward Linears, dgrads) and "
                          "simt_wgrad_kernel (wgrads)")
        roof["peak_source"] = F32_ALU_SOURCE
    else:
        roof["kernel"] = ("tcgen05 grouped GEMMs: tc_grouped_gemm_kernel / "
                          "tc2_grouped_gemm_kernel (forward Linear 1 keeping its "
                          "pre-activation, Linear 2; dgrads on CTA pairs) and "
                          "tc_bwd_gemm_kernel (dgrads, wgrads)")
        roof["peak_source"] = pk["source"] + " (burst)"
    roof["per_launch"] = {n: {"ms": ms, "tflops": gemm_flop / (ms * 1e-3) / 1e12}
                          for n, ms in gemm_names}
    train_flop = 6.0 * gemm_flop + 3 * 2.0 * T * wl.d_model * wl.n_experts
    res = {
        "metric": TRAIN_METRIC, "value": job_tokens_per_s(T, K, world, total_ms),
        "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if wl.dtype == 1 else "f32", "data": "synthetic",
        "config": run_config(wl, world, train=True),
        "launch": "moe_forward + moe_backward captured once as a CUDA graph, replayed; "
                  "per-kernel times from direct *_profiled calls",
        "tflops": train_flop / (total_ms / K * 1e-3) / 1e12,
        "forward_stage_ms": fmean, "backward_stage_ms": bmean,
        "roofline": roof,
        # the backward skips its recompute launch (the forward kept the
        # pre-activation from its epilogue)
        "gpu_launches": (B.forward_launch_count(cfg) + B.backward_launch_count(cfg) - 1) * K,
        "clocks": clk,
    }
    del flops
    if not args.no_e2e:
        xh = x.cpu().pin_memory()
        dyh = dy.cpu().pin_memory()
        xd, dyd = torch.empty_like(x), torch.empty_like(dy)
        dxh = torch.empty(grads.dx.shape, dtype=grads.dx.dtype).pin_memory()
        cur = torch.cuda.current_stream(dev)

        def e2e_step():
            xd.copy_(xh, non_blocking=True)
            dyd.copy_(dyh, non_blocking=True)
            B.forward(cfg, xd, layer.weights, out, layer.workspace, cur)
            B.backward(cfg, xd, layer.weights, out, layer.workspace, dyd, AUX_WEIGHT, grads,
                       bws, cur)
            dxh.copy_(grads.dx, non_blocking=True)
            cur.synchronize()

        for _ in range(3):
            e2e_step()
        t0 = time.perf_counter()
        for _ in range(K):
            e2e_step()
        dt = time.perf_counter() - t0
        res["e2e"] = {"value": T * K / dt, "unit": "tokens/s",
                      "h2d_bytes_per_step": 2 * T * wl.d_model * es,
                      "d2h_bytes_per_step": T * wl.d_model * es,
                      "api": "moe_forward + moe_backward between pinned host copies of x, dy "
                             "and dx on one stream (synchronous)"}
    if rank == 0 and cpu_budget_s:
        host = host_copy(tensors)
        del tensors, layer, out, grads, bws
        res["cpu_baseline"] = cpu_baseline(wl, host, cpu_budget_s, train=True)
    return res


def measure_e2e(args, layer, wl, dev):
    """Same metric through moe_forward_host: tokens copied in from pinned host
    memory and the results copied back inside the timed call."""
    import torch

    from sparse_mixture_experts_68_b300 import binding as B
    cfg = layer.cfg
    ws = torch.empty(B.host_workspace_size(cfg), dtype=torch.uint8, device=dev)
    xh = layer.t["x"].cpu().pin_memory()
    oh = B.alloc_outputs(cfg, "cpu", pin_memory=True)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        B.forward_host(cfg, xh, layer.weights, oh, ws, stream)
    K = args.steps
    t0 = time.perf_counter()
    for _ in range(K):
        B.forward_host(cfg, xh, layer.weights, oh, ws, stream)
    dt = time.perf_counter() - t0
    es = wl.elem_bytes
    T, k, N = cfg.T, cfg.top_k, cfg.n_experts
    h2d = T * wl.d_model * es
    d2h = T * wl.d_model * es + T * k * 8 + N * 12 + 8
    return {"value": T * K / dt, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "api": "moe_forward_host (host buffers, synchronous)"}


def measure_e2e_ec(args, calls, wl, dev):
    """Expert-choice layer end to end: x copied in from pinned host memory,
    moe_ec_forward, y and the per-expert picks copied back, all on one stream
    and inside the timed loop."""
    import torch
    cfg = calls.cfg
    stream = torch.cuda.current_stream(dev)
    xh = calls.layer.t["x"].cpu().pin_memory()
    xd = torch.empty_like(calls.layer.t["x"])
    o = calls.out
    yh = torch.empty(o.y.shape, dtype=o.y.dtype).pin_memory()
    th = torch.empty(o.ec_token.shape, dtype=o.ec_token.dtype).pin_memory()
    gh = torch.empty(o.ec_gate.shape, dtype=o.ec_gate.dtype).pin_memory()

    def step():
        xd.copy_(xh, non_blocking=True)
        calls.forward(xd, stream)
        yh.copy_(o.y, non_blocking=True)
        th.copy_(o.ec_token, non_blocking=True)
        gh.copy_(o.ec_gate, non_blocking=True)
        stream.synchronize()

    for _ in range(3):
        step()
    K = args.steps
    t0 = time.perf_counter()
    for _ in range(K):
        step()
    dt = time.perf_counter() - t0
    es = wl.elem_bytes
    T = cfg.T
    return {"value": T * K / dt, "unit": "tokens/s", "h2d_bytes_per_step": T * wl.d_model * es,
            "d2h_bytes_per_step": T * wl.d_model * es + th.numel() * 4 + gh.numel() * 4,
            "api": "moe_ec_forward between pinned host copies on its stream (synchronous)"}


def main():
    args = parse()
    from sparse_mixture_experts_68_b300.workloads import WORKLOADS
    wl = WORKLOADS[args.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        res = run_reference(args, wl, rank, world)
        if rank == 0 and res is not None:
            print(json.dumps(res), flush=True)
        return

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    import torch
    cpu = not args.no_cpu_baseline
    if args.mode == "train":
        res = run_train(args, wl, rank, world, local_rank, cpu_budget_s=24.0 if cpu else None)
    else:
        res = run_ours(args, wl, rank, world, local_rank, cpu_budget_s=24.0 if cpu else None)
        subs = [n for n in args.sub_workloads.split(",") if n and n != "none" and n != wl.name]
        if subs:
            res["per_workload"] = {}
        for name in subs:
            torch.cuda.empty_cache()
            res["per_workload"][name] = run_ours(args, WORKLOADS[name], rank, world, local_rank,
                                                 cpu_budget_s=6.0 if cpu else None)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
