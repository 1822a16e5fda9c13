// C ABI of libmoe (declared in include/moe.h): host-side validation,
// workspace layout, and the sequence of launches of one layer.
#include <cuda.h>
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {

__device__ int32_t g_device_status = MOE_OK;

namespace {

std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};

// One NVTX range (a profiler's timeline label) for the scope of a call or a
// step; nothing happens unless a profiler is attached.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t elem_bytes(const moe_config& c) { return c.dtype == MOE_F32 ? 4 : 2; }

moe_status check_config(const moe_config* cfg) {
  if (!cfg) return MOE_ERR_INVALID_ARG;
  const moe_config& c = *cfg;
  if (c.T < 0 || c.d_model <= 0 || c.d_ff <= 0 || c.n_experts < 1 || c.top_k < 1 ||
      c.top_k > c.n_experts || c.d_ff_shared < 0 || c.reserved != 0)
    return MOE_ERR_INVALID_ARG;
  if (c.dtype != MOE_F32 && c.dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c.act != MOE_ACT_GELU_ERF && c.act != MOE_ACT_RELU) return MOE_ERR_INVALID_ARG;
  if (c.renormalize != 0 && c.renormalize != 1) return MOE_ERR_INVALID_ARG;
  if (c.n_experts > 1024) return MOE_ERR_UNSUPPORTED;
  if (c.d_model % 8 != 0 || c.d_ff % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (c.dtype == MOE_BF16 && (c.d_model % 64 != 0 || c.d_ff % 64 != 0))
    return MOE_ERR_UNSUPPORTED;
  if (c.d_ff_shared != 0 && c.d_ff_shared != c.d_ff) return MOE_ERR_UNSUPPORTED;
  // 32-bit row indices inside the kernels
  const int64_t rows = c.T * c.top_k + c.n_experts * (kGroupAlign - 1) + c.T + kGroupAlign;
  if (rows >= (int64_t(1) << 31) || c.T * c.top_k >= (int64_t(1) << 31))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int64_t rows_max_of(const moe_config& c) {
  int64_t r = c.T * c.top_k + c.n_experts * (kGroupAlign - 1);
  if (c.d_ff_shared > 0) r += round_up(c.T, kGroupAlign);
  return r;
}

int64_t router_blocks_of(const moe_config& c) { return router_partial_rows(c); }

// Workspace of moe_forward: every region 256-byte aligned.
struct Workspace {
  float* logits;
  float* prob_partials;
  int32_t* offsets;
  int32_t* row_token;
  int32_t* token_row;
  void* scratch;
  size_t scratch_bytes;
  void* Xp;
  void* H;
  void* Yp;
  float* front_part;      // small-batch front end: router score slices (or nullptr)
  float* sk_partials;     // stream-K decode tiles (nullptr when the layer has none)
  int32_t* sk_counters;
  int64_t sk_counter_ints;
  size_t bytes;
  // checks build: a 256-byte guard after every region (offsets from the base)
  static constexpr int kMaxGuards = 16;
  int64_t guard[kMaxGuards];
  int32_t n_guards;
};

#ifdef MOE_CHECKS
constexpr size_t kGuardBytes = 256;
#else
constexpr size_t kGuardBytes = 0;
#endif

Workspace layout(const moe_config& c, void* base) {
  Workspace w{};
  uintptr_t p = reinterpret_cast<uintptr_t>(base);
  size_t off = 0;
  auto take = [&](size_t n) {
    const size_t at = off;
    off += (n + 255) / 256 * 256;
    if (kGuardBytes > 0 && w.n_guards < Workspace::kMaxGuards) {
      w.guard[w.n_guards++] = int64_t(off);
      off += kGuardBytes;
    }
    return reinterpret_cast<void*>(p + at);
  };
  const int64_t rows = rows_max_of(c);
  const int64_t es = elem_bytes(c);
  w.logits = static_cast<float*>(take(size_t(c.T * c.n_experts) * 4));
  w.prob_partials = static_cast<float*>(take(size_t(router_blocks_of(c) * c.n_experts) * 4));
  w.offsets = static_cast<int32_t*>(take(size_t(c.n_experts + 2) * 4));
  w.row_token = static_cast<int32_t*>(take(size_t(rows) * 4));
  w.token_row = static_cast<int32_t*>(take(size_t(c.T * c.top_k) * 4));
  w.scratch_bytes = permute_scratch_bytes(c);
  w.scratch = take(w.scratch_bytes);
  w.Xp = take(size_t(rows * c.d_model * es));
  w.H = take(size_t(rows * c.d_ff * es));
  w.Yp = take(size_t(rows * c.d_model * es));
  const int64_t fp = small_front_partial_floats(c);
  if (fp > 0) w.front_part = static_cast<float*>(take(size_t(fp) * 4));
  const size_t skp = sk_partial_bytes(c);
  if (skp > 0) {
    w.sk_counter_ints = sk_counter_ints(c, 1) + sk_counter_ints(c, 2);
    w.sk_partials = static_cast<float*>(take(skp));
    w.sk_counters = static_cast<int32_t*>(take(size_t(w.sk_counter_ints) * 4));
  }
  w.bytes = off;
  return w;
}

// ---- backward ----

struct BwdWorkspace {
  void* dO;
  void* A1;
  void* dA;
  void* dXp;
  float* dz;
  float* dw;
  float* dxr;
  void* dz_bf;
  void* dxr_bf;
  int32_t* rgrp;
  float* part;
  float* bpart;
  size_t bytes;
};

BwdWorkspace bwd_layout(const moe_config& c, void* base) {
  BwdWorkspace w{};
  uintptr_t p = reinterpret_cast<uintptr_t>(base);
  size_t off = 0;
  auto take = [&](size_t n) {
    const size_t at = off;
    off += (n + 255) / 256 * 256;
    return reinterpret_cast<void*>(p + at);
  };
  const int64_t rows = rows_max_of(c);
  const int64_t es = elem_bytes(c);
  w.dO = take(size_t(rows * c.d_model * es));
  w.A1 = take(size_t(rows * c.d_ff * es));
  w.dA = take(size_t(rows * c.d_ff * es));
  w.dXp = take(size_t(rows * c.d_model * es));
  w.dz = static_cast<float*>(take(size_t(c.T * c.n_experts) * 4));
  w.dw = static_cast<float*>(take(size_t(c.T * c.top_k) * 4));
  w.dxr = static_cast<float*>(take(size_t(c.T * c.d_model) * 4));
  w.dz_bf = take(size_t(c.T * c.n_experts) * 2);
  w.dxr_bf = take(size_t(round_up(c.T, kGroupAlign) * c.d_model) * 2);
  w.rgrp = static_cast<int32_t*>(take(16));
  w.part = static_cast<float*>(take(router_bwd_partial_bytes(c)));
  w.bpart = static_cast<float*>(take(bias_partial_bytes(c, rows)));
  w.bytes = off;
  return w;
}

moe_status check_bwd_config(const moe_config* cfg) { return check_config(cfg); }

// ---- expert-choice routing ----

int64_t ec_tokens_of(const moe_config& c) {
  return c.capacity <= 0 ? c.T : (c.capacity < c.T ? c.capacity : c.T);
}

int64_t ec_rows_max_of(const moe_config& c) {
  int64_t r = c.n_experts * ec_group_rows(ec_tokens_of(c));
  if (c.d_ff_shared > 0) r += round_up(c.T, kGroupAlign);
  return r;
}

// the top-k fields are not read; everything else as for top-k routing
moe_status check_ec_config(const moe_config* cfg) {
  if (!cfg) return MOE_ERR_INVALID_ARG;
  moe_config c = *cfg;
  c.top_k = 1;
  c.renormalize = 1;
  const moe_status st = check_config(&c);
  if (st != MOE_OK) return st;
  if (ec_rows_max_of(c) >= (int64_t(1) << 31) || c.T * c.n_experts >= (int64_t(1) << 31))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// the layer configuration the shared kernels see: one combine slot per expert
moe_config ec_kernel_config(const moe_config& c) {
  moe_config k = c;
  k.top_k = c.n_experts;
  k.capacity = 0;
  k.renormalize = 1;
  return k;
}

struct EcWorkspace {
  float* logits;
  float* probT;
  float* prob_partials;
  int32_t* offsets;
  int32_t* counts;
  int32_t* row_token;
  int32_t* token_row;
  float* token_w;
  int32_t* scratch;
  void* Xp;
  void* H;
  void* Yp;
  size_t bytes;
};

EcWorkspace ec_layout(const moe_config& c, void* base) {
  EcWorkspace w{};
  uintptr_t p = reinterpret_cast<uintptr_t>(base);
  size_t off = 0;
  auto take = [&](size_t n) {
    const size_t at = off;
    off += (n + 255) / 256 * 256;
    return reinterpret_cast<void*>(p + at);
  };
  const int64_t rows = ec_rows_max_of(c);
  const int64_t es = elem_bytes(c);
  const size_t tn = size_t(c.T * c.n_experts) * 4;
  w.logits = static_cast<float*>(take(tn));
  w.probT = static_cast<float*>(take(tn));
  w.prob_partials = static_cast<float*>(take(size_t(router_blocks_of(c) * c.n_experts) * 4));
  w.offsets = static_cast<int32_t*>(take(size_t(c.n_experts + 2) * 4));
  w.counts = static_cast<int32_t*>(take(size_t(c.n_experts) * 4));
  w.row_token = static_cast<int32_t*>(take(size_t(rows) * 4));
  w.token_row = static_cast<int32_t*>(take(tn));
  w.token_w = static_cast<float*>(take(tn));
  w.scratch = static_cast<int32_t*>(take(4));
  w.Xp = take(size_t(rows * c.d_model * es));
  w.H = take(size_t(rows * c.d_ff * es));
  w.Yp = take(size_t(rows * c.d_model * es));
  w.bytes = off;
  return w;
}

}  // namespace

// Unique id of the calling thread's current CUDA context, 0 when none is
// current or the driver cannot say.  Per-device caches of device addresses and
// kernel attributes belong to one context; after cudaDeviceReset the device's
// next context has a new id, so a cache keyed on it is refilled.
uint64_t context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  CUcontext c = nullptr;
  if (!get_current || !get_id || get_current(&c) != CUDA_SUCCESS || c == nullptr) return 0;
  unsigned long long id = 0;
  return get_id(c, &id) == CUDA_SUCCESS ? uint64_t(id) : 0;
}

namespace {

// Device status word address and SM count, per device (and context).
struct DeviceInfo {
  int32_t* status = nullptr;
  int num_sms = 0;
  uint64_t ctx = 0;
};

bool device_info(DeviceInfo* out) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(mu);
  const uint64_t ctx = context_id();
  if (!cache[dev].status || (ctx != 0 && ctx != cache[dev].ctx)) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_device_status) != cudaSuccess) return false;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return false;
    cache[dev].status = static_cast<int32_t*>(ptr);
    cache[dev].num_sms = sms;
    cache[dev].ctx = context_id();       // current now: the lookup made it so
  }
  *out = cache[dev];
  return true;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

moe_status check_weights(const moe_config& c, const moe_weights* w, bool router, bool experts) {
  if (!w) return MOE_ERR_INVALID_ARG;
  if (router && (!w->W_g || !w->b_g || !aligned16(w->W_g) || !aligned16(w->b_g)))
    return MOE_ERR_INVALID_ARG;
  if (experts) {
    const void* ps[] = {w->W1, w->b1, w->W2, w->b2};
    for (const void* q : ps)
      if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
    if (c.d_ff_shared > 0) {
      const void* ss[] = {w->W1s, w->b1s, w->W2s, w->b2s};
      for (const void* q : ss)
        if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
    }
  }
  return MOE_OK;
}

__global__ void bounded_wait_selftest_kernel(uint64_t limit_ns, int32_t* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // nothing arrives on `bar`: the wait runs out after limit_ns
    mbar_wait_bounded(&bar, 0, limit_ns, status);
  }
}

__global__ void activation_kernel(int act, const float* __restrict__ x, float* __restrict__ y,
                                  int64_t n) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x)
    y[i] = apply_act(x[i], act);
}

}  // namespace

moe_status validate_config(const moe_config* cfg) { return check_config(cfg); }
int64_t rows_max_for(const moe_config& c) { return rows_max_of(c); }

cudaError_t launch_bounded_wait_selftest(uint64_t limit_ns, int32_t* status, cudaStream_t s) {
  bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace moe

namespace moe {

cudaError_t record_event(void* event, cudaStream_t s) {
  if (!event) return cudaSuccess;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cs);
  if (e != cudaSuccess) return e;
  return cudaEventRecordWithFlags(static_cast<cudaEvent_t>(event), s,
                                  cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal
                                                                      : cudaEventRecordDefault);
}

}  // namespace moe

using namespace moe;

extern "C" {

int32_t moe_version(void) { return 1; }

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported layer shape";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

void moe_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns); }
uint64_t moe_get_wait_limit_ns(void) { return g_wait_limit_ns.load(); }

int64_t moe_rows_max(const moe_config* cfg) {
  if (check_config(cfg) != MOE_OK) return -1;
  return rows_max_of(*cfg);
}

int64_t moe_router_blocks(const moe_config* cfg) {
  if (check_config(cfg) != MOE_OK) return -1;
  return router_blocks_of(*cfg);
}

size_t moe_permute_scratch_size(const moe_config* cfg) {
  if (check_config(cfg) != MOE_OK) return 0;
  return permute_scratch_bytes(*cfg);
}

size_t moe_workspace_size(const moe_config* cfg) {
  if (check_config(cfg) != MOE_OK) return 0;
  return layout(*cfg, nullptr).bytes;
}

moe_status moe_router_topk(const moe_config* cfg, const void* x, const void* W_g,
                           const void* b_g, float* logits, int32_t* topk_idx, float* topk_w,
                           float* prob_partials, void* stream) {
  moe_status st = check_config(cfg);
  if (st != MOE_OK) return st;
  const void* ps[] = {x, W_g, b_g, logits, topk_idx, topk_w, prob_partials};
  for (const void* q : ps)
    if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  DeviceInfo di;
  if (!device_info(&di)) return MOE_ERR_CUDA;
  return cuda_status(launch_router(*cfg, x, W_g, b_g, logits, topk_idx, topk_w, prob_partials,
                                   di.num_sms, di.status, g_wait_limit_ns.load(),
                                   static_cast<cudaStream_t>(stream)));
}

moe_status moe_permute(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                       int32_t* counts, int32_t* kept, int32_t* offsets, int32_t* row_token,
                       int32_t* token_row, void* Xp, void* scratch, size_t scratch_bytes,
                       void* stream) {
  moe_status st = check_config(cfg);
  if (st != MOE_OK) return st;
  const void* ps[] = {x, topk_idx, counts, kept, offsets, row_token, token_row, Xp, scratch};
  for (const void* q : ps)
    if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  if (scratch_bytes < permute_scratch_bytes(*cfg)) return MOE_ERR_WORKSPACE;
  return cuda_status(launch_permute(*cfg, x, topk_idx, counts, kept, offsets, row_token,
                                    token_row, Xp, scratch, rows_max_of(*cfg),
                                    static_cast<cudaStream_t>(stream), nullptr, nullptr, 0));
}

moe_status moe_grouped_ffn(const moe_config* cfg, const void* Xp, const int32_t* offsets,
                           const int32_t* kept, const moe_weights* w, void* H, void* Yp,
                           void* stream) {
  moe_status st = check_config(cfg);
  if (st != MOE_OK) return st;
  st = check_weights(*cfg, w, false, true);
  if (st != MOE_OK) return st;
  const void* ps[] = {Xp, offsets, kept, H, Yp};
  for (const void* q : ps)
    if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  DeviceInfo di;
  if (!device_info(&di)) return MOE_ERR_CUDA;
  GroupedFfnArgs a{};
  a.Xp = Xp; a.offsets = offsets; a.kept = kept; a.w = w; a.H = H; a.Yp = Yp;
  a.rows_max = rows_max_of(*cfg);
  a.status = di.status;
  a.wait_limit_ns = g_wait_limit_ns.load();
  a.num_sms = di.num_sms;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return cuda_status(cfg->dtype == MOE_F32 ? launch_grouped_ffn_f32(*cfg, a, s)
                                           : launch_grouped_ffn_bf16(*cfg, a, s));
}

moe_status moe_combine(const moe_config* cfg, const void* Yp, const int32_t* token_row,
                       const float* topk_w, const int32_t* offsets, void* y, void* stream) {
  moe_status st = check_config(cfg);
  if (st != MOE_OK) return st;
  const void* ps[] = {Yp, token_row, topk_w, offsets, y};
  for (const void* q : ps)
    if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(*cfg, Yp, token_row, topk_w, offsets, y,
                                    static_cast<cudaStream_t>(stream)));
}

moe_status moe_load_stats(const moe_config* cfg, const float* prob_partials,
                          const int32_t* counts, const int32_t* kept, float* mean_prob,
                          float* balance, int32_t* dropped, float* cv_squared,
                          void* stream) {
  moe_status st = check_config(cfg);
  if (st != MOE_OK) return st;
  const void* ps[] = {prob_partials, counts, kept, mean_prob, balance, dropped};
  for (const void* q : ps)
    if (!q) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_load_stats(*cfg, prob_partials, counts, kept, mean_prob, balance,
                                       dropped, cv_squared, static_cast<cudaStream_t>(stream)));
}

// One token chunk of a batch (moe_forward_host): the router writes its
// probability partial-sum rows to prob_rows, and the chunk computes no
// statistics (counts and kept are still written; the batch's statistics come
// after the last chunk).
struct ChunkMode {
  float* prob_rows;
};

static moe_status forward_impl(const moe_config* cfg, const void* x, const moe_weights* w,
                               const moe_outputs* out, void* workspace, size_t workspace_bytes,
                               void* const* events, void* stream,
                               const ChunkMode* chunk = nullptr) {
  moe_status st = check_config(cfg);
  if (st != MOE_OK) return st;
  const moe_config& c = *cfg;
  st = check_weights(c, w, true, true);
  if (st != MOE_OK) return st;
  // token-sized buffers may be NULL when there are no tokens
  auto token_buf_ok = [&](const void* q) { return c.T == 0 || (q && aligned16(q)); };
  if (!out || !token_buf_ok(x) || !workspace ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return MOE_ERR_INVALID_ARG;
  if (!token_buf_ok(out->y) || !token_buf_ok(out->topk_idx) || !token_buf_ok(out->topk_w))
    return MOE_ERR_INVALID_ARG;
  const void* ps[] = {out->counts, out->kept};
  for (const void* q : ps)
    if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  if (!out->dropped || !out->mean_prob || !out->balance) return MOE_ERR_INVALID_ARG;
  if (out->logits && !aligned16(out->logits)) return MOE_ERR_INVALID_ARG;
  if (out->pre_act && !aligned16(out->pre_act)) return MOE_ERR_INVALID_ARG;
  Workspace ws = layout(c, workspace);
  if (workspace_bytes < ws.bytes) return MOE_ERR_WORKSPACE;
  DeviceInfo di;
  if (!device_info(&di)) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* logits = out->logits ? out->logits : ws.logits;
  void* const none[7] = {};
  void* const* ev = events ? events : none;

  const NvtxRange call_range("moe_forward");
  // a few tokens and experts: router, sort and statistics in the two
  // front-end kernels, then the row copy
  const bool front = ws.front_part != nullptr && chunk == nullptr;
  float* prob_rows = chunk ? chunk->prob_rows : ws.prob_partials;
  cudaError_t e = record_event(ev[0], s);
  if (e == cudaSuccess) {
    const NvtxRange r("router_topk");
    if (front)
      e = launch_small_front(c, x, w->W_g, w->b_g, ws.front_part, logits, out->topk_idx,
                             out->topk_w, out->counts, out->kept, ws.offsets, ws.row_token,
                             ws.token_row, out->mean_prob, out->balance, out->dropped,
                             out->cv_squared, s);
    else
      e = launch_router(c, x, w->W_g, w->b_g, logits, out->topk_idx, out->topk_w,
                        prob_rows, di.num_sms, di.status, g_wait_limit_ns.load(), s);
  }
  if (e == cudaSuccess) e = record_event(ev[1], s);
  // small layers: the one-block permutation also computes the load statistics
  const bool fused_stats = chunk == nullptr && (front || permute_fuses_stats(c));
  const StatsArgs stats{ws.prob_partials, int(router_blocks_of(c)), out->mean_prob,
                        out->balance, out->dropped, out->cv_squared};
  if (e == cudaSuccess) {
    const NvtxRange r("permute");
    if (front)
      e = launch_row_copy(c, x, ws.offsets, ws.row_token, ws.Xp, rows_max_of(c), s,
                          ws.sk_counters, ws.sk_counter_ints);
    else
      e = launch_permute(c, x, out->topk_idx, out->counts, out->kept, ws.offsets,
                         ws.row_token, ws.token_row, ws.Xp, ws.scratch, rows_max_of(c), s,
                         fused_stats ? &stats : nullptr, ws.sk_counters, ws.sk_counter_ints);
  }
  if (e == cudaSuccess) e = record_event(ev[2], s);
  if (e == cudaSuccess) {
    const NvtxRange r("grouped_ffn");
    GroupedFfnArgs a{};
    a.Xp = ws.Xp; a.offsets = ws.offsets; a.kept = out->kept; a.w = w; a.H = ws.H;
    a.Yp = ws.Yp; a.rows_max = rows_max_of(c); a.status = di.status;
    a.wait_limit_ns = g_wait_limit_ns.load(); a.num_sms = di.num_sms;
    a.mid_event = ev[3];
    a.pre_out = out->pre_act;
    a.sk_partials = ws.sk_partials;
    a.sk_counters = ws.sk_counters;
    e = c.dtype == MOE_F32 ? launch_grouped_ffn_f32(c, a, s) : launch_grouped_ffn_bf16(c, a, s);
  }
  if (e == cudaSuccess) e = record_event(ev[4], s);
  if (e == cudaSuccess) {
    const NvtxRange r("combine");
    e = launch_combine(c, ws.Yp, ws.token_row, out->topk_w, ws.offsets, out->y, s);
  }
  if (e == cudaSuccess) e = record_event(ev[5], s);
  if (e == cudaSuccess && !fused_stats && chunk == nullptr) {
    const NvtxRange r("load_stats");
    e = launch_load_stats(c, ws.prob_partials, out->counts, out->kept, out->mean_prob,
                          out->balance, out->dropped, out->cv_squared, s);
  }
  if (e == cudaSuccess) e = record_event(ev[6], s);
  return cuda_status(e);
}

moe_status moe_forward(const moe_config* cfg, const void* x, const moe_weights* w,
                       const moe_outputs* out, void* workspace, size_t workspace_bytes,
                       void* stream) {
  return forward_impl(cfg, x, w, out, workspace, workspace_bytes, nullptr, stream);
}

moe_status moe_forward_profiled(const moe_config* cfg, const void* x, const moe_weights* w,
                                const moe_outputs* out, void* workspace,
                                size_t workspace_bytes, void* const* events, void* stream) {
  if (!events) return MOE_ERR_INVALID_ARG;
  // kernels run back to back without overlapping, so each event pair times one step
  pdl_enabled() = false;
  const moe_status st = forward_impl(cfg, x, w, out, workspace, workspace_bytes, events, stream);
  pdl_enabled() = true;
  return st;
}

int32_t moe_forward_launch_count(const moe_config* cfg) {
  if (check_config(cfg) != MOE_OK) return -1;
  const moe_config& c = *cfg;
  const int ffn = rows_max_of(c) > 0 ? 2 : 0;
  if (small_front_fits(c)) return 2 + (rows_max_of(c) > 0 ? 1 : 0) + ffn + 1;
  return router_launch_count(c) + permute_launch_count(c) + ffn + (c.T > 0 ? 1 : 0) +
         (permute_fuses_stats(c) ? 0 : 1);
}

const char* moe_ffn_kernel_name(const moe_config* cfg, int32_t linear) {
  if (check_config(cfg) != MOE_OK || (linear != 1 && linear != 2)) return nullptr;
  return grouped_linear_kernel_name(*cfg, linear, 0);
}

// Chunk halves: tokens [0, T0) and [T0, T), T0 a multiple of 4 so that every
// per-token array of the second chunk starts on a 16-byte boundary.
static moe_config chunk_cfg(const moe_config& c, int i) {
  moe_config h = c;
  const int64_t t0 = (c.T / 2) & ~int64_t(3);
  h.T = i == 0 ? t0 : c.T - t0;
  return h;
}

// moe_forward_host overlaps its copies with the layer by running the batch as
// two token chunks on the caller's stream, with the copies on a second stream:
// chunk 1's tokens go in while chunk 0 runs, chunk 0's results come out while
// chunk 1 runs.  Per token nothing changes -- routing, the grouped rows and the
// combine are per token, and a half runs the same grouped-FFN kernels as the
// whole batch -- so it is only done when that holds: no capacity (which would
// depend on the whole batch), at least 1024 tokens, the same kernels, and
// either FFN work above the ridge for a half (>= 256 rows per expert) or
// weights small enough to be read twice (<= 96 MB).  The statistics of the
// whole batch come from both chunks' partial sums after the second chunk.
static int host_chunks(const moe_config& c) {
  if (c.capacity > 0 || c.T < 1024 || c.dtype != MOE_BF16) return 1;
  const moe_config h = chunk_cfg(c, 0);
  if (small_front_fits(h)) return 1;
  for (int linear = 1; linear <= 2; ++linear) {
    const char* a = grouped_linear_kernel_name(c, linear, 0);
    const char* b = grouped_linear_kernel_name(h, linear, 0);
    if (a == nullptr || b == nullptr || std::strcmp(a, b) != 0) return 1;
  }
  if (linear_saves_pre(c) != linear_saves_pre(h)) return 1;
  const double rows_per_group = double(h.T * h.top_k) / double(c.n_experts);
  const double wbytes = 4.0 * double(c.n_experts + (c.d_ff_shared > 0 ? 1 : 0)) *
                        double(c.d_model) * double(c.d_ff);   // both Linears, bf16
  if (rows_per_group < 256.0 && wbytes > 96.0 * 1024 * 1024) return 1;
  return 2;
}

// Bytes of the chunked path's scratch: both chunks' probability partial-sum
// rows, their counts and kept counts, and per-chunk statistics outputs the
// chunks do not fill.
static size_t chunk_scratch_bytes(const moe_config& c) {
  if (host_chunks(c) < 2) return 0;
  auto r = [](size_t n) { return (n + 255) / 256 * 256; };
  const size_t N = size_t(c.n_experts);
  const size_t rows = size_t(router_partial_rows(chunk_cfg(c, 0)) +
                             router_partial_rows(chunk_cfg(c, 1)));
  return r(rows * N * 4) + 5 * r(N * 4) + 3 * r(4);
}

size_t moe_host_workspace_size(const moe_config* cfg) {
  if (check_config(cfg) != MOE_OK) return 0;
  const moe_config& c = *cfg;
  auto r = [](size_t n) { return (n + 255) / 256 * 256; };
  const size_t es = size_t(elem_bytes(c));
  return layout(c, nullptr).bytes + 2 * r(size_t(c.T * c.d_model) * es) +
         2 * r(size_t(c.T * c.top_k) * 4) + 3 * r(size_t(c.n_experts) * 4) + 3 * r(4) +
         r(size_t(c.T * c.n_experts) * 4) +   // dropped, balance, cv_squared; logits
         chunk_scratch_bytes(c);
}

int32_t moe_forward_host_chunks(const moe_config* cfg) {
  if (check_config(cfg) != MOE_OK) return -1;
  return host_chunks(*cfg);
}

// The second stream and the events of the chunked path, one set per device and
// context; a call holds its device's lock from the first copy to the final
// synchronise, so concurrent callers do not share them.
struct HostPipe {
  uint64_t ctx = 0;
  cudaStream_t copy = nullptr;
  cudaEvent_t ev[6] = {};
  std::mutex mu;
};

static HostPipe* host_pipe(int dev) {
  static HostPipe pipes[64];
  if (dev < 0 || dev >= 64) return nullptr;
  return &pipes[dev];
}

static bool host_pipe_ready(HostPipe* hp) {
  const uint64_t ctx = context_id();
  if (hp->copy != nullptr && hp->ctx == ctx) return true;
  if (cudaStreamCreateWithFlags(&hp->copy, cudaStreamNonBlocking) != cudaSuccess) return false;
  for (cudaEvent_t& e : hp->ev)
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return false;
  hp->ctx = ctx;
  return true;
}

moe_status moe_forward_host(const moe_config* cfg, const void* x_host, const moe_weights* w,
                            const moe_outputs* oh, void* workspace, size_t workspace_bytes,
                            void* stream) {
  moe_status st = check_config(cfg);
  if (st != MOE_OK) return st;
  if (!x_host || !oh || !oh->y || !oh->topk_idx || !oh->topk_w || !oh->counts || !oh->kept ||
      !oh->dropped || !oh->mean_prob || !oh->balance || !workspace ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return MOE_ERR_INVALID_ARG;
  const moe_config& c = *cfg;
  if (workspace_bytes < moe_host_workspace_size(cfg)) return MOE_ERR_WORKSPACE;
  const size_t base = layout(c, nullptr).bytes;
  uint8_t* p = static_cast<uint8_t*>(workspace) + base;
  auto take = [&](size_t n) {
    uint8_t* at = p;
    p += (n + 255) / 256 * 256;
    return static_cast<void*>(at);
  };
  const size_t es = size_t(elem_bytes(c));
  const size_t xb = size_t(c.T * c.d_model) * es, kb = size_t(c.T * c.top_k) * 4,
               nb = size_t(c.n_experts) * 4, lb = size_t(c.T * c.n_experts) * 4;
  void* xd = take(xb);
  moe_outputs od{};
  od.y = take(xb);
  od.topk_idx = static_cast<int32_t*>(take(kb));
  od.topk_w = static_cast<float*>(take(kb));
  od.counts = static_cast<int32_t*>(take(nb));
  od.kept = static_cast<int32_t*>(take(nb));
  od.mean_prob = static_cast<float*>(take(nb));
  od.dropped = static_cast<int32_t*>(take(4));
  od.balance = static_cast<float*>(take(4));
  od.logits = oh->logits ? static_cast<float*>(take(lb)) : nullptr;
  od.cv_squared = oh->cv_squared ? static_cast<float*>(take(4)) : nullptr;
  od.pre_act = nullptr;                              // device-only: not kept here
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  struct Copy { void* dst; const void* src; size_t n; };
  const Copy small[] = {{oh->counts, od.counts, nb},
                        {oh->kept, od.kept, nb},
                        {oh->mean_prob, od.mean_prob, nb},
                        {oh->dropped, od.dropped, 4},
                        {oh->balance, od.balance, 4},
                        {oh->cv_squared, od.cv_squared, oh->cv_squared ? size_t(4) : 0}};

  if (host_chunks(c) < 2) {
    if (xb && cudaMemcpyAsync(xd, x_host, xb, cudaMemcpyHostToDevice, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    st = moe_forward(cfg, xd, w, &od, workspace, base, stream);
    if (st != MOE_OK) return st;
    const Copy big[] = {{oh->y, od.y, xb},
                        {oh->topk_idx, od.topk_idx, kb},
                        {oh->topk_w, od.topk_w, kb},
                        {oh->logits, od.logits, oh->logits ? lb : 0}};
    for (const Copy& cp : big)
      if (cp.n && cudaMemcpyAsync(cp.dst, cp.src, cp.n, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    for (const Copy& cp : small)
      if (cp.n && cudaMemcpyAsync(cp.dst, cp.src, cp.n, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return cuda_status(cudaStreamSynchronize(s));
  }

  // two chunks: scratch for their partial sums, counts and unused statistics
  const size_t N = size_t(c.n_experts);
  const moe_config ch[2] = {chunk_cfg(c, 0), chunk_cfg(c, 1)};
  const int64_t rows0 = router_partial_rows(ch[0]), rows1 = router_partial_rows(ch[1]);
  float* prob_rows = static_cast<float*>(take(size_t(rows0 + rows1) * N * 4));
  int32_t* counts_ch[2] = {static_cast<int32_t*>(take(N * 4)), static_cast<int32_t*>(take(N * 4))};
  int32_t* kept_ch[2] = {static_cast<int32_t*>(take(N * 4)), static_cast<int32_t*>(take(N * 4))};
  float* scratch_mean = static_cast<float*>(take(N * 4));
  int32_t* scratch_dropped = static_cast<int32_t*>(take(4));
  float* scratch_balance = static_cast<float*>(take(4));
  float* scratch_cv = static_cast<float*>(take(4));

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  HostPipe* hp = host_pipe(dev);
  if (!hp) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(hp->mu);
  if (!host_pipe_ready(hp)) return MOE_ERR_CUDA;
  cudaStream_t cs = hp->copy;
  cudaEvent_t fork = hp->ev[0], in_done[2] = {hp->ev[1], hp->ev[2]},
              out_ready[2] = {hp->ev[3], hp->ev[4]}, stats_done = hp->ev[5];
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  // the copies start after the caller's earlier work on `stream`
  if (!ok(cudaEventRecord(fork, s)) || !ok(cudaStreamWaitEvent(cs, fork, 0))) return MOE_ERR_CUDA;
  const size_t row_bytes = size_t(c.d_model) * es;
  int64_t t0 = 0;
  for (int i = 0; i < 2; ++i) {
    const size_t n = size_t(ch[i].T) * row_bytes;
    if (!ok(cudaMemcpyAsync(static_cast<uint8_t*>(xd) + t0 * row_bytes,
                            static_cast<const uint8_t*>(x_host) + t0 * row_bytes, n,
                            cudaMemcpyHostToDevice, cs)) ||
        !ok(cudaEventRecord(in_done[i], cs)))
      return MOE_ERR_CUDA;
    t0 += ch[i].T;
  }
  t0 = 0;
  for (int i = 0; i < 2; ++i) {
    const int64_t Ti = ch[i].T, k = c.top_k;
    moe_outputs oc{};
    oc.y = static_cast<uint8_t*>(od.y) + t0 * row_bytes;
    oc.topk_idx = od.topk_idx + t0 * k;
    oc.topk_w = od.topk_w + t0 * k;
    oc.counts = counts_ch[i];
    oc.kept = kept_ch[i];
    oc.mean_prob = scratch_mean;
    oc.dropped = scratch_dropped;
    oc.balance = scratch_balance;
    oc.cv_squared = scratch_cv;
    oc.logits = od.logits ? od.logits + t0 * int64_t(N) : nullptr;
    oc.pre_act = nullptr;
    const ChunkMode mode{prob_rows + (i == 0 ? 0 : rows0) * int64_t(N)};
    if (!ok(cudaStreamWaitEvent(s, in_done[i], 0))) return MOE_ERR_CUDA;
    st = forward_impl(&ch[i], static_cast<uint8_t*>(xd) + t0 * row_bytes, w, &oc, workspace,
                      base, nullptr, stream, &mode);
    if (st != MOE_OK) return st;
    if (!ok(cudaEventRecord(out_ready[i], s)) || !ok(cudaStreamWaitEvent(cs, out_ready[i], 0)))
      return MOE_ERR_CUDA;
    const Copy out[] = {{static_cast<uint8_t*>(oh->y) + t0 * row_bytes, oc.y, size_t(Ti) * row_bytes},
                        {static_cast<int32_t*>(oh->topk_idx) + t0 * k, oc.topk_idx, size_t(Ti * k) * 4},
                        {static_cast<float*>(oh->topk_w) + t0 * k, oc.topk_w, size_t(Ti * k) * 4},
                        {oh->logits ? static_cast<float*>(oh->logits) + t0 * int64_t(N) : nullptr,
                         oc.logits, oh->logits ? size_t(Ti) * N * 4 : 0}};
    for (const Copy& cp : out)
      if (cp.n && !ok(cudaMemcpyAsync(cp.dst, cp.src, cp.n, cudaMemcpyDeviceToHost, cs)))
        return MOE_ERR_CUDA;
    t0 += Ti;
  }
  if (!ok(launch_chunk_stats(c, prob_rows, int(rows0 + rows1), counts_ch[0], kept_ch[0],
                             counts_ch[1], kept_ch[1], od.counts, od.kept, od.mean_prob,
                             od.balance, od.dropped, od.cv_squared, s)) ||
      !ok(cudaEventRecord(stats_done, s)) || !ok(cudaStreamWaitEvent(cs, stats_done, 0)))
    return MOE_ERR_CUDA;
  for (const Copy& cp : small)
    if (cp.n && !ok(cudaMemcpyAsync(cp.dst, cp.src, cp.n, cudaMemcpyDeviceToHost, cs)))
      return MOE_ERR_CUDA;
  // every copy is on `cs`, after all of the layer's work on `stream`
  return cuda_status(cudaStreamSynchronize(cs));
}

// ---- backward ----------------------------------------------------------------------

size_t moe_backward_workspace_size(const moe_config* cfg) {
  if (check_bwd_config(cfg) != MOE_OK) return 0;
  return bwd_layout(*cfg, nullptr).bytes;
}

int32_t moe_backward_launch_count(const moe_config* cfg) {
  if (check_bwd_config(cfg) != MOE_OK) return -1;
  return backward_launch_count(*cfg);
}

static moe_status backward_impl(const moe_config* cfg, const void* x, const moe_weights* w,
                                const moe_outputs* fwd, void* fwd_workspace,
                                size_t fwd_workspace_bytes, const void* dy, float aux_weight,
                                const moe_grads* grads, void* workspace, size_t workspace_bytes,
                                void* const* events, void* stream) {
  const NvtxRange call_range("moe_backward");
  moe_status st = check_bwd_config(cfg);
  if (st != MOE_OK) return st;
  const moe_config& c = *cfg;
  st = check_weights(c, w, true, true);
  if (st != MOE_OK) return st;
  if (!fwd || !grads || !fwd_workspace || !workspace ||
      (reinterpret_cast<uintptr_t>(fwd_workspace) & 255u) != 0 ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return MOE_ERR_INVALID_ARG;
  auto ok16 = [](const void* q) { return q && aligned16(q); };
  auto tok = [&](const void* q) { return c.T == 0 || ok16(q); };
  if (!tok(x) || !tok(dy) || !tok(grads->dx) || !tok(fwd->topk_idx) || !tok(fwd->topk_w))
    return MOE_ERR_INVALID_ARG;
  const void* need[] = {grads->dW_g, grads->db_g, grads->dW1, grads->db1, grads->dW2,
                        grads->db2, fwd->kept, fwd->mean_prob};
  for (const void* q : need)
    if (!ok16(q)) return MOE_ERR_INVALID_ARG;
  if (c.d_ff_shared > 0) {
    const void* ss[] = {grads->dW1s, grads->db1s, grads->dW2s, grads->db2s};
    for (const void* q : ss)
      if (!ok16(q)) return MOE_ERR_INVALID_ARG;
  }
  if (!std::isfinite(aux_weight)) return MOE_ERR_INVALID_ARG;
  const Workspace fws = layout(c, fwd_workspace);
  if (fwd_workspace_bytes < fws.bytes) return MOE_ERR_WORKSPACE;
  const BwdWorkspace ws = bwd_layout(c, workspace);
  if (workspace_bytes < ws.bytes) return MOE_ERR_WORKSPACE;
  DeviceInfo di;
  if (!device_info(&di)) return MOE_ERR_CUDA;
  BackwardArgs a{};
  a.w = w; a.g = grads; a.x = x; a.dy = dy;
  a.Yp = fws.Yp; a.H = fws.H; a.Xp = fws.Xp; a.offsets = fws.offsets; a.kept = fwd->kept;
  a.token_row = fws.token_row; a.topk_idx = fwd->topk_idx; a.topk_w = fwd->topk_w;
  a.logits = fwd->logits ? fwd->logits : fws.logits; a.mean_prob = fwd->mean_prob;
  a.aux_weight = aux_weight;
  a.dO = ws.dO; a.dA = ws.dA; a.dXp = ws.dXp;
  // the forward's kept pre-activation, else recomputed into the workspace
  if (fwd->pre_act && !aligned16(fwd->pre_act)) return MOE_ERR_INVALID_ARG;
  a.A1 = fwd->pre_act ? fwd->pre_act : ws.A1;
  a.recompute_A1 = fwd->pre_act == nullptr;
  a.dz = grads->dz ? grads->dz : ws.dz;
  a.dw = grads->dw ? grads->dw : ws.dw;
  a.dxr = ws.dxr;
  a.dz_bf = ws.dz_bf;
  a.dxr_bf = ws.dxr_bf;
  a.rgrp = ws.rgrp;
  a.part = ws.part;
  a.bpart = ws.bpart;
  a.rows_max = rows_max_of(c);
  a.status = di.status; a.wait_limit_ns = g_wait_limit_ns.load(); a.num_sms = di.num_sms;
  return cuda_status(launch_backward(c, a, events, static_cast<cudaStream_t>(stream)));
}

moe_status moe_backward(const moe_config* cfg, const void* x, const moe_weights* w,
                        const moe_outputs* fwd, void* fwd_workspace, size_t fwd_workspace_bytes,
                        const void* dy, float aux_weight, const moe_grads* grads,
                        void* workspace, size_t workspace_bytes, void* stream) {
  return backward_impl(cfg, x, w, fwd, fwd_workspace, fwd_workspace_bytes, dy, aux_weight,
                       grads, workspace, workspace_bytes, nullptr, stream);
}

moe_status moe_backward_profiled(const moe_config* cfg, const void* x, const moe_weights* w,
                                 const moe_outputs* fwd, void* fwd_workspace,
                                 size_t fwd_workspace_bytes, const void* dy, float aux_weight,
                                 const moe_grads* grads, void* workspace,
                                 size_t workspace_bytes, void* const* events, void* stream) {
  if (!events) return MOE_ERR_INVALID_ARG;
  pdl_enabled() = false;
  const moe_status st = backward_impl(cfg, x, w, fwd, fwd_workspace, fwd_workspace_bytes, dy,
                                      aux_weight, grads, workspace, workspace_bytes, events,
                                      stream);
  pdl_enabled() = true;
  return st;
}

// ---- expert-choice routing --------------------------------------------------------

int64_t moe_ec_tokens_per_expert(const moe_config* cfg) {
  if (check_ec_config(cfg) != MOE_OK) return -1;
  return ec_tokens_of(*cfg);
}

int64_t moe_ec_rows_max(const moe_config* cfg) {
  if (check_ec_config(cfg) != MOE_OK) return -1;
  return ec_rows_max_of(*cfg);
}

size_t moe_ec_workspace_size(const moe_config* cfg) {
  if (check_ec_config(cfg) != MOE_OK) return 0;
  return ec_layout(*cfg, nullptr).bytes;
}

int32_t moe_ec_forward_launch_count(const moe_config* cfg) {
  if (check_ec_config(cfg) != MOE_OK) return -1;
  const moe_config& c = *cfg;
  if (c.T == 0) return 2;                          // selection (group offsets), statistics
  const int router = (c.dtype == MOE_BF16 && c.n_experts % 64 == 0) ? 2
                                                                      : router_launch_count(c);
  return router + 1 + 1 + 2 + 1 + 1;   // router, select, row copy, two Linears, combine, stats
}

moe_status moe_ec_router(const moe_config* cfg, const void* x, const void* W_g, const void* b_g,
                         float* logits, float* probT, int32_t* token_picks,
                         float* prob_partials, void* stream) {
  moe_status st = check_ec_config(cfg);
  if (st != MOE_OK) return st;
  if (cfg->T == 0) return MOE_OK;
  const void* ps[] = {x, W_g, b_g, logits, probT, token_picks, prob_partials};
  for (const void* q : ps)
    if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  DeviceInfo di;
  if (!device_info(&di)) return MOE_ERR_CUDA;
  return cuda_status(launch_router_probs(*cfg, x, W_g, b_g, logits, probT, token_picks,
                                         prob_partials, di.num_sms, di.status,
                                         g_wait_limit_ns.load(),
                                         static_cast<cudaStream_t>(stream)));
}

moe_status moe_ec_select(const moe_config* cfg, const float* probT, int32_t* ec_token,
                         float* ec_gate, int32_t* offsets, int32_t* counts, int32_t* row_token,
                         int32_t* token_row, float* token_w, int32_t* token_picks,
                         void* stream) {
  moe_status st = check_ec_config(cfg);
  if (st != MOE_OK) return st;
  const moe_config& c = *cfg;
  if (!offsets || !counts || !aligned16(offsets) || !aligned16(counts) ||
      (ec_rows_max_of(c) > 0 && (!row_token || !aligned16(row_token))))
    return MOE_ERR_INVALID_ARG;
  if (c.T > 0) {
    const void* ps[] = {probT, ec_token, ec_gate, token_row, token_w, token_picks};
    for (const void* q : ps)
      if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  }
  return cuda_status(launch_ec_select(c, ec_tokens_of(c), probT, ec_token, ec_gate, offsets,
                                      counts, row_token, token_row, token_w, token_picks,
                                      static_cast<cudaStream_t>(stream)));
}

static moe_status ec_forward_impl(const moe_config* cfg, const void* x, const moe_weights* w,
                                  const moe_ec_outputs* out, void* workspace,
                                  size_t workspace_bytes, void* const* events, void* stream) {
  const NvtxRange call_range("moe_ec_forward");
  moe_status st = check_ec_config(cfg);
  if (st != MOE_OK) return st;
  const moe_config& c = *cfg;
  st = check_weights(c, w, true, true);
  if (st != MOE_OK) return st;
  auto token_buf_ok = [&](const void* q) { return c.T == 0 || (q && aligned16(q)); };
  if (!out || !token_buf_ok(x) || !workspace ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return MOE_ERR_INVALID_ARG;
  if (!token_buf_ok(out->y) || !token_buf_ok(out->ec_token) || !token_buf_ok(out->ec_gate) ||
      !token_buf_ok(out->token_picks))
    return MOE_ERR_INVALID_ARG;
  if (!out->unpicked || !out->mean_prob || !out->balance || !aligned16(out->mean_prob))
    return MOE_ERR_INVALID_ARG;
  if (out->logits && !aligned16(out->logits)) return MOE_ERR_INVALID_ARG;
  const EcWorkspace ws = ec_layout(c, workspace);
  if (workspace_bytes < ws.bytes) return MOE_ERR_WORKSPACE;
  DeviceInfo di;
  if (!device_info(&di)) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* logits = out->logits ? out->logits : ws.logits;
  void* const none[7] = {};
  void* const* ev = events ? events : none;
  const int64_t C = ec_tokens_of(c), rows = ec_rows_max_of(c);
  const moe_config kc = ec_kernel_config(c);

  cudaError_t e = record_event(ev[0], s);
  if (e == cudaSuccess)
    e = launch_router_probs(c, x, w->W_g, w->b_g, logits, ws.probT, out->token_picks,
                            ws.prob_partials, di.num_sms, di.status, g_wait_limit_ns.load(), s);
  if (e == cudaSuccess) e = record_event(ev[1], s);
  if (e == cudaSuccess)
    e = launch_ec_select(c, C, ws.probT, out->ec_token, out->ec_gate, ws.offsets, ws.counts,
                         ws.row_token, ws.token_row, ws.token_w, out->token_picks, s);
  if (e == cudaSuccess && c.T > 0)
    e = launch_row_copy(c, x, ws.offsets, ws.row_token, ws.Xp, rows, s);
  if (e == cudaSuccess) e = record_event(ev[2], s);
  if (e == cudaSuccess && c.T > 0) {
    GroupedFfnArgs a{};
    a.Xp = ws.Xp; a.offsets = ws.offsets; a.kept = ws.counts; a.w = w; a.H = ws.H;
    a.Yp = ws.Yp; a.rows_max = rows; a.status = di.status;
    a.wait_limit_ns = g_wait_limit_ns.load(); a.num_sms = di.num_sms;
    a.mid_event = ev[3];
    a.routed_rows = c.n_experts * C;
    e = c.dtype == MOE_F32 ? launch_grouped_ffn_f32(kc, a, s) : launch_grouped_ffn_bf16(kc, a, s);
  }
  if (e == cudaSuccess) e = record_event(ev[4], s);
  if (e == cudaSuccess)
    e = launch_combine(kc, ws.Yp, ws.token_row, ws.token_w, ws.offsets, out->y, s);
  if (e == cudaSuccess) e = record_event(ev[5], s);
  if (e == cudaSuccess)
    e = launch_ec_stats(c, ws.prob_partials, ws.counts, out->token_picks, out->mean_prob,
                        out->balance, ws.scratch, out->unpicked, s);
  if (e == cudaSuccess) e = record_event(ev[6], s);
  return cuda_status(e);
}

moe_status moe_ec_forward(const moe_config* cfg, const void* x, const moe_weights* w,
                          const moe_ec_outputs* out, void* workspace, size_t workspace_bytes,
                          void* stream) {
  return ec_forward_impl(cfg, x, w, out, workspace, workspace_bytes, nullptr, stream);
}

moe_status moe_ec_forward_profiled(const moe_config* cfg, const void* x, const moe_weights* w,
                                   const moe_ec_outputs* out, void* workspace,
                                   size_t workspace_bytes, void* const* events, void* stream) {
  if (!events) return MOE_ERR_INVALID_ARG;
  pdl_enabled() = false;
  const moe_status st =
      ec_forward_impl(cfg, x, w, out, workspace, workspace_bytes, events, stream);
  pdl_enabled() = true;
  return st;
}

int32_t moe_build_flags(void) {
#ifdef MOE_CHECKS
  return MOE_BUILD_CHECKS;
#else
  return 0;
#endif
}

int32_t moe_workspace_guards(const moe_config* cfg, int64_t* offsets, int32_t max_guards) {
  if (check_config(cfg) != MOE_OK) return -1;
  const Workspace w = layout(*cfg, nullptr);
  for (int32_t i = 0; i < w.n_guards && i < max_guards && offsets; ++i) offsets[i] = w.guard[i];
  return w.n_guards;
}

moe_status moe_checks_read(int32_t* fails, int32_t* site, int32_t* line, int32_t clear) {
  if (!fails || !site || !line) return MOE_ERR_INVALID_ARG;
  cudaError_t (*readers[])(CheckRecord*, bool) = {
      checks_read_router, checks_read_permute, checks_read_combine,
      checks_read_expert_choice, checks_read_backward, checks_read_grouped_bwd,
      checks_read_grouped_ffn_f32, checks_read_grouped_ffn, checks_read_front_small};
  *fails = 0;
  *site = 0;
  *line = 0;
  for (auto rd : readers) {
    CheckRecord r{};
    if (rd(&r, clear != 0) != cudaSuccess) return MOE_ERR_CUDA;
    if (r.fails > 0 && *fails == 0) {
      *site = r.site;
      *line = r.line;
    }
    *fails += r.fails;
  }
  return MOE_OK;
}

moe_status moe_get_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  int32_t v = MOE_OK;
  const int32_t zero = MOE_OK;
  if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(v)) != cudaSuccess) return MOE_ERR_CUDA;
  if (v != MOE_OK && cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return v;
}

moe_status moe_activation(int32_t act, const float* x, float* y, int64_t n, void* stream) {
  if (act != MOE_ACT_GELU_ERF && act != MOE_ACT_RELU) return MOE_ERR_INVALID_ARG;
  if (n < 0 || (n > 0 && (!x || !y))) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  const int64_t blocks64 = ceil_div(n, 256);
  const unsigned blocks = unsigned(blocks64 < 4096 ? blocks64 : 4096);
  activation_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(act, x, y, n);
  return cuda_status(cudaGetLastError());
}

moe_status moe_selftest_bounded_wait(uint64_t limit_ns, void* stream) {
  DeviceInfo di;
  if (!device_info(&di)) return MOE_ERR_CUDA;
  return cuda_status(
      launch_bounded_wait_selftest(limit_ns, di.status, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
