// Internal launchers of libmoe's kernels (host functions, one per step).
// The C ABI in api.cu validates arguments and calls these; each returns the
// cudaError_t of its launches.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// Whether launch_pdl may overlap a kernel with its predecessor on the stream
// (per host thread).  moe_forward_profiled turns it off so that the events
// it records between kernels time each kernel alone.
inline bool& pdl_enabled() {
  static thread_local bool on = true;
  return on;
}

// Launches `kern`, with programmatic stream serialisation when enabled: the
// kernel may start while the previous kernel on the stream is finishing (see
// pdl_* in common.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ---- router (router.cu) ------------------------------------------------------

constexpr int kRouterTokensPerBlock = 8;    // tokens per router pass (one per warp)
constexpr int kRouterMaxBlocks = 296;       // router blocks (grid-stride over 8-token groups)

// bf16 layers with 64 experts: the tensor-core router GEMM also takes the
// softmax, top-k and gates in its epilogue (k <= 8).
inline bool router_tc_topk(const moe_config& c) {
  return c.dtype == MOE_BF16 && c.n_experts == 64 && c.top_k >= 1 && c.top_k <= 8;
}

// Rows of the router's probability partial sums: one per router block (one
// per 128-token tile for the tensor-core router with the top-k epilogue).
inline int64_t router_partial_rows(const moe_config& c) {
  if (router_tc_topk(c)) return (c.T + 127) / 128;
  const int64_t groups = (c.T + kRouterTokensPerBlock - 1) / kRouterTokensPerBlock;
  return groups < kRouterMaxBlocks ? groups : kRouterMaxBlocks;
}

cudaError_t launch_router_logits(const moe_config& c, const void* x, const void* W_g,
                                 const void* b_g, float* logits, cudaStream_t s);
// k == 0 with probT set: no top-k; writes probT [N, T] and zeroes picks [T]
cudaError_t launch_router_softmax_topk(const moe_config& c, int k, const float* logits,
                                       int32_t* topk_idx, float* topk_w,
                                       float* prob_partials, float* probT, int32_t* picks,
                                       cudaStream_t s);
// router scores on the tensor cores, fp32 out (grouped_ffn_sm103.cu)
cudaError_t launch_router_logits_tc(const moe_config& c, const void* x, const void* W_g,
                                    const void* b_g, float* logits, int num_sms,
                                    int32_t* status, uint64_t wait_limit_ns, cudaStream_t s);
// the whole router step, kernels chosen by shape
cudaError_t launch_router(const moe_config& c, const void* x, const void* W_g,
                          const void* b_g, float* logits, int32_t* topk_idx, float* topk_w,
                          float* prob_partials, int num_sms, int32_t* status,
                          uint64_t wait_limit_ns, cudaStream_t s);

// ---- permutation (permute.cu) ------------------------------------------------

constexpr int kPermuteTokensPerBlock = 128;  // tokens per histogram / rank block

// Load statistics computed at the end of the permutation (moe_forward only).
struct StatsArgs {
  const float* prob_partials;   // nullptr: no statistics
  int nblk;
  float* mean_prob;
  float* balance;
  int32_t* dropped;
  float* cv_squared;            // nullptr: not computed
};

size_t permute_scratch_bytes(const moe_config& c);
// true when launch_permute can also produce the load statistics
bool permute_fuses_stats(const moe_config& c);
// zero / n_zero: int32 counters the row copy sets to 0 for the kernels after it
// (nullptr / 0: none)
cudaError_t launch_permute(const moe_config& c, const void* x, const int32_t* topk_idx,
                           int32_t* counts, int32_t* kept, int32_t* offsets,
                           int32_t* row_token, int32_t* token_row, void* Xp, void* scratch,
                           int64_t rows_max, cudaStream_t s, const StatsArgs* stats,
                           int32_t* zero, int64_t n_zero);

// ---- expert-choice routing (router.cu, expert_choice.cu) -------------------------

// Xp[r] = x[row_token[r]] for the routed rows [0, offsets[N]) (-1: padding,
// left as is), Xp[offsets[N] + t] = x[t] for the shared group (permute.cu)
// zero / n_zero as in launch_permute.
cudaError_t launch_row_copy(const moe_config& c, const void* x, const int32_t* offsets,
                            const int32_t* row_token, void* Xp, int64_t rows_max,
                            cudaStream_t s, int32_t* zero = nullptr, int64_t n_zero = 0);

// ---- small-batch front end (front_small.cu) --------------------------------------

// Whether moe_forward routes, sorts and computes the statistics of this layer
// with the two front-end kernels (a few tokens and experts).
bool small_front_fits(const moe_config& c);
// fp32 slice sums of the router scores it keeps in the workspace (0: not used)
int64_t small_front_partial_floats(const moe_config& c);
// Router scores, softmax, top-k and gates, the counting sort (counts, kept,
// offsets, row_token, token_row) and the load statistics; part: scratch of
// small_front_partial_floats(c) floats.
cudaError_t launch_small_front(const moe_config& c, const void* x, const void* W_g,
                               const void* b_g, float* part, float* logits, int32_t* topk_idx,
                               float* topk_w, int32_t* counts, int32_t* kept, int32_t* offsets,
                               int32_t* row_token, int32_t* token_row, float* mean_prob,
                               float* balance, int32_t* dropped, float* cv_squared,
                               cudaStream_t s);

// scores, expert-major probabilities probT [N, T] (and picks [T] zeroed), block
// sums of p: the router without its top-k
cudaError_t launch_router_probs(const moe_config& c, const void* x, const void* W_g,
                                const void* b_g, float* logits, float* probT, int32_t* picks,
                                float* prob_partials, int num_sms, int32_t* status,
                                uint64_t wait_limit_ns, cudaStream_t s);
// every expert's C picked tokens, grouped in Cpad-row groups (plus the shared
// expert's T rows), with the per-token slot view token_row / token_w [T, N]
cudaError_t launch_ec_select(const moe_config& c, int64_t C, const float* probT,
                             int32_t* ec_token, float* ec_gate, int32_t* offsets,
                             int32_t* counts, int32_t* row_token, int32_t* token_row,
                             float* token_w, int32_t* picks, cudaStream_t s);
// mean_prob, balance and the tokens no expert picked
cudaError_t launch_ec_stats(const moe_config& c, const float* prob_partials,
                            const int32_t* counts, const int32_t* picks, float* mean_prob,
                            float* balance, int32_t* scratch, int32_t* unpicked,
                            cudaStream_t s);
// rows of one expert's group: C rounded up to the group alignment
inline int64_t ec_group_rows(int64_t C) {
  return (C + MOE_GROUP_ALIGN - 1) / MOE_GROUP_ALIGN * MOE_GROUP_ALIGN;
}

// ---- grouped expert FFN ----------------------------------------------------------

struct GroupedFfnArgs {
  const void* Xp;
  const int32_t* offsets;   // [N + 2]
  const int32_t* kept;      // [N]
  const moe_weights* w;
  void* H;
  void* Yp;
  int64_t rows_max;
  int32_t* status;          // device status word
  uint64_t wait_limit_ns;
  int num_sms;
  void* mid_event;          // cudaEvent_t recorded between the two Linears, or nullptr
  int64_t routed_rows;      // live routed rows for the tile heuristics; 0: T * top_k
  void* pre_out;            // [rows_max, d_ff]: also keep the first Linear's
                            // pre-activation (for the backward), or nullptr
  // stream-K scratch (both nullptr: whole tiles per CTA): per-CTA fp32
  // partial accumulators, and per-tile counters that start at 0
  // (sk_counter_ints(c, 1) for Linear 1, then those of Linear 2)
  float* sk_partials;
  int32_t* sk_counters;
};
// Stream-K bookkeeping of moe_forward's grouped Linears: counters of Linear
// 1 or 2 (0 when that Linear runs whole tiles), and the partial-accumulator
// bytes (0 when neither runs stream-K).
int64_t sk_counter_ints(const moe_config& c, int linear);

size_t sk_partial_bytes(const moe_config& c);
// whether the bf16 first Linear stores its pre-activation from its epilogue
// (else a second pass does)
bool linear_saves_pre(const moe_config& c);
// Unique id of the calling thread's current CUDA context (0: none current).
uint64_t context_id();
// Device-check records of each translation unit (zeros in the ordinary build).
struct CheckRecord;
cudaError_t checks_read_router(CheckRecord* out, bool clear);
cudaError_t checks_read_permute(CheckRecord* out, bool clear);
cudaError_t checks_read_combine(CheckRecord* out, bool clear);
cudaError_t checks_read_expert_choice(CheckRecord* out, bool clear);
cudaError_t checks_read_backward(CheckRecord* out, bool clear);
cudaError_t checks_read_grouped_bwd(CheckRecord* out, bool clear);
cudaError_t checks_read_grouped_ffn_f32(CheckRecord* out, bool clear);
cudaError_t checks_read_grouped_ffn(CheckRecord* out, bool clear);
cudaError_t checks_read_front_small(CheckRecord* out, bool clear);
// Kernel (and tile) of grouped Linear 1 or 2 for this layer; routed_rows 0: T * top_k.
const char* grouped_linear_kernel_name(const moe_config& c, int linear, int64_t routed_rows);

// Records a caller's event on s (as an external node while s is capturing).
cudaError_t record_event(void* event, cudaStream_t s);

// fp32 path on CUDA cores (grouped_ffn_f32.cu)
cudaError_t launch_grouped_ffn_f32(const moe_config& c, const GroupedFfnArgs& a, cudaStream_t s);
// bf16 path on tcgen05 tensor cores (grouped_ffn_sm103.cu)
cudaError_t launch_grouped_ffn_bf16(const moe_config& c, const GroupedFfnArgs& a, cudaStream_t s);

// ---- combine and statistics (combine.cu) ----------------------------------------

cudaError_t launch_combine(const moe_config& c, const void* Yp, const int32_t* token_row,
                           const float* topk_w, const int32_t* offsets, void* y,
                           cudaStream_t s);
cudaError_t launch_load_stats(const moe_config& c, const float* prob_partials,
                              const int32_t* counts, const int32_t* kept, float* mean_prob,
                              float* balance, int32_t* dropped, float* cv_squared,
                              cudaStream_t s);
// Statistics of a batch run as two consecutive token chunks: counts and kept
// summed from the chunks' arrays, then the statistics of the whole batch
// (c.T tokens) from nblk partial-sum rows (both chunks' rows).
cudaError_t launch_chunk_stats(const moe_config& c, const float* prob_rows, int nblk,
                               const int32_t* counts0, const int32_t* kept0,
                               const int32_t* counts1, const int32_t* kept1, int32_t* counts,
                               int32_t* kept, float* mean_prob, float* balance,
                               int32_t* dropped, float* cv_squared, cudaStream_t s);

// ---- kernels launched per step, for the chosen dispatch ------------------------------
// Router scores, softmax, top-k, gates and the per-tile sums of p for 64
// experts in one tensor-core launch (router_tc_topk) (grouped_ffn_sm103.cu).
cudaError_t launch_router_topk_tc(const moe_config& c, const void* x, const void* W_g,
                                  const void* b_g, float* logits, int32_t* topk_idx,
                                  float* topk_w, float* prob_rows, int num_sms,
                                  int32_t* status, uint64_t wait_limit_ns, cudaStream_t s);
int router_launch_count(const moe_config& c);
int permute_launch_count(const moe_config& c);

// ---- host-side checks shared with entry points outside api.cu -------------------------
moe_status validate_config(const moe_config* cfg);   // as every moe_* entry checks cfg
int64_t rows_max_for(const moe_config& c);             // moe_rows_max without the check

// ---- self test of the bounded wait (api.cu) ---------------------------------------
cudaError_t launch_bounded_wait_selftest(uint64_t limit_ns, int32_t* status, cudaStream_t s);

// ---- backward (grouped_bwd_sm103.cu, backward.cu) --------------------------------

struct BwdGemmArgs {
  const int32_t* offsets;   // [N + 2]
  const int32_t* kept;      // [N]
  int64_t rows_max;
  int32_t* status;
  uint64_t wait_limit_ns;
  int num_sms;
};
// out = dOut . W[e] per group ([K, Nd] weights as stored), times act'(pre)
// when act >= 0; group padding rows written as zeros
cudaError_t launch_bwd_dgrad(const moe_config& c, const BwdGemmArgs& g, const void* dOut,
                             const void* W, const void* Ws, int64_t K, int64_t Nd, int act,
                             const void* pre, void* out, cudaStream_t s);
// the same dgrad on CTA-pair 256 x 256 tiles (grouped_ffn_sm103.cu), used when
// bwd_dgrad_on_pair: groups of >= 256 rows, Nd % 256 == 0, K >= 2048
bool bwd_dgrad_on_pair(const moe_config& c, int64_t K, int64_t Nd);
cudaError_t launch_bwd_dgrad_pair(const moe_config& c, const BwdGemmArgs& g, const void* dOut,
                                  const void* W, const void* Ws, int64_t K, int64_t Nd,
                                  int act, const void* pre, void* out, cudaStream_t s);
// out[e] = L[group e]^T . R[group e] ([Md, Nd] per group; shared into out_s)
cudaError_t launch_bwd_wgrad(const moe_config& c, const BwdGemmArgs& g, const void* Lm,
                             int64_t Md, const void* Rm, int64_t Nd, void* out, void* out_s,
                             cudaStream_t s);
struct BackwardArgs {
  const moe_weights* w;
  const moe_grads* g;
  const void* x;            // [T, d]
  const void* dy;           // [T, d]
  // saved by the forward
  const void* Yp;           // [rows_max, d]
  void* H;                  // [rows_max, d_ff] (bf16: padding rows up to each group's next
                            // multiple of 16 zeroed here)
  void* Xp;                 // [rows_max, d] (the same)
  const int32_t* offsets;
  const int32_t* kept;
  const int32_t* token_row;
  const int32_t* topk_idx;
  const float* topk_w;
  const float* logits;
  const float* mean_prob;
  float aux_weight;
  // backward scratch
  void* dO;                 // [rows_max, d]
  void* A1;                 // [rows_max, d_ff] the first Linear's pre-activation
  bool recompute_A1;        // false: A1 holds the forward's kept pre-activation
  void* dA;                 // [rows_max, d_ff]
  void* dXp;                // [rows_max, d]
  float* dz;                // [T, N]
  float* dw;                // [T, k]
  float* dxr;               // [T, d] fp32 (router part of dx on CUDA cores)
  void* dz_bf;              // [T, N] bf16 (router GEMMs on tensor cores)
  void* dxr_bf;             // [round_up(T, 128), d] bf16 (router part of dx on tensor cores)
  int32_t* rgrp;            // 4 ints: the router GEMMs' one-group offsets and row count
  float* part;              // split-K partial sums of dW_g on CUDA cores
  float* bpart;             // [ceil(rows_max / 128), d + d_ff] bias column-sum partials
  int64_t rows_max;
  int32_t* status;
  uint64_t wait_limit_ns;
  int num_sms;
};
// events: NULL or 8 cudaEvent_t recorded at the step boundaries (see moe_backward_profiled)
cudaError_t launch_backward(const moe_config& c, const BackwardArgs& a, void* const* events,
                            cudaStream_t s);
int backward_launch_count(const moe_config& c);
// router gradients on the tensor cores (N % 64 == 0), else CUDA cores with split K
bool router_bwd_on_tensor_cores(const moe_config& c);
size_t router_bwd_partial_bytes(const moe_config& c);
// the bias column sums' per-chunk partials
size_t bias_partial_bytes(const moe_config& c, int64_t rows_max);

// fp32 layers: the same three backward GEMMs on CUDA cores (grouped_ffn_f32.cu)
cudaError_t launch_grouped_linear_f32(const moe_config& c, const BwdGemmArgs& g, const void* A,
                                      const void* W, const void* Ws, const void* bias,
                                      const void* bias_s, void* out, int64_t K, int64_t Nd,
                                      cudaStream_t s);
cudaError_t launch_bwd_dgrad_f32(const moe_config& c, const BwdGemmArgs& g, const void* dOut,
                                 const void* W, const void* Ws, int64_t K, int64_t Nd, int act,
                                 const void* pre, void* out, cudaStream_t s);
cudaError_t launch_bwd_wgrad_f32(const moe_config& c, const BwdGemmArgs& g, const void* Lm,
                                 int64_t Md, const void* Rm, int64_t Nd, void* out, void* out_s,
                                 cudaStream_t s);

// the first Linear without its activation: out = A W^T + b per group (bf16)
cudaError_t launch_grouped_linear_bf16(const moe_config& c, const GroupedFfnArgs& g,
                                       const void* A, const void* W, const void* Ws,
                                       const void* bias, const void* bias_s, void* out,
                                       int64_t K, int64_t Nd, cudaStream_t s);

}  // namespace moe
