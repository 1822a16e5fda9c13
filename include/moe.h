/*
 * moe.h -- C ABI of libmoe.so: the forward pass of a sparse Mixture-of-Experts
 * FFN layer on one NVIDIA B300 (sm_103a).
 *
 * The layer (botmartz.com "Mixture of Experts (MoE) and Mixtral: Scaling
 * Without Dense Computation", sections "MoE Architecture" and "Expert
 * Routing"; roadtointelligence.com "Mixture of Experts (MoE)", router formula
 * and output equation; matteuscruz.github.io "What is a Mixture of Experts?",
 * section "Architecture: router + experts"):
 *
 *   z   = x . W_g^T + b_g                       router scores, fp32   [T, N]
 *   p   = softmax(z) over the N experts                                [T, N]
 *   idx = the k experts with the largest z (ties: lower index; slot 0 largest)
 *   w   = softmax over the kept k scores (= kept p renormalised to sum 1),
 *         or the kept p themselves when renormalize == 0
 *   y[t] = sum_j [kept] w[t,j] * E_idx[t,j](x[t])  (+ E_shared(x[t]))
 *   E_e(v) = W2[e] . act(W1[e] . v + b1[e]) + b2[e],  act = GELU(erf) | ReLU
 *
 * With a capacity C > 0 (roadtointelligence.com "Keeping the experts busy";
 * matteuscruz.github.io "Load balancing: the core training challenge"), the
 * (token, slot) assignments of each expert are ranked in token-major order
 * and those with rank >= C are dropped: they contribute 0 to y (the token
 * passes on through the caller's residual connection).
 *
 * Conventions for every call below
 *   - Pointers named x, y, W*, b*, and all index / statistic arrays are DEVICE
 *     pointers (except in moe_forward_host, which says otherwise).  The caller
 *     owns every buffer; the library allocates no memory.  `cfg` and the
 *     structs are read during the call only.
 *   - Layouts are row-major.  x, y: [T, d_model].  Weights follow
 *     nn.Linear's [out, in]: W_g [N, d_model], W1 [N, d_ff, d_model],
 *     W2 [N, d_model, d_ff], W1s [d_ff, d_model], W2s [d_model, d_ff];
 *     biases b_g [N], b1 [N, d_ff], b2 [N, d_model], b1s [d_ff], b2s [d_model].
 *     x, y, weights and biases share one element type, cfg->dtype.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and never synchronise, except moe_forward_host and
 *     moe_get_device_status.
 *   - Arguments are validated on the host before anything is launched; a
 *     failed check returns a status and leaves every buffer untouched.  A
 *     failed launch returns MOE_ERR_CUDA.  There is no CPU fallback.
 *   - Every device pointer must be 16-byte aligned.  Requirements on sizes:
 *     1 <= top_k <= n_experts <= 1024, T >= 0, d_model % 8 == 0; for bf16
 *     also d_model % 64 == 0 and d_ff % 64 == 0; d_ff_shared is 0 or d_ff.
 *     Otherwise MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED.
 *   - Kernels that wait on on-chip barriers give up after a time limit
 *     (moe_set_wait_limit_ns), record MOE_ERR_TIMEOUT in a device status word
 *     and return; moe_get_device_status reports it.
 *   - All kernels are deterministic: the same inputs give bit-identical
 *     outputs (no order-dependent atomics).
 *   - The library's only global state is that status word, the wait limit
 *     and the fixed scratch array of moe_permute_noalloc.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t moe_status;
enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null / misaligned pointer, bad size */
  MOE_ERR_UNSUPPORTED = 2,   /* valid layer the library does not run (shape rule) */
  MOE_ERR_WORKSPACE = 3,     /* workspace or scratch smaller than required */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
  MOE_ERR_TIMEOUT = 5        /* a device-side barrier wait ran out of time */
};

enum { MOE_F32 = 0, MOE_BF16 = 1 };           /* moe_config.dtype */
enum { MOE_ACT_GELU_ERF = 0, MOE_ACT_RELU = 1 };  /* moe_config.act  */

/* Rows of the expert-grouped buffers are padded per expert to this multiple. */
#define MOE_GROUP_ALIGN 128

typedef struct moe_config {
  int64_t T;            /* tokens (batch x sequence), >= 0                     */
  int64_t d_model;      /* model width d                                        */
  int64_t d_ff;         /* hidden width of each routed expert                   */
  int64_t n_experts;    /* N routed experts                                     */
  int64_t top_k;        /* k experts per token                                  */
  int64_t capacity;     /* assignments kept per expert; <= 0 means unlimited    */
  int64_t d_ff_shared;  /* 0: no shared expert; else its hidden width (= d_ff)  */
  int32_t renormalize;  /* 1: gates = softmax over the kept k scores; 0: raw p  */
  int32_t act;          /* MOE_ACT_*                                            */
  int32_t dtype;        /* MOE_F32 or MOE_BF16 for x, y, weights, biases        */
  int32_t reserved;     /* set to 0                                             */
} moe_config;

typedef struct moe_weights {
  const void *W_g, *b_g;              /* router                                 */
  const void *W1, *b1, *W2, *b2;      /* routed experts, stacked over N         */
  const void *W1s, *b1s, *W2s, *b2s;  /* shared expert (NULL if d_ff_shared=0)  */
} moe_weights;

typedef struct moe_outputs {
  void    *y;          /* [T, d_model], cfg->dtype                      required */
  int32_t *topk_idx;   /* [T, k] expert of each slot, slot 0 largest    required */
  float   *topk_w;     /* [T, k] gate of each slot                      required */
  int32_t *counts;     /* [N] assignments routed to each expert         required */
  int32_t *kept;       /* [N] assignments kept (min(counts, capacity))  required */
  int32_t *dropped;    /* [1] total dropped assignments                 required */
  float   *mean_prob;  /* [N] mean over tokens of p                     required */
  float   *balance;    /* [1] std_unbiased(mean_prob)^2                 required */
  float   *logits;     /* [T, N] router scores z; NULL = keep in workspace      */
  float   *cv_squared; /* [1] var_unbiased(counts) / mean(counts)^2; NULL = skip */
  void    *pre_act;    /* [moe_rows_max(cfg), d_ff], cfg->dtype: the first Linear's
                          pre-activation in the grouped row layout, kept for
                          moe_backward (which then skips recomputing it);
                          NULL = not kept.  Device memory (moe_forward_host
                          ignores it). */
} moe_outputs;

/* ---- sizes --------------------------------------------------------------- */

/* Upper bound on the rows of the expert-grouped buffers Xp / H / Yp:
 * T*k + N*(MOE_GROUP_ALIGN-1), plus T rounded up to MOE_GROUP_ALIGN when there
 * is a shared expert.  Returns -1 for an invalid config. */
int64_t moe_rows_max(const moe_config* cfg);

/* Rows of the router's per-block probability partial sums ([rows, N] fp32). */
int64_t moe_router_blocks(const moe_config* cfg);

/* Bytes of scratch moe_permute needs (per-block counts, bases or ranks). */
size_t moe_permute_scratch_size(const moe_config* cfg);

/* Bytes of workspace moe_forward needs; 0 for an invalid config. */
size_t moe_workspace_size(const moe_config* cfg);

/* Number of kernels one moe_forward call launches for this layer (the
 * kernels are chosen by shape); -1 for an invalid config. */
int32_t moe_forward_launch_count(const moe_config* cfg);

/* Name of the kernel, with its tile shape, that moe_forward launches for
 * grouped Linear `linear` (1: Xp -> H, 2: H -> Yp) of this layer; the choice
 * depends on the shape only.  A static string owned by the library; NULL for
 * an invalid config or `linear` outside {1, 2}.  A host-side query for
 * profiling reports: the pages have no counterpart. */
const char* moe_ffn_kernel_name(const moe_config* cfg, int32_t linear);

/* ---- the steps of the layer ------------------------------------------------ */

/* Router scores, softmax over all N experts, top-k and gates
 * (botmartz.com "Expert Routing": router Linear, softmax, topk, renormalise;
 * roadtointelligence.com router formula Softmax(TopK(x . W_g))).
 *   x [T, d] dtype; W_g [N, d] dtype; b_g [N] dtype
 *   logits        out [T, N] fp32: z, accumulated in fp32
 *   topk_idx      out [T, k] int32, slot 0 = largest score, ties -> lower index
 *   topk_w        out [T, k] fp32 gates
 *   prob_partials out [moe_router_blocks(cfg), N] fp32: per token-block sums
 *                 of p, consumed by moe_load_stats. */
moe_status moe_router_topk(const moe_config* cfg, const void* x, const void* W_g,
                           const void* b_g, float* logits, int32_t* topk_idx,
                           float* topk_w, float* prob_partials, void* stream);

/* Group the (token, slot) assignments by expert, in token-major order, apply
 * the capacity and copy the kept tokens' rows into per-expert contiguous
 * groups (matteuscruz.github.io "Distributed training and inference":
 * grouping tokens by expert; "Load balancing": capacity buffer).
 *   topk_idx  in  [T, k]
 *   counts    out [N] routed assignments per expert
 *   kept      out [N] kept assignments per expert
 *   offsets   out [N + 2] first row of each group in Xp; groups padded to
 *             MOE_GROUP_ALIGN rows; offsets[N] = end of the routed groups,
 *             offsets[N+1] = end of the shared expert's group (rows
 *             offsets[N] + t hold token t) or offsets[N] without one
 *   row_token out [moe_rows_max] token of each routed row; -1 for padding
 *   token_row out [T, k] row of each assignment in Xp; -1 when dropped
 *   Xp        out [moe_rows_max, d] dtype; padding rows are left unwritten
 *   scratch   device scratch of moe_permute_scratch_size(cfg) bytes. */
moe_status moe_permute(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                       int32_t* counts, int32_t* kept, int32_t* offsets,
                       int32_t* row_token, int32_t* token_row, void* Xp,
                       void* scratch, size_t scratch_bytes, void* stream);

/* moe_permute for callers that cannot allocate device memory -- for example a
 * plugin whose host framework owns every byte of device memory and forbids
 * allocation in its execution path, or a latency-bound loop where a
 * cudaMalloc would synchronise the device.  The pages have no counterpart:
 * this is an interface convenience, not a step of the layer.
 *
 * Same arguments and results as moe_permute, minus the scratch: the
 * per-block counts, bases or ranks live in a fixed array inside the library,
 * MOE_PERMUTE_STATIC_SCRATCH_INTS int32 (1 MiB) large, which every GPU that
 * loads the library holds until the process exits.  Layers whose scratch
 * need (moe_permute_scratch_size) exceeds it return MOE_ERR_WORKSPACE and
 * launch nothing.  Layers of 2048 to 65536 assignments (T * k) with at most
 * 384 experts always fit; other layers need ceil(T/128) * N <= 131072 (for
 * example T = 16384 with N = 1024 still fits).
 *
 * The array is shared by every call on a device: two calls whose kernels
 * overlap on the GPU (different streams, no ordering) race on it, so order
 * them on one stream or with events.  Nothing in it needs clearing between
 * calls: every entry is written before it is read.  The first call on each
 * device looks up the array's device address (cudaGetSymbolAddress) and
 * caches it; the lookup is repeated when the device's context has changed
 * (for example after cudaDeviceReset).  Make the first call on a device, and
 * the first after such a change, before any stream capture.  No memory is
 * allocated by this call. */
#define MOE_PERMUTE_STATIC_SCRATCH_INTS (1 << 18)
moe_status moe_permute_noalloc(const moe_config* cfg, const void* x,
                               const int32_t* topk_idx, int32_t* counts, int32_t* kept,
                               int32_t* offsets, int32_t* row_token, int32_t* token_row,
                               void* Xp, void* stream);

/* Run every expert on its group (botmartz.com "Expert Routing": Linear ->
 * GELU -> Linear; codingnowai.in "Code": Linear -> ReLU -> Linear):
 *   H  = act(Xp[group e] . W1[e]^T + b1[e])   stored in dtype  [rows_max, d_ff]
 *   Yp = H[group e] . W2[e]^T + b2[e]          stored in dtype  [rows_max, d]
 * Only the kept[e] leading rows of each group are computed and written; the
 * shared expert's group (when present) has T rows.  offsets/kept as written
 * by moe_permute.  bf16 runs on the tensor cores (fp32 accumulate), fp32 on
 * CUDA cores. */
moe_status moe_grouped_ffn(const moe_config* cfg, const void* Xp, const int32_t* offsets,
                           const int32_t* kept, const moe_weights* w, void* H, void* Yp,
                           void* stream);

/* Gate-weighted combine back to token order (roadtointelligence.com output
 * equation; botmartz.com "Expert Routing" outputs[mask] += prob * expert(x)):
 *   y[t] = sum_j [token_row[t,j] >= 0] topk_w[t,j] * Yp[token_row[t,j]]
 *          (+ Yp[offsets[N] + t] with weight 1 for the shared expert)
 * accumulated in fp32 in slot order, stored in dtype.  A token with every
 * slot dropped and no shared expert gets y[t] = 0. */
moe_status moe_combine(const moe_config* cfg, const void* Yp, const int32_t* token_row,
                       const float* topk_w, const int32_t* offsets, void* y, void* stream);

/* Load statistics (botmartz.com "Load Balancing: The Hidden Challenge"):
 *   mean_prob[e] = (1/T) sum_t p[t, e]            (from prob_partials)
 *   balance      = sum_e (mean_prob[e] - 1/N)^2 / (N - 1)   (0 when N == 1)
 *                = torch.std(mean_prob)**2 with the unbiased default
 *   dropped      = sum_e (counts[e] - kept[e])
 *   cv_squared   = var(counts) / mean(counts)^2, unbiased variance over the N
 *                  routed counts; 0 when N == 1 or nothing is routed.  The
 *                  coefficient of variation the auxiliary loss penalises
 *                  (matteuscruz.github.io "Load balancing: the core training
 *                  challenge"; invest-in.ai "MoE - Mixture of Experts",
 *                  "Common Usage Examples": cv_squared(expert_counts)); the
 *                  pages give no formula, this is the plain reading.
 *                  Optional: NULL skips it.
 * One block; sums in a fixed order (compensated fp32 for the probabilities,
 * exact integers for the counts), so results are deterministic. */
moe_status moe_load_stats(const moe_config* cfg, const float* prob_partials,
                          const int32_t* counts, const int32_t* kept, float* mean_prob,
                          float* balance, int32_t* dropped, float* cv_squared, void* stream);

/* The whole layer: router_topk -> permute -> grouped_ffn -> combine ->
 * load_stats on `stream`, with intermediates carved from `workspace`
 * (device, >= moe_workspace_size(cfg) bytes, 256-byte aligned). */
moe_status moe_forward(const moe_config* cfg, const void* x, const moe_weights* w,
                       const moe_outputs* out, void* workspace, size_t workspace_bytes,
                       void* stream);

/* moe_forward that also records seven caller-owned CUDA events (cudaEvent_t,
 * timing enabled) on `stream` at the step boundaries, for per-kernel timing:
 *   events[0] before the router      events[4] after the second Linear
 *   events[1] after the router        events[5] after the combine
 *   events[2] after the permutation   events[6] after the statistics
 *   events[3] after the first Linear (H)
 * (when the permutation runs as a single block it also computes the
 * statistics, and events[5] and events[6] then bracket no work) 
 * A NULL entry is skipped.  While `stream` is being captured into a CUDA
 * graph, the events become external event-record nodes, so every replay of
 * the graph records them.  Otherwise identical to moe_forward, except that
 * its kernels do not overlap their neighbours (moe_forward lets each kernel
 * start while the previous one finishes), so each interval times one step. */
moe_status moe_forward_profiled(const moe_config* cfg, const void* x, const moe_weights* w,
                                const moe_outputs* out, void* workspace,
                                size_t workspace_bytes, void* const* events, void* stream);

/* moe_forward for callers holding tokens and results in HOST memory: x and
 * every non-NULL pointer in `out` are host pointers (page-locked memory makes
 * the copies asynchronous); weights and workspace stay on the device.  The
 * call copies x in, runs the layer, copies the results out and synchronises
 * before returning; when it returns, all of its work on `stream` is done.
 * The workspace must hold moe_workspace_size(cfg) bytes plus room for x,
 * every output and the chunk scratch below (moe_host_workspace_size).
 *
 * Layers of at least 1024 tokens without capacity, whose halves run the same
 * grouped-FFN kernels as the whole batch and either keep >= 256 rows per
 * expert or have <= 96 MB of expert weights, run as two token chunks so that
 * the copies overlap the layer: chunk 1's tokens are copied in while chunk 0
 * runs, and chunk 0's results copied out while chunk 1 runs (the copies on a
 * second stream the library keeps per device; calls on one device take turns).
 * Per token the results are those of moe_forward bit for bit; counts, kept
 * and dropped are exact; mean_prob, balance and cv_squared come from both
 * chunks' partial sums and may differ from moe_forward's in the last bits.
 * This division of the work is an implementation choice: the pages have no
 * counterpart.  moe_forward_host_chunks gives the number of chunks (1 or 2;
 * -1 for an invalid config). */
size_t moe_host_workspace_size(const moe_config* cfg);
int32_t moe_forward_host_chunks(const moe_config* cfg);
moe_status moe_forward_host(const moe_config* cfg, const void* x_host, const moe_weights* w,
                            const moe_outputs* out_host, void* workspace,
                            size_t workspace_bytes, void* stream);

/* The expert activation exactly as the FFN kernels evaluate it, applied
 * elementwise to n fp32 values (device pointers): y[i] = act(x[i]).  GELU is
 * the exact erf form, 0.5 x (1 + erf(x / sqrt 2)) (botmartz.com "Expert
 * Routing": nn.GELU()), with erf evaluated by Abramowitz & Stegun's formula
 * 7.1.26 (absolute error <= 1.5e-7); ReLU is max(x, 0) (codingnowai.in
 * "Code").  Lets callers check the activation against other implementations. */
moe_status moe_activation(int32_t act, const float* x, float* y, int64_t n, void* stream);

/* ---- backward pass ----------------------------------------------------------
 *
 * Gradients of the training loss total = task + aux_weight * balance
 * (botmartz.com "Load Balancing: The Hidden Challenge": total_loss = task_loss
 * + 0.01 * balance_loss; roadtointelligence.com "Keeping the experts busy":
 * coefficient 0.01) with respect to x and every parameter, given
 * dy = d task / d y.  The chain rule runs back through the forward of the
 * same call sequence: combine, expert FFNs (the first Linear's
 * pre-activation is recomputed), gates (softmax over the k selected scores,
 * or the raw probabilities), the balance statistic and the router.  The top-k
 * choice and the capacity drops pass no gradient.  Top-k routing only.  bf16
 * layers run their GEMMs on the tensor cores, fp32 layers on CUDA cores in
 * fp32.  Gradients are written in the layer dtype, accumulated in fp32. */

typedef struct moe_grads {
  void  *dx;                          /* [T, d_model]                      required */
  void  *dW_g, *db_g;                 /* [N, d_model], [N]                 required */
  void  *dW1, *db1, *dW2, *db2;       /* shapes of W1, b1, W2, b2          required */
  void  *dW1s, *db1s, *dW2s, *db2s;   /* shared expert (NULL without one)           */
  float *dz;                          /* [T, N] d total / d z (scores); NULL = skip */
  float *dw;                          /* [T, k] d total / d gate; NULL = skip       */
} moe_grads;

/* Bytes of device workspace moe_backward needs; 0 for an invalid config. */
size_t moe_backward_workspace_size(const moe_config* cfg);
/* Kernels one moe_backward launches without a kept pre-activation (one fewer
 * when the forward kept it in moe_outputs.pre_act); -1 for an invalid config. */
int32_t moe_backward_launch_count(const moe_config* cfg);

/* The backward pass.  `fwd` and `fwd_workspace` are the outputs and the
 * workspace of the moe_forward call on the same cfg, x and weights (the
 * backward reads the saved grouping, the expert rows Xp, H and Yp, the
 * scores, gates and mean_prob from them; it writes nothing there; padding
 * rows of the grouped buffers are never read as data).  dy [T, d_model] in
 * the layer dtype.  `workspace`
 * (device, >= moe_backward_workspace_size(cfg) bytes, 256-byte aligned) holds
 * the backward's intermediates. */
moe_status moe_backward(const moe_config* cfg, const void* x, const moe_weights* w,
                        const moe_outputs* fwd, void* fwd_workspace, size_t fwd_workspace_bytes,
                        const void* dy, float aux_weight, const moe_grads* grads,
                        void* workspace, size_t workspace_bytes, void* stream);

/* moe_backward with eight caller-owned CUDA events recorded on `stream` at
 * the step boundaries (kernels not overlapping their neighbours):
 *   events[0] start                     events[4] after dXp = dA W1
 *   events[1] after the gate step       events[5] after dW2 = dO^T H
 *                                       events[6] after dW1 = dA^T Xp
 *   events[2] after the recomputed A1   events[7] after the bias sums, the
 *   events[3] after dA = (dO W2) act'(A1)         router gradients and dx
 * A NULL entry is skipped. */
moe_status moe_backward_profiled(const moe_config* cfg, const void* x, const moe_weights* w,
                                 const moe_outputs* fwd, void* fwd_workspace,
                                 size_t fwd_workspace_bytes, const void* dy, float aux_weight,
                                 const moe_grads* grads, void* workspace,
                                 size_t workspace_bytes, void* const* events, void* stream);

/* ---- expert-choice routing -------------------------------------------------
 *
 * matteuscruz.github.io "What is a Mixture of Experts?", "Load balancing: the
 * core training challenge": expert choice routing (Zhou et al., 2022) turns
 * the routing around -- every expert selects the tokens it scores highest
 * rather than every token selecting its top-k experts -- so each expert gets
 * the same load by construction, and a token may be processed by any number
 * of experts (none included).  The page gives only the idea; this library
 * reads it as follows (the same readings as its CPU oracle):
 *   - the score of token t for expert e is the router probability
 *     p[t, e] = softmax over the N experts of z[t, :], z = x . W_g^T + b_g;
 *   - every expert takes C = moe_ec_tokens_per_expert(cfg) tokens:
 *     cfg->capacity clamped to T, or all T when capacity <= 0;
 *   - among equal scores the lower token index is taken first;
 *   - a picked token's gate is p[t, e], and
 *       y[t] = sum over the experts e that picked t of p[t, e] * expert_e(x[t])
 *     (+ the shared expert's output with weight 1), so a token no expert
 *     picked gets y[t] = 0 (+ shared).
 * cfg->top_k and cfg->renormalize are not read; every other field means what
 * it does for top-k routing.  The routed rows live in N groups of
 * round_up(C, MOE_GROUP_ALIGN) rows (expert e from row e * that), each in
 * ascending token order, then the shared group as for top-k routing. */

typedef struct moe_ec_outputs {
  void    *y;           /* [T, d_model], cfg->dtype                         required */
  int32_t *ec_token;    /* [N, C] tokens each expert picked, ascending       required */
  float   *ec_gate;     /* [N, C] p[ec_token, e]: the gate of each pick      required */
  int32_t *token_picks; /* [T] number of experts that picked each token      required */
  int32_t *unpicked;    /* [1] tokens no expert picked                       required */
  float   *mean_prob;   /* [N] mean over tokens of p                         required */
  float   *balance;     /* [1] std_unbiased(mean_prob)^2                     required */
  float   *logits;      /* [T, N] router scores z; NULL = keep in workspace         */
} moe_ec_outputs;

/* C, the tokens every expert takes; -1 for an invalid config. */
int64_t moe_ec_tokens_per_expert(const moe_config* cfg);
/* Rows of the grouped buffers: N * round_up(C, MOE_GROUP_ALIGN), plus T rounded
 * up to MOE_GROUP_ALIGN with a shared expert; -1 for an invalid config. */
int64_t moe_ec_rows_max(const moe_config* cfg);
/* Bytes of device workspace moe_ec_forward needs; 0 for an invalid config. */
size_t moe_ec_workspace_size(const moe_config* cfg);
/* Kernels one moe_ec_forward launches; -1 for an invalid config. */
int32_t moe_ec_forward_launch_count(const moe_config* cfg);

/* Router step without the top-k: scores, probabilities and their block sums.
 *   logits        out [T, N] fp32 scores z
 *   probT         out [N, T] fp32 probabilities, expert-major (probT[e*T + t] = p[t, e])
 *   token_picks   out [T] int32, set to 0 (moe_ec_select counts into it)
 *   prob_partials out [moe_router_blocks(cfg), N] fp32, as for moe_router_topk */
moe_status moe_ec_router(const moe_config* cfg, const void* x, const void* W_g, const void* b_g,
                         float* logits, float* probT, int32_t* token_picks,
                         float* prob_partials, void* stream);

/* Selection and grouping: every expert's C highest-probability tokens.
 *   probT       in  [N, T] fp32, p >= 0 (as moe_ec_router writes it)
 *   ec_token    out [N, C] int32, ascending per expert
 *   ec_gate     out [N, C] fp32, probT[e, ec_token[e, i]]
 *   offsets     out [N + 2] int32: offsets[e] = e * round_up(C, 128); offsets[N]
 *               = end of the routed groups; offsets[N + 1] = end of the shared group
 *   counts      out [N] int32, all C
 *   row_token   out [moe_ec_rows_max(cfg)] int32, token of each grouped row (-1 = padding)
 *   token_row   out [T, N] int32, grouped row of (t, e), -1 where e did not pick t
 *   token_w     out [T, N] fp32, p[t, e] where e picked t, else 0
 *   token_picks in/out [T] int32, incremented once per pick: zero it first
 * Exact: the selection compares the fp32 bit patterns, so it is reproducible
 * and equal to a stable sort of each expert's column by (-p, t). */
moe_status moe_ec_select(const moe_config* cfg, const float* probT, int32_t* ec_token,
                         float* ec_gate, int32_t* offsets, int32_t* counts, int32_t* row_token,
                         int32_t* token_row, float* token_w, int32_t* token_picks,
                         void* stream);

/* The whole expert-choice layer: ec_router -> ec_select -> row copy ->
 * grouped FFN (the same kernels as top-k routing, every group C rows) ->
 * combine (one slot per expert) -> statistics, on `stream`; workspace as for
 * moe_forward but moe_ec_workspace_size(cfg) bytes. */
moe_status moe_ec_forward(const moe_config* cfg, const void* x, const moe_weights* w,
                          const moe_ec_outputs* out, void* workspace, size_t workspace_bytes,
                          void* stream);

/* moe_ec_forward with seven events at the step boundaries, as in
 * moe_forward_profiled (events[2] follows the selection and the row copy,
 * events[5] the combine, events[6] the statistics). */
moe_status moe_ec_forward_profiled(const moe_config* cfg, const void* x, const moe_weights* w,
                                   const moe_ec_outputs* out, void* workspace,
                                   size_t workspace_bytes, void* const* events, void* stream);

/* ---- status ---------------------------------------------------------------- */

/* Synchronises `stream`, returns (and clears) the device status word:
 * MOE_OK or MOE_ERR_TIMEOUT; MOE_ERR_CUDA if the synchronisation failed. */
moe_status moe_get_device_status(void* stream);

/* Time after which a device-side barrier wait gives up (default 2 s). */
void moe_set_wait_limit_ns(uint64_t ns);
uint64_t moe_get_wait_limit_ns(void);

/* Launches one block that waits on an on-chip barrier nothing will complete,
 * for at most `limit_ns`, then records MOE_ERR_TIMEOUT and returns: exercises
 * the bounded-wait path without hanging the GPU. */
moe_status moe_selftest_bounded_wait(uint64_t limit_ns, void* stream);

const char* moe_status_string(moe_status s);
int32_t moe_version(void);

/* ---- build variants and device checks ----------------------------------------
 *
 * The library can be built with -DMOE_CHECKS (libmoe_checks.so): every kernel
 * then checks the indices it gathers or scatters through (expert ids, token
 * rows, group extents) before the access, and a failed check is counted in a
 * device record -- the kernel carries on with its accesses bounded, nothing
 * traps.  The forward workspace also gets a 256-byte guard gap after each of
 * its regions, so a test can fill the workspace with a pattern and see that no
 * kernel wrote outside its region.  Test and debugging aids: the pages have no
 * counterpart.
 *
 * moe_build_flags: MOE_BUILD_CHECKS when this is the checks build, else 0.
 * moe_workspace_guards: the guard gaps of moe_forward's workspace for this
 *   layer (offsets in bytes from its start, each 256 bytes long), up to
 *   max_guards of them written to offsets; returns their number (0 in the
 *   ordinary build) or -1 for an invalid config.
 * moe_checks_read: the number of failed checks since the last clear, with the
 *   site (MOE_CHECK_* below) and source line of the first; clear != 0 resets
 *   the records.  Synchronous with the device; always 0 in the ordinary build. */
#define MOE_BUILD_CHECKS 1
enum {
  MOE_CHECK_ROUTER_TOPK = 1, MOE_CHECK_SORT_EXPERT = 2, MOE_CHECK_COPY_TOKEN = 3,
  MOE_CHECK_ROWS_TOTAL = 4, MOE_CHECK_COMBINE_ROW = 5, MOE_CHECK_GEMM_ROWS = 6,
  MOE_CHECK_EC_PICK = 7
};
int32_t moe_build_flags(void);
int32_t moe_workspace_guards(const moe_config* cfg, int64_t* offsets, int32_t max_guards);
moe_status moe_checks_read(int32_t* fails, int32_t* site, int32_t* line, int32_t clear);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
