/* CPU oracle for the sparse Mixture-of-Experts FFN layer: plain single-threaded
 * C++ in double precision.
 *
 * TEST INFRASTRUCTURE ONLY.  The library (libmoe.so and its Python binding)
 * never includes, links or calls this code; only the tests, the smoke check
 * and the benchmark's CPU-baseline leg do.  It shares no header, helper, table
 * or constant with the CUDA path.
 *
 * Every function is the plain definition of one step, in the order the pages
 * give them (each .cpp function cites its passage):
 *   router scores, softmax over all N experts, top-k, gates (renormalised or
 *   raw), grouping of (token, slot) assignments by expert with a capacity,
 *   expert FFN Linear -> activation -> Linear, gate-weighted combine, the
 *   balance statistic and cv^2 of the counts; expert-choice routing; the
 *   backward pass of task + alpha * balance.
 *
 * Conventions: row-major arrays; weights in nn.Linear's [out, in] layout,
 * stacked over experts (W1 [N, f, d], W2 [N, d, f]); every input may be
 * float32, bfloat16 (raw 16-bit patterns) or float64 and is upcast to double
 * exactly as it is read; every result is double (indices int64).  Functions
 * return 0, or -1 on an invalid argument.  Nothing here keeps state: calls on
 * disjoint outputs may run at the same time from several threads. */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F64 = 2 };
enum { ORC_ACT_GELU_ERF = 0, ORC_ACT_RELU = 1 };

typedef struct {
  const void* data;   /* NULL: absent */
  int32_t dtype;      /* ORC_F32, ORC_BF16 or ORC_F64 */
  int32_t reserved;
} orc_tensor;

typedef struct {
  int64_t T, d, f, N, k;
  int64_t f_shared;           /* 0: no shared expert */
  int32_t act;                /* ORC_ACT_* */
  int32_t round_hidden_bf16;  /* 1: the hidden activation is rounded to bf16 */
  orc_tensor x, W_g, b_g, W1, b1, W2, b2, W1s, b1s, W2s, b2s;
} orc_layer;

/* ---- number formats and elementwise definitions ---------------------------- */
double orc_round_bf16(double v);
void orc_round_bf16_array(const double* v, double* out, int64_t n);
void orc_upcast(orc_tensor a, int64_t n, double* out);
int orc_activation(int32_t act, const double* a, double* out, int64_t n);
int orc_activation_grad(int32_t act, const double* a, double* out, int64_t n);

/* ---- router ----------------------------------------------------------------- */
/* z[t, e] = sum_i x[t, i] W_g[e, i] + b_g[e] for the tokens t0 <= t < t1 (z rows t0..t1-1). */
int orc_router_logits(const orc_layer* L, int64_t t0, int64_t t1, double* z);
int orc_softmax_rows(int64_t rows, int64_t n, const double* z, double* p);
/* k largest of each row, largest first; equal scores -> lower index first. */
int orc_topk(int64_t rows, int64_t n, int64_t k, const double* z, int64_t* idx);
/* k-th minus (k+1)-th largest score per row; +inf when k >= n. */
int orc_topk_gap(int64_t rows, int64_t n, int64_t k, const double* z, double* gap);
/* gates as the softmax over the kept scores (Softmax(TopK(z))). */
int orc_gates_softmax_of_topk(int64_t rows, int64_t n, int64_t k, const double* z,
                              const int64_t* idx, double* w);
/* gates as the kept probabilities divided by their sum. */
int orc_gates_renormalised_probs(int64_t rows, int64_t n, int64_t k, const double* p,
                                 const int64_t* idx, double* w);
/* gates as the raw kept probabilities. */
int orc_gates_raw_probs(int64_t rows, int64_t n, int64_t k, const double* p,
                        const int64_t* idx, double* w);

/* ---- capacity, grouping and statistics ------------------------------------ */
int64_t orc_capacity(double capacity_factor, int64_t T, int64_t N);
/* Walk (t, j) token-major; rank = earlier assignments to the same expert;
 * kept when capacity <= 0 or rank < capacity.  order [T*k]: kept assignment
 * ids t*k + j grouped by expert (ascending), each group in rank order;
 * group_start [N+1]: where each group starts in order.  Returns the number
 * dropped, or -1. */
int64_t orc_group(int64_t T, int64_t k, int64_t N, int64_t capacity, const int64_t* idx,
                  int64_t* counts, int64_t* kept, int64_t* rank, uint8_t* keep,
                  int64_t* order, int64_t* group_start);
/* mean_prob[e] = mean_t p[t, e]; balance = unbiased variance of mean_prob. */
int orc_balance(int64_t T, int64_t N, const double* p, double* mean_prob, double* balance);
double orc_cv_squared(int64_t N, const int64_t* counts);

/* Router, softmax, top-k (or idx_override), gates, grouping and statistics
 * for all T tokens.  z_in: the scores when already computed (else NULL). */
int orc_route(const orc_layer* L, int64_t capacity, int32_t renormalize,
              const int64_t* idx_override, const double* z_in, double* z, double* p,
              int64_t* idx, double* w, int64_t* counts, int64_t* kept, int64_t* rank,
              uint8_t* keep, int64_t* order, int64_t* group_start, int64_t* dropped,
              double* mean_prob, double* balance, double* cv_squared);

/* ---- experts and the layer -------------------------------------------------- */
/* Expert e (e == N: the shared expert) on the rows x[tokens[r]]:
 * pre = W1 x + b1, h = act(pre) (bf16-rounded if the layer says so),
 * o = W2 h + b2.  Any output may be NULL. */
int orc_expert_rows(const orc_layer* L, int64_t e, const int64_t* tokens, int64_t n,
                    double* pre, double* h, double* o);
/* y[r] = sum over kept slots j of w[t, j] expert_idx[t,j](x[t]) (+ shared), t = tokens[r]. */
int orc_combine_rows(const orc_layer* L, const int64_t* idx, const double* w,
                     const uint8_t* keep, const int64_t* tokens, int64_t n, double* y);
/* orc_route + orc_combine_rows over `tokens` (NULL: all T, n ignored). */
int orc_forward(const orc_layer* L, int64_t capacity, int32_t renormalize,
                const int64_t* idx_override, const int64_t* tokens, int64_t n, double* z,
                double* p, int64_t* idx, double* w, int64_t* counts, int64_t* kept,
                int64_t* rank, uint8_t* keep, int64_t* order, int64_t* group_start,
                int64_t* dropped, double* mean_prob, double* balance, double* cv_squared,
                double* y);
/* Every expert on every token, then masks and weights per (slot, expert),
 * with gates as renormalised probabilities and the capacity mask from a
 * direct recount.  Tiny inputs only.  y [T, d]. */
int orc_bruteforce(const orc_layer* L, int64_t capacity, int32_t renormalize, double* y);

/* ---- expert-choice routing -------------------------------------------------- */
int64_t orc_ec_tokens(int64_t T, int64_t capacity);
/* sel [N, C]: per expert the C tokens of largest p[t, e] (lower token first
 * among equal scores), listed in ascending token order. */
int orc_ec_select(int64_t T, int64_t N, int64_t C, const double* p, int64_t* sel);
int orc_ec_gap(int64_t T, int64_t N, int64_t C, const double* p, double* gap);
/* picks [T]: how many experts picked each token; returns the number of
 * tokens no expert picked, or -1. */
int64_t orc_ec_picks(int64_t T, int64_t N, int64_t C, const int64_t* sel, int64_t* picks);
/* y[r] = sum over experts e that picked t of p[t, e] expert_e(x[t]) (+ shared). */
int orc_ec_combine_rows(const orc_layer* L, int64_t C, const int64_t* sel, const double* p,
                        const int64_t* tokens, int64_t n, double* y);

/* ---- backward pass of total = <dy, y> + aux_weight * balance ----------------
 * The routing (z, p, idx, w, keep, order, group_start) comes from orc_route. */
int orc_backward(const orc_layer* L, int64_t capacity, int32_t renormalize,
                 const int64_t* idx_override, orc_tensor dy, double aux_weight, double* dx,
                 double* dW_g, double* db_g, double* dW1, double* db1, double* dW2,
                 double* db2, double* dW1s, double* db1s, double* dW2s, double* db2s,
                 double* dz, double* dw);
/* dW_g [N, d] = dz^T x and db_g [N] = sum_t dz for the score gradients dz [T, N]. */
int orc_router_weight_grads(const orc_layer* L, const double* dz, double* dW_g, double* db_g);
/* Expert e's (e == N: shared) weight gradients from its rows (tokens[r],
 * gates[r]): dO_r = gates[r] dy[t_r].  Only hidden units `units` (NULL: all
 * f): dW1_rows [n_units, d], db1 [n_units], dW2_cols [d, n_units]; db2 [d]. */
int orc_expert_weight_grads(const orc_layer* L, int64_t e, const int64_t* tokens,
                            const double* gates, int64_t n_rows, orc_tensor dy,
                            const int64_t* units, int64_t n_units, double* dW1_rows,
                            double* db1, double* dW2_cols, double* db2);
/* For the listed tokens only: dw [n, k], dz [n, N], dx [n, d], from the
 * routing of all T tokens (p for the balance term). */
int orc_token_grads(const orc_layer* L, int32_t renormalize, const double* p,
                    const int64_t* idx, const double* w, const uint8_t* keep, orc_tensor dy,
                    double aux_weight, const int64_t* tokens, int64_t n, double* dw,
                    double* dz, double* dx);

#ifdef __cplusplus
}
#endif
#endif /* MOE_ORACLE_H */
