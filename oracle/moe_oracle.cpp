// CPU oracle for the sparse Mixture-of-Experts FFN layer (declarations and
// conventions in moe_oracle.h).  TEST INFRASTRUCTURE ONLY: plain
// single-threaded C++ in double precision, the definitions written out with no
// blocking, fusion or reordering beyond what each definition states.
//
// Sources (site, page title, section):
//   botmartz.com "Mixture of Experts (MoE) and Mixtral: Scaling Without Dense
//     Computation": "Expert Routing" (router nn.Linear, softmax, top-k,
//     renormalise, expert Linear -> GELU -> Linear, masked weighted sum);
//     "Load Balancing: The Hidden Challenge" (balance = std(mean router
//     probability)^2, total_loss = task_loss + 0.01 balance_loss).
//   roadtointelligence.com "Mixture of Experts (MoE)": router formula
//     G(x) = Softmax(TopK(x W_g)), output y = sum_i G(x)_i E_i(x), the tiny
//     worked example; "Keeping the experts busy" (capacity, dropped tokens
//     pass through the residual); "Total versus active parameters" (one
//     shared expert).
//   matteuscruz.github.io "What is a Mixture of Experts?": "Architecture:
//     router + experts"; "Load balancing: the core training challenge"
//     (capacity = capacity factor x batch / experts; coefficient of variation
//     of the load; expert-choice routing: each expert selects its tokens).
//   codingnowai.in "Mixture of Experts": "Code" (raw softmax probability as
//     the gate, Linear -> ReLU -> Linear experts).
//   invest-in.ai "MoE - Mixture of Experts": "Common Usage Examples"
//     (cv_squared(expert_counts)).
//
// Readings where the pages are silent: ties in the top-k go to the lower
// expert index and slot 0 holds the largest score; capacity priority is
// token-major; the capacity is ceil(factor * T / N); a dropped slot adds 0;
// the shared expert has the routed experts' form and gate 1; expert choice
// scores are the router probabilities, ties to the lower token, gate p[t, e].
#include "moe_oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <limits>
#include <numeric>
#include <vector>

namespace {

using Vec = std::vector<double>;

// an int64 count as a container size (also keeps declarations like
// `Vec v(sz(n))` from parsing as function declarations)
size_t sz(int64_t n) { return static_cast<size_t>(n); }
const double kInf = std::numeric_limits<double>::infinity();

bool valid(const orc_tensor& a) {
  return a.data != nullptr && (a.dtype == ORC_F32 || a.dtype == ORC_BF16 || a.dtype == ORC_F64);
}

// bfloat16 is the upper half of a float32: its value is that float32's.
double bf16_value(uint16_t bits) {
  const uint32_t u = uint32_t(bits) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return double(f);
}

double at(const orc_tensor& a, int64_t i) {
  switch (a.dtype) {
    case ORC_F32: return double(static_cast<const float*>(a.data)[i]);
    case ORC_BF16: return bf16_value(static_cast<const uint16_t*>(a.data)[i]);
    default: return static_cast<const double*>(a.data)[i];
  }
}

// n consecutive elements starting at element `off`, upcast to double
void read(const orc_tensor& a, int64_t off, int64_t n, double* out) {
  switch (a.dtype) {
    case ORC_F32: {
      const float* s = static_cast<const float*>(a.data) + off;
      for (int64_t i = 0; i < n; ++i) out[i] = double(s[i]);
      return;
    }
    case ORC_BF16: {
      const uint16_t* s = static_cast<const uint16_t*>(a.data) + off;
      for (int64_t i = 0; i < n; ++i) out[i] = bf16_value(s[i]);
      return;
    }
    default: {
      const double* s = static_cast<const double*>(a.data) + off;
      for (int64_t i = 0; i < n; ++i) out[i] = s[i];
    }
  }
}

double dot(const double* a, const double* b, int64_t n) {
  double s = 0.0;
  for (int64_t i = 0; i < n; ++i) s += a[i] * b[i];
  return s;
}

// nn.GELU() default (exact erf form), botmartz.com "Expert Routing";
// ReLU, codingnowai.in "Code".
double act_value(int32_t act, double a) {
  if (act == ORC_ACT_GELU_ERF) return 0.5 * a * (1.0 + std::erf(a / std::sqrt(2.0)));
  return a > 0.0 ? a : 0.0;
}

// GELU(a) = a Phi(a): GELU'(a) = Phi(a) + a phi(a), phi the normal density.
double act_derivative(int32_t act, double a) {
  if (act == ORC_ACT_GELU_ERF) {
    const double cdf = 0.5 * (1.0 + std::erf(a / std::sqrt(2.0)));
    const double pdf = std::exp(-0.5 * a * a) / std::sqrt(2.0 * 3.14159265358979323846);
    return cdf + a * pdf;
  }
  return a > 0.0 ? 1.0 : 0.0;
}

bool layer_ok(const orc_layer* L) {
  return L && L->T >= 0 && L->d > 0 && L->f > 0 && L->N > 0 && L->k > 0 && L->k <= L->N &&
         (L->act == ORC_ACT_GELU_ERF || L->act == ORC_ACT_RELU) && L->f_shared >= 0;
}

// One expert's weights inside the stacked tensors (e == N: the shared expert).
struct Expert {
  orc_tensor W1, b1, W2, b2;
  int64_t o1, ob1, o2, ob2, f;
};

bool expert_of(const orc_layer& L, int64_t e, Expert* E) {
  if (e < 0 || e > L.N) return false;
  if (e == L.N) {
    if (L.f_shared <= 0 || !valid(L.W1s) || !valid(L.b1s) || !valid(L.W2s) || !valid(L.b2s))
      return false;
    *E = {L.W1s, L.b1s, L.W2s, L.b2s, 0, 0, 0, 0, L.f_shared};
    return true;
  }
  if (!valid(L.W1) || !valid(L.b1) || !valid(L.W2) || !valid(L.b2)) return false;
  *E = {L.W1, L.b1, L.W2, L.b2, e * L.f * L.d, e * L.f, e * L.d * L.f, e * L.d, L.f};
  return true;
}

// The expert FFN on one token row xr: pre = W1 xr + b1, h = act(pre) (rounded
// to bf16 when the layer stores its hidden activation in bf16),
// o = W2 h + b2 (o may be null).  buf holds max(d, f) doubles.
void expert_forward(const orc_layer& L, const Expert& E, const double* xr, double* pre,
                    double* h, double* o, double* buf) {
  const int64_t d = L.d, f = E.f;
  for (int64_t i = 0; i < f; ++i) {
    read(E.W1, E.o1 + i * d, d, buf);
    const double a = dot(buf, xr, d) + at(E.b1, E.ob1 + i);
    pre[i] = a;
    const double v = act_value(L.act, a);
    h[i] = L.round_hidden_bf16 ? orc_round_bf16(v) : v;
  }
  if (!o) return;
  for (int64_t c = 0; c < d; ++c) {
    read(E.W2, E.o2 + c * f, f, buf);
    o[c] = dot(buf, h, f) + at(E.b2, E.ob2 + c);
  }
}

// dh = W2^T dO (a row of W2 per output feature c), then da = dh * act'(pre).
void expert_hidden_grad(const orc_layer& L, const Expert& E, const double* dO,
                        const double* pre, double* da, double* buf) {
  const int64_t d = L.d, f = E.f;
  std::fill(da, da + f, 0.0);
  for (int64_t c = 0; c < d; ++c) {
    read(E.W2, E.o2 + c * f, f, buf);
    for (int64_t i = 0; i < f; ++i) da[i] += buf[i] * dO[c];
  }
  for (int64_t i = 0; i < f; ++i) da[i] *= act_derivative(L.act, pre[i]);
}

// dx += W1^T da
void expert_input_grad(const orc_layer& L, const Expert& E, const double* da, double* dx,
                       double* buf) {
  const int64_t d = L.d, f = E.f;
  for (int64_t i = 0; i < f; ++i) {
    read(E.W1, E.o1 + i * d, d, buf);
    for (int64_t m = 0; m < d; ++m) dx[m] += da[i] * buf[m];
  }
}

}  // namespace

extern "C" {

// ---- number formats and elementwise definitions ------------------------------

// Nearest value with 8 significant bits, ties to even (bfloat16 keeps float32's
// exponent range and 8 significant bits).  Zeros, infinities and NaNs pass
// through; the layer's values stay far from bf16's overflow and subnormals.
double orc_round_bf16(double v) {
  if (v == 0.0 || !std::isfinite(v)) return v;
  int e = 0;
  const double m = std::frexp(v, &e);          // v = m 2^e, 0.5 <= |m| < 1
  const double q = std::nearbyint(m * 256.0);  // default mode: to nearest, ties even
  return std::ldexp(q / 256.0, e);
}

void orc_round_bf16_array(const double* v, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_round_bf16(v[i]);
}

void orc_upcast(orc_tensor a, int64_t n, double* out) {
  if (valid(a)) read(a, 0, n, out);
}

int orc_activation(int32_t act, const double* a, double* out, int64_t n) {
  if (act != ORC_ACT_GELU_ERF && act != ORC_ACT_RELU) return -1;
  for (int64_t i = 0; i < n; ++i) out[i] = act_value(act, a[i]);
  return 0;
}

int orc_activation_grad(int32_t act, const double* a, double* out, int64_t n) {
  if (act != ORC_ACT_GELU_ERF && act != ORC_ACT_RELU) return -1;
  for (int64_t i = 0; i < n; ++i) out[i] = act_derivative(act, a[i]);
  return 0;
}

// ---- router -------------------------------------------------------------------

// Router scores: nn.Linear(d_model, N) (botmartz.com "Expert Routing";
// roadtointelligence.com router formula, x . W_g).
int orc_router_logits(const orc_layer* L, int64_t t0, int64_t t1, double* z) {
  if (!layer_ok(L) || !valid(L->x) || !valid(L->W_g) || !valid(L->b_g) || t0 < 0 || t1 < t0 ||
      t1 > L->T)
    return -1;
  const int64_t d = L->d, N = L->N;
  Vec Wg(sz(N * d)), xr(sz(d));
  read(L->W_g, 0, N * d, Wg.data());
  for (int64_t t = t0; t < t1; ++t) {
    read(L->x, t * d, d, xr.data());
    for (int64_t e = 0; e < N; ++e)
      z[(t - t0) * N + e] = dot(&Wg[sz(e * d)], xr.data(), d) + at(L->b_g, e);
  }
  return 0;
}

// Softmax over the N experts, max-subtracted (botmartz.com "Expert Routing";
// codingnowai.in "The Routing Formula").
int orc_softmax_rows(int64_t rows, int64_t n, const double* z, double* p) {
  if (rows < 0 || n <= 0) return -1;
  for (int64_t r = 0; r < rows; ++r) {
    const double* zr = z + r * n;
    double m = zr[0];
    for (int64_t e = 1; e < n; ++e) m = std::max(m, zr[e]);
    double s = 0.0;
    for (int64_t e = 0; e < n; ++e) s += std::exp(zr[e] - m);
    for (int64_t e = 0; e < n; ++e) p[r * n + e] = std::exp(zr[e] - m) / s;
  }
  return 0;
}

// Top-k (botmartz.com "Expert Routing": torch.topk of the probabilities).  The
// softmax is increasing in each score, so selecting on z selects the same
// experts.  A stable sort by descending score keeps equal scores in index order.
int orc_topk(int64_t rows, int64_t n, int64_t k, const double* z, int64_t* idx) {
  if (rows < 0 || n <= 0 || k <= 0 || k > n) return -1;
  std::vector<int64_t> o(sz(n));
  for (int64_t r = 0; r < rows; ++r) {
    const double* zr = z + r * n;
    std::iota(o.begin(), o.end(), int64_t(0));
    std::stable_sort(o.begin(), o.end(), [&](int64_t a, int64_t b) { return zr[a] > zr[b]; });
    for (int64_t j = 0; j < k; ++j) idx[r * k + j] = o[sz(j)];
  }
  return 0;
}

int orc_topk_gap(int64_t rows, int64_t n, int64_t k, const double* z, double* gap) {
  if (rows < 0 || n <= 0 || k <= 0) return -1;
  Vec s(sz(n));
  for (int64_t r = 0; r < rows; ++r) {
    if (k >= n) {
      gap[r] = kInf;
      continue;
    }
    std::copy(z + r * n, z + (r + 1) * n, s.begin());
    std::sort(s.begin(), s.end(), [](double a, double b) { return a > b; });
    gap[r] = s[sz(k - 1)] - s[sz(k)];
  }
  return 0;
}

// Gates as Softmax(TopK(z)): the scores outside the top-k count as minus
// infinity, so the softmax runs over the kept k scores only
// (roadtointelligence.com router formula and tiny worked example).
int orc_gates_softmax_of_topk(int64_t rows, int64_t n, int64_t k, const double* z,
                              const int64_t* idx, double* w) {
  if (rows < 0 || n <= 0 || k <= 0 || k > n) return -1;
  for (int64_t r = 0; r < rows; ++r) {
    double m = -kInf;
    for (int64_t j = 0; j < k; ++j) m = std::max(m, z[r * n + idx[r * k + j]]);
    double s = 0.0;
    for (int64_t j = 0; j < k; ++j) s += std::exp(z[r * n + idx[r * k + j]] - m);
    for (int64_t j = 0; j < k; ++j) w[r * k + j] = std::exp(z[r * n + idx[r * k + j]] - m) / s;
  }
  return 0;
}

// Gates as the kept probabilities over their sum (botmartz.com "Expert
// Routing": topk_probs / topk_probs.sum(); matteuscruz.github.io
// "Architecture: router + experts").
int orc_gates_renormalised_probs(int64_t rows, int64_t n, int64_t k, const double* p,
                                 const int64_t* idx, double* w) {
  if (rows < 0 || n <= 0 || k <= 0 || k > n) return -1;
  for (int64_t r = 0; r < rows; ++r) {
    double s = 0.0;
    for (int64_t j = 0; j < k; ++j) s += p[r * n + idx[r * k + j]];
    for (int64_t j = 0; j < k; ++j) w[r * k + j] = p[r * n + idx[r * k + j]] / s;
  }
  return 0;
}

// Gates as the raw kept probabilities (codingnowai.in "Code").
int orc_gates_raw_probs(int64_t rows, int64_t n, int64_t k, const double* p, const int64_t* idx,
                        double* w) {
  if (rows < 0 || n <= 0 || k <= 0 || k > n) return -1;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t j = 0; j < k; ++j) w[r * k + j] = p[r * n + idx[r * k + j]];
  return 0;
}

// ---- capacity, grouping and statistics ----------------------------------------

// capacity factor x batch size / number of experts (matteuscruz.github.io
// "Load balancing: the core training challenge"), rounded up.
int64_t orc_capacity(double capacity_factor, int64_t T, int64_t N) {
  if (N <= 0) return -1;
  return int64_t(std::ceil(capacity_factor * double(T) / double(N)));
}

// Tokens grouped by expert (matteuscruz.github.io "Distributed training and
// inference"); over-capacity assignments dropped (roadtointelligence.com
// "Keeping the experts busy").
int64_t orc_group(int64_t T, int64_t k, int64_t N, int64_t capacity, const int64_t* idx,
                  int64_t* counts, int64_t* kept, int64_t* rank, uint8_t* keep, int64_t* order,
                  int64_t* group_start) {
  if (T < 0 || k <= 0 || N <= 0) return -1;
  for (int64_t a = 0; a < T * k; ++a)
    if (idx[a] < 0 || idx[a] >= N) return -1;
  std::fill(counts, counts + N, int64_t(0));
  for (int64_t t = 0; t < T; ++t)
    for (int64_t j = 0; j < k; ++j) {
      const int64_t a = t * k + j, e = idx[a];
      rank[a] = counts[e];
      counts[e] += 1;
      keep[a] = (capacity <= 0 || rank[a] < capacity) ? 1 : 0;
    }
  int64_t dropped = 0;
  group_start[0] = 0;
  for (int64_t e = 0; e < N; ++e) {
    kept[e] = (capacity <= 0 || counts[e] < capacity) ? counts[e] : capacity;
    dropped += counts[e] - kept[e];
    group_start[e + 1] = group_start[e] + kept[e];
  }
  // each group in rank order = the token-major walk restricted to expert e
  std::vector<int64_t> fill(group_start, group_start + N);
  for (int64_t a = 0; a < T * k; ++a)
    if (keep[a]) order[fill[sz(idx[a])]++] = a;
  return dropped;
}

// std(mean over tokens of the router probabilities)^2 with torch.std's default
// unbiased estimator (botmartz.com "Load Balancing: The Hidden Challenge").
int orc_balance(int64_t T, int64_t N, const double* p, double* mean_prob, double* balance) {
  if (T < 0 || N <= 0) return -1;
  for (int64_t e = 0; e < N; ++e) {
    double s = 0.0;
    for (int64_t t = 0; t < T; ++t) s += p[t * N + e];
    mean_prob[e] = T > 0 ? s / double(T) : 0.0;
  }
  *balance = 0.0;
  if (N < 2 || T == 0) return 0;
  double mean = 0.0;
  for (int64_t e = 0; e < N; ++e) mean += mean_prob[e];
  mean /= double(N);
  double v = 0.0;
  for (int64_t e = 0; e < N; ++e) v += (mean_prob[e] - mean) * (mean_prob[e] - mean);
  *balance = v / double(N - 1);
  return 0;
}

// Squared coefficient of variation of the counts: unbiased variance over the
// N experts divided by the squared mean (matteuscruz.github.io "Load
// balancing"; invest-in.ai "Common Usage Examples" names cv_squared).
double orc_cv_squared(int64_t N, const int64_t* counts) {
  if (N < 2) return 0.0;
  double mean = 0.0;
  for (int64_t e = 0; e < N; ++e) mean += double(counts[e]);
  mean /= double(N);
  if (mean == 0.0) return 0.0;
  double v = 0.0;
  for (int64_t e = 0; e < N; ++e) v += (double(counts[e]) - mean) * (double(counts[e]) - mean);
  return v / double(N - 1) / (mean * mean);
}

int orc_route(const orc_layer* L, int64_t capacity, int32_t renormalize,
              const int64_t* idx_override, const double* z_in, double* z, double* p,
              int64_t* idx, double* w, int64_t* counts, int64_t* kept, int64_t* rank,
              uint8_t* keep, int64_t* order, int64_t* group_start, int64_t* dropped,
              double* mean_prob, double* balance, double* cv_squared) {
  if (!layer_ok(L)) return -1;
  const int64_t T = L->T, N = L->N, k = L->k;
  if (z_in)
    std::copy(z_in, z_in + T * N, z);
  else if (orc_router_logits(L, 0, T, z) != 0)
    return -1;
  if (orc_softmax_rows(T, N, z, p) != 0) return -1;
  if (idx_override)
    std::copy(idx_override, idx_override + T * k, idx);
  else if (orc_topk(T, N, k, z, idx) != 0)
    return -1;
  const int g = renormalize ? orc_gates_softmax_of_topk(T, N, k, z, idx, w)
                            : orc_gates_raw_probs(T, N, k, p, idx, w);
  if (g != 0) return -1;
  const int64_t dr = orc_group(T, k, N, capacity, idx, counts, kept, rank, keep, order,
                               group_start);
  if (dr < 0) return -1;
  *dropped = dr;
  if (orc_balance(T, N, p, mean_prob, balance) != 0) return -1;
  *cv_squared = orc_cv_squared(N, counts);
  return 0;
}

// ---- experts and the layer -----------------------------------------------------

int orc_expert_rows(const orc_layer* L, int64_t e, const int64_t* tokens, int64_t n,
                    double* pre, double* h, double* o) {
  Expert E;
  if (!layer_ok(L) || !valid(L->x) || !expert_of(*L, e, &E)) return -1;
  const int64_t d = L->d, f = E.f;
  Vec xr(sz(d)), a(sz(f)), hh(sz(f)), oo(sz(d)), buf(sz(std::max(d, f)));
  for (int64_t r = 0; r < n; ++r) {
    if (tokens[r] < 0 || tokens[r] >= L->T) return -1;
    read(L->x, tokens[r] * d, d, xr.data());
    expert_forward(*L, E, xr.data(), a.data(), hh.data(), o ? oo.data() : nullptr, buf.data());
    if (pre) std::copy(a.begin(), a.end(), pre + r * f);
    if (h) std::copy(hh.begin(), hh.end(), h + r * f);
    if (o) std::copy(oo.begin(), oo.end(), o + r * d);
  }
  return 0;
}

// y = sum over the kept slots of gate * expert(x) (roadtointelligence.com output
// equation; botmartz.com "Expert Routing": output[mask] += weight * expert(x)),
// plus the shared expert with weight 1 (roadtointelligence.com "Total versus
// active parameters").  A dropped slot adds nothing.
int orc_combine_rows(const orc_layer* L, const int64_t* idx, const double* w,
                     const uint8_t* keep, const int64_t* tokens, int64_t n, double* y) {
  if (!layer_ok(L) || !valid(L->x)) return -1;
  const int64_t d = L->d, k = L->k;
  const int64_t fmax = std::max(L->f, L->f_shared);
  Vec xr(sz(d)), a(sz(fmax)), h(sz(fmax)), o(sz(d)),
      buf(sz(std::max(d, fmax)));
  for (int64_t r = 0; r < n; ++r) {
    const int64_t t = tokens[r];
    if (t < 0 || t >= L->T) return -1;
    read(L->x, t * d, d, xr.data());
    double* yr = y + r * d;
    std::fill(yr, yr + d, 0.0);
    for (int64_t j = 0; j < k; ++j) {
      if (!keep[t * k + j]) continue;
      Expert E;
      if (!expert_of(*L, idx[t * k + j], &E) || idx[t * k + j] == L->N) return -1;
      expert_forward(*L, E, xr.data(), a.data(), h.data(), o.data(), buf.data());
      for (int64_t c = 0; c < d; ++c) yr[c] += w[t * k + j] * o[sz(c)];
    }
    if (L->f_shared > 0) {
      Expert S;
      if (!expert_of(*L, L->N, &S)) return -1;
      expert_forward(*L, S, xr.data(), a.data(), h.data(), o.data(), buf.data());
      for (int64_t c = 0; c < d; ++c) yr[c] += o[sz(c)];
    }
  }
  return 0;
}

int orc_forward(const orc_layer* L, int64_t capacity, int32_t renormalize,
                const int64_t* idx_override, const int64_t* tokens, int64_t n, double* z,
                double* p, int64_t* idx, double* w, int64_t* counts, int64_t* kept,
                int64_t* rank, uint8_t* keep, int64_t* order, int64_t* group_start,
                int64_t* dropped, double* mean_prob, double* balance, double* cv_squared,
                double* y) {
  if (orc_route(L, capacity, renormalize, idx_override, nullptr, z, p, idx, w, counts, kept,
                rank, keep, order, group_start, dropped, mean_prob, balance, cv_squared) != 0)
    return -1;
  std::vector<int64_t> all;
  if (!tokens) {
    all.resize(sz(L->T));
    std::iota(all.begin(), all.end(), int64_t(0));
    tokens = all.data();
    n = L->T;
  }
  return orc_combine_rows(L, idx, w, keep, tokens, n, y);
}

// The pages' loop, written as masks: every expert runs on every token, then
// for each (slot, expert) pair the rows routed there are added with their
// weight (botmartz.com "Expert Routing"; codingnowai.in "Code").  The gates
// are the renormalised probabilities (or the raw ones), and the capacity mask
// recounts, for each assignment, the earlier assignments to its expert.
int orc_bruteforce(const orc_layer* L, int64_t capacity, int32_t renormalize, double* y) {
  if (!layer_ok(L)) return -1;
  const int64_t T = L->T, N = L->N, k = L->k, d = L->d;
  Vec z(sz(T * N)), p(sz(T * N)), w(sz(T * k));
  std::vector<int64_t> idx(sz(T * k));
  if (orc_router_logits(L, 0, T, z.data()) || orc_softmax_rows(T, N, z.data(), p.data()) ||
      orc_topk(T, N, k, z.data(), idx.data()))
    return -1;
  if (renormalize)
    orc_gates_renormalised_probs(T, N, k, p.data(), idx.data(), w.data());
  else
    orc_gates_raw_probs(T, N, k, p.data(), idx.data(), w.data());
  std::vector<uint8_t> keep(sz(T * k));
  for (int64_t a = 0; a < T * k; ++a) {
    int64_t earlier = 0;
    for (int64_t b = 0; b < a; ++b) earlier += idx[sz(b)] == idx[sz(a)] ? 1 : 0;
    keep[sz(a)] = (capacity <= 0 || earlier < capacity) ? 1 : 0;
  }
  std::vector<int64_t> all(sz(T));
  std::iota(all.begin(), all.end(), int64_t(0));
  std::vector<Vec> out(sz(N), Vec(sz(T * d)));
  for (int64_t e = 0; e < N; ++e)
    if (orc_expert_rows(L, e, all.data(), T, nullptr, nullptr, out[sz(e)].data())) return -1;
  std::fill(y, y + T * d, 0.0);
  for (int64_t j = 0; j < k; ++j)
    for (int64_t e = 0; e < N; ++e)
      for (int64_t t = 0; t < T; ++t)
        if (idx[sz(t * k + j)] == e && keep[sz(t * k + j)])
          for (int64_t c = 0; c < d; ++c)
            y[t * d + c] += w[sz(t * k + j)] * out[sz(e)][sz(t * d + c)];
  if (L->f_shared > 0) {
    Vec s(sz(T * d));
    if (orc_expert_rows(L, N, all.data(), T, nullptr, nullptr, s.data())) return -1;
    for (int64_t i = 0; i < T * d; ++i) y[i] += s[sz(i)];
  }
  return 0;
}

// ---- expert-choice routing (matteuscruz.github.io "Load balancing": each
// expert selects the tokens it scores highest) -------------------------------------

int64_t orc_ec_tokens(int64_t T, int64_t capacity) {
  return capacity <= 0 ? T : std::min(capacity, T);
}

int orc_ec_select(int64_t T, int64_t N, int64_t C, const double* p, int64_t* sel) {
  if (T < 0 || N <= 0 || C < 0 || C > T) return -1;
  std::vector<int64_t> o(sz(T));
  for (int64_t e = 0; e < N; ++e) {
    std::iota(o.begin(), o.end(), int64_t(0));
    std::stable_sort(o.begin(), o.end(),
                     [&](int64_t a, int64_t b) { return p[a * N + e] > p[b * N + e]; });
    std::sort(o.begin(), o.begin() + C);
    std::copy(o.begin(), o.begin() + C, sel + e * C);
  }
  return 0;
}

// How many experts picked each token; returns the number of tokens no expert picked.
int64_t orc_ec_picks(int64_t T, int64_t N, int64_t C, const int64_t* sel, int64_t* picks) {
  if (T < 0 || N <= 0 || C < 0) return -1;
  std::fill(picks, picks + T, int64_t(0));
  for (int64_t i = 0; i < N * C; ++i) {
    if (sel[i] < 0 || sel[i] >= T) return -1;
    picks[sel[i]] += 1;
  }
  int64_t unpicked = 0;
  for (int64_t t = 0; t < T; ++t) unpicked += picks[t] == 0 ? 1 : 0;
  return unpicked;
}

int orc_ec_gap(int64_t T, int64_t N, int64_t C, const double* p, double* gap) {
  if (T < 0 || N <= 0 || C < 0) return -1;
  Vec s(sz(T));
  for (int64_t e = 0; e < N; ++e) {
    if (C <= 0 || C >= T) {
      gap[e] = kInf;
      continue;
    }
    for (int64_t t = 0; t < T; ++t) s[sz(t)] = p[t * N + e];
    std::sort(s.begin(), s.end(), [](double a, double b) { return a > b; });
    gap[e] = s[sz(C - 1)] - s[sz(C)];
  }
  return 0;
}

int orc_ec_combine_rows(const orc_layer* L, int64_t C, const int64_t* sel, const double* p,
                        const int64_t* tokens, int64_t n, double* y) {
  if (!layer_ok(L) || !valid(L->x) || C < 0) return -1;
  const int64_t d = L->d, N = L->N;
  const int64_t fmax = std::max(L->f, L->f_shared);
  Vec xr(sz(d)), a(sz(fmax)), h(sz(fmax)), o(sz(d)),
      buf(sz(std::max(d, fmax)));
  for (int64_t r = 0; r < n; ++r) {
    const int64_t t = tokens[r];
    if (t < 0 || t >= L->T) return -1;
    read(L->x, t * d, d, xr.data());
    double* yr = y + r * d;
    std::fill(yr, yr + d, 0.0);
    for (int64_t e = 0; e < N; ++e) {
      if (!std::binary_search(sel + e * C, sel + (e + 1) * C, t)) continue;
      Expert E;
      if (!expert_of(*L, e, &E)) return -1;
      expert_forward(*L, E, xr.data(), a.data(), h.data(), o.data(), buf.data());
      for (int64_t c = 0; c < d; ++c) yr[c] += p[t * N + e] * o[sz(c)];
    }
    if (L->f_shared > 0) {
      Expert S;
      if (!expert_of(*L, N, &S)) return -1;
      expert_forward(*L, S, xr.data(), a.data(), h.data(), o.data(), buf.data());
      for (int64_t c = 0; c < d; ++c) yr[c] += o[sz(c)];
    }
  }
  return 0;
}

// ---- backward pass ------------------------------------------------------------------
//
// total = <dy, y> + aux_weight * balance (botmartz.com "Load Balancing":
// total_loss = task_loss + 0.01 * balance_loss; dy stands for d task / d y).
// Each step is the chain rule through the matching forward step; the top-k
// choice and the capacity drops are piecewise constant and pass no gradient.

namespace {

// Gradient of the router scores of one token from its gate gradients dw [k]
// and the balance term: renormalised gates are a softmax over the k selected
// scores, dz_sel = w (dw - <w, dw>); raw gates are p[selected], so the
// gradient runs through the softmax over all N, dz = p (dp - <p, dp>).  The
// balance sum_e (m_e - 1/N)^2 / (N - 1), m_e = mean_t p[t, e], adds
// dp[t, e] = aux 2 (m_e - 1/N) / ((N - 1) T) through the softmax.
void score_grad(int64_t N, int64_t k, int64_t T, int32_t renormalize, const double* pt,
                const int64_t* it, const double* wt, const double* dwt, const double* mean_prob,
                double aux_weight, double* dzt) {
  std::fill(dzt, dzt + N, 0.0);
  if (renormalize) {
    double s = 0.0;
    for (int64_t j = 0; j < k; ++j) s += wt[j] * dwt[j];
    for (int64_t j = 0; j < k; ++j) dzt[it[j]] += wt[j] * (dwt[j] - s);
  } else {
    Vec dp(sz(N), 0.0);
    for (int64_t j = 0; j < k; ++j) dp[sz(it[j])] += dwt[j];
    double s = 0.0;
    for (int64_t e = 0; e < N; ++e) s += pt[e] * dp[sz(e)];
    for (int64_t e = 0; e < N; ++e) dzt[e] += pt[e] * (dp[sz(e)] - s);
  }
  if (aux_weight != 0.0 && N > 1 && T > 0) {
    Vec dp(sz(N));
    for (int64_t e = 0; e < N; ++e)
      dp[sz(e)] = aux_weight * 2.0 * (mean_prob[e] - 1.0 / double(N)) / double(N - 1) /
                      double(T);
    double s = 0.0;
    for (int64_t e = 0; e < N; ++e) s += pt[e] * dp[sz(e)];
    for (int64_t e = 0; e < N; ++e) dzt[e] += pt[e] * (dp[sz(e)] - s);
  }
}

}  // namespace

int orc_backward(const orc_layer* L, int64_t capacity, int32_t renormalize,
                 const int64_t* idx_override, orc_tensor dy, double aux_weight, double* dx,
                 double* dW_g, double* db_g, double* dW1, double* db1, double* dW2,
                 double* db2, double* dW1s, double* db1s, double* dW2s, double* db2s,
                 double* dz, double* dw) {
  if (!layer_ok(L) || !valid(dy) || !valid(L->x)) return -1;
  const int64_t T = L->T, N = L->N, k = L->k, d = L->d, f = L->f;
  Vec z(sz(T * N)), p(sz(T * N)), w(sz(T * k)), mean_prob(sz(N));
  std::vector<int64_t> idx(sz(T * k)), counts(sz(N)), kept(sz(N)),
      rank(sz(T * k)), order(sz(T * k)), start(sz(N + 1));
  std::vector<uint8_t> keep(sz(T * k));
  int64_t dropped = 0;
  double balance = 0.0, cv2 = 0.0;
  if (orc_route(L, capacity, renormalize, idx_override, nullptr, z.data(), p.data(),
                idx.data(), w.data(), counts.data(), kept.data(), rank.data(), keep.data(),
                order.data(), start.data(), &dropped, mean_prob.data(), &balance, &cv2) != 0)
    return -1;
  std::fill(dx, dx + T * d, 0.0);
  std::fill(dw, dw + T * k, 0.0);
  std::fill(dW1, dW1 + N * f * d, 0.0);
  std::fill(db1, db1 + N * f, 0.0);
  std::fill(dW2, dW2 + N * d * f, 0.0);
  std::fill(db2, db2 + N * d, 0.0);
  const int64_t fmax = std::max(f, L->f_shared);
  Vec xr(sz(d)), dyr(sz(d)), dO(sz(d)), a(sz(fmax)), h(sz(fmax)),
      o(sz(d)), da(sz(fmax)), buf(sz(std::max(d, fmax)));

  // one row of an expert: forward, then dW2 += dO h^T, db2 += dO,
  // da = (W2^T dO) * act'(a), dW1 += da x^T, db1 += da, dx += W1^T da
  auto row_backward = [&](const Expert& E, int64_t t, double gate, double* gW1, double* gb1,
                          double* gW2, double* gb2, double* dw_out) {
    const int64_t fe = E.f;
    read(L->x, t * d, d, xr.data());
    read(dy, t * d, d, dyr.data());
    expert_forward(*L, E, xr.data(), a.data(), h.data(), dw_out ? o.data() : nullptr,
                   buf.data());
    if (dw_out) *dw_out = dot(dyr.data(), o.data(), d);
    for (int64_t c = 0; c < d; ++c) dO[sz(c)] = gate * dyr[sz(c)];
    for (int64_t c = 0; c < d; ++c) {
      for (int64_t i = 0; i < fe; ++i) gW2[c * fe + i] += dO[sz(c)] * h[sz(i)];
      gb2[c] += dO[sz(c)];
    }
    expert_hidden_grad(*L, E, dO.data(), a.data(), da.data(), buf.data());
    for (int64_t i = 0; i < fe; ++i) {
      for (int64_t m = 0; m < d; ++m) gW1[i * d + m] += da[sz(i)] * xr[sz(m)];
      gb1[i] += da[sz(i)];
    }
    expert_input_grad(*L, E, da.data(), dx + t * d, buf.data());
  };

  for (int64_t e = 0; e < N; ++e) {
    Expert E;
    if (!expert_of(*L, e, &E)) return -1;
    for (int64_t r = start[sz(e)]; r < start[sz(e + 1)]; ++r) {
      const int64_t asg = order[sz(r)], t = asg / k;
      row_backward(E, t, w[sz(asg)], dW1 + e * f * d, db1 + e * f, dW2 + e * d * f,
                   db2 + e * d, &dw[asg]);
    }
  }
  if (L->f_shared > 0) {
    Expert S;
    if (!expert_of(*L, N, &S) || !dW1s || !db1s || !dW2s || !db2s) return -1;
    const int64_t fs = L->f_shared;
    std::fill(dW1s, dW1s + fs * d, 0.0);
    std::fill(db1s, db1s + fs, 0.0);
    std::fill(dW2s, dW2s + d * fs, 0.0);
    std::fill(db2s, db2s + d, 0.0);
    for (int64_t t = 0; t < T; ++t) row_backward(S, t, 1.0, dW1s, db1s, dW2s, db2s, nullptr);
  }
  // router scores, then z = x W_g^T + b_g: dW_g = dz^T x, db_g = sum_t dz, dx += dz W_g
  Vec Wg(sz(N * d));
  read(L->W_g, 0, N * d, Wg.data());
  std::fill(dW_g, dW_g + N * d, 0.0);
  std::fill(db_g, db_g + N, 0.0);
  for (int64_t t = 0; t < T; ++t) {
    double* dzt = dz + t * N;
    score_grad(N, k, T, renormalize, &p[sz(t * N)], &idx[sz(t * k)], &w[sz(t * k)],
               dw + t * k, mean_prob.data(), aux_weight, dzt);
    read(L->x, t * d, d, xr.data());
    for (int64_t e = 0; e < N; ++e) {
      for (int64_t m = 0; m < d; ++m) {
        dW_g[e * d + m] += dzt[e] * xr[sz(m)];
        dx[t * d + m] += dzt[e] * Wg[sz(e * d + m)];
      }
      db_g[e] += dzt[e];
    }
  }
  return 0;
}

// Router weight gradients from the score gradients: z = x W_g^T + b_g gives
// dW_g = dz^T x and db_g = sum_t dz.
int orc_router_weight_grads(const orc_layer* L, const double* dz, double* dW_g, double* db_g) {
  if (!layer_ok(L) || !valid(L->x)) return -1;
  const int64_t T = L->T, N = L->N, d = L->d;
  Vec xr(sz(d));
  std::fill(dW_g, dW_g + N * d, 0.0);
  std::fill(db_g, db_g + N, 0.0);
  for (int64_t t = 0; t < T; ++t) {
    read(L->x, t * d, d, xr.data());
    for (int64_t e = 0; e < N; ++e) {
      for (int64_t m = 0; m < d; ++m) dW_g[e * d + m] += dz[t * N + e] * xr[sz(m)];
      db_g[e] += dz[t * N + e];
    }
  }
  return 0;
}

int orc_expert_weight_grads(const orc_layer* L, int64_t e, const int64_t* tokens,
                            const double* gates, int64_t n_rows, orc_tensor dy,
                            const int64_t* units, int64_t n_units, double* dW1_rows,
                            double* db1, double* dW2_cols, double* db2) {
  Expert E;
  if (!layer_ok(L) || !valid(dy) || !valid(L->x) || !expert_of(*L, e, &E)) return -1;
  const int64_t d = L->d, f = E.f;
  std::vector<int64_t> all;
  if (!units) {
    all.resize(sz(f));
    std::iota(all.begin(), all.end(), int64_t(0));
    units = all.data();
    n_units = f;
  }
  for (int64_t u = 0; u < n_units; ++u)
    if (units[u] < 0 || units[u] >= f) return -1;
  std::fill(dW1_rows, dW1_rows + n_units * d, 0.0);
  std::fill(db1, db1 + n_units, 0.0);
  std::fill(dW2_cols, dW2_cols + d * n_units, 0.0);
  std::fill(db2, db2 + d, 0.0);
  Vec xr(sz(d)), dO(sz(d)), buf(sz(std::max(d, f))), a(sz(f)), h(sz(f)),
      da(sz(f));
  const bool full = !all.empty();
  for (int64_t r = 0; r < n_rows; ++r) {
    const int64_t t = tokens[r];
    if (t < 0 || t >= L->T) return -1;
    read(L->x, t * d, d, xr.data());
    read(dy, t * d, d, dO.data());
    for (int64_t c = 0; c < d; ++c) dO[sz(c)] *= gates[r];
    if (full) {   // every hidden unit: the row-wise products
      expert_forward(*L, E, xr.data(), a.data(), h.data(), nullptr, buf.data());
      expert_hidden_grad(*L, E, dO.data(), a.data(), da.data(), buf.data());
    }
    for (int64_t u = 0; u < n_units; ++u) {
      const int64_t i = units[u];
      double ai, hi, dai;
      if (full) {
        ai = a[sz(i)];
        hi = h[sz(i)];
        dai = da[sz(i)];
      } else {    // one hidden unit: a row of W1, a column of W2
        read(E.W1, E.o1 + i * d, d, buf.data());
        ai = dot(buf.data(), xr.data(), d) + at(E.b1, E.ob1 + i);
        const double v = act_value(L->act, ai);
        hi = L->round_hidden_bf16 ? orc_round_bf16(v) : v;
        double dh = 0.0;
        for (int64_t c = 0; c < d; ++c) dh += at(E.W2, E.o2 + c * f + i) * dO[sz(c)];
        dai = dh * act_derivative(L->act, ai);
      }
      for (int64_t m = 0; m < d; ++m) dW1_rows[u * d + m] += dai * xr[sz(m)];
      db1[u] += dai;
      for (int64_t c = 0; c < d; ++c) dW2_cols[c * n_units + u] += dO[sz(c)] * hi;
    }
    for (int64_t c = 0; c < d; ++c) db2[c] += dO[sz(c)];
  }
  return 0;
}

int orc_token_grads(const orc_layer* L, int32_t renormalize, const double* p,
                    const int64_t* idx, const double* w, const uint8_t* keep, orc_tensor dy,
                    double aux_weight, const int64_t* tokens, int64_t n, double* dw, double* dz,
                    double* dx) {
  if (!layer_ok(L) || !valid(dy) || !valid(L->x) || !valid(L->W_g)) return -1;
  const int64_t T = L->T, N = L->N, k = L->k, d = L->d;
  Vec mean_prob(sz(N));
  double balance = 0.0;
  if (orc_balance(T, N, p, mean_prob.data(), &balance) != 0) return -1;
  Vec Wg(sz(N * d));
  read(L->W_g, 0, N * d, Wg.data());
  const int64_t fmax = std::max(L->f, L->f_shared);
  Vec xr(sz(d)), dyr(sz(d)), dO(sz(d)), a(sz(fmax)), h(sz(fmax)),
      o(sz(d)), da(sz(fmax)), buf(sz(std::max(d, fmax)));
  for (int64_t r = 0; r < n; ++r) {
    const int64_t t = tokens[r];
    if (t < 0 || t >= T) return -1;
    read(L->x, t * d, d, xr.data());
    read(dy, t * d, d, dyr.data());
    double* dxr = dx + r * d;
    std::fill(dxr, dxr + d, 0.0);
    for (int64_t j = 0; j < k; ++j) {
      dw[r * k + j] = 0.0;
      if (!keep[t * k + j]) continue;
      Expert E;
      if (!expert_of(*L, idx[t * k + j], &E) || idx[t * k + j] == N) return -1;
      expert_forward(*L, E, xr.data(), a.data(), h.data(), o.data(), buf.data());
      dw[r * k + j] = dot(dyr.data(), o.data(), d);
      for (int64_t c = 0; c < d; ++c) dO[sz(c)] = w[t * k + j] * dyr[sz(c)];
      expert_hidden_grad(*L, E, dO.data(), a.data(), da.data(), buf.data());
      expert_input_grad(*L, E, da.data(), dxr, buf.data());
    }
    if (L->f_shared > 0) {
      Expert S;
      if (!expert_of(*L, N, &S)) return -1;
      expert_forward(*L, S, xr.data(), a.data(), h.data(), nullptr, buf.data());
      expert_hidden_grad(*L, S, dyr.data(), a.data(), da.data(), buf.data());
      expert_input_grad(*L, S, da.data(), dxr, buf.data());
    }
    score_grad(N, k, T, renormalize, p + t * N, idx + t * k, w + t * k, dw + r * k,
               mean_prob.data(), aux_weight, dz + r * N);
    for (int64_t e = 0; e < N; ++e)
      for (int64_t m = 0; m < d; ++m) dxr[m] += dz[r * N + e] * Wg[sz(e * d + m)];
  }
  return 0;
}

}  // extern "C"
