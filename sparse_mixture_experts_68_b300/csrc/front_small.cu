// Front end of the forward pass for a small batch (decoding: a few tokens,
// a few experts): the router scores z = x . W_g^T + b_g, the softmax, the
// top-k and its gates (botmartz.com "Mixture of Experts (MoE) and Mixtral",
// section "Expert Routing"; codingnowai.in "Mixture of Experts", section
// "Code", for gates without renormalisation), the stable counting sort of the
// assignments into padded expert groups with capacity dropping, and the load
// statistics -- in two launches.
//
// With a handful of tokens the router reads only x (T rows) and W_g (N rows),
// a few hundred KB, and the usual one-warp-per-token router leaves that to two
// or three blocks whose loads come back one latency at a time.  Here the
// reduction over d is cut into G slices of 64 columns, one block each, so
// every byte is requested in the first wave of loads across the SMs:
//
//   front_scores_kernel (G blocks): part[b][t][e] = sum over the b-th slice of
//       d of x[t][i] * W_g[e][i], in column order.
//   front_route_kernel (one block of 1024 threads): z = the slices' sums in
//       slice order + b_g; softmax, top-k and gates per token; per-expert
//       counts, kept counts, padded group offsets and the row maps; the load
//       statistics.  The same results as the router and the one-block sort up
//       to the order of the fp32 additions in z.
#include <float.h>

#include "common.cuh"
#include "kernels.h"
#include "stats.cuh"

namespace moe {
namespace {

constexpr int kFrontSlice = 64;          // columns of d per scores block
constexpr int kFrontMaxT = 32;           // tokens
constexpr int kFrontMaxN = 64;           // experts
constexpr int kFrontMaxA = 256;          // assignments T * k
constexpr int kFrontMaxBlocks = 148;     // slices of d

template <typename TIn>
__global__ void __launch_bounds__(256)
    front_scores_kernel(const TIn* __restrict__ x, const TIn* __restrict__ W_g, int T, int d,
                        int N, float* __restrict__ part) {
  constexpr int V = Vec16<TIn>::n;
  constexpr int kPitch = kFrontSlice + 1;       // padded rows: conflict-free columns
  __shared__ float xs[kFrontMaxT * kPitch];
  __shared__ float ws[kFrontMaxN * kPitch];
  pdl_launch_dependents();
  pdl_wait_previous();
  const int c0 = blockIdx.x * kFrontSlice;
  const int len = min(kFrontSlice, d - c0);     // a multiple of V
  const int nv = len / V;
  for (int i = threadIdx.x; i < (T + N) * nv; i += blockDim.x) {
    const int r = i / nv, v = i - r * nv;
    float f[V];
    if (r < T) {
      Vec16<TIn>::load(x + int64_t(r) * d + c0 + v * V, f);
#pragma unroll
      for (int u = 0; u < V; ++u) xs[r * kPitch + v * V + u] = f[u];
    } else {
      Vec16<TIn>::load(W_g + int64_t(r - T) * d + c0 + v * V, f);
#pragma unroll
      for (int u = 0; u < V; ++u) ws[(r - T) * kPitch + v * V + u] = f[u];
    }
  }
  __syncthreads();
  for (int pr = threadIdx.x; pr < T * N; pr += blockDim.x) {
    const int t = pr / N, e = pr - t * N;
    const float* xr = xs + t * kPitch;
    const float* wr = ws + e * kPitch;
    float acc = 0.f;
    for (int i = 0; i < len; ++i) acc = fmaf(xr[i], wr[i], acc);
    part[(int64_t(blockIdx.x) * T + t) * N + e] = acc;
  }
}

// part[b0 .. b1)[q] added in slice order; the loads of eight slices and
// their additions are unconditional (an index past b1 reads slice b1 - 1 and
// a select adds 0 instead), so the loads are in flight together rather than
// one round trip each.
__device__ __forceinline__ float sum_slices(const float* __restrict__ part, int P, int q,
                                            int b0, int b1) {
  float acc = 0.f;
  for (int b = b0; b < b1; b += 8) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = __ldcg(part + int64_t(min(b + u, b1 - 1)) * P + q);
#pragma unroll
    for (int u = 0; u < 8; ++u) acc += b + u < b1 ? v[u] : 0.f;   // + 0 changes nothing
  }
  return acc;
}

template <typename TIn>
__global__ void __launch_bounds__(1024)
    front_route_kernel(const float* __restrict__ part, int G, const TIn* __restrict__ b_g,
                       int T, int N, int k, int64_t capacity, int renorm, int has_shared,
                       float* __restrict__ logits, int32_t* __restrict__ topk_idx,
                       float* __restrict__ topk_w, int32_t* __restrict__ counts,
                       int32_t* __restrict__ kept, int32_t* __restrict__ offsets,
                       int32_t* __restrict__ row_token, int32_t* __restrict__ token_row,
                       float* __restrict__ mean_prob, float* __restrict__ balance,
                       int32_t* __restrict__ dropped, float* __restrict__ cv_squared) {
  __shared__ float red[1024];                        // slice-group sums, then z
  __shared__ float ps[kFrontMaxT * kFrontMaxN];      // probabilities [t][e]
  __shared__ int32_t ids[kFrontMaxA];                // expert of each assignment
  __shared__ int32_t cnt_s[kFrontMaxN], kept_s[kFrontMaxN], off_s[kFrontMaxN];
  __shared__ float psum[kFrontMaxN];                 // sum over tokens of p, per expert
  pdl_launch_dependents();
  pdl_wait_previous();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int P = T * N, A = T * k;
  // 1. z: thread (pair, group) sums the group's slices in order; the groups'
  //    sums are then added in order
  const int S = P >= 1024 ? 1 : 1024 / P;            // slice groups
  const int Gs = (G + S - 1) / S;
  float zsum[2] = {0.f, 0.f};
  {
    const int pr = tid % P, grp = tid / P;
    if (P <= 1024 && grp < S) {
      const int b0 = grp * Gs, b1 = min(G, b0 + Gs);
      red[grp * P + pr] = sum_slices(part, P, pr, b0, b1);
    } else if (P > 1024) {
      // P <= 2048: two pairs per thread, all slices
      for (int h = 0; h < 2; ++h) {
        const int q = tid + h * 1024;
        zsum[h] = q < P ? sum_slices(part, P, q, 0, G) : 0.f;
      }
    }
  }
  __syncthreads();
  float zv[2];
  for (int h = 0; h < 2; ++h) {
    const int q = tid + h * 1024;
    zv[h] = 0.f;
    if (q >= P) continue;
    float acc;
    if (P <= 1024) {
      acc = 0.f;
      for (int g = 0; g < S; ++g) acc += red[g * P + q];
    } else {
      acc = zsum[h];
    }
    const int e = q % N;
    zv[h] = acc + to_f32(b_g[e]);
    logits[q] = zv[h];
    ps[q] = zv[h];                                    // z, replaced by p below
  }
  __syncthreads();
  // 2. softmax, top-k and gates: warp t takes token t, lane l experts l and
  //    l + 32 (the larger score first, then the lower expert)
  if (warp < T) {
    const int t = warp;
    float z[2], m = -FLT_MAX;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int e = lane + 32 * i;
      z[i] = e < N ? ps[t * N + e] : -INFINITY;
      m = fmaxf(m, z[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float ex[2], ssum = 0.f;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      ex[i] = lane + 32 * i < N ? expf(z[i] - m) : 0.f;
      ssum += ex[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
    const float inv = 1.0f / ssum;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int e = lane + 32 * i;
      if (e < N) ps[t * N + e] = ex[i] * inv;
    }
    uint32_t taken = 0;
    float kept_sum = 0.f, my_g = 0.f;
    int my_e = 0;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int e = lane + 32 * i;
        if (e < N && !((taken >> i) & 1u) && (z[i] > bv || (z[i] == bv && e < be))) {
          bv = z[i];
          be = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
      }
      if (be == lane) taken |= 1u;
      if (be == lane + 32) taken |= 2u;
      const float g = expf(bv - m);
      kept_sum += g;
      if (lane == 0) MOE_CHECK(be >= 0 && be < N, CK_ROUTER_TOPK);
      if (lane == j) { my_e = be; my_g = g; }         // k <= 8: slot j on lane j
    }
    const float scale = renorm ? 1.0f / kept_sum : inv;
    if (lane < k) {
      topk_idx[t * k + lane] = my_e;
      topk_w[t * k + lane] = my_g * scale;
      ids[t * k + lane] = (my_e >= 0 && my_e < N) ? my_e : -1;
    }
  }
  __syncthreads();
  // 3. per expert: routed and kept counts, the sum of p over tokens (in token
  //    order); thread 0 then lays out the padded groups
  if (tid < N) {
    int32_t c = 0;
    for (int a = 0; a < A; ++a) c += ids[a] == tid ? 1 : 0;
    const int32_t kp = (capacity > 0 && int64_t(c) > capacity) ? int32_t(capacity) : c;
    cnt_s[tid] = c;
    kept_s[tid] = kp;
    counts[tid] = c;
    kept[tid] = kp;
    float sp = 0.f;
    for (int t = 0; t < T; ++t) sp += ps[t * N + tid];
    psum[tid] = sp;
  }
  __syncthreads();
  if (tid == 0) {
    int32_t off = 0;
    for (int e = 0; e < N; ++e) {
      off_s[e] = off;
      offsets[e] = off;
      off += int32_t(round_up(kept_s[e], kGroupAlign));
    }
    offsets[N] = off;
    offsets[N + 1] = off + (has_shared ? int32_t(round_up(T, kGroupAlign)) : 0);
  }
  __syncthreads();
  // 4. rows: an assignment's rank is the number of earlier assignments to its
  //    expert (stable in token, then slot order); padding rows are -1
  for (int a = tid; a < A; a += blockDim.x) {
    const int e = ids[a];
    int32_t row = -1;
    if (e >= 0) {
      int32_t rank = 0;
      for (int b = 0; b < a; ++b) rank += ids[b] == e ? 1 : 0;
      if (capacity <= 0 || rank < capacity) {
        row = off_s[e] + rank;
        row_token[row] = a / k;
      }
    }
    token_row[a] = row;
  }
  for (int e = 0; e < N; ++e) {
    const int32_t r0 = off_s[e] + kept_s[e];
    const int32_t r1 = off_s[e] + int32_t(round_up(kept_s[e], kGroupAlign));
    for (int32_t r = r0 + tid; r < r1; r += blockDim.x) row_token[r] = -1;
  }
  // 5. load statistics from the per-expert sums (one partial row)
  __syncthreads();
  block_load_stats(psum, 1, N, T, cnt_s, kept_s, mean_prob, balance, dropped, cv_squared);
}

}  // namespace

bool small_front_fits(const moe_config& c) {
  return c.T >= 1 && c.T <= kFrontMaxT && c.n_experts <= kFrontMaxN && c.top_k <= 8 &&
         c.T * c.top_k <= kFrontMaxA &&
         ceil_div(c.d_model, int64_t(kFrontSlice)) <= kFrontMaxBlocks;
}

int64_t small_front_partial_floats(const moe_config& c) {
  if (!small_front_fits(c)) return 0;
  return ceil_div(c.d_model, int64_t(kFrontSlice)) * c.T * c.n_experts;
}

cudaError_t launch_small_front(const moe_config& c, const void* x, const void* W_g,
                               const void* b_g, float* part, float* logits, int32_t* topk_idx,
                               float* topk_w, int32_t* counts, int32_t* kept, int32_t* offsets,
                               int32_t* row_token, int32_t* token_row, float* mean_prob,
                               float* balance, int32_t* dropped, float* cv_squared,
                               cudaStream_t s) {
  const int G = int(ceil_div(c.d_model, int64_t(kFrontSlice)));
  const int T = int(c.T), d = int(c.d_model), N = int(c.n_experts), k = int(c.top_k);
  cudaError_t e;
  if (c.dtype == MOE_F32)
    e = launch_pdl(front_scores_kernel<float>, dim3(G), dim3(256), 0, s,
                   static_cast<const float*>(x), static_cast<const float*>(W_g), T, d, N, part);
  else
    e = launch_pdl(front_scores_kernel<__nv_bfloat16>, dim3(G), dim3(256), 0, s,
                   static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(W_g),
                   T, d, N, part);
  if (e != cudaSuccess) return e;
  const int rn = c.renormalize ? 1 : 0, sh = c.d_ff_shared > 0 ? 1 : 0;
  if (c.dtype == MOE_F32)
    return launch_pdl(front_route_kernel<float>, dim3(1), dim3(1024), 0, s,
                      static_cast<const float*>(part), G, static_cast<const float*>(b_g), T, N,
                      k, c.capacity, rn, sh, logits, topk_idx, topk_w, counts, kept, offsets,
                      row_token, token_row, mean_prob, balance, dropped, cv_squared);
  return launch_pdl(front_route_kernel<__nv_bfloat16>, dim3(1), dim3(1024), 0, s,
                    static_cast<const float*>(part), G,
                    static_cast<const __nv_bfloat16*>(b_g), T, N, k, c.capacity, rn, sh, logits,
                    topk_idx, topk_w, counts, kept, offsets, row_token, token_row, mean_prob,
                    balance, dropped, cv_squared);
}

MOE_CHECKS_UNIT(front_small)

}  // namespace moe
