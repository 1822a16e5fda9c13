// Gate-weighted combine back to token order and the load statistics.
//
// Combine (roadtointelligence.com "Mixture of Experts (MoE)", output equation
// y = sum over top-K of G(x)_i E_i(x); botmartz.com "Mixture of Experts (MoE)
// and Mixtral", "Expert Routing", outputs[mask] += prob * expert(x)): a gather,
// one warp per token, fp32 accumulation in slot order, 16-byte vectors.
// Dropped slots (token_row < 0) add nothing; the shared expert's row adds
// with weight 1 (roadtointelligence.com "Total versus active parameters").
//
// Load statistics (botmartz.com "Load Balancing: The Hidden Challenge"):
// mean over tokens of the router probabilities and its unbiased variance.
#include "kernels.h"
#include "common.cuh"

namespace moe {

namespace {

constexpr int kCombineWarps = 8;

template <typename T>
__global__ void __launch_bounds__(kCombineWarps * 32)
    combine_kernel(const T* __restrict__ Yp, const int32_t* __restrict__ token_row,
                   const float* __restrict__ topk_w, const int32_t* __restrict__ offsets,
                   int Ttok, int k, int N, int has_shared, int64_t d, T* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const int64_t t = int64_t(blockIdx.x) * kCombineWarps + (threadIdx.x >> 5);
  if (t >= Ttok) return;
  constexpr int V = Vec16<T>::n;
  const int64_t shared_row = has_shared ? int64_t(offsets[N]) + t : -1;
  for (int64_t c = int64_t(lane) * V; c < d; c += 32 * V) {
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;
    for (int j = 0; j < k; ++j) {
      const int32_t r = token_row[t * k + j];
      if (r < 0) continue;
      const float g = topk_w[t * k + j];
      float v[V];
      Vec16<T>::load(Yp + int64_t(r) * d + c, v);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] = fmaf(g, v[i], acc[i]);
    }
    if (shared_row >= 0) {
      float v[V];
      Vec16<T>::load(Yp + shared_row * d + c, v);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] += v[i];
    }
    Vec16<T>::store(y + t * d + c, acc);
  }
}

// One block of 256 threads; fp64 sums in a fixed order.
__global__ void __launch_bounds__(256)
    load_stats_kernel(const float* __restrict__ prob_partials, int nblk, int N, int Ttok,
                      const int32_t* __restrict__ counts, const int32_t* __restrict__ kept,
                      float* __restrict__ mean_prob, float* __restrict__ balance,
                      int32_t* __restrict__ dropped) {
  __shared__ double sq[256];
  __shared__ long long dr[256];
  double my_sq = 0.0;
  long long my_dr = 0;
  const double invN = 1.0 / double(N);
  for (int e = threadIdx.x; e < N; e += blockDim.x) {
    double s = 0.0;
    for (int b = 0; b < nblk; ++b) s += double(prob_partials[int64_t(b) * N + e]);
    const double m = Ttok > 0 ? s / double(Ttok) : 0.0;
    mean_prob[e] = float(m);
    my_sq += (m - invN) * (m - invN);
    my_dr += counts[e] - kept[e];
  }
  sq[threadIdx.x] = my_sq;
  dr[threadIdx.x] = my_dr;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if (threadIdx.x < o) {
      sq[threadIdx.x] += sq[threadIdx.x + o];
      dr[threadIdx.x] += dr[threadIdx.x + o];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    *balance = (N > 1 && Ttok > 0) ? float(sq[0] / double(N - 1)) : 0.f;
    *dropped = int32_t(dr[0]);
  }
}

}  // namespace

cudaError_t launch_combine(const moe_config& c, const void* Yp, const int32_t* token_row,
                           const float* topk_w, const int32_t* offsets, void* y,
                           cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  const unsigned blocks = unsigned(ceil_div(c.T, kCombineWarps));
  const int hs = c.d_ff_shared > 0 ? 1 : 0;
  if (c.dtype == MOE_F32)
    combine_kernel<float><<<blocks, kCombineWarps * 32, 0, s>>>(
        static_cast<const float*>(Yp), token_row, topk_w, offsets, int(c.T), int(c.top_k),
        int(c.n_experts), hs, c.d_model, static_cast<float*>(y));
  else
    combine_kernel<__nv_bfloat16><<<blocks, kCombineWarps * 32, 0, s>>>(
        static_cast<const __nv_bfloat16*>(Yp), token_row, topk_w, offsets, int(c.T),
        int(c.top_k), int(c.n_experts), hs, c.d_model, static_cast<__nv_bfloat16*>(y));
  return cudaGetLastError();
}

cudaError_t launch_load_stats(const moe_config& c, const float* prob_partials,
                              const int32_t* counts, const int32_t* kept, float* mean_prob,
                              float* balance, int32_t* dropped, cudaStream_t s) {
  const int nblk = int(ceil_div(c.T, kRouterTokensPerBlock));
  load_stats_kernel<<<1, 256, 0, s>>>(prob_partials, nblk, int(c.n_experts), int(c.T),
                                      counts, kept, mean_prob, balance, dropped);
  return cudaGetLastError();
}

}  // namespace moe
