// Gate-weighted combine back to token order and the load statistics.
//
// Combine (roadtointelligence.com "Mixture of Experts (MoE)", output equation
// y = sum over top-K of G(x)_i E_i(x); botmartz.com "Mixture of Experts (MoE)
// and Mixtral", "Expert Routing", outputs[mask] += prob * expert(x)): a gather,
// one warp per token, fp32 accumulation in slot order, 16-byte vectors.
// Dropped slots (token_row < 0) add nothing; the shared expert's row adds
// with weight 1 (roadtointelligence.com "Total versus active parameters").
// The warp first reads its token's slots 32 at a time and keeps the live
// ones (and the shared row), in slot order, in shared memory, so that the
// column passes walk only those, two rows' loads in flight at a time.
//
// Load statistics: see stats.cuh.
#include "kernels.h"
#include "stats.cuh"

namespace moe {

namespace {

constexpr int kCombineWarps = 8;

template <typename T>
__global__ void __launch_bounds__(kCombineWarps * 32, 4)   // 4 blocks per SM: latency-bound gathers
    combine_kernel(const T* __restrict__ Yp, const int32_t* __restrict__ token_row,
                   const float* __restrict__ topk_w, const int32_t* __restrict__ offsets,
                   int Ttok, int k, int N, int has_shared, int64_t d, T* __restrict__ y) {
  constexpr int V = Vec16<T>::n;
  constexpr int CB = 4;                            // 16-byte columns per lane per pass
  extern __shared__ int2 live[];                   // [kCombineWarps][k + 1] (row, gate)
  pdl_launch_dependents();
  pdl_wait_previous();
  const int lane = threadIdx.x & 31;
  const int64_t t = int64_t(blockIdx.x) * kCombineWarps + (threadIdx.x >> 5);
  if (t >= Ttok) return;
  // the token's kept rows in slot order, then the shared expert's (gate 1):
  // all slots read at once, so that the row loads below depend on one round trip
  int2* mine = live + (threadIdx.x >> 5) * (k + 1);
  int n_live = 0;
  const int routed_end = offsets[N];             // rows past it are not routed rows
  for (int j0 = 0; j0 < k; j0 += 32) {
    const int j = j0 + lane;
    int r = j < k ? token_row[t * k + j] : -1;
    MOE_CHECK(r < routed_end, CK_COMBINE_ROW);
    if (r >= routed_end) r = -1;
    const float g = j < k ? topk_w[t * k + j] : 0.f;
    const uint32_t m = __ballot_sync(0xffffffffu, r >= 0);
    if (r >= 0) mine[n_live + __popc(m & ((1u << lane) - 1u))] = make_int2(r, __float_as_int(g));
    n_live += __popc(m);
  }
  if (has_shared) {
    if (lane == 0) mine[n_live] = make_int2(offsets[N] + int(t), __float_as_int(1.f));
    ++n_live;
  }
  __syncwarp();
  const int64_t nv = d / V;
  // few tokens (decode): the columns are split over gridDim.y blocks per token group
  const int64_t per = (nv + gridDim.y - 1) / gridDim.y;
  const int64_t c_end = min(nv, per * (blockIdx.y + 1));
  for (int64_t c0 = per * blockIdx.y + lane; c0 < c_end; c0 += 32 * CB) {
    float acc[CB][V];
#pragma unroll
    for (int b = 0; b < CB; ++b)
#pragma unroll
      for (int i = 0; i < V; ++i) acc[b][i] = 0.f;
    // two rows' loads in flight, accumulated in slot order
    for (int j = 0; j < n_live; j += 2) {
      const bool two = j + 1 < n_live;
      const int2 rg0 = mine[j];
      const int2 rg1 = two ? mine[j + 1] : rg0;
      const uint4* row0 = reinterpret_cast<const uint4*>(Yp + int64_t(rg0.x) * d);
      const uint4* row1 = reinterpret_cast<const uint4*>(Yp + int64_t(rg1.x) * d);
      uint4 q0[CB], q1[CB];
#pragma unroll
      for (int b = 0; b < CB; ++b) {
        const int64_t c = c0 + 32 * b;
        q0[b] = c < c_end ? __ldg(row0 + c) : make_uint4(0, 0, 0, 0);
        q1[b] = (two && c < c_end) ? __ldg(row1 + c) : make_uint4(0, 0, 0, 0);
      }
      const float g0 = __int_as_float(rg0.y), g1 = __int_as_float(rg1.y);
#pragma unroll
      for (int b = 0; b < CB; ++b) {
        float v[V];
        Vec16<T>::load(reinterpret_cast<const T*>(&q0[b]), v);
#pragma unroll
        for (int i = 0; i < V; ++i) acc[b][i] = fmaf(g0, v[i], acc[b][i]);
      }
      if (two) {
#pragma unroll
        for (int b = 0; b < CB; ++b) {
          float v[V];
          Vec16<T>::load(reinterpret_cast<const T*>(&q1[b]), v);
#pragma unroll
          for (int i = 0; i < V; ++i) acc[b][i] = fmaf(g1, v[i], acc[b][i]);
        }
      }
    }
#pragma unroll
    for (int b = 0; b < CB; ++b) {
      const int64_t c = c0 + 32 * b;
      if (c < c_end) Vec16<T>::store(y + t * d + c * V, acc[b]);
    }
  }
}

__global__ void __launch_bounds__(kStatsThreads)
    load_stats_kernel(const float* __restrict__ prob_partials, int nblk, int N, int Ttok,
                      const int32_t* __restrict__ counts, const int32_t* __restrict__ kept,
                      float* __restrict__ mean_prob, float* __restrict__ balance,
                      int32_t* __restrict__ dropped, float* __restrict__ cv_squared) {
  pdl_launch_dependents();
  pdl_wait_previous();
  block_load_stats(prob_partials, nblk, N, Ttok, counts, kept, mean_prob, balance, dropped,
                   cv_squared);
}

// Statistics of a batch run as two consecutive token chunks (moe_forward_host):
// the chunks' routed and kept counts added per expert, then the statistics
// from both chunks' probability partial-sum rows.
__global__ void __launch_bounds__(kStatsThreads)
    chunk_stats_kernel(const float* __restrict__ prob_rows, int nblk, int N, int Ttok,
                       const int32_t* __restrict__ counts0, const int32_t* __restrict__ kept0,
                       const int32_t* __restrict__ counts1, const int32_t* __restrict__ kept1,
                       int32_t* __restrict__ counts, int32_t* __restrict__ kept,
                       float* __restrict__ mean_prob, float* __restrict__ balance,
                       int32_t* __restrict__ dropped, float* __restrict__ cv_squared) {
  pdl_launch_dependents();
  pdl_wait_previous();
  for (int e = threadIdx.x; e < N; e += blockDim.x) {
    counts[e] = counts0[e] + counts1[e];
    kept[e] = kept0[e] + kept1[e];
  }
  __syncthreads();
  block_load_stats(prob_rows, nblk, N, Ttok, counts, kept, mean_prob, balance, dropped,
                   cv_squared);
}

}  // namespace

cudaError_t launch_chunk_stats(const moe_config& c, const float* prob_rows, int nblk,
                               const int32_t* counts0, const int32_t* kept0,
                               const int32_t* counts1, const int32_t* kept1, int32_t* counts,
                               int32_t* kept, float* mean_prob, float* balance,
                               int32_t* dropped, float* cv_squared, cudaStream_t s) {
  return launch_pdl(chunk_stats_kernel, dim3(1), dim3(kStatsThreads), 0, s, prob_rows, nblk,
                    int(c.n_experts), int(c.T), counts0, kept0, counts1, kept1, counts, kept,
                    mean_prob, balance, dropped, cv_squared);
}

cudaError_t launch_combine(const moe_config& c, const void* Yp, const int32_t* token_row,
                           const float* topk_w, const int32_t* offsets, void* y,
                           cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  const unsigned blocks = unsigned(ceil_div(c.T, kCombineWarps));
  // few tokens: split each token's columns into chunks of at least one
  // warp pass (32 lanes x 4 x 16 bytes), until there are about eight warps per SM
  const int64_t vec = c.dtype == MOE_F32 ? 4 : 8;
  const int64_t passes = ceil_div(c.d_model / vec, 32 * 4);
  int64_t split = ceil_div(148 * 8, int64_t(blocks) * kCombineWarps);
  if (split > passes) split = passes;
  if (split < 1) split = 1;
  const int hs = c.d_ff_shared > 0 ? 1 : 0;
  const size_t smem = size_t(kCombineWarps) * size_t(c.top_k + 1) * sizeof(int2);
  auto go = [&](auto kern, auto* Yt, auto* yt) -> cudaError_t {
    if (smem > 48 * 1024) {
      const cudaError_t e =
          cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
      if (e != cudaSuccess) return e;
    }
    return launch_pdl(kern, dim3(blocks, unsigned(split)), dim3(kCombineWarps * 32), smem, s,
                      Yt, token_row,
                      topk_w, offsets, int(c.T), int(c.top_k), int(c.n_experts), hs,
                      c.d_model, yt);
  };
  if (c.dtype == MOE_F32) {
    const float* Yt = static_cast<const float*>(Yp);
    float* yt = static_cast<float*>(y);
    return go(combine_kernel<float>, Yt, yt);
  }
  const __nv_bfloat16* Yt = static_cast<const __nv_bfloat16*>(Yp);
  __nv_bfloat16* yt = static_cast<__nv_bfloat16*>(y);
  return go(combine_kernel<__nv_bfloat16>, Yt, yt);
}

cudaError_t launch_load_stats(const moe_config& c, const float* prob_partials,
                              const int32_t* counts, const int32_t* kept, float* mean_prob,
                              float* balance, int32_t* dropped, float* cv_squared,
                              cudaStream_t s) {
  const int nblk = int(router_partial_rows(c));
  return launch_pdl(load_stats_kernel, dim3(1), dim3(kStatsThreads), 0, s, prob_partials, nblk,
                    int(c.n_experts), int(c.T), counts, kept, mean_prob, balance, dropped,
                    cv_squared);
}

MOE_CHECKS_UNIT(combine)

}  // namespace moe
