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
  constexpr int V = Vec16<T>::n;
  constexpr int CB = 4;                            // 16-byte columns per lane per pass
  const int lane = threadIdx.x & 31;
  const int64_t t = int64_t(blockIdx.x) * kCombineWarps + (threadIdx.x >> 5);
  if (t >= Ttok) return;
  const int64_t shared_row = has_shared ? int64_t(offsets[N]) + t : -1;
  const int64_t nv = d / V;
  for (int64_t c0 = lane; c0 < nv; c0 += 32 * CB) {
    float acc[CB][V];
#pragma unroll
    for (int b = 0; b < CB; ++b)
#pragma unroll
      for (int i = 0; i < V; ++i) acc[b][i] = 0.f;
    for (int j = 0; j <= k; ++j) {
      int64_t r;
      float g;
      if (j < k) {
        r = token_row[t * k + j];
        g = topk_w[t * k + j];
      } else {
        r = shared_row;                            // the shared expert, weight 1
        g = 1.f;
      }
      if (r < 0) continue;
      const uint4* row = reinterpret_cast<const uint4*>(Yp + r * d);
      uint4 q[CB];
#pragma unroll
      for (int b = 0; b < CB; ++b) {
        const int64_t c = c0 + 32 * b;
        q[b] = c < nv ? __ldg(row + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int b = 0; b < CB; ++b) {
        float v[V];
        Vec16<T>::load(reinterpret_cast<const T*>(&q[b]), v);
#pragma unroll
        for (int i = 0; i < V; ++i) acc[b][i] = fmaf(g, v[i], acc[b][i]);
      }
    }
#pragma unroll
    for (int b = 0; b < CB; ++b) {
      const int64_t c = c0 + 32 * b;
      if (c < nv) Vec16<T>::store(y + t * d + c * V, acc[b]);
    }
  }
}

// One block of 1024 threads, all sums in a fixed order and in fp32 (B300's
// fp64 rate is low, and an fp64 division alone costs microseconds); accuracy
// comes from compensated arithmetic instead.  The partial-sum rows are split
// into RG row groups and the experts into 32-wide chunks; warp w takes (row
// group w % RG, chunk w / RG) with lane = expert, so every load is a
// coalesced 128-byte row segment, eight of them in flight.  Each warp keeps a
// Kahan sum per expert; the row groups are combined in order with
// error-free additions (two-sum).  The deviation from the uniform load is
// taken as (S - T/N) / T with S the compensated sum, so it keeps its
// accuracy when the load is nearly uniform.
constexpr int kStatsThreads = 1024;
constexpr int kStatsWarps = kStatsThreads / 32;

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& err) {
  s = a + b;
  const float bb = s - a;
  err = (a - (s - bb)) + (b - bb);
}

__device__ __forceinline__ void kahan_add(float v, float& s, float& comp) {
  const float y = v - comp;
  const float t = s + y;
  comp = (t - s) - y;
  s = t;
}

__global__ void __launch_bounds__(kStatsThreads)
    load_stats_kernel(const float* __restrict__ prob_partials, int nblk, int N, int Ttok,
                      const int32_t* __restrict__ counts, const int32_t* __restrict__ kept,
                      float* __restrict__ mean_prob, float* __restrict__ balance,
                      int32_t* __restrict__ dropped) {
  __shared__ float2 part[kStatsWarps][32];        // (sum, -compensation) per warp, lane
  __shared__ float2 sq[kStatsWarps];              // Kahan sum of squared deviations
  __shared__ int dr[kStatsWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nchunks = (N + 31) / 32;
  const float invT = Ttok > 0 ? 1.0f / float(Ttok) : 0.f;
  const float tN = float(Ttok) / float(N);        // the per-expert sum of a uniform router
  float sq_s = 0.f, sq_c = 0.f;
  int my_dr = 0;
  const int RG = nchunks >= kStatsWarps ? 1 : kStatsWarps / nchunks;
  const int chunks_per_pass = kStatsWarps / RG;
  for (int c0 = 0; c0 < nchunks; c0 += chunks_per_pass) {
    const int rg = warp % RG, chunk = c0 + warp / RG;
    const int e = chunk * 32 + lane;
    const bool live = chunk < nchunks && warp / RG < chunks_per_pass && e < N;
    float s = 0.f, comp = 0.f;
    if (live) {
      const int rows = (nblk + RG - 1) / RG;
      const int b0 = rg * rows, b1 = min(nblk, b0 + rows);
      int b = b0;
      for (; b + 8 <= b1; b += 8) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = prob_partials[int64_t(b + u) * N + e];
#pragma unroll
        for (int u = 0; u < 8; ++u) kahan_add(v[u], s, comp);
      }
      for (; b < b1; ++b) kahan_add(prob_partials[int64_t(b) * N + e], s, comp);
    }
    part[warp][lane] = make_float2(s, -comp);
    __syncthreads();
    if (rg == 0 && live) {
      const int slot = warp / RG;
      float hi = 0.f, lo = 0.f;
      for (int g = 0; g < RG; ++g) {
        const float2 pv = part[slot * RG + g][lane];
        float ns, ne;
        two_sum(hi, pv.x, ns, ne);
        hi = ns;
        lo += ne + pv.y;
      }
      mean_prob[e] = (hi + lo) * invT;
      float dhi, dlo;
      two_sum(hi, -tN, dhi, dlo);
      const float dev = (dhi + (dlo + lo)) * invT;
      kahan_add(dev * dev, sq_s, sq_c);
      my_dr += counts[e] - kept[e];
    }
    __syncthreads();
  }
  // lanes, then warps, in a fixed order
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float os = __shfl_xor_sync(0xffffffffu, sq_s, o);
    const float oc = __shfl_xor_sync(0xffffffffu, sq_c, o);
    float ns, ne;
    two_sum(sq_s, os, ns, ne);
    sq_s = ns;
    sq_c = sq_c + oc - ne;
    my_dr += __shfl_xor_sync(0xffffffffu, my_dr, o);
  }
  if (lane == 0) {
    sq[warp] = make_float2(sq_s, sq_c);
    dr[warp] = my_dr;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float v = 0.f, vc = 0.f;
    int w = 0;
    for (int i = 0; i < kStatsWarps; ++i) {
      kahan_add(sq[i].x, v, vc);
      vc += sq[i].y;
      w += dr[i];
    }
    *balance = (N > 1 && Ttok > 0) ? (v - vc) / float(N - 1) : 0.f;
    *dropped = w;
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
  const int nblk = int(router_partial_rows(c));
  load_stats_kernel<<<1, kStatsThreads, 0, s>>>(prob_partials, nblk, int(c.n_experts), int(c.T),
                                      counts, kept, mean_prob, balance, dropped);
  return cudaGetLastError();
}

}  // namespace moe
