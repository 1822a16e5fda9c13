// Router: scores z = x . W_g^T + b_g, softmax over the N experts, top-k and
// the gates (botmartz.com "Mixture of Experts (MoE) and Mixtral", section
// "Expert Routing"; roadtointelligence.com "Mixture of Experts (MoE)", router
// formula G(x) = Softmax(TopK(x . W_g)); codingnowai.in "Mixture of Experts",
// section "Code", for gates without renormalisation).
#include <float.h>

#include "kernels.h"
#include "simt_gemm.cuh"

namespace moe {

cudaError_t launch_router_logits(const moe_config& c, const void* x, const void* W_g,
                                 const void* b_g, float* logits, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  SimtGemmArgs a{};
  a.A = x; a.B = W_g; a.bias = b_g; a.C = logits;
  a.rows = c.T; a.K = c.d_model; a.Nc = c.n_experts;
  a.act = -1;
  dim3 grid(unsigned(ceil_div(c.n_experts, kSimtBN)), unsigned(ceil_div(c.T, kSimtBM)));
  if (c.dtype == MOE_F32)
    simt_gemm_kernel<float, float><<<grid, kSimtThreads, 0, s>>>(a);
  else
    simt_gemm_kernel<__nv_bfloat16, float><<<grid, kSimtThreads, 0, s>>>(a);
  return cudaGetLastError();
}

// One warp per token.  Lane l holds the scores of experts l, l+32, ...,
// (NPL of them).  The softmax's max and sum are warp shuffles; the top-k is
// k rounds of a warp-wide arg-max (larger score first, then lower expert).
// Each block also sums p over its tokens for the load statistic, in a fixed
// order so the result is reproducible.
constexpr int kRouterWarps = 8;

template <int NPL>
__global__ void __launch_bounds__(kRouterWarps * 32)
    router_softmax_topk_kernel(const float* __restrict__ logits, int T, int N, int k,
                               int renorm, int32_t* __restrict__ topk_idx,
                               float* __restrict__ topk_w, float* __restrict__ prob_partials) {
  extern __shared__ float red[];                 // [kRouterWarps][N]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kTokPerWarp = kRouterTokensPerBlock / kRouterWarps;
  float psum[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) psum[i] = 0.f;

  for (int q = 0; q < kTokPerWarp; ++q) {
    const int t = blockIdx.x * kRouterTokensPerBlock + warp * kTokPerWarp + q;
    if (t >= T) break;
    const float* zr = logits + int64_t(t) * N;
    float z[NPL];
    float m = -FLT_MAX;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      z[i] = e < N ? zr[e] : -INFINITY;
      m = fmaxf(m, z[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float ex[NPL], ssum = 0.f;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      ex[i] = (lane + 32 * i < N) ? expf(z[i] - m) : 0.f;
      ssum += ex[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
    const float inv = 1.0f / ssum;
#pragma unroll
    for (int i = 0; i < NPL; ++i) psum[i] += ex[i] * inv;

    // top-k by repeated warp arg-max over the not yet selected experts
    uint32_t taken = 0;                          // bit i: expert lane + 32 i selected
    float kept_sum = 0.f;
    int32_t* out_i = topk_idx + int64_t(t) * k;
    float* out_w = topk_w + int64_t(t) * k;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
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
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      const float g = expf(bv - m);              // m is the largest score: slot 0's
      kept_sum += g;
      if (lane == 0) {
        out_i[j] = be;
        out_w[j] = renorm ? g : g * inv;
      }
    }
    if (renorm && lane == 0) {
      const float r = 1.0f / kept_sum;
      for (int j = 0; j < k; ++j) out_w[j] *= r;
    }
  }

  // block partial sums of p: per warp in registers, then warps in order
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    if (e < N) red[warp * N + e] = psum[i];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += blockDim.x) {
    float v = 0.f;
    for (int w = 0; w < kRouterWarps; ++w) v += red[w * N + e];
    prob_partials[int64_t(blockIdx.x) * N + e] = v;
  }
}

cudaError_t launch_router_softmax_topk(const moe_config& c, const float* logits,
                                       int32_t* topk_idx, float* topk_w,
                                       float* prob_partials, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  const int N = int(c.n_experts);
  const unsigned blocks = unsigned(ceil_div(c.T, kRouterTokensPerBlock));
  const size_t smem = size_t(kRouterWarps) * N * sizeof(float);
  const int T = int(c.T), k = int(c.top_k), rn = c.renormalize ? 1 : 0;
#define MOE_ROUTER_CASE(NPL)                                                              \
  {                                                                                        \
    auto kern = router_softmax_topk_kernel<NPL>;                                           \
    if (smem > 48 * 1024) {                                                                \
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                           int(smem));                                     \
      if (e != cudaSuccess) return e;                                                      \
    }                                                                                      \
    kern<<<blocks, kRouterWarps * 32, smem, s>>>(logits, T, N, k, rn, topk_idx, topk_w,   \
                                                 prob_partials);                           \
    return cudaGetLastError();                                                             \
  }
  if (N <= 32) MOE_ROUTER_CASE(1)
  if (N <= 64) MOE_ROUTER_CASE(2)
  if (N <= 128) MOE_ROUTER_CASE(4)
  if (N <= 256) MOE_ROUTER_CASE(8)
  if (N <= 512) MOE_ROUTER_CASE(16)
  MOE_ROUTER_CASE(32)
#undef MOE_ROUTER_CASE
}

}  // namespace moe
