// Router: scores z = x . W_g^T + b_g, softmax over the N experts, top-k and
// the gates (botmartz.com "Mixture of Experts (MoE) and Mixtral", section
// "Expert Routing"; roadtointelligence.com "Mixture of Experts (MoE)", router
// formula G(x) = Softmax(TopK(x . W_g)); codingnowai.in "Mixture of Experts",
// section "Code", for gates without renormalisation).
#include <float.h>

#include "common.cuh"
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
  if (c.dtype == MOE_F32) return launch_simt_gemm<float, float>(a, c.T, 0, s);
  return launch_simt_gemm<__nv_bfloat16, float>(a, c.T, 0, s);
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
                               float* __restrict__ topk_w, float* __restrict__ prob_partials,
                               float* __restrict__ probT, int32_t* __restrict__ picks) {
  extern __shared__ float red[];                 // [kRouterWarps][N]
  pdl_launch_dependents();
  pdl_wait_previous();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kTokPerWarp = kRouterTokensPerBlock / kRouterWarps;
  float psum[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) psum[i] = 0.f;

  const int groups = (T + kRouterTokensPerBlock - 1) / kRouterTokensPerBlock;
  for (int grp = blockIdx.x; grp < groups; grp += gridDim.x)
  for (int q = 0; q < kTokPerWarp; ++q) {
    const int t = grp * kRouterTokensPerBlock + warp * kTokPerWarp + q;
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
    if (probT) {                                 // expert-major probabilities
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        const int e = lane + 32 * i;
        if (e < N) probT[int64_t(e) * T + t] = ex[i] * inv;
      }
      if (lane == 0) picks[t] = 0;
    }

    // top-k by repeated warp arg-max over the not yet selected experts
    uint32_t taken = 0;                          // bit i: expert lane + 32 i selected
    float kept_sum = 0.f;
    int my_e = 0;
    float my_g = 0.f;
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
      if (lane == 0) MOE_CHECK(be >= 0 && be < N, CK_ROUTER_TOPK);
      if (lane == (j & 31)) { my_e = be; my_g = g; }   // slot j is held by lane j % 32
      if (k > 32 && ((j & 31) == 31 || j == k - 1)) {  // k > 32: flush 32 slots at a time
        const int j0 = j & ~31;
        if (lane <= j - j0) {
          out_i[j0 + lane] = my_e;
          out_w[j0 + lane] = my_g;                      // unnormalised for now
        }
      }
    }
    // gate = exp(z - max) / (sum over the kept k), or / (sum over all N)
    const float scale = renorm ? 1.0f / kept_sum : inv;
    if (k <= 32) {
      if (lane < k) {
        out_i[lane] = my_e;
        out_w[lane] = my_g * scale;
      }
    } else {
      for (int j = lane; j < k; j += 32) out_w[j] *= scale;  // each lane rescales its own writes
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

// Fused router for small expert counts (N <= 64) whose W_g fits in shared
// memory.  One warp per token: lanes split d in 16-byte vectors (up to 16 of
// them loaded at once) against W_g staged in shared memory, padded with zero
// rows to NE experts (8, 16, 32 or 64).  A butterfly reduce-scatter then
// leaves each expert's score in DUP = 32/NE adjacent lanes (NE <= 32) or two
// experts per lane (NE = 64); the softmax, the top-k and the gates follow as
// above.  One pass over x, no score round trip.  WF32 (bf16 layers with at
// most 16 experts whose W_g takes <= 48 KB as fp32): W_g is staged converted to
// fp32, laid out [NE][2][d / 8][4] so that a lane's two 16-byte reads of an
// 8-element vector are each contiguous across the warp; the inner loop then
// reads weights without converting them.  WG (bf16, at most 8 experts, W_g at
// most 16 KB): no staging; the inner loop reads W_g from global memory, where
// it stays in L1, so the x loads start without waiting for a staged copy.
template <typename TIn, int NE, bool WF32 = false, bool WG = false>
__global__ void __launch_bounds__(kRouterWarps * 32, (WF32 || WG) ? 2 : 1)
    router_fused_kernel(const TIn* __restrict__ x, const TIn* __restrict__ W_g,
                        const TIn* __restrict__ b_g, int T, int d, int N, int k, int renorm,
                        float* __restrict__ logits, int32_t* __restrict__ topk_idx,
                        float* __restrict__ topk_w, float* __restrict__ prob_partials,
                        float* __restrict__ probT, int32_t* __restrict__ picks) {
  constexpr int V = Vec16<TIn>::n;
  constexpr int NPL = NE > 32 ? NE / 32 : 1;          // experts per lane after the reduce
  constexpr int DUP = NE < 32 ? 32 / NE : 1;          // lanes holding the same expert
  constexpr int kBatch = (WF32 || WG) ? 8 : (NE <= 16 ? 16 : (NE == 32 ? 8 : 2));   // x loads in flight
  extern __shared__ uint4 wsm[];                      // W_g [NE][d] (zero rows), then sums
  pdl_launch_dependents();
  pdl_wait_previous();
  const int dv = d / V;
  const int nvec = N * dv, nvec_pad = NE * dv;
  const uint4* wsrc = reinterpret_cast<const uint4*>(W_g);
  float4* wsf = reinterpret_cast<float4*>(wsm);       // WF32: [NE][2][dv] float4
  if constexpr (WG) {
    // W_g read straight from global memory (L1-resident) in the inner loop
  } else if constexpr (WF32) {
    for (int i = threadIdx.x; i < nvec_pad; i += blockDim.x) {
      const int e = i / dv, c = i - e * dv;
      float v[8];
      if (i < nvec) {
        Vec16<TIn>::load(reinterpret_cast<const TIn*>(wsrc + i), v);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = 0.f;
      }
      wsf[(2 * e) * dv + c] = make_float4(v[0], v[1], v[2], v[3]);
      wsf[(2 * e + 1) * dv + c] = make_float4(v[4], v[5], v[6], v[7]);
    }
  } else {
    int i = threadIdx.x;
    for (; i + 3 * int(blockDim.x) < nvec; i += 4 * blockDim.x) {
      const uint4 a0 = __ldg(wsrc + i), a1 = __ldg(wsrc + i + blockDim.x),
                  a2 = __ldg(wsrc + i + 2 * blockDim.x), a3 = __ldg(wsrc + i + 3 * blockDim.x);
      wsm[i] = a0; wsm[i + blockDim.x] = a1; wsm[i + 2 * blockDim.x] = a2;
      wsm[i + 3 * blockDim.x] = a3;
    }
    for (; i < nvec; i += blockDim.x) wsm[i] = __ldg(wsrc + i);
    for (int j = nvec + int(threadIdx.x); j < nvec_pad; j += blockDim.x)
      wsm[j] = make_uint4(0, 0, 0, 0);
  }
  float* red = WG     ? reinterpret_cast<float*>(wsm)
               : WF32 ? reinterpret_cast<float*>(wsf + 2 * nvec_pad)
                      : reinterpret_cast<float*>(wsm + nvec_pad);   // [kRouterWarps][NE]
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // experts held by this lane after the reduce: e0 .. e0 + NPL - 1
  const int e0 = NE > 32 ? lane * NPL : lane / DUP;
  const bool owner = (lane % DUP) == 0;               // one lane per expert writes
  float psum[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) psum[i] = 0.f;

  const int groups = (T + kRouterTokensPerBlock - 1) / kRouterTokensPerBlock;
  // a warp takes TPW of its grid-stride groups' tokens at once, so that each
  // staged weight vector is read and converted once for TPW tokens; every
  // token's sums run in the same order as with one token per pass
  constexpr int TPW = (!WF32 && !WG && NE <= 16 && sizeof(TIn) == 2) ? 2 : 1;
  constexpr int kB = kBatch / TPW;                    // x loads in flight per token
  for (int grp = blockIdx.x; grp < groups; grp += TPW * gridDim.x) {
    int tok[TPW];
    bool live[TPW];
#pragma unroll
    for (int u = 0; u < TPW; ++u) {
      const int g = grp + u * int(gridDim.x);
      tok[u] = g * kRouterTokensPerBlock + warp;
      live[u] = g < groups && tok[u] < T;
    }
    if (!live[0]) break;
    float accs[TPW][NE];
#pragma unroll
    for (int u = 0; u < TPW; ++u)
#pragma unroll
      for (int e = 0; e < NE; ++e) accs[u][e] = 0.f;
    for (int c0 = lane; c0 < dv; c0 += kB * 32) {
      uint4 xq[TPW][kB];
#pragma unroll
      for (int u = 0; u < TPW; ++u) {
        const uint4* xr = reinterpret_cast<const uint4*>(x + int64_t(live[u] ? tok[u] : tok[0]) * d);
#pragma unroll
        for (int b = 0; b < kB; ++b) {
          const int c = c0 + 32 * b;
          xq[u][b] = (c < dv && live[u]) ? __ldg(xr + c) : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int b = 0; b < kB; ++b) {
        const int c = c0 + 32 * b;
        if (c >= dv) break;
        float xv[TPW][V];
#pragma unroll
        for (int u = 0; u < TPW; ++u)
          Vec16<TIn>::load(reinterpret_cast<const TIn*>(&xq[u][b]), xv[u]);
#pragma unroll
        for (int e = 0; e < NE; ++e) {
          float wv[V];
          if constexpr (WF32) {
            const float4 lo = wsf[(2 * e) * dv + c], hi = wsf[(2 * e + 1) * dv + c];
            wv[0] = lo.x; wv[1] = lo.y; wv[2] = lo.z; wv[3] = lo.w;
            wv[4] = hi.x; wv[5] = hi.y; wv[6] = hi.z; wv[7] = hi.w;
          } else if constexpr (WG) {
            const uint4 q = e < N ? __ldg(wsrc + e * dv + c) : make_uint4(0, 0, 0, 0);
            Vec16<TIn>::load(reinterpret_cast<const TIn*>(&q), wv);
          } else {
            Vec16<TIn>::load(reinterpret_cast<const TIn*>(wsm + e * dv + c), wv);
          }
#pragma unroll
          for (int u = 0; u < TPW; ++u)
#pragma unroll
            for (int i = 0; i < V; ++i) accs[u][e] = fmaf(xv[u][i], wv[i], accs[u][e]);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < TPW; ++u) {
      if (!live[u]) break;
      const int t = tok[u];
      float (&acc)[NE] = accs[u];
      // reduce-scatter while more than NPL values remain, then all-reduce
      // across the DUP lanes that share an expert
      constexpr int kRsSteps = NE > 32 ? 5 : (NE == 32 ? 5 : (NE == 16 ? 4 : 3));
#pragma unroll
      for (int step = 0; step < 5; ++step) {
        const int o = 16 >> step;
        if (step < kRsSteps) {
          const int S = NE >> step;                     // values still held per lane
          const bool upper = (lane & o) != 0;
#pragma unroll
          for (int i = 0; i < S / 2; ++i) {
            const float send = upper ? acc[i] : acc[i + S / 2];
            const float keep = upper ? acc[i + S / 2] : acc[i];
            acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
          }
        } else {
          acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], o);
        }
      }
      float z[NPL];
      float m = -FLT_MAX;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        const int e = e0 + i;
        z[i] = e < N ? acc[i] + to_f32(b_g[e]) : -INFINITY;
        if (e < N && owner) logits[int64_t(t) * N + e] = z[i];
        m = fmaxf(m, z[i]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float ex[NPL], ssum = 0.f;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        ex[i] = (e0 + i < N) ? expf(z[i] - m) : 0.f;
        if (owner) ssum += ex[i];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
      const float inv = 1.0f / ssum;
#pragma unroll
      for (int i = 0; i < NPL; ++i) psum[i] += ex[i] * inv;
      if (probT) {                                       // expert-major probabilities
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
          const int e = e0 + i;
          if (e < N && owner) probT[int64_t(e) * T + t] = ex[i] * inv;
        }
        if (lane == 0) picks[t] = 0;
      }

      uint32_t taken = 0;                                // bit i: expert e0 + i selected
      float kept_sum = 0.f;
      int my_e = 0;
      float my_g = 0.f;
      int32_t* out_i = topk_idx + int64_t(t) * k;
      float* out_w = topk_w + int64_t(t) * k;
      for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
          const int e = e0 + i;
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
        if (be >= e0 && be < e0 + NPL) taken |= 1u << (be - e0);
        const float g = expf(bv - m);
        kept_sum += g;
        if (lane == 0) MOE_CHECK(be >= 0 && be < N, CK_ROUTER_TOPK);
        if (lane == (j & 31)) { my_e = be; my_g = g; }   // slot j is held by lane j % 32
        if (k > 32 && ((j & 31) == 31 || j == k - 1)) {  // k > 32: flush 32 slots at a time
          const int j0 = j & ~31;
          if (lane <= j - j0) {
            out_i[j0 + lane] = my_e;
            out_w[j0 + lane] = my_g;                      // unnormalised for now
          }
        }
      }
      const float scale = renorm ? 1.0f / kept_sum : inv;
      if (k <= 32) {
        if (lane < k) {
          out_i[lane] = my_e;
          out_w[lane] = my_g * scale;
        }
      } else {
        for (int j = lane; j < k; j += 32) out_w[j] *= scale;
      }
    }
  }

#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = e0 + i;
    if (e < N && owner) red[warp * NE + e] = psum[i];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += blockDim.x) {
    float v = 0.f;
    for (int w = 0; w < kRouterWarps; ++w) v += red[w * NE + e];
    prob_partials[int64_t(blockIdx.x) * N + e] = v;
  }
}

int fused_ne(int64_t n) { return n <= 8 ? 8 : n <= 16 ? 16 : n <= 32 ? 32 : 64; }

constexpr size_t kFusedRouterSmemLimit = 200 * 1024;

// bf16 layers stage W_g as fp32 when that takes at most 48 KB (several blocks
// per SM still fit)
constexpr size_t kFusedRouterF32Limit = 48 * 1024;

// bf16 layers of at most 8 experts whose W_g takes at most 16 KB read it from
// global memory in the inner loop (it stays in L1) instead of staging it first
constexpr size_t kFusedRouterGlobalLimit = 16 * 1024;

bool fused_router_wg(const moe_config& c) {
  return c.dtype == MOE_BF16 && fused_ne(c.n_experts) <= 8 &&
         size_t(c.n_experts * c.d_model) * 2 <= kFusedRouterGlobalLimit;
}

bool fused_router_wf32(const moe_config& c) {
  return c.dtype == MOE_BF16 && fused_ne(c.n_experts) <= 16 && !fused_router_wg(c) &&
         size_t(fused_ne(c.n_experts) * c.d_model) * 4 <= kFusedRouterF32Limit;
}

size_t fused_router_smem(const moe_config& c) {
  const int ne = fused_ne(c.n_experts);
  const size_t red = size_t(kRouterWarps) * ne * sizeof(float);
  if (fused_router_wg(c)) return red;
  const size_t es = (c.dtype == MOE_F32 || fused_router_wf32(c)) ? 4 : 2;
  return size_t(ne * c.d_model) * es + red;
}

bool fused_router_fits(const moe_config& c) {
  return c.n_experts <= 64 && fused_router_smem(c) <= kFusedRouterSmemLimit;
}

// k == 0 with probT set: probabilities only (expert-choice routing)
cudaError_t launch_router_fused(const moe_config& c, int k, const void* x, const void* W_g,
                                const void* b_g, float* logits, int32_t* topk_idx,
                                float* topk_w, float* prob_partials, float* probT,
                                int32_t* picks, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  const unsigned blocks = unsigned(router_partial_rows(c));
  const size_t smem = fused_router_smem(c);
  const int T = int(c.T), d = int(c.d_model), N = int(c.n_experts);
  const int rn = c.renormalize ? 1 : 0;
#define MOE_FUSED_CASE(TIN, NPAD, WF, ...)                                                 \
  {                                                                                        \
    auto kern = router_fused_kernel<TIN, NPAD, WF, ##__VA_ARGS__>;                         \
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,  \
                                         int(smem));                                       \
    if (e != cudaSuccess) return e;                                                        \
    return launch_pdl(kern, dim3(blocks), dim3(kRouterWarps * 32), smem, s,                \
                      static_cast<const TIN*>(x), static_cast<const TIN*>(W_g),            \
                      static_cast<const TIN*>(b_g), T, d, N, k, rn, logits, topk_idx,      \
                      topk_w, prob_partials, probT, picks);                                \
  }
  if (c.dtype == MOE_F32) {
    if (N <= 8) MOE_FUSED_CASE(float, 8, false)
    if (N <= 16) MOE_FUSED_CASE(float, 16, false)
    if (N <= 32) MOE_FUSED_CASE(float, 32, false)
    MOE_FUSED_CASE(float, 64, false)
  }
  if (fused_router_wg(c)) MOE_FUSED_CASE(__nv_bfloat16, 8, false, true)
  if (fused_router_wf32(c)) {
    if (N <= 8) MOE_FUSED_CASE(__nv_bfloat16, 8, true)
    MOE_FUSED_CASE(__nv_bfloat16, 16, true)
  }
  if (N <= 8) MOE_FUSED_CASE(__nv_bfloat16, 8, false)
  if (N <= 16) MOE_FUSED_CASE(__nv_bfloat16, 16, false)
  if (N <= 32) MOE_FUSED_CASE(__nv_bfloat16, 32, false)
  MOE_FUSED_CASE(__nv_bfloat16, 64, false)
#undef MOE_FUSED_CASE
}

cudaError_t launch_router_softmax_topk(const moe_config& c, int k, const float* logits,
                                       int32_t* topk_idx, float* topk_w,
                                       float* prob_partials, float* probT, int32_t* picks,
                                       cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  const int N = int(c.n_experts);
  const unsigned blocks = unsigned(router_partial_rows(c));
  const size_t smem = size_t(kRouterWarps) * N * sizeof(float);
  const int T = int(c.T), rn = c.renormalize ? 1 : 0;
#define MOE_ROUTER_CASE(NPL)                                                              \
  {                                                                                        \
    auto kern = router_softmax_topk_kernel<NPL>;                                           \
    if (smem > 48 * 1024) {                                                                \
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                           int(smem));                                     \
      if (e != cudaSuccess) return e;                                                      \
    }                                                                                      \
    return launch_pdl(kern, dim3(blocks), dim3(kRouterWarps * 32), smem, s, logits, T, N,  \
                      k, rn, topk_idx, topk_w, prob_partials, probT, picks);               \
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

namespace moe {

int router_launch_count(const moe_config& c) {
  if (c.T == 0) return 0;
  if (router_tc_topk(c)) return 1;
  if (c.dtype == MOE_BF16 && c.n_experts % 64 == 0) return 2;
  return fused_router_fits(c) ? 1 : 2;
}

// Scores + softmax + top-k for one layer, choosing the kernels by shape:
// bf16 with 64 experts (k <= 8): the tensor-core GEMM with the softmax, top-k
// and gates in its epilogue; bf16 with N a multiple of 64: the tensor-core
// GEMM (fp32 scores) then the softmax/top-k kernel; otherwise, when N <= 64
// and W_g fits in shared
// memory, the fused warp-per-token kernel; otherwise the CUDA-core GEMM then
// the softmax/top-k kernel.
cudaError_t launch_router(const moe_config& c, const void* x, const void* W_g,
                          const void* b_g, float* logits, int32_t* topk_idx, float* topk_w,
                          float* prob_partials, int num_sms, int32_t* status,
                          uint64_t wait_limit_ns, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  cudaError_t e;
  const int k = int(c.top_k);
  if (router_tc_topk(c))
    return launch_router_topk_tc(c, x, W_g, b_g, logits, topk_idx, topk_w, prob_partials,
                                 num_sms, status, wait_limit_ns, s);
  if (c.dtype == MOE_BF16 && c.n_experts % 64 == 0)
    e = launch_router_logits_tc(c, x, W_g, b_g, logits, num_sms, status, wait_limit_ns, s);
  else if (fused_router_fits(c))
    return launch_router_fused(c, k, x, W_g, b_g, logits, topk_idx, topk_w, prob_partials,
                               nullptr, nullptr, s);
  else
    e = launch_router_logits(c, x, W_g, b_g, logits, s);
  if (e != cudaSuccess) return e;
  return launch_router_softmax_topk(c, k, logits, topk_idx, topk_w, prob_partials, nullptr,
                                    nullptr, s);
}

// The same kernels without the top-k: scores, the expert-major probabilities
// probT [N, T] and the block sums of p (expert-choice routing).
cudaError_t launch_router_probs(const moe_config& c, const void* x, const void* W_g,
                                const void* b_g, float* logits, float* probT, int32_t* picks,
                                float* prob_partials, int num_sms, int32_t* status,
                                uint64_t wait_limit_ns, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  cudaError_t e;
  if (c.dtype == MOE_BF16 && c.n_experts % 64 == 0)
    e = launch_router_logits_tc(c, x, W_g, b_g, logits, num_sms, status, wait_limit_ns, s);
  else if (fused_router_fits(c))
    return launch_router_fused(c, 0, x, W_g, b_g, logits, nullptr, nullptr, prob_partials,
                               probT, picks, s);
  else
    e = launch_router_logits(c, x, W_g, b_g, logits, s);
  if (e != cudaSuccess) return e;
  return launch_router_softmax_topk(c, 0, logits, nullptr, nullptr, prob_partials, probT,
                                    picks, s);
}

MOE_CHECKS_UNIT(router)

}  // namespace moe
