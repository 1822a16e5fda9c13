// Backward pass of the layer for the training loss total = task + alpha *
// balance (botmartz.com "Mixture of Experts (MoE) and Mixtral", "Load
// Balancing: The Hidden Challenge": total_loss = task_loss + 0.01 *
// balance_loss; roadtointelligence.com "Keeping the experts busy": coefficient
// 0.01).  The task loss enters as dy = d task / d y; the rest is the chain rule
// through the forward, step by step:
//
//   gate step      per token: dw_j = <dy, Yp[row_j]>, dO[row_j] = w_j dy
//                  (shared row: dy); the gates' softmax (over the k selected
//                  scores, or the raw probabilities), plus the balance term
//                  d p[t, e] = alpha 2 (m_e - 1/N) / ((N - 1) T), through the
//                  softmax over all N -> dz [T, N]
//   expert FFNs    A1 recomputed (first Linear without its activation), then
//                  dA = (dO W2) act'(A1), dXp = dA W1, dW2 = dO^T H,
//                  dW1 = dA^T Xp on the tensor cores (grouped_bwd_sm103.cu);
//                  db2, db1 = column sums of dO, dA over each group's rows
//   router         dW_g = dz^T x, db_g = sum_t dz, dx_router = dz W_g
//                  (CUDA-core GEMMs: K or M is the expert count)
//   dx             dx[t] = sum of dXp over t's kept rows (+ the shared row)
//                  + dx_router[t]
//
// The top-k choice and the capacity drops are piecewise constant and pass no
// gradient.  Every sum runs in a fixed order, so the gradients are
// reproducible bit for bit.
#include <float.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

// ---- zero the padding rows of grouped buffers ------------------------------------------

struct PadBufs {
  void* buf[3];
  int64_t vec16[3];          // 16-byte words per row
  int n;
};

// Blocks (g, y): rows offsets[g] + live_g + y, + gridDim.y, ... below offsets[g + 1].
__global__ void __launch_bounds__(256)
    zero_pad_rows_kernel(const int32_t* __restrict__ offsets, const int32_t* __restrict__ kept,
                         int n_routed, int shared_rows, PadBufs b) {
  pdl_launch_dependents();
  pdl_wait_previous();
  const int g = blockIdx.x;
  const int64_t live = g < n_routed ? kept[g] : shared_rows;
  const int64_t r1 = offsets[g + 1];
  for (int64_t r = offsets[g] + live + blockIdx.y; r < r1; r += gridDim.y)
    for (int i = 0; i < b.n; ++i) {
      const int64_t nv = b.vec16[i];
      uint4* row = static_cast<uint4*>(b.buf[i]) + r * nv;
      for (int64_t j = threadIdx.x; j < nv; j += blockDim.x) row[j] = make_uint4(0, 0, 0, 0);
    }
}

// ---- gate step ------------------------------------------------------------------------

constexpr int kGateWarps = 8;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// One warp per token.  Shared memory per warp: p [N], dp [N], dz [N], dw [k].
// E: the layer's element type (dy, Yp, dO).
template <typename E>
__global__ void __launch_bounds__(kGateWarps * 32)
    bwd_gate_kernel(const E* __restrict__ dy, const E* __restrict__ Yp,
                    const int32_t* __restrict__ token_row, const int32_t* __restrict__ topk_idx,
                    const float* __restrict__ topk_w, const float* __restrict__ logits,
                    const float* __restrict__ mean_prob, const int32_t* __restrict__ offsets,
                    int T, int64_t d, int N, int k, int renorm, int has_shared, float aux,
                    E* __restrict__ dO, float* __restrict__ dz_out,
                    float* __restrict__ dw_out, __nv_bfloat16* __restrict__ dz_bf,
                    int32_t* __restrict__ rgrp) {
  extern __shared__ float gsm[];
  pdl_launch_dependents();
  pdl_wait_previous();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (rgrp && blockIdx.x == 0 && threadIdx.x == 0) {
    // the router's tensor-core GEMMs see one group of T rows
    const int32_t tp = (T + 127) / 128 * 128;
    rgrp[0] = 0; rgrp[1] = tp; rgrp[2] = tp; rgrp[3] = T;
  }
  const int t = blockIdx.x * kGateWarps + warp;
  if (t >= T) return;
  float* P = gsm + size_t(warp) * (3 * N + k);
  float* DP = P + N;
  float* DZ = DP + N;
  float* DW = DZ + N;
  constexpr int V = Vec16<E>::n;
  const int64_t nv = d / V;
  const E* dyr = dy + int64_t(t) * d;

  // dw_j = <dy, o_j> and dO rows
  for (int j = 0; j < k; ++j) {
    const int64_t r = token_row[int64_t(t) * k + j];
    float dot = 0.f;
    if (r >= 0) {
      const float wj = topk_w[int64_t(t) * k + j];
      const E* orow = Yp + r * d;
      E* drow = dO + r * d;
      for (int64_t c = lane; c < nv; c += 32) {
        float av[V], ov[V], q[V];
        Vec16<E>::load(dyr + c * V, av);
        Vec16<E>::load(orow + c * V, ov);
#pragma unroll
        for (int i = 0; i < V; ++i) {
          dot = fmaf(av[i], ov[i], dot);
          q[i] = wj * av[i];
        }
        Vec16<E>::store(drow + c * V, q);
      }
      dot = warp_sum(dot);
    }
    if (lane == 0) DW[j] = dot;
    if (dw_out && lane == 0) dw_out[int64_t(t) * k + j] = dot;
  }
  if (has_shared) {                           // the shared expert's gate is 1
    E* drow = dO + (int64_t(offsets[N]) + t) * d;
    for (int64_t c = lane; c < nv; c += 32) {
      float av[V];
      Vec16<E>::load(dyr + c * V, av);
      Vec16<E>::store(drow + c * V, av);
    }
  }

  // p = softmax(z) over all N
  const float* zr = logits + int64_t(t) * N;
  float m = -FLT_MAX;
  for (int e = lane; e < N; e += 32) m = fmaxf(m, zr[e]);
  m = warp_max(m);
  float ssum = 0.f;
  for (int e = lane; e < N; e += 32) {
    const float ex = __expf(zr[e] - m);
    P[e] = ex;
    ssum += ex;
  }
  ssum = warp_sum(ssum);
  const float inv = 1.0f / ssum;
  // balance term: d p[t, e] = alpha 2 (m_e - 1/N) / ((N - 1) T)
  const float cb = (aux != 0.f && N > 1) ? aux * 2.0f / (float(N - 1) * float(T)) : 0.f;
  for (int e = lane; e < N; e += 32) {
    P[e] *= inv;
    DP[e] = cb * (mean_prob[e] - 1.0f / float(N));
    DZ[e] = 0.f;
  }
  __syncwarp();
  // gates
  if (renorm) {
    float sd = 0.f;
    for (int j = lane; j < k; j += 32) sd += topk_w[int64_t(t) * k + j] * DW[j];
    sd = warp_sum(sd);
    for (int j = lane; j < k; j += 32) {
      const float wj = topk_w[int64_t(t) * k + j];
      DZ[topk_idx[int64_t(t) * k + j]] = wj * (DW[j] - sd);
    }
  } else {
    for (int j = lane; j < k; j += 32) DP[topk_idx[int64_t(t) * k + j]] += DW[j];
  }
  __syncwarp();
  // through the softmax over all N: p (dp - <p, dp>)
  float pd = 0.f;
  for (int e = lane; e < N; e += 32) pd += P[e] * DP[e];
  pd = warp_sum(pd);
  float* dzr = dz_out + int64_t(t) * N;
  for (int e = lane; e < N; e += 32) {
    const float v = DZ[e] + P[e] * (DP[e] - pd);
    dzr[e] = v;
    if (dz_bf) dz_bf[int64_t(t) * N + e] = __float2bfloat16_rn(v);
  }
}

// ---- column sums of groups (bias gradients) -----------------------------------------------

// Block (g, chunk): columns chunk*32V .. +32V-1 of group g's live rows (V
// elements per 16-byte word); eight warps take every eighth row, lanes one word
// each; warps combine in order.
template <typename T>
__global__ void __launch_bounds__(256)
    group_colsum_kernel(const T* __restrict__ src, int64_t width,
                        const int32_t* __restrict__ offsets, const int32_t* __restrict__ kept,
                        int n_routed, int shared_rows, T* __restrict__ out, T* __restrict__ out_s) {
  constexpr int V = Vec16<T>::n;
  __shared__ float part[8][32 * V];
  pdl_launch_dependents();
  pdl_wait_previous();
  const int g = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t c0 = int64_t(blockIdx.y) * 32 * V + lane * V;
  const int64_t live = g < n_routed ? kept[g] : shared_rows;
  const int64_t r0 = offsets[g];
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  if (c0 < width) {
    for (int64_t r = warp; r < live; r += 8) {
      float v[V];
      Vec16<T>::load(src + (r0 + r) * width + c0, v);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] += v[i];
    }
  }
#pragma unroll
  for (int i = 0; i < V; ++i) part[warp][lane * V + i] = acc[i];
  __syncthreads();
  for (int col = threadIdx.x; col < 32 * V; col += blockDim.x) {
    const int64_t cc = int64_t(blockIdx.y) * 32 * V + col;
    if (cc < width) {
      float s = 0.f;
      for (int w = 0; w < 8; ++w) s += part[w][col];
      T* dst = g < n_routed ? out + int64_t(g) * width : out_s;
      dst[cc] = from_f32<T>(s);
    }
  }
}

// db_g[e] = sum_t dz[t, e] (fp32 in, bf16 out): block b takes experts
// 32 b .. 32 b + 31 (one per lane), its eight warps every eighth token, and
// the warps combine in order.
template <typename TO>
__global__ void __launch_bounds__(256)
    router_bias_grad_kernel(const float* __restrict__ dz, int T, int N, TO* __restrict__ db_g) {
  __shared__ float part[8][32];
  pdl_launch_dependents();
  pdl_wait_previous();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 32 + lane;
  float s = 0.f;
  if (e < N)
    for (int t = warp; t < T; t += 8) s += dz[int64_t(t) * N + e];
  part[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && e < N) {
    float v = 0.f;
    for (int w = 0; w < 8; ++w) v += part[w][lane];
    db_g[e] = from_f32<TO>(v);
  }
}

// ---- router GEMMs on CUDA cores ---------------------------------------------------------------
//
// C[m, n] = sum_k A(m, k) B[k, n] with A fp32 addressed by strides (am, ak)
// and B bf16 row-major [K, ldb]; C fp32 or bf16 row-major [M, ldc].
constexpr int kRg = 64, kRk = 16;
constexpr int kRouterMaxSplits = 32;

// blockIdx.z splits K into chunks of kc; split z writes its partial sums to
// C + z * M * ldc (fp32), summed afterwards by splitk_reduce_kernel.
template <typename TB, typename TOut>
__global__ void __launch_bounds__(256)
    router_grad_gemm_kernel(const float* __restrict__ A, int64_t am, int64_t ak,
                            const TB* __restrict__ B, int64_t ldb, int64_t M,
                            int64_t Nn, int64_t K, int64_t kc, TOut* __restrict__ C,
                            int64_t ldc) {
  __shared__ float As[kRk][kRg + 4];
  __shared__ float Bs[kRk][kRg + 4];
  pdl_launch_dependents();
  pdl_wait_previous();
  const int64_t m0 = int64_t(blockIdx.y) * kRg, n0 = int64_t(blockIdx.x) * kRg;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int64_t kb = int64_t(blockIdx.z) * kc;
  const int64_t ke = kb + kc < K ? kb + kc : K;
  C += int64_t(blockIdx.z) * M * ldc;
  float acc[4][4] = {};
  for (int64_t k0 = kb; k0 < ke; k0 += kRk) {
    // A tile 64 x 16: along m when A is m-contiguous, else along k
    for (int i = tid; i < kRg * kRk; i += 256) {
      int mm, kk;
      if (am == 1) { mm = i % kRg; kk = i / kRg; } else { kk = i % kRk; mm = i / kRk; }
      const int64_t gm = m0 + mm, gk = k0 + kk;
      As[kk][mm] = (gm < M && gk < ke) ? A[gm * am + gk * ak] : 0.f;
    }
    for (int i = tid; i < kRg * kRk; i += 256) {
      const int nn = i % kRg, kk = i / kRg;
      const int64_t gn = n0 + nn, gk = k0 + kk;
      Bs[kk][nn] = (gn < Nn && gk < ke) ? to_f32(B[gk * ldb + gn]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kRk; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t gm = m0 + ty + 16 * i;
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t gn = n0 + tx + 16 * j;
      if (gn < Nn) C[gm * ldc + gn] = from_f32<TOut>(acc[i][j]);
    }
  }
}

// out[i] = sum over the S splits of part[z * n + i], in split order.
template <typename TO>
__global__ void __launch_bounds__(256)
    splitk_reduce_kernel(const float* __restrict__ part, int S, int64_t n, TO* __restrict__ out) {
  pdl_launch_dependents();
  pdl_wait_previous();
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x) {
    float v = 0.f;
    for (int z = 0; z < S; ++z) v += part[int64_t(z) * n + i];
    out[i] = from_f32<TO>(v);
  }
}

// ---- dx -----------------------------------------------------------------------------------------

constexpr int kDxWarps = 8;

// dx[t] = dxr[t] (the router's part, fp32 or bf16) + sum over t's kept rows
// of dXp (slot order) + the shared row; T: the layer's element type.
template <typename TR, typename T>
__global__ void __launch_bounds__(kDxWarps * 32)
    bwd_dx_kernel(const T* __restrict__ dXp, const int32_t* __restrict__ token_row,
                  const int32_t* __restrict__ offsets, const TR* __restrict__ dxr, int Ttok,
                  int k, int N, int has_shared, int64_t d, T* __restrict__ dx) {
  constexpr int V = Vec16<T>::n;
  pdl_launch_dependents();
  pdl_wait_previous();
  const int lane = threadIdx.x & 31;
  const int64_t t = int64_t(blockIdx.x) * kDxWarps + (threadIdx.x >> 5);
  if (t >= Ttok) return;
  const int64_t nv = d / V;
  for (int64_t c = lane; c < nv; c += 32) {
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = to_f32(dxr[t * d + c * V + i]);
    for (int j = 0; j <= k; ++j) {
      int64_t r;
      if (j < k) r = token_row[t * k + j];
      else r = has_shared ? int64_t(offsets[N]) + t : -1;
      if (r < 0) continue;
      float v[V];
      Vec16<T>::load(dXp + r * d + c * V, v);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] += v[i];
    }
    Vec16<T>::store(dx + t * d + c * V, acc);
  }
}

template <typename TB, typename TOut>
cudaError_t launch_router_grad_gemm(const float* A, int64_t am, int64_t ak, const TB* B,
                                    int64_t ldb, int64_t M, int64_t Nn, int64_t K, TOut* C,
                                    int64_t ldc, cudaStream_t s) {
  if (M == 0 || Nn == 0) return cudaSuccess;
  dim3 grid(unsigned((Nn + kRg - 1) / kRg), unsigned((M + kRg - 1) / kRg));
  return launch_pdl(router_grad_gemm_kernel<TB, TOut>, grid, dim3(256), 0, s, A, am, ak, B,
                    ldb, M, Nn, K, K, C, ldc);
}

// Splits of K for dW_g = dz^T x on CUDA cores: enough blocks for two waves.
int router_splits(const moe_config& c) {
  const int64_t tiles = ((c.d_model + kRg - 1) / kRg) * ((c.n_experts + kRg - 1) / kRg);
  int64_t S = (2 * 148 + tiles - 1) / tiles;
  const int64_t by_k = (c.T + 255) / 256;
  if (S > by_k) S = by_k;
  if (S > kRouterMaxSplits) S = kRouterMaxSplits;
  return int(S < 1 ? 1 : S);
}

// n zeros of T: 16-byte words, then the tail element by element.
template <typename T>
__global__ void __launch_bounds__(256) fill_zero_kernel(T* __restrict__ p, int64_t n) {
  constexpr int V = Vec16<T>::n;
  pdl_launch_dependents();
  pdl_wait_previous();
  const int64_t n16 = n / V;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const int64_t i0 = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  for (int64_t i = i0; i < n16; i += stride)
    reinterpret_cast<uint4*>(p)[i] = make_uint4(0, 0, 0, 0);
  for (int64_t i = n16 * V + i0; i < n; i += stride) p[i] = from_f32<T>(0.f);
}

// No tokens: every parameter gradient is zero.
cudaError_t zero_param_grads(const moe_config& c, const moe_grads* g, cudaStream_t s) {
  const int64_t N = c.n_experts, d = c.d_model, f = c.d_ff;
  struct Buf { void* p; int64_t n; };
  const Buf bufs[] = {{g->dW_g, N * d}, {g->db_g, N},     {g->dW1, N * f * d}, {g->db1, N * f},
                      {g->dW2, N * d * f}, {g->db2, N * d}, {g->dW1s, f * d},  {g->db1s, f},
                      {g->dW2s, d * f},  {g->db2s, d}};
  const int nb = c.d_ff_shared > 0 ? 10 : 6;
  for (int i = 0; i < nb; ++i) {
    const int64_t want = (bufs[i].n / 4 + 255) / 256 + 1;
    const dim3 grid(unsigned(want < 1184 ? want : 1184));
    const cudaError_t e =
        c.dtype == MOE_F32
            ? launch_pdl(fill_zero_kernel<float>, grid, dim3(256), 0, s,
                         static_cast<float*>(bufs[i].p), bufs[i].n)
            : launch_pdl(fill_zero_kernel<__nv_bfloat16>, grid, dim3(256), 0, s,
                         static_cast<__nv_bfloat16*>(bufs[i].p), bufs[i].n);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

bool router_bwd_on_tensor_cores(const moe_config& c) {
  return c.dtype == MOE_BF16 && c.n_experts % 64 == 0;
}

size_t router_bwd_partial_bytes(const moe_config& c) {
  return router_bwd_on_tensor_cores(c)
             ? 0
             : size_t(router_splits(c)) * size_t(c.n_experts * c.d_model) * sizeof(float);
}

int backward_launch_count(const moe_config& c) {
  if (c.T == 0) return c.d_ff_shared > 0 ? 10 : 6;    // zero parameter gradients
  // gate, padding (bf16 only), A1, dA, dXp, dW2, dW1, db2, db1, dx_router,
  // dW_g (+ split-K reduce on CUDA cores), db_g, dx
  return (router_bwd_on_tensor_cores(c) ? 13 : 14) - (c.dtype == MOE_F32 ? 1 : 0);
}

namespace {

// The backward for layers of element type T (bf16: tensor-core GEMMs; fp32:
// CUDA-core GEMMs), with the events of moe_backward_profiled.
template <typename E>
cudaError_t backward_t(const moe_config& c, const BackwardArgs& a, void* const* events,
                       cudaStream_t s) {
  constexpr bool kBf16 = sizeof(E) == 2;
  void* const none[8] = {};
  void* const* ev = events ? events : none;
  cudaError_t er = record_event(ev[0], s);
  if (er != cudaSuccess) return er;
  if (c.T == 0) {
    er = zero_param_grads(c, a.g, s);
    for (int i = 1; i < 8 && er == cudaSuccess; ++i) er = record_event(ev[i], s);
    return er;
  }
  const int N = int(c.n_experts), k = int(c.top_k), T = int(c.T);
  const int64_t d = c.d_model, f = c.d_ff;
  const int hs = c.d_ff_shared > 0 ? 1 : 0;
  const moe_weights* w = a.w;
  const int groups = N + hs;

  // gate step: dO rows, dz
  {
    const size_t smem = size_t(kGateWarps) * (3 * N + k) * sizeof(float);
    if (smem > 48 * 1024) {
      const cudaError_t e = cudaFuncSetAttribute(
          bwd_gate_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
      if (e != cudaSuccess) return e;
    }
    const bool tcr = router_bwd_on_tensor_cores(c);
    const cudaError_t e = launch_pdl(
        bwd_gate_kernel<E>, dim3(unsigned((T + kGateWarps - 1) / kGateWarps)),
        dim3(kGateWarps * 32), smem, s, static_cast<const E*>(a.dy),
        static_cast<const E*>(a.Yp), a.token_row, a.topk_idx, a.topk_w, a.logits,
        a.mean_prob, a.offsets, T, d, N, k, c.renormalize ? 1 : 0, hs, a.aux_weight,
        static_cast<E*>(a.dO), a.dz, a.dw, tcr ? static_cast<__nv_bfloat16*>(a.dz_bf) : nullptr,
        tcr ? a.rgrp : nullptr);
    if (e != cudaSuccess) return e;
  }
  if (kBf16) {
    // padding rows of dO, H and Xp -> 0 (the wgrads run K over whole 64-row blocks)
    PadBufs pb{};
    pb.buf[0] = a.dO; pb.vec16[0] = d / 8;
    pb.buf[1] = a.H; pb.vec16[1] = f / 8;
    pb.buf[2] = a.Xp; pb.vec16[2] = d / 8;
    pb.n = 3;
    const cudaError_t e = launch_pdl(zero_pad_rows_kernel, dim3(unsigned(groups), 16),
                                     dim3(256), 0, s, a.offsets, a.kept, N, hs ? T : 0, pb);
    if (e != cudaSuccess) return e;
  }
  er = record_event(ev[1], s);
  if (er != cudaSuccess) return er;
  GroupedFfnArgs ga{};
  ga.offsets = a.offsets; ga.kept = a.kept; ga.w = w; ga.rows_max = a.rows_max;
  ga.status = a.status; ga.wait_limit_ns = a.wait_limit_ns; ga.num_sms = a.num_sms;
  BwdGemmArgs bg{};
  bg.offsets = a.offsets; bg.kept = a.kept; bg.rows_max = a.rows_max; bg.status = a.status;
  bg.wait_limit_ns = a.wait_limit_ns; bg.num_sms = a.num_sms;
  cudaError_t e;
  // A1 = Xp W1^T + b1 (the pre-activation), unless the forward kept it
  e = cudaSuccess;
  if (a.recompute_A1)
    e = kBf16
            ? launch_grouped_linear_bf16(c, ga, a.Xp, w->W1, w->W1s, w->b1, w->b1s, a.A1, d, f, s)
            : launch_grouped_linear_f32(c, bg, a.Xp, w->W1, w->W1s, w->b1, w->b1s, a.A1, d, f, s);
  if (e == cudaSuccess) e = record_event(ev[2], s);
  if (e != cudaSuccess) return e;
  // dA = (dO . W2) act'(A1);  dXp = dA . W1
  auto dgrad = kBf16 ? launch_bwd_dgrad : launch_bwd_dgrad_f32;
  e = dgrad(c, bg, a.dO, w->W2, w->W2s, d, f, c.act, a.A1, a.dA, s);
  if (e == cudaSuccess) e = record_event(ev[3], s);
  if (e != cudaSuccess) return e;
  e = dgrad(c, bg, a.dA, w->W1, w->W1s, f, d, -1, nullptr, a.dXp, s);
  if (e == cudaSuccess) e = record_event(ev[4], s);
  if (e != cudaSuccess) return e;
  // dW2 = dO^T H [d, f];  dW1 = dA^T Xp [f, d]
  auto wgrad = kBf16 ? launch_bwd_wgrad : launch_bwd_wgrad_f32;
  e = wgrad(c, bg, a.dO, d, a.H, f, a.g->dW2, a.g->dW2s, s);
  if (e == cudaSuccess) e = record_event(ev[5], s);
  if (e != cudaSuccess) return e;
  e = wgrad(c, bg, a.dA, f, a.Xp, d, a.g->dW1, a.g->dW1s, s);
  if (e == cudaSuccess) e = record_event(ev[6], s);
  if (e != cudaSuccess) return e;
  // db2, db1
  constexpr int kColsPerBlock = 32 * Vec16<E>::n;
  e = launch_pdl(group_colsum_kernel<E>,
                 dim3(unsigned(groups), unsigned((d + kColsPerBlock - 1) / kColsPerBlock)),
                 dim3(256), 0, s, static_cast<const E*>(a.dO), d, a.offsets, a.kept, N,
                 hs ? T : 0, static_cast<E*>(a.g->db2), static_cast<E*>(a.g->db2s));
  if (e != cudaSuccess) return e;
  e = launch_pdl(group_colsum_kernel<E>,
                 dim3(unsigned(groups), unsigned((f + kColsPerBlock - 1) / kColsPerBlock)),
                 dim3(256), 0, s, static_cast<const E*>(a.dA), f, a.offsets, a.kept, N,
                 hs ? T : 0, static_cast<E*>(a.g->db1), static_cast<E*>(a.g->db1s));
  if (e != cudaSuccess) return e;
  // router: dx_router = dz W_g [T, d]; dW_g = dz^T x [N, d]; db_g = sum_t dz
  const bool tc_router = router_bwd_on_tensor_cores(c);
  if (tc_router) {
    // the dgrad / wgrad kernels on one group of T rows, dz rounded to bf16
    moe_config rc = c;
    rc.n_experts = 1;
    rc.d_ff_shared = 0;
    BwdGemmArgs rg = bg;
    rg.offsets = a.rgrp;
    rg.kept = a.rgrp + 3;
    rg.rows_max = T;
    e = launch_bwd_dgrad(rc, rg, a.dz_bf, w->W_g, nullptr, N, d, -1, nullptr, a.dxr_bf, s);
    if (e != cudaSuccess) return e;
    e = launch_bwd_wgrad(rc, rg, a.dz_bf, N, a.x, d, a.g->dW_g, nullptr, s);
    if (e != cudaSuccess) return e;
  } else {
    e = launch_router_grad_gemm<E, float>(a.dz, N, 1, static_cast<const E*>(w->W_g), d, T, d,
                                          N, a.dxr, d, s);
    if (e != cudaSuccess) return e;
    const int S = router_splits(c);
    const int64_t kc = ((T + S - 1) / S + kRk - 1) / kRk * kRk;
    dim3 grid(unsigned((d + kRg - 1) / kRg), unsigned((N + kRg - 1) / kRg), unsigned(S));
    e = launch_pdl(router_grad_gemm_kernel<E, float>, grid, dim3(256), 0, s,
                   static_cast<const float*>(a.dz), int64_t(1), int64_t(N),
                   static_cast<const E*>(a.x), d, int64_t(N), d, int64_t(T), kc, a.part, d);
    if (e != cudaSuccess) return e;
    const int64_t n = int64_t(N) * d;
    const int64_t blocks = (n + 255) / 256;
    e = launch_pdl(splitk_reduce_kernel<E>, dim3(unsigned(blocks < 1184 ? blocks : 1184)),
                   dim3(256), 0, s, static_cast<const float*>(a.part), S, n,
                   static_cast<E*>(a.g->dW_g));
    if (e != cudaSuccess) return e;
  }
  e = launch_pdl(router_bias_grad_kernel<E>, dim3(unsigned((N + 31) / 32)), dim3(256), 0, s,
                 static_cast<const float*>(a.dz), T, N, static_cast<E*>(a.g->db_g));
  if (e != cudaSuccess) return e;
  // dx
  if (tc_router)
    e = launch_pdl(bwd_dx_kernel<__nv_bfloat16, E>,
                   dim3(unsigned((T + kDxWarps - 1) / kDxWarps)), dim3(kDxWarps * 32), 0, s,
                   static_cast<const E*>(a.dXp), a.token_row, a.offsets,
                   static_cast<const __nv_bfloat16*>(a.dxr_bf), T, k, N, hs, d,
                   static_cast<E*>(a.g->dx));
  else
    e = launch_pdl(bwd_dx_kernel<float, E>, dim3(unsigned((T + kDxWarps - 1) / kDxWarps)),
                   dim3(kDxWarps * 32), 0, s, static_cast<const E*>(a.dXp), a.token_row,
                   a.offsets, static_cast<const float*>(a.dxr), T, k, N, hs, d,
                   static_cast<E*>(a.g->dx));
  if (e != cudaSuccess) return e;
  return record_event(ev[7], s);
}

}  // namespace

cudaError_t launch_backward(const moe_config& c, const BackwardArgs& a, void* const* events,
                            cudaStream_t s) {
  return c.dtype == MOE_F32 ? backward_t<float>(c, a, events, s)
                            : backward_t<__nv_bfloat16>(c, a, events, s);
}

}  // namespace moe
