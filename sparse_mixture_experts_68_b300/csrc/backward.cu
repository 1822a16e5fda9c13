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
//   expert FFNs    A1 (the forward's kept pre-activation, or recomputed by
//                  the first Linear without its activation), then
//                  dA = (dO W2) act'(A1), dXp = dA W1, dW2 = dO^T H,
//                  dW1 = dA^T Xp on the tensor cores (grouped_bwd_sm103.cu;
//                  CUDA cores for fp32 layers); db2, db1 = column sums of
//                  dO, dA over each group's rows
//   router         dW_g = dz^T x, db_g = sum_t dz, dx_router = dz W_g
//                  (tensor cores when N % 64 == 0; else CUDA cores, with
//                  dx_router folded into dx for N <= 32)
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
                    int32_t* __restrict__ rgrp, const int32_t* __restrict__ kept,
                    E* __restrict__ H, E* __restrict__ Xp, int64_t f, int pad_groups) {
  extern __shared__ float gsm[];
  pdl_launch_dependents();
  pdl_wait_previous();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tok_blocks = (T + kGateWarps - 1) / kGateWarps;
  if (int(blockIdx.x) >= tok_blocks) {
    // blocks past the tokens: group g's padding rows [live, round_up(live, 16))
    // of dO, H and Xp -> 0, the rows the tensor-core wgrads' last K step reads
    const int g = int(blockIdx.x) - tok_blocks;
    if (g >= pad_groups) return;
    const int64_t live = g < N ? kept[g] : T;
    const int64_t r0 = int64_t(offsets[g]) + live, r1 = int64_t(offsets[g]) + (live + 15) / 16 * 16;
    const int64_t nd = d * int64_t(sizeof(E)) / 16, nf = f * int64_t(sizeof(E)) / 16;
    for (int64_t r = r0; r < r1; ++r) {
      uint4* a = reinterpret_cast<uint4*>(dO + r * d);
      uint4* b = reinterpret_cast<uint4*>(Xp + r * d);
      uint4* c = reinterpret_cast<uint4*>(H + r * f);
      for (int64_t j = threadIdx.x; j < nd; j += blockDim.x) {
        a[j] = make_uint4(0, 0, 0, 0);
        b[j] = make_uint4(0, 0, 0, 0);
      }
      for (int64_t j = threadIdx.x; j < nf; j += blockDim.x) c[j] = make_uint4(0, 0, 0, 0);
    }
    return;
  }
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
//
// db2[g] = sum of dO's live rows of group g, db1[g] the same over dA.  Groups
// start on 128-row boundaries, so each 128-row chunk of the grouped row space
// lies in one group.  Pass 1: block (c, y) sums chunk c's live rows over one
// column block (32 lanes x one 16-byte word) of dO (y < the dO column
// blocks) or of dA; its eight warps take every eighth row and combine in order;
// fp32 partials part[c][col], col over dO's d then dA's f columns.  Pass 2:
// each output sums its group's chunks in order.  Rows past a group's live rows
// (padding, never read) do not enter.
constexpr int kChunkRows = MOE_GROUP_ALIGN;

template <typename T>
__global__ void __launch_bounds__(256)
    colsum_partial_kernel(const T* __restrict__ m2, int64_t w2, const T* __restrict__ m1,
                          int64_t w1, const int32_t* __restrict__ offsets,
                          const int32_t* __restrict__ kept, int n_routed, int shared_rows,
                          int n_groups, float* __restrict__ part) {
  constexpr int V = Vec16<T>::n;
  __shared__ float red[8][32 * V];
  __shared__ int s_live;
  pdl_launch_dependents();
  pdl_wait_previous();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t r0 = int64_t(blockIdx.x) * kChunkRows;
  if (threadIdx.x == 0) {
    int nl = 0;
    if (r0 < offsets[n_groups]) {
      int lo = 0, hi = n_groups - 1;            // the last group starting at or before r0
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (offsets[mid] <= r0) lo = mid; else hi = mid - 1;
      }
      const int64_t live = lo < n_routed ? kept[lo] : shared_rows;
      const int64_t n = int64_t(offsets[lo]) + live - r0;
      nl = int(n < 0 ? 0 : (n > kChunkRows ? kChunkRows : n));
    }
    s_live = nl;
  }
  __syncthreads();
  const int nlive = s_live;
  const int64_t cb2 = (w2 + 32 * V - 1) / (32 * V);
  const bool second = blockIdx.y >= cb2;
  const T* src = second ? m1 : m2;
  const int64_t width = second ? w1 : w2;
  const int64_t cblk = second ? blockIdx.y - cb2 : blockIdx.y;
  const int64_t c0 = cblk * 32 * V + lane * V;
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  if (c0 < width) {
    int r = warp;
    for (; r + 24 < nlive; r += 32) {            // four rows in flight per lane
      float v[4][V];
#pragma unroll
      for (int u = 0; u < 4; ++u) Vec16<T>::load(src + (r0 + r + 8 * u) * width + c0, v[u]);
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] += v[u][i];
    }
    for (; r < nlive; r += 8) {
      float v[V];
      Vec16<T>::load(src + (r0 + r) * width + c0, v);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] += v[i];
    }
  }
#pragma unroll
  for (int i = 0; i < V; ++i) red[warp][lane * V + i] = acc[i];
  __syncthreads();
  float* dst = part + int64_t(blockIdx.x) * (w2 + w1) + (second ? w2 : 0);
  for (int col = threadIdx.x; col < 32 * V; col += blockDim.x) {
    const int64_t cc = cblk * 32 * V + col;
    if (cc < width) {
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) sum += red[w][col];
      dst[cc] = sum;
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256)
    colsum_reduce_kernel(const float* __restrict__ part, int64_t w2, int64_t w1,
                         const int32_t* __restrict__ offsets, int n_routed, int n_groups,
                         T* __restrict__ db2, T* __restrict__ db2s, T* __restrict__ db1,
                         T* __restrict__ db1s) {
  pdl_launch_dependents();
  pdl_wait_previous();
  const int64_t W = w2 + w1;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n_groups * W;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int g = int(i / W);
    const int64_t col = i - int64_t(g) * W;
    const int c0 = offsets[g] / kChunkRows, c1 = offsets[g + 1] / kChunkRows;
    float v[4] = {0.f, 0.f, 0.f, 0.f};          // chunks c0 + 4j + u, combined in order
    int c = c0;
    for (; c + 3 < c1; c += 4) {
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] += part[int64_t(c + u) * W + col];
    }
    for (; c < c1; ++c) v[0] += part[int64_t(c) * W + col];
    const float sum = (v[0] + v[1]) + (v[2] + v[3]);
    if (col < w2) (g < n_routed ? db2 + int64_t(g) * w2 : db2s)[col] = from_f32<T>(sum);
    else (g < n_routed ? db1 + int64_t(g) * w1 : db1s)[col - w2] = from_f32<T>(sum);
  }
}

// db_g[e] = sum_t dz[t, e] (fp32 in): block b takes experts 32 b .. 32 b + 31
// (one per lane), its 32 warps every 32nd token with four tokens in flight,
// and the warps combine in order.
constexpr int kBiasWarps = 32;

template <typename TO>
__global__ void __launch_bounds__(kBiasWarps * 32)
    router_bias_grad_kernel(const float* __restrict__ dz, int T, int N, TO* __restrict__ db_g) {
  __shared__ float part[kBiasWarps][32];
  pdl_launch_dependents();
  pdl_wait_previous();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 32 + lane;
  float s = 0.f;
  if (e < N) {
    int t = warp;
    for (; t + 3 * kBiasWarps < T; t += 4 * kBiasWarps) {
      float v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = dz[int64_t(t + u * kBiasWarps) * N + e];
      s += (v[0] + v[1]) + (v[2] + v[3]);
    }
    for (; t < T; t += kBiasWarps) s += dz[int64_t(t) * N + e];
  }
  part[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && e < N) {
    float v = 0.f;
    for (int w = 0; w < kBiasWarps; ++w) v += part[w][lane];
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

// ---- router gradients for few experts (N <= 32) on CUDA cores -----------------------------------
//
// dW_g[e, i] = sum_t dz[t, e] x[t, i] and db_g[e] = sum_t dz[t, e].  Block
// (cb, z): tokens [z*tc, (z+1)*tc), columns cb*256*CPT ...; each thread keeps
// NMAX x CPT accumulators for its CPT columns (NMAX * CPT <= 64, experts
// n..NMAX-1 read zeros); the chunk's dz rows are staged in shared memory.
// Partial sums per chunk, summed afterwards in chunk order
// (splitk_reduce2_kernel): [S][n*d] for dW_g, then [S][n] for db_g.
constexpr int kRouterSmallMaxN = 32;
constexpr int kRouterSmallRows = 64;            // dz rows staged per pass

template <typename T, int NMAX, int CPT>
__global__ void __launch_bounds__(256)
    router_grad_small_kernel(const float* __restrict__ dz, const T* __restrict__ x, int Ttok,
                             int n, int64_t d, int tc, float* __restrict__ part) {
  __shared__ float dzs[kRouterSmallRows][NMAX];
  pdl_launch_dependents();
  for (int i = threadIdx.x; i < kRouterSmallRows * NMAX; i += 256) (&dzs[0][0])[i] = 0.f;
  pdl_wait_previous();
  const int z = blockIdx.y, S = gridDim.y;
  const int t0 = z * tc, t1 = min(Ttok, t0 + tc);
  const int64_t col0 = (int64_t(blockIdx.x) * 256 + threadIdx.x) * CPT;
  float acc[NMAX][CPT];
#pragma unroll
  for (int e = 0; e < NMAX; ++e)
#pragma unroll
    for (int j = 0; j < CPT; ++j) acc[e][j] = 0.f;
  float bacc = 0.f;                               // db_g: thread e < n of block x = 0
  for (int tb = t0; tb < t1; tb += kRouterSmallRows) {
    const int nr = min(kRouterSmallRows, t1 - tb);
    __syncthreads();
    for (int i = threadIdx.x; i < nr * n; i += 256) dzs[i / n][i % n] = dz[int64_t(tb) * n + i];
    __syncthreads();
    if (blockIdx.x == 0 && threadIdx.x < n)
      for (int rr = 0; rr < nr; ++rr) bacc += dzs[rr][threadIdx.x];
    if (col0 < d) {
      // four rows of x in flight (past nr: the last row again, weighted 0)
      for (int rr = 0; rr < nr; rr += 4) {
        float xv[4][CPT];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int row = tb + min(rr + u, nr - 1);
          const T* xr = x + int64_t(row) * d + col0;
          if constexpr (CPT % Vec16<T>::n == 0) {
#pragma unroll
            for (int j = 0; j < CPT; j += Vec16<T>::n) Vec16<T>::load(xr + j, xv[u] + j);
          } else {
#pragma unroll
            for (int j = 0; j < CPT; ++j) xv[u][j] = to_f32(xr[j]);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const bool in = rr + u < nr;
#pragma unroll
          for (int e = 0; e < NMAX; ++e) {
            const float g = in ? dzs[rr + u][e] : 0.f;
#pragma unroll
            for (int j = 0; j < CPT; ++j) acc[e][j] = fmaf(g, xv[u][j], acc[e][j]);
          }
        }
      }
    }
  }
  if (col0 < d) {
#pragma unroll
    for (int e = 0; e < NMAX; ++e)
      if (e < n)
#pragma unroll
        for (int j = 0; j < CPT; ++j)
          part[int64_t(z) * n * d + int64_t(e) * d + col0 + j] = acc[e][j];
  }
  if (blockIdx.x == 0 && threadIdx.x < n)
    part[int64_t(S) * n * d + int64_t(z) * n + threadIdx.x] = bacc;
}

// out1[i] = sum_z part[z * n1 + i] (i < n1), out2[i] = sum_z part[S * n1 + z * n2 + i]
template <typename TO>
__global__ void __launch_bounds__(256)
    splitk_reduce2_kernel(const float* __restrict__ part, int S, int64_t n1,
                          TO* __restrict__ out1, int64_t n2, TO* __restrict__ out2) {
  pdl_launch_dependents();
  pdl_wait_previous();
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n1 + n2;
       i += int64_t(gridDim.x) * blockDim.x) {
    // four running sums (chunks z mod 4), combined in a fixed order
    const float* src = i < n1 ? part + i : part + int64_t(S) * n1 + (i - n1);
    const int64_t stride = i < n1 ? n1 : n2;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    int z = 0;
    for (; z + 3 < S; z += 4) {
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] += src[int64_t(z + u) * stride];
    }
    for (; z < S; ++z) v[0] += src[int64_t(z) * stride];
    const float sum = (v[0] + v[1]) + (v[2] + v[3]);
    if (i < n1) out1[i] = from_f32<TO>(sum);
    else out2[i - n1] = from_f32<TO>(sum);
  }
}

// ---- dx -----------------------------------------------------------------------------------------

constexpr int kDxWarps = 8;

// dx[t] = dxr[t] (the router's part, fp32 or bf16; or, with dxr == nullptr,
// dz[t] W_g computed here) + sum over t's kept rows of dXp (slot order) + the
// shared row; T: the layer's element type.  Warp (token, column chunk): each
// lane takes kDxVec 16-byte words of the chunk, 32 words apart, so that every
// row read keeps kDxVec loads in flight.
constexpr int kDxVec = 4;

template <typename TR, typename T>
__global__ void __launch_bounds__(kDxWarps * 32)
    bwd_dx_kernel(const T* __restrict__ dXp, const int32_t* __restrict__ token_row,
                  const int32_t* __restrict__ offsets, const TR* __restrict__ dxr, int Ttok,
                  int k, int N, int has_shared, int64_t d, T* __restrict__ dx,
                  const float* __restrict__ dz, const T* __restrict__ W_g) {
  constexpr int V = Vec16<T>::n;
  __shared__ float dzs[kDxWarps][32];
  pdl_launch_dependents();
  pdl_wait_previous();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t t = int64_t(blockIdx.x) * kDxWarps + warp;
  if (t >= Ttok) return;
  if (!dxr) {                                   // few experts (N <= 32): dz[t] per warp
    dzs[warp][lane] = lane < N ? dz[t * N + lane] : 0.f;
    __syncwarp();
  }
  const int64_t nv = d / V;
  const int64_t cbase = int64_t(blockIdx.y) * 32 * kDxVec + lane;
  float acc[kDxVec][V];
#pragma unroll
  for (int u = 0; u < kDxVec; ++u)
#pragma unroll
    for (int i = 0; i < V; ++i) acc[u][i] = 0.f;
  for (int j = 0; j <= k; ++j) {
    int64_t r;
    if (j < k) r = token_row[t * k + j];
    else r = has_shared ? int64_t(offsets[N]) + t : -1;
    if (r < 0) continue;
    float v[kDxVec][V];
#pragma unroll
    for (int u = 0; u < kDxVec; ++u) {
      const int64_t c = cbase + 32 * u;
      if (c < nv) Vec16<T>::load(dXp + r * d + c * V, v[u]);
    }
#pragma unroll
    for (int u = 0; u < kDxVec; ++u)
      if (cbase + 32 * u < nv)
#pragma unroll
        for (int i = 0; i < V; ++i) acc[u][i] += v[u][i];
  }
  if (dxr) {
#pragma unroll
    for (int u = 0; u < kDxVec; ++u) {
      const int64_t c = cbase + 32 * u;
      if (c < nv)
#pragma unroll
        for (int i = 0; i < V; ++i) acc[u][i] += to_f32(dxr[t * d + c * V + i]);
    }
  } else {
    // the router's part dz[t] W_g (W_g of few experts stays in cache)
    float rt[kDxVec][V];
#pragma unroll
    for (int u = 0; u < kDxVec; ++u)
#pragma unroll
      for (int i = 0; i < V; ++i) rt[u][i] = 0.f;
    for (int e = 0; e < N; ++e) {
      const float g = dzs[warp][e];
      float wv[kDxVec][V];
#pragma unroll
      for (int u = 0; u < kDxVec; ++u) {
        const int64_t c = cbase + 32 * u;
        if (c < nv) Vec16<T>::load(W_g + int64_t(e) * d + c * V, wv[u]);
      }
#pragma unroll
      for (int u = 0; u < kDxVec; ++u)
        if (cbase + 32 * u < nv)
#pragma unroll
          for (int i = 0; i < V; ++i) rt[u][i] = fmaf(g, wv[u][i], rt[u][i]);
    }
#pragma unroll
    for (int u = 0; u < kDxVec; ++u)
#pragma unroll
      for (int i = 0; i < V; ++i) acc[u][i] += rt[u][i];
  }
#pragma unroll
  for (int u = 0; u < kDxVec; ++u) {
    const int64_t c = cbase + 32 * u;
    if (c < nv) Vec16<T>::store(dx + t * d + c * V, acc[u]);
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

// Chunks of T for router_grad_small_kernel: about two waves of blocks.
int router_small_chunks(const moe_config& c) {
  const int N = int(c.n_experts);
  const int cpt = N <= 8 ? 8 : (N <= 16 ? 4 : 2);
  const int64_t cblocks = (c.d_model + 256 * cpt - 1) / (256 * cpt);
  int64_t S = (2 * 148 + cblocks - 1) / cblocks;
  const int64_t by_t = (c.T + 31) / 32;           // at least 32 tokens a chunk
  if (S > by_t) S = by_t;
  return int(S < 1 ? 1 : S);
}

template <typename E>
cudaError_t launch_router_small(const moe_config& c, const float* dz, const E* x, float* part,
                                E* dW_g, E* db_g, cudaStream_t s) {
  const int N = int(c.n_experts), T = int(c.T);
  const int64_t d = c.d_model;
  const int S = router_small_chunks(c);
  const int tc = (T + S - 1) / S;
  cudaError_t e;
#define MOE_ROUTER_SMALL(NN, CPT)                                                          \
  {                                                                                        \
    const dim3 grid(unsigned((d + 256 * CPT - 1) / (256 * CPT)), unsigned(S));            \
    e = launch_pdl(router_grad_small_kernel<E, NN, CPT>, grid, dim3(256), 0, s, dz, x, T, N, \
                   d, tc, part);                                                           \
  }
  if (N <= 1) MOE_ROUTER_SMALL(1, 8)
  else if (N <= 2) MOE_ROUTER_SMALL(2, 8)
  else if (N <= 4) MOE_ROUTER_SMALL(4, 8)
  else if (N <= 8) MOE_ROUTER_SMALL(8, 8)
  else if (N <= 16) MOE_ROUTER_SMALL(16, 4)
  else MOE_ROUTER_SMALL(32, 2)
#undef MOE_ROUTER_SMALL
  if (e != cudaSuccess) return e;
  const int64_t n1 = int64_t(N) * d, n2 = N;
  const int64_t blocks = (n1 + n2 + 255) / 256;
  return launch_pdl(splitk_reduce2_kernel<E>, dim3(unsigned(blocks < 1184 ? blocks : 1184)),
                    dim3(256), 0, s, static_cast<const float*>(part), S, n1, dW_g, n2, db_g);
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

size_t bias_partial_bytes(const moe_config& c, int64_t rows_max) {
  return size_t((rows_max + kChunkRows - 1) / kChunkRows) * size_t(c.d_model + c.d_ff) *
         sizeof(float);
}

size_t router_bwd_partial_bytes(const moe_config& c) {
  if (router_bwd_on_tensor_cores(c)) return 0;
  if (c.n_experts <= kRouterSmallMaxN)
    return size_t(router_small_chunks(c)) * size_t(c.n_experts * (c.d_model + 1)) *
           sizeof(float);
  return size_t(router_splits(c)) * size_t(c.n_experts * c.d_model) * sizeof(float);
}

int backward_launch_count(const moe_config& c) {
  if (c.T == 0) return c.d_ff_shared > 0 ? 10 : 6;    // zero parameter gradients
  // gate, A1, dA, dXp, dW2, dW1, the bias column sums (partials, reduction),
  // then the router: tensor cores dx_router + dW_g + db_g; few experts (<= 32)
  // dW_g with db_g + their reduction (dx_router inside dx); otherwise
  // dx_router, split-K dW_g + reduction, db_g; then dx
  const int router = router_bwd_on_tensor_cores(c) ? 3
                     : c.n_experts <= kRouterSmallMaxN ? 2 : 4;
  return 8 + router + 1;
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
    // bf16: one more block per group zeroes the padding rows its wgrads read
    const int pad_groups = kBf16 ? groups : 0;
    const cudaError_t e = launch_pdl(
        bwd_gate_kernel<E>, dim3(unsigned((T + kGateWarps - 1) / kGateWarps + pad_groups)),
        dim3(kGateWarps * 32), smem, s, static_cast<const E*>(a.dy),
        static_cast<const E*>(a.Yp), a.token_row, a.topk_idx, a.topk_w, a.logits,
        a.mean_prob, a.offsets, T, d, N, k, c.renormalize ? 1 : 0, hs, a.aux_weight,
        static_cast<E*>(a.dO), a.dz, a.dw, tcr ? static_cast<__nv_bfloat16*>(a.dz_bf) : nullptr,
        tcr ? a.rgrp : nullptr, a.kept, static_cast<E*>(a.H), static_cast<E*>(a.Xp), f,
        pad_groups);
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
  // db2, db1: chunk partials, then each group's chunks in order
  {
    constexpr int kColsPerBlock = 32 * Vec16<E>::n;
    const int64_t cb = (d + kColsPerBlock - 1) / kColsPerBlock +
                       (f + kColsPerBlock - 1) / kColsPerBlock;
    const int64_t chunks = (a.rows_max + kChunkRows - 1) / kChunkRows;
    e = launch_pdl(colsum_partial_kernel<E>, dim3(unsigned(chunks), unsigned(cb)), dim3(256), 0,
                   s, static_cast<const E*>(a.dO), d, static_cast<const E*>(a.dA), f,
                   a.offsets, a.kept, N, hs ? T : 0, groups, a.bpart);
    if (e != cudaSuccess) return e;
    const int64_t outs = int64_t(groups) * (d + f);
    const int64_t blocks = (outs + 255) / 256;
    e = launch_pdl(colsum_reduce_kernel<E>, dim3(unsigned(blocks < 4096 ? blocks : 4096)),
                   dim3(256), 0, s, static_cast<const float*>(a.bpart), d, f, a.offsets, N,
                   groups, static_cast<E*>(a.g->db2), static_cast<E*>(a.g->db2s),
                   static_cast<E*>(a.g->db1), static_cast<E*>(a.g->db1s));
    if (e != cudaSuccess) return e;
  }
  // router: dx_router = dz W_g [T, d]; dW_g = dz^T x [N, d]; db_g = sum_t dz
  const bool tc_router = router_bwd_on_tensor_cores(c);
  const bool small_router = !tc_router && N <= kRouterSmallMaxN;
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
  } else if (small_router) {
    e = launch_router_small<E>(c, a.dz, static_cast<const E*>(a.x), a.part,
                               static_cast<E*>(a.g->dW_g), static_cast<E*>(a.g->db_g), s);
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
  if (!small_router) {
    e = launch_pdl(router_bias_grad_kernel<E>, dim3(unsigned((N + 31) / 32)),
                   dim3(kBiasWarps * 32), 0, s, static_cast<const float*>(a.dz), T, N,
                   static_cast<E*>(a.g->db_g));
    if (e != cudaSuccess) return e;
  }
  // dx
  const dim3 dx_grid(unsigned((T + kDxWarps - 1) / kDxWarps),
                     unsigned((d / Vec16<E>::n + 32 * kDxVec - 1) / (32 * kDxVec)));
  if (tc_router)
    e = launch_pdl(bwd_dx_kernel<__nv_bfloat16, E>, dx_grid, dim3(kDxWarps * 32), 0, s,
                   static_cast<const E*>(a.dXp), a.token_row, a.offsets,
                   static_cast<const __nv_bfloat16*>(a.dxr_bf), T, k, N, hs, d,
                   static_cast<E*>(a.g->dx), static_cast<const float*>(nullptr),
                   static_cast<const E*>(nullptr));
  else
    e = launch_pdl(bwd_dx_kernel<float, E>, dx_grid, dim3(kDxWarps * 32), 0, s,
                   static_cast<const E*>(a.dXp), a.token_row,
                   a.offsets, small_router ? nullptr : static_cast<const float*>(a.dxr), T, k,
                   N, hs, d, static_cast<E*>(a.g->dx), static_cast<const float*>(a.dz),
                   static_cast<const E*>(w->W_g));
  if (e != cudaSuccess) return e;
  return record_event(ev[7], s);
}

}  // namespace

cudaError_t launch_backward(const moe_config& c, const BackwardArgs& a, void* const* events,
                            cudaStream_t s) {
  return c.dtype == MOE_F32 ? backward_t<float>(c, a, events, s)
                            : backward_t<__nv_bfloat16>(c, a, events, s);
}

MOE_CHECKS_UNIT(backward)

}  // namespace moe
