// Tiled CUDA-core GEMM C = A . B^T (+ bias, activation), fp32 accumulate.
//
// A [rows, K] and B [Nc, K] are row-major (both K-contiguous, the nn.Linear
// layout).  With `offsets` set the rows are expert groups: group g occupies
// rows [offsets[g], offsets[g+1]) of A and C, of which the first kept_g are
// live; it multiplies B_g (the routed expert g for g < n_routed, else the
// shared expert).  Used for the router scores and for the fp32 expert FFN.
#pragma once

#include "common.cuh"

namespace moe {

struct SimtGemmArgs {
  const void* A;
  const void* B;            // [n_routed, Nc, K] (or [Nc, K] without groups)
  const void* Bs;           // shared expert's [Nc, K] or nullptr
  const void* bias;         // [n_routed, Nc] (or [Nc]) or nullptr
  const void* bias_s;       // shared expert's [Nc] or nullptr
  void* C;
  int64_t rows;             // rows of A / C when offsets == nullptr
  int64_t K, Nc;
  const int32_t* offsets;   // nullptr: one group of `rows` rows
  const int32_t* kept;      // [n_routed]
  int32_t n_routed;
  int32_t shared_rows;      // live rows of the shared group (0: none)
  int32_t act;              // -1: none, else MOE_ACT_*
  // backward: B stored [K, Nc] (the weight as is) instead of [Nc, K], and
  // the result multiplied by act'(pre[row, col]) when pre is set (no bias)
  int32_t b_kn;
  int32_t dact;             // MOE_ACT_* of act' (read only when pre is set)
  const void* pre;          // [rows, Nc] or nullptr
};

constexpr int kSimtBM = 64, kSimtBN = 64, kSimtBK = 16, kSimtThreads = 256;

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(kSimtThreads) simt_gemm_kernel(SimtGemmArgs a) {
  __shared__ float As[kSimtBK][kSimtBM + 4];
  __shared__ float Bs[kSimtBK][kSimtBN + 4];
  pdl_launch_dependents();
  pdl_wait_previous();

  const int64_t row0 = int64_t(blockIdx.y) * kSimtBM;
  const int64_t col0 = int64_t(blockIdx.x) * kSimtBN;
  const TIn* B = static_cast<const TIn*>(a.B);
  const TIn* bias = static_cast<const TIn*>(a.bias);
  int64_t row_end;                     // one past the last live row of this tile's group
  if (a.offsets == nullptr) {
    row_end = a.rows;
  } else {
    const int ng = a.n_routed + (a.shared_rows > 0 ? 1 : 0);
    if (row0 >= a.offsets[ng]) return;
    int lo = 0, hi = ng - 1;           // last group g with offsets[g] <= row0
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.offsets[mid] <= row0) lo = mid; else hi = mid - 1;
    }
    const int g = lo;
    if (g < a.n_routed) {
      row_end = a.offsets[g] + a.kept[g];
      B += int64_t(g) * a.Nc * a.K;
      if (bias) bias += int64_t(g) * a.Nc;
    } else {
      row_end = a.offsets[g] + a.shared_rows;
      B = static_cast<const TIn*>(a.Bs);
      bias = static_cast<const TIn*>(a.bias_s);
    }
  }
  if (row0 >= row_end) return;         // padding tile

  const TIn* A = static_cast<const TIn*>(a.A);
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int lr = tid >> 2;             // loader: row within the tile
  const int lk = (tid & 3) * 4;        // loader: first of 4 k values

  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int64_t k0 = 0; k0 < a.K; k0 += kSimtBK) {
    {
      const int64_t r = row0 + lr, kk = k0 + lk;
      const bool ok = r < row_end && kk < a.K;   // K % 4 == 0: 4 values all in or all out
#pragma unroll
      for (int q = 0; q < 4; ++q) As[lk + q][lr] = ok ? to_f32(A[r * a.K + kk + q]) : 0.f;
      if (a.b_kn) {
        // B[k, n]: 64 consecutive columns of 4 K-rows per pass of 256 threads
        const int nn = tid & 63, kq = tid >> 6;
        const int64_t c = col0 + nn;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int64_t kr = k0 + 4 * kq + q;
          Bs[4 * kq + q][nn] = (c < a.Nc && kr < a.K) ? to_f32(B[kr * a.Nc + c]) : 0.f;
        }
      } else {
        const int64_t c = col0 + lr;
        const bool okb = c < a.Nc && kk < a.K;
#pragma unroll
        for (int q = 0; q < 4; ++q) Bs[lk + q][lr] = okb ? to_f32(B[c * a.K + kk + q]) : 0.f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kSimtBK; ++kk) {
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

  TOut* C = static_cast<TOut*>(a.C);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t r = row0 + ty + 16 * i;
    if (r >= row_end) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t c = col0 + tx + 16 * j;
      if (c >= a.Nc) continue;
      float v = acc[i][j];
      if (bias) v += to_f32(bias[c]);
      if (a.act >= 0) v = apply_act(v, a.act);
      if (a.pre) {
        const float pa = to_f32(static_cast<const TIn*>(a.pre)[r * a.Nc + c]);
        v *= a.dact == MOE_ACT_RELU ? (pa > 0.f ? 1.f : 0.f) : gelu_erf_grad(pa);
      }
      C[r * a.Nc + c] = from_f32<TOut>(v);
    }
  }
}

// Grouped weight gradient on CUDA cores: for group g (blockIdx.z),
// C_g[m, n] = sum over the group's live rows r of L[r, m] R[r, n]
// (L [rows, Md], R [rows, Nd], both row-major; C_g [Md, Nd] at C + g Md Nd,
// the shared group's at Cs).  The K loop covers exactly the live rows.
struct SimtWgradArgs {
  const void* L;
  const void* R;
  void* C;
  void* Cs;
  int64_t Md, Nd;
  const int32_t* offsets;
  const int32_t* kept;
  int32_t n_routed;
  int32_t shared_rows;
};

template <typename T>
__global__ void __launch_bounds__(kSimtThreads) simt_wgrad_kernel(SimtWgradArgs a) {
  __shared__ float Ls[kSimtBK][kSimtBM + 4];
  __shared__ float Rs[kSimtBK][kSimtBN + 4];
  pdl_launch_dependents();
  pdl_wait_previous();
  const int g = blockIdx.z;
  const int64_t m0 = int64_t(blockIdx.y) * kSimtBM, n0 = int64_t(blockIdx.x) * kSimtBN;
  const int64_t r0 = a.offsets[g];
  const int64_t live = g < a.n_routed ? a.kept[g] : a.shared_rows;
  const T* L = static_cast<const T*>(a.L);
  const T* R = static_cast<const T*>(a.R);
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int cc = tid & 63, kq = tid >> 6;       // loaders: 64 columns x 4 rows per pass
  float acc[4][4] = {};
  for (int64_t k0 = 0; k0 < live; k0 += kSimtBK) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int64_t r = k0 + 4 * kq + q;
      const bool okr = r < live;
      Ls[4 * kq + q][cc] = (okr && m0 + cc < a.Md) ? to_f32(L[(r0 + r) * a.Md + m0 + cc]) : 0.f;
      Rs[4 * kq + q][cc] = (okr && n0 + cc < a.Nd) ? to_f32(R[(r0 + r) * a.Nd + n0 + cc]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kSimtBK; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = Ls[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = Rs[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
  T* C = g < a.n_routed ? static_cast<T*>(a.C) + int64_t(g) * a.Md * a.Nd : static_cast<T*>(a.Cs);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + ty + 16 * i;
    if (m >= a.Md) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = n0 + tx + 16 * j;
      if (n < a.Nd) C[m * a.Nd + n] = from_f32<T>(acc[i][j]);
    }
  }
}

}  // namespace moe
