// Tiled CUDA-core GEMM C = A . B^T (+ bias, activation), fp32 accumulate.
//
// A [rows, K] and B [Nc, K] are row-major (both K-contiguous, the nn.Linear
// layout).  With `offsets` set the rows are expert groups: group g occupies
// rows [offsets[g], offsets[g+1]) of A and C, of which the first kept_g are
// live; it multiplies B_g (the routed expert g for g < n_routed, else the
// shared expert).  Used for the router scores and for the fp32 expert FFN.
#pragma once

#include "common.cuh"
#include "kernels.h"

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
  void* C_pre;              // with act >= 0: also store the pre-activation here (or nullptr)
};

constexpr int kSimtThreads = 256;

// L consecutive elements (L = 2 or 4, aligned to L) as fp32.
template <typename TIn, int L>
__device__ __forceinline__ void simt_load(const TIn* p, float (&v)[L]) {
  if constexpr (sizeof(TIn) == 4) {
    if constexpr (L == 4) {
      const float4 q = *reinterpret_cast<const float4*>(p);
      v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    } else {
      const float2 q = *reinterpret_cast<const float2*>(p);
      v[0] = q.x; v[1] = q.y;
    }
  } else {
    if constexpr (L == 4) {
      const uint2 q = *reinterpret_cast<const uint2*>(p);
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.x));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.y));
      v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
    } else {
      const uint32_t q = *reinterpret_cast<const uint32_t*>(p);
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q));
      v[0] = a.x; v[1] = a.y;
    }
  }
}

// Row (column) of a thread's i-th output in a BM (BN) tile: 4-wide groups,
// BM / 2 (BN / 2) apart when a thread holds 8.
template <int BM>
__device__ __forceinline__ int simt_trow(int ty, int i) {
  return (i >> 2) * (BM / 2) + ty * 4 + (i & 3);
}

// The shared K loop of the register-tiled kernels: `fetch(k0)` loads the
// k-step at k0 into registers, `stash(buf)` writes them to buffer buf; the
// next step's loads are in flight while the current step is multiplied.
template <int BM, int BN, class Fetch, class Stash>
__device__ __forceinline__ void simt_mainloop(float (&As)[2][8][BM + 4],
                                              float (&Bs)[2][8][BN + 4], int64_t K,
                                              Fetch&& fetch, Stash&& stash,
                                              float (&acc)[BM / 16][BN / 16], int tx, int ty) {
  constexpr int BK = 8, TM = BM / 16, TN = BN / 16;
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
  if (K <= 0) return;
  fetch(0);
  stash(0);
  __syncthreads();
  int buf = 0;
  for (int64_t k0 = 0; k0 < K; k0 += BK) {
    const bool more = k0 + BK < K;
    if (more) fetch(k0 + BK);
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float av[TM], bv[TN];
#pragma unroll
      for (int i = 0; i < TM; i += 4) {
        const float4 q = *reinterpret_cast<const float4*>(&As[buf][kk][simt_trow<BM>(ty, i)]);
        av[i] = q.x; av[i + 1] = q.y; av[i + 2] = q.z; av[i + 3] = q.w;
      }
#pragma unroll
      for (int j = 0; j < TN; j += 4) {
        const float4 q = *reinterpret_cast<const float4*>(&Bs[buf][kk][simt_trow<BN>(tx, j)]);
        bv[j] = q.x; bv[j + 1] = q.y; bv[j + 2] = q.z; bv[j + 3] = q.w;
      }
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    if (more) stash(buf ^ 1);
    __syncthreads();
    buf ^= 1;
  }
}

// Register-tiled CUDA-core GEMM: a BM x BN tile per block of 256 threads as
// 16 x 16 threads of TM x TN outputs (TM = BM / 16, TN = BN / 16, each 4 or
// 8), K in steps of 8 through two shared-memory buffers (the next step's
// global loads are in flight while the current one is multiplied; one
// barrier per step).  A (and B in the [Nc, K] layout) is stored transposed,
// [k][row] with rows padded by 4 floats, so that the loader's writes are free
// of bank conflicts.  A thread's rows (columns) are groups of 4 consecutive
// ones, BM / 2 (BN / 2) apart when it holds 8: its 16-byte reads then cover
// 16 consecutive words across the warp, free of bank conflicts.  Rows past
// the group's live rows read as zeros and are not stored; K % 8 == 0.
template <typename TIn, typename TOut, int BM, int BN>
__global__ void __launch_bounds__(kSimtThreads, 2) simt_gemm_kernel(SimtGemmArgs a) {
  constexpr int BK = 8;
  constexpr int TM = BM / 16, TN = BN / 16;
  constexpr int LA = BM / 32, LB = BN / 32;       // elements per thread per k-step
  __shared__ __align__(16) float As[2][BK][BM + 4];
  __shared__ __align__(16) float Bs[2][BK][BN + 4];
  pdl_launch_dependents();
  pdl_wait_previous();

  const int64_t row0 = int64_t(blockIdx.y) * BM;
  const int64_t col0 = int64_t(blockIdx.x) * BN;
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
  // loaders: A row a_r, k offset a_k; B as [Nc, K] the same with LB; B as
  // [K, Nc]: k-row kn_k, columns kn_c .. kn_c + LB - 1
  const int a_r = tid / (BK / LA), a_k = (tid % (BK / LA)) * LA;
  const int b_r = tid / (BK / LB), b_k = (tid % (BK / LB)) * LB;
  const int kn_k = tid / (BN / LB), kn_c = (tid % (BN / LB)) * LB;
  const bool a_ok = row0 + a_r < row_end;
  const bool b_ok = a.b_kn ? true : col0 + b_r < a.Nc;
  float ra[LA], rb[LB];

  auto fetch = [&](int64_t k0) {
    if (a_ok) {
      simt_load<TIn, LA>(A + (row0 + a_r) * a.K + k0 + a_k, ra);
    } else {
#pragma unroll
      for (int q = 0; q < LA; ++q) ra[q] = 0.f;
    }
    if (a.b_kn) {
      const int64_t c = col0 + kn_c;
      const TIn* src = B + (k0 + kn_k) * a.Nc + c;
      if (c + LB <= a.Nc && (a.Nc % LB) == 0) {
        simt_load<TIn, LB>(src, rb);
      } else {
#pragma unroll
        for (int q = 0; q < LB; ++q) rb[q] = c + q < a.Nc ? to_f32(src[q]) : 0.f;
      }
    } else if (b_ok) {
      simt_load<TIn, LB>(B + (col0 + b_r) * a.K + k0 + b_k, rb);
    } else {
#pragma unroll
      for (int q = 0; q < LB; ++q) rb[q] = 0.f;
    }
  };
  auto stash = [&](int buf) {
#pragma unroll
    for (int q = 0; q < LA; ++q) As[buf][a_k + q][a_r] = ra[q];
    if (a.b_kn) {
      if constexpr (LB == 4)
        *reinterpret_cast<float4*>(&Bs[buf][kn_k][kn_c]) = make_float4(rb[0], rb[1], rb[2], rb[3]);
      else
        *reinterpret_cast<float2*>(&Bs[buf][kn_k][kn_c]) = make_float2(rb[0], rb[1]);
    } else {
#pragma unroll
      for (int q = 0; q < LB; ++q) Bs[buf][b_k + q][b_r] = rb[q];
    }
  };

  float acc[TM][TN];
  simt_mainloop<BM, BN>(As, Bs, a.K, fetch, stash, acc, tx, ty);

  TOut* C = static_cast<TOut*>(a.C);
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int64_t r = row0 + simt_trow<BM>(ty, i);
    if (r >= row_end) continue;
#pragma unroll
    for (int j = 0; j < TN; ++j) {
      const int64_t c = col0 + simt_trow<BN>(tx, j);
      if (c >= a.Nc) continue;
      float v = acc[i][j];
      if (bias) v += to_f32(bias[c]);
      if (a.C_pre) static_cast<TOut*>(a.C_pre)[r * a.Nc + c] = from_f32<TOut>(v);
      if (a.act >= 0) v = apply_act(v, a.act);
      if (a.pre) {
        const float pa = to_f32(static_cast<const TIn*>(a.pre)[r * a.Nc + c]);
        v *= a.dact == MOE_ACT_RELU ? (pa > 0.f ? 1.f : 0.f) : gelu_erf_grad(pa);
      }
      acc[i][j] = v;
    }
#pragma unroll
    for (int j = 0; j < TN; j += 4) {
      const int64_t cb = col0 + simt_trow<BN>(tx, j);   // 4 consecutive columns
      if constexpr (sizeof(TOut) == 4) {
        if (cb + 4 <= a.Nc && (a.Nc % 4) == 0) {
          *reinterpret_cast<float4*>(C + r * a.Nc + cb) =
              make_float4(acc[i][j], acc[i][j + 1], acc[i][j + 2], acc[i][j + 3]);
          continue;
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (cb + q < a.Nc) C[r * a.Nc + cb + q] = from_f32<TOut>(acc[i][j + q]);
    }
  }
}

// Launches simt_gemm_kernel over `rows` rows (grouped: the grouped row count)
// with the widest tile that still gives about two blocks per SM.
template <typename TIn, typename TOut>
cudaError_t launch_simt_gemm(const SimtGemmArgs& a, int64_t rows, int num_sms, cudaStream_t s) {
  auto blocks = [&](int bm, int bn) { return ceil_div(a.Nc, bn) * ceil_div(rows, bm); };
  const int64_t want = 2 * int64_t(num_sms > 0 ? num_sms : 148);
  if (blocks(128, 128) >= want)
    return launch_pdl(simt_gemm_kernel<TIn, TOut, 128, 128>,
                      dim3(unsigned(ceil_div(a.Nc, 128)), unsigned(ceil_div(rows, 128))),
                      dim3(kSimtThreads), 0, s, a);
  if (blocks(128, 64) >= want)
    return launch_pdl(simt_gemm_kernel<TIn, TOut, 128, 64>,
                      dim3(unsigned(ceil_div(a.Nc, 64)), unsigned(ceil_div(rows, 128))),
                      dim3(kSimtThreads), 0, s, a);
  return launch_pdl(simt_gemm_kernel<TIn, TOut, 64, 64>,
                    dim3(unsigned(ceil_div(a.Nc, 64)), unsigned(ceil_div(rows, 64))),
                    dim3(kSimtThreads), 0, s, a);
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

// The weight gradient on the register-tiled loop: block (n-tile, m-tile,
// group g) computes its BM x BN tile of C_g = L_g^T R_g, K = the group's live
// rows in steps of 8 (rows past them read as zeros).  Both operands are
// [rows, M] row-major, so each k-step loads 16-byte runs along M and N and
// stores them as they are.  A group with no rows writes zeros.  Md % 4 == 0,
// Nd % 4 == 0.
template <typename T, int BM, int BN>
__global__ void __launch_bounds__(kSimtThreads, 2) simt_wgrad_kernel(SimtWgradArgs a) {
  constexpr int TM = BM / 16, TN = BN / 16;
  constexpr int LA = BM / 32, LB = BN / 32;
  __shared__ __align__(16) float As[2][8][BM + 4];
  __shared__ __align__(16) float Bs[2][8][BN + 4];
  pdl_launch_dependents();
  pdl_wait_previous();
  const int g = blockIdx.z;
  const int64_t m0 = int64_t(blockIdx.y) * BM, n0 = int64_t(blockIdx.x) * BN;
  const int64_t r0 = a.offsets[g];
  const int64_t live = g < a.n_routed ? a.kept[g] : a.shared_rows;
  const T* L = static_cast<const T*>(a.L);
  const T* R = static_cast<const T*>(a.R);
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int ka = tid / (BM / LA), ma = (tid % (BM / LA)) * LA;   // k-row, first m
  const int kb = tid / (BN / LB), nb = (tid % (BN / LB)) * LB;   // k-row, first n
  const bool a_ok = m0 + ma + LA <= a.Md, b_ok = n0 + nb + LB <= a.Nd;
  float ra[LA], rb[LB];
  auto fetch = [&](int64_t k0) {
    const bool ka_in = k0 + ka < live, kb_in = k0 + kb < live;
    if (ka_in && a_ok) {
      simt_load<T, LA>(L + (r0 + k0 + ka) * a.Md + m0 + ma, ra);
    } else {
#pragma unroll
      for (int q = 0; q < LA; ++q) ra[q] = 0.f;
    }
    if (kb_in && b_ok) {
      simt_load<T, LB>(R + (r0 + k0 + kb) * a.Nd + n0 + nb, rb);
    } else {
#pragma unroll
      for (int q = 0; q < LB; ++q) rb[q] = 0.f;
    }
  };
  auto stash = [&](int buf) {
    if constexpr (LA == 4)
      *reinterpret_cast<float4*>(&As[buf][ka][ma]) = make_float4(ra[0], ra[1], ra[2], ra[3]);
    else
      *reinterpret_cast<float2*>(&As[buf][ka][ma]) = make_float2(ra[0], ra[1]);
    if constexpr (LB == 4)
      *reinterpret_cast<float4*>(&Bs[buf][kb][nb]) = make_float4(rb[0], rb[1], rb[2], rb[3]);
    else
      *reinterpret_cast<float2*>(&Bs[buf][kb][nb]) = make_float2(rb[0], rb[1]);
  };
  float acc[TM][TN];
  simt_mainloop<BM, BN>(As, Bs, live, fetch, stash, acc, tx, ty);

  T* C = g < a.n_routed ? static_cast<T*>(a.C) + int64_t(g) * a.Md * a.Nd : static_cast<T*>(a.Cs);
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int64_t m = m0 + simt_trow<BM>(ty, i);
    if (m >= a.Md) continue;
#pragma unroll
    for (int j = 0; j < TN; j += 4) {
      const int64_t n = n0 + simt_trow<BN>(tx, j);    // 4 consecutive columns
      if constexpr (sizeof(T) == 4) {
        if (n + 4 <= a.Nd) {
          *reinterpret_cast<float4*>(C + m * a.Nd + n) =
              make_float4(acc[i][j], acc[i][j + 1], acc[i][j + 2], acc[i][j + 3]);
          continue;
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (n + q < a.Nd) C[m * a.Nd + n + q] = from_f32<T>(acc[i][j + q]);
    }
  }
}

}  // namespace moe
