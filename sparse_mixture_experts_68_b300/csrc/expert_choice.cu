// Expert-choice routing (matteuscruz.github.io "What is a Mixture of Experts?",
// "Load balancing: the core training challenge"; Zhou et al., 2022, as the page
// describes it): instead of every token taking its top-k experts, every expert
// takes the C tokens it scores highest, so each expert gets exactly C tokens.
// The score is the router probability p[t, e]; equal scores go to the lower
// token index; a picked token's gate is p[t, e].
//
// Selection: one 1024-thread block per expert over its row of the
// expert-major probabilities probT [N, T].  p >= 0, so the fp32 bit patterns
// order like the values, and a four-pass radix select (8 bits a pass, from the
// top) finds the bit pattern of the C-th largest score exactly.  A pass in
// token order then keeps every score above it plus the first `need` tokens
// equal to it, with two block scans per 4096 tokens.  The picked tokens land
// in ascending token order in the expert's group of Cpad = round_up(C, 128)
// rows, ready for the row copy and the grouped FFN of top-k routing; the
// per-token view token_row / token_w [T, N] (-1 / 0 where not picked) feeds
// the combine with one slot per expert.
#include "kernels.h"
#include "stats.cuh"

namespace moe {

namespace {

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;     // 32: one warp-0 lane per warp
constexpr int kSelPerThread = 4;
constexpr int kSelChunk = kSelThreads * kSelPerThread;

// Exclusive prefix of v over the block's threads; `total` = the block sum.
// scratch: kSelWarps + 1 ints of shared memory.
__device__ __forceinline__ int sel_block_scan(int v, int* scratch, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = scratch[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += u;
    }
    scratch[lane] = wi - w;
    if (lane == 31) scratch[kSelWarps] = wi;
  }
  __syncthreads();
  const int r = scratch[warp] + incl - v;
  total = scratch[kSelWarps];
  __syncthreads();                               // scratch is reused by the next scan
  return r;
}

__global__ void __launch_bounds__(kSelThreads)
    ec_select_kernel(const float* __restrict__ probT, int T, int N, int C, int Cpad,
                     int has_shared, int32_t* __restrict__ ec_token,
                     float* __restrict__ ec_gate, int32_t* __restrict__ offsets,
                     int32_t* __restrict__ counts, int32_t* __restrict__ row_token,
                     int32_t* __restrict__ token_row, float* __restrict__ token_w,
                     int32_t* __restrict__ picks) {
  __shared__ int hist[256];
  __shared__ int scan[kSelWarps + 1];
  __shared__ uint32_t s_digit;
  __shared__ int s_need;
  pdl_launch_dependents();
  pdl_wait_previous();
  const int e = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t routed_end = int64_t(N) * Cpad;
  if (e == N) {                                  // the shared expert: every token, in order
    const int64_t Tpad = int64_t(T + kGroupAlign - 1) / kGroupAlign * kGroupAlign;
    for (int64_t r = tid; r < Tpad; r += kSelThreads)
      row_token[routed_end + r] = r < T ? int32_t(r) : -1;
    return;
  }
  if (e == 0 && tid == 0) {
    offsets[N] = int32_t(routed_end);
    offsets[N + 1] = int32_t(routed_end + (has_shared ? int64_t(T + kGroupAlign - 1) /
                                                            kGroupAlign * kGroupAlign
                                                      : 0));
  }
  const int64_t base = int64_t(e) * Cpad;
  if (tid == 0) {
    offsets[e] = int32_t(base);
    counts[e] = C;
  }
  for (int r = C + tid; r < Cpad; r += kSelThreads) row_token[base + r] = -1;   // padding
  if (C == 0) return;
  const uint32_t* key = reinterpret_cast<const uint32_t*>(probT + int64_t(e) * T);

  // radix select: the bit pattern of the C-th largest score
  uint32_t prefix = 0, mask = 0;
  int need = C;                                  // still to take at or below the prefix
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kSelThreads) hist[i] = 0;
    if (tid == 0) {
      s_digit = 0;
      s_need = need;
    }
    __syncthreads();
    for (int t0 = 0; t0 < T; t0 += kSelThreads) {          // uniform trip count per warp
      const int t = t0 + tid;
      const uint32_t k = t < T ? key[t] : 0u;
      const bool in = t < T && (k & mask) == prefix;
      const int digit = int((k >> shift) & 255u);
      const uint32_t peers = __match_any_sync(0xffffffffu, in ? digit : -1);
      if (in && (__ffs(peers) - 1) == lane) atomicAdd(&hist[digit], __popc(peers));
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns digits 8l .. 8l+7; count the keys above each lane's range
      int h[8], sl = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        h[j] = hist[lane * 8 + j];
        sl += h[j];
      }
      int incl = sl;                             // keys in this lane's digits and above
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += u;
      }
      const int above = incl - sl;
      if (above < need && need <= incl) {        // exactly one lane
        int run = above;
        for (int j = 7; j >= 0; --j) {
          if (run + h[j] >= need) {
            s_digit = uint32_t(lane * 8 + j);
            s_need = need - run;
            break;
          }
          run += h[j];
        }
      }
    }
    __syncthreads();
    prefix |= s_digit << shift;
    mask |= 255u << shift;
    need = s_need;
    __syncthreads();
  }
  const uint32_t thr = prefix;

  // keep, in token order, every key above thr and the first `need` equal to it
  int carry_eq = 0, carry_take = 0;
  for (int t0 = 0; t0 < T; t0 += kSelChunk) {
    const int tb = t0 + tid * kSelPerThread;
    uint32_t kv[kSelPerThread];
    int n_eq = 0;
#pragma unroll
    for (int j = 0; j < kSelPerThread; ++j) {
      kv[j] = tb + j < T ? key[tb + j] : 0u;
      n_eq += (tb + j < T && kv[j] == thr) ? 1 : 0;
    }
    int tot_eq;
    int eq_rank = carry_eq + sel_block_scan(n_eq, scan, tot_eq);
    bool take[kSelPerThread];
    int n_take = 0;
#pragma unroll
    for (int j = 0; j < kSelPerThread; ++j) {
      const bool valid = tb + j < T;
      const bool eq = valid && kv[j] == thr;
      take[j] = valid && (kv[j] > thr || (eq && eq_rank < need));
      eq_rank += eq ? 1 : 0;
      n_take += take[j] ? 1 : 0;
    }
    int tot_take;
    int pos = carry_take + sel_block_scan(n_take, scan, tot_take);
#pragma unroll
    for (int j = 0; j < kSelPerThread; ++j) {
      const int t = tb + j;
      if (t >= T) break;
      const int64_t slot = int64_t(t) * N + e;
      if (take[j] && pos < C) {                  // exactly C are taken; the bound is a guard
        const float pv = __uint_as_float(kv[j]);
        MOE_CHECK(t >= 0 && t < T, CK_EC_PICK);
        ec_token[int64_t(e) * C + pos] = t;
        ec_gate[int64_t(e) * C + pos] = pv;
        row_token[base + pos] = t;
        token_row[slot] = int32_t(base + pos);
        token_w[slot] = pv;
        atomicAdd(&picks[t], 1);
        ++pos;
      } else {
        token_row[slot] = -1;
        token_w[slot] = 0.f;
      }
    }
    carry_eq += tot_eq;
    carry_take += tot_take;
  }
}

__global__ void __launch_bounds__(kStatsThreads)
    ec_stats_kernel(const float* __restrict__ prob_partials, int nblk, int N, int T,
                    const int32_t* __restrict__ counts, const int32_t* __restrict__ picks,
                    float* __restrict__ mean_prob, float* __restrict__ balance,
                    int32_t* __restrict__ scratch, int32_t* __restrict__ unpicked) {
  __shared__ int part[kStatsWarps];
  pdl_launch_dependents();
  pdl_wait_previous();
  // every expert keeps all it picked: kept = counts, nothing dropped
  block_load_stats(prob_partials, nblk, N, T, counts, counts, mean_prob, balance, scratch,
                   nullptr);
  int n = 0;
  for (int t = threadIdx.x; t < T; t += kStatsThreads) n += picks[t] == 0 ? 1 : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = n;
  __syncthreads();
  if (threadIdx.x == 0) {
    int s = 0;
    for (int w = 0; w < kStatsWarps; ++w) s += part[w];
    *unpicked = s;
  }
}

}  // namespace

cudaError_t launch_ec_select(const moe_config& c, int64_t C, const float* probT,
                             int32_t* ec_token, float* ec_gate, int32_t* offsets,
                             int32_t* counts, int32_t* row_token, int32_t* token_row,
                             float* token_w, int32_t* picks, cudaStream_t s) {
  const int has_shared = c.d_ff_shared > 0 ? 1 : 0;
  const unsigned blocks = unsigned(c.n_experts + has_shared);
  return launch_pdl(ec_select_kernel, dim3(blocks), dim3(kSelThreads), 0, s, probT, int(c.T),
                    int(c.n_experts), int(C), int(ec_group_rows(C)), has_shared, ec_token,
                    ec_gate, offsets, counts, row_token, token_row, token_w, picks);
}

cudaError_t launch_ec_stats(const moe_config& c, const float* prob_partials,
                            const int32_t* counts, const int32_t* picks, float* mean_prob,
                            float* balance, int32_t* scratch, int32_t* unpicked,
                            cudaStream_t s) {
  const int nblk = int(router_partial_rows(c));
  return launch_pdl(ec_stats_kernel, dim3(1), dim3(kStatsThreads), 0, s, prob_partials, nblk,
                    int(c.n_experts), int(c.T), counts, picks, mean_prob, balance, scratch,
                    unpicked);
}

MOE_CHECKS_UNIT(expert_choice)

}  // namespace moe
