// Load statistics (botmartz.com "Mixture of Experts (MoE) and Mixtral",
// "Load Balancing: The Hidden Challenge"): mean over tokens of the router
// probabilities, the unbiased variance of those means, and the dropped count;
// also the squared coefficient of variation of the routed counts
// (matteuscruz.github.io "Load balancing: the core training challenge";
// invest-in.ai "MoE - Mixture of Experts", cv_squared(expert_counts)).
// A block-wide device function so that the statistics can run either as
// their own kernel or at the end of the one-block permutation.
#pragma once

#include "common.cuh"

namespace moe {

// One block of 1024 threads, all sums in a fixed order and in fp32 (B300's
// fp64 rate is low, and an fp64 division alone costs microseconds); accuracy
// comes from compensated arithmetic instead.  The partial-sum rows are split
// into RG row groups and the experts into 32-wide chunks; warp w takes (row
// group w % RG, chunk w / RG) with lane = expert, so every load is a
// coalesced 128-byte row segment, kStatsBatch of them in flight.  The loads
// are unconditional (a row index past the warp's range is clamped to its last
// row, and the sum skips it): with each load under the same bounds test as its
// addition the compiler issued them one round trip at a time, which took 33 us
// for 296 x 256 partial sums.  The function is not inlined, so that every
// caller gets the same schedule.  Each warp keeps a
// Kahan sum per expert; the row groups are combined in order with
// error-free additions (two-sum).  The deviation from the uniform load is
// taken as (S - T/N) / T with S the compensated sum, so it keeps its
// accuracy when the load is nearly uniform.  The counts' statistic is exact
// integer arithmetic up to its last step: with S = sum c and Q = sum c^2,
// var/mean^2 = N (N Q - S^2) / ((N - 1) S^2), N Q - S^2 in 128-bit integers.
constexpr int kStatsThreads = 1024;
constexpr int kStatsWarps = kStatsThreads / 32;
constexpr int kStatsBatch = 16;                   // partial-sum rows loaded at once

__device__ __forceinline__ void stats_two_sum(float a, float b, float& s, float& err) {
  s = a + b;
  const float bb = s - a;
  err = (a - (s - bb)) + (b - bb);
}

__device__ __forceinline__ void stats_kahan_add(float v, float& s, float& comp) {
  const float y = v - comp;
  const float t = s + y;
  comp = (t - s) - y;
  s = t;
}

// var(c) / mean(c)^2 = N (N Q - S^2) / ((N - 1) S^2) from S = sum c, Q = sum c^2:
// N Q - S^2 exactly in 128-bit integers; numerator a and denominator b in
// fp64 products, and the quotient without an fp64 division: q0 = a / b in
// fp32, then one correction q0 + (a - q0 b) / b with the residual exact in
// an fp64 fma and its quotient needing only fp32 accuracy; then one rounding.
__device__ __forceinline__ float cv_squared_of(int N, long long S, long long Q) {
  if (N <= 1 || S <= 0) return 0.f;
  const unsigned __int128 nq = (unsigned __int128)(unsigned long long)N * (unsigned long long)Q;
  const unsigned __int128 s2 = (unsigned __int128)(unsigned long long)S * (unsigned long long)S;
  const unsigned __int128 num = nq - s2;                   // >= 0 (Cauchy-Schwarz)
  const double numd = double((unsigned long long)(num >> 64)) * 18446744073709551616.0 +
                      double((unsigned long long)num);
  const double sd = double(S);
  const double a = double(N) * numd, b = double(N - 1) * sd * sd;
  const float bf = float(b);
  const float q0 = float(a) / bf;
  const double r = fma(-double(q0), b, a);
  return float(double(q0) + r * double(1.0f / bf));
}

// Runs on all kStatsThreads threads of a block (blockDim.x == kStatsThreads).
static __device__ __noinline__ void block_load_stats(const float* __restrict__ prob_partials,
                                                 int nblk, int N, int Ttok,
                                                 const int32_t* __restrict__ counts,
                                                 const int32_t* __restrict__ kept,
                                                 float* __restrict__ mean_prob,
                                                 float* __restrict__ balance,
                                                 int32_t* __restrict__ dropped,
                                                 float* __restrict__ cv_squared) {
  __shared__ float2 part[kStatsWarps][32];        // (sum, -compensation) per warp, lane
  __shared__ float2 sq[kStatsWarps];              // Kahan sum of squared deviations
  __shared__ int dr[kStatsWarps];
  __shared__ long long cs[kStatsWarps], cq[kStatsWarps];   // sum c, sum c^2
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nchunks = (N + 31) / 32;
  const float invT = Ttok > 0 ? 1.0f / float(Ttok) : 0.f;
  const float tN = float(Ttok) / float(N);        // the per-expert sum of a uniform router
  if (nchunks == 1) {
    // N <= 32: warp g sums row group g (every 32nd... rows g*R .. g*R + R-1)
    // for all experts (lane = expert); warp e then combines expert e's 32
    // groups and warp 0 the experts, both as shuffle trees of error-free
    // additions (a fixed order, so the result is reproducible).
    {
      const int rows = (nblk + kStatsWarps - 1) / kStatsWarps;
      const int b0 = warp * rows, b1 = min(nblk, b0 + rows);
      float s = 0.f, comp = 0.f;
      if (lane < N) {
        for (int b = b0; b < b1; b += kStatsBatch) {   // loads in flight, added in order
          float v[kStatsBatch];
#pragma unroll
          for (int u = 0; u < kStatsBatch; ++u)
            v[u] = prob_partials[int64_t(min(b + u, b1 - 1)) * N + lane];
#pragma unroll
          for (int u = 0; u < kStatsBatch; ++u)
            if (b + u < b1) stats_kahan_add(v[u], s, comp);
        }
      }
      part[warp][lane] = make_float2(s, -comp);
    }
    __syncthreads();
    if (warp < N) {
      const int e = warp;
      const float2 pv = part[lane][e];            // lane = row group
      float hi = pv.x, lo = pv.y;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ohi = __shfl_xor_sync(0xffffffffu, hi, o);
        const float olo = __shfl_xor_sync(0xffffffffu, lo, o);
        float ns, ne;
        stats_two_sum(hi, ohi, ns, ne);
        hi = ns;
        lo = lo + olo + ne;
      }
      if (lane == 0) {
        mean_prob[e] = (hi + lo) * invT;
        float dhi, dlo;
        stats_two_sum(hi, -tN, dhi, dlo);
        const float dev = (dhi + (dlo + lo)) * invT;
        sq[e] = make_float2(dev * dev, 0.f);
        const int ce = counts[e];
        dr[e] = ce - kept[e];
        cs[e] = ce;
        cq[e] = (long long)ce * ce;
      }
    }
    __syncthreads();
    if (warp == 0) {
      float v = lane < N ? sq[lane].x : 0.f, vc = 0.f;
      int w = lane < N ? dr[lane] : 0;
      long long S = lane < N ? cs[lane] : 0, Q = lane < N ? cq[lane] : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const float oc = __shfl_xor_sync(0xffffffffu, vc, o);
        float ns, ne;
        stats_two_sum(v, ov, ns, ne);
        v = ns;
        vc = vc + oc + ne;
        w += __shfl_xor_sync(0xffffffffu, w, o);
        S += __shfl_xor_sync(0xffffffffu, S, o);
        Q += __shfl_xor_sync(0xffffffffu, Q, o);
      }
      if (lane == 0) {
        *balance = (N > 1 && Ttok > 0) ? (v + vc) / float(N - 1) : 0.f;
        *dropped = w;
        if (cv_squared) *cv_squared = cv_squared_of(N, S, Q);
      }
    }
    return;
  }
  float sq_s = 0.f, sq_c = 0.f;
  int my_dr = 0;
  long long my_cs = 0, my_cq = 0;
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
      for (int b = b0; b < b1; b += kStatsBatch) {     // loads in flight, added in order
        float v[kStatsBatch];
#pragma unroll
        for (int u = 0; u < kStatsBatch; ++u)
          v[u] = prob_partials[int64_t(min(b + u, b1 - 1)) * N + e];
#pragma unroll
        for (int u = 0; u < kStatsBatch; ++u)
          if (b + u < b1) stats_kahan_add(v[u], s, comp);
      }
    }
    part[warp][lane] = make_float2(s, -comp);
    __syncthreads();
    if (rg == 0 && live) {
      const int slot = warp / RG;
      float hi = 0.f, lo = 0.f;
      for (int g = 0; g < RG; ++g) {
        const float2 pv = part[slot * RG + g][lane];
        float ns, ne;
        stats_two_sum(hi, pv.x, ns, ne);
        hi = ns;
        lo += ne + pv.y;
      }
      mean_prob[e] = (hi + lo) * invT;
      float dhi, dlo;
      stats_two_sum(hi, -tN, dhi, dlo);
      const float dev = (dhi + (dlo + lo)) * invT;
      stats_kahan_add(dev * dev, sq_s, sq_c);
      const long long ce = counts[e];
      my_dr += int(ce) - kept[e];
      my_cs += ce;
      my_cq += ce * ce;
    }
    __syncthreads();
  }
  // lanes, then warps, in a fixed order
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float os = __shfl_xor_sync(0xffffffffu, sq_s, o);
    const float oc = __shfl_xor_sync(0xffffffffu, sq_c, o);
    float ns, ne;
    stats_two_sum(sq_s, os, ns, ne);
    sq_s = ns;
    sq_c = sq_c + oc - ne;
    my_dr += __shfl_xor_sync(0xffffffffu, my_dr, o);
    my_cs += __shfl_xor_sync(0xffffffffu, my_cs, o);
    my_cq += __shfl_xor_sync(0xffffffffu, my_cq, o);
  }
  if (lane == 0) {
    sq[warp] = make_float2(sq_s, sq_c);
    dr[warp] = my_dr;
    cs[warp] = my_cs;
    cq[warp] = my_cq;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float v = 0.f, vc = 0.f;
    int w = 0;
    long long S = 0, Q = 0;
    for (int i = 0; i < kStatsWarps; ++i) {
      stats_kahan_add(sq[i].x, v, vc);
      vc += sq[i].y;
      w += dr[i];
      S += cs[i];
      Q += cq[i];
    }
    *balance = (N > 1 && Ttok > 0) ? (v - vc) / float(N - 1) : 0.f;
    *dropped = w;
    if (cv_squared) *cv_squared = cv_squared_of(N, S, Q);
  }
}

}  // namespace moe
