// Permutation of the (token, slot) assignments into per-expert contiguous
// groups with an optional capacity (matteuscruz.github.io "What is a Mixture
// of Experts?", sections "Distributed training and inference" -- grouping
// tokens by expert -- and "Load balancing" -- capacity factor x batch /
// experts, overflow dropped; roadtointelligence.com "Mixture of Experts
// (MoE)", "Keeping the experts busy").
//
// A stable counting sort in four launches, with no order-dependent atomics:
//   hist  : per token-block, per expert assignment counts
//   scan  : per expert, exclusive scan over blocks (the block's base rank),
//           totals, capacity clamp, padded group offsets (one block)
//   rank  : per token-block, one warp walks the block's assignments in
//           token-major order; rank = base + earlier matches in the block
//   copy  : one warp per grouped row copies the token's x row (16-byte
//           vectors); the shared expert's group is x in token order
#include <mutex>

#include "kernels.h"
#include "stats.cuh"

namespace moe {

namespace {

struct PermuteScratch {
  int32_t* block_counts;  // [nblk][N]
  int32_t* block_base;    // [nblk][N]
};

inline int64_t permute_blocks(const moe_config& c) {
  return ceil_div(c.T, kPermuteTokensPerBlock);
}

PermuteScratch carve(const moe_config& c, void* scratch) {
  const int64_t n = permute_blocks(c) * c.n_experts;
  PermuteScratch p;
  p.block_counts = static_cast<int32_t*>(scratch);
  p.block_base = p.block_counts + round_up(n, 64);
  return p;
}

__global__ void __launch_bounds__(256)
    permute_hist_kernel(const int32_t* __restrict__ topk_idx, int T, int k, int N,
                        int32_t* __restrict__ block_counts) {
  extern __shared__ int32_t cnt[];
  pdl_launch_dependents();
  pdl_wait_previous();
  for (int e = threadIdx.x; e < N; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int64_t a0 = int64_t(blockIdx.x) * kPermuteTokensPerBlock * k;
  const int64_t a1 = min(int64_t(T) * k, a0 + int64_t(kPermuteTokensPerBlock) * k);
  for (int64_t a = a0 + threadIdx.x; a < a1; a += blockDim.x) {
    const int e = topk_idx[a];
    MOE_CHECK(e >= 0 && e < N, CK_SORT_EXPERT);
    if (e >= 0 && e < N) atomicAdd(&cnt[e], 1);  // out-of-range experts are not counted
  }
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += blockDim.x)
    block_counts[int64_t(blockIdx.x) * N + e] = cnt[e];
}

// One block of 1024 threads.  Thread e owns expert e (N <= 1024).
__global__ void __launch_bounds__(1024)
    permute_scan_kernel(const int32_t* __restrict__ block_counts, int nblk, int N, int T,
                        int64_t capacity, int has_shared, int32_t* __restrict__ block_base,
                        int32_t* __restrict__ counts, int32_t* __restrict__ kept,
                        int32_t* __restrict__ offsets, int32_t* __restrict__ row_token) {
  __shared__ int32_t warp_tot[32];
  pdl_launch_dependents();
  pdl_wait_previous();
  const int e = threadIdx.x;
  int32_t total = 0, kp = 0, padded = 0;
  if (e < N) {
    for (int b = 0; b < nblk; ++b) {
      block_base[int64_t(b) * N + e] = total;
      total += block_counts[int64_t(b) * N + e];
    }
    kp = (capacity > 0 && int64_t(total) > capacity) ? int32_t(capacity) : total;
    padded = int32_t(round_up(kp, kGroupAlign));
    counts[e] = total;
    kept[e] = kp;
  }
  // exclusive scan of padded over e (warp shuffles, then warp totals)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t incl = padded;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int32_t w = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += v;
    }
    warp_tot[lane] = w;                          // inclusive over warps
  }
  __syncthreads();
  const int32_t excl = incl - padded + (warp > 0 ? warp_tot[warp - 1] : 0);
  if (e < N) {
    offsets[e] = excl;
    for (int32_t r = excl + kp; r < excl + padded; ++r) row_token[r] = -1;   // padding rows
  }
  if (e == N - 1) {
    const int32_t end = excl + padded;
    offsets[N] = end;
    offsets[N + 1] = end + (has_shared ? int32_t(round_up(T, kGroupAlign)) : 0);
  }
}

// One warp per block walks the block's assignments in token-major order.
__global__ void __launch_bounds__(32)
    permute_rank_kernel(const int32_t* __restrict__ topk_idx, int T, int k, int N,
                        int64_t capacity, const int32_t* __restrict__ block_base,
                        const int32_t* __restrict__ offsets, int32_t* __restrict__ row_token,
                        int32_t* __restrict__ token_row) {
  extern __shared__ int32_t run[];              // next rank per expert
  pdl_launch_dependents();
  pdl_wait_previous();
  const int lane = threadIdx.x;
  for (int e = lane; e < N; e += 32) run[e] = block_base[int64_t(blockIdx.x) * N + e];
  __syncwarp();
  const int64_t a0 = int64_t(blockIdx.x) * kPermuteTokensPerBlock * k;
  const int64_t a1 = min(int64_t(T) * k, a0 + int64_t(kPermuteTokensPerBlock) * k);
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int64_t base = a0; base < a1; base += 32) {
    const int64_t a = base + lane;
    const int e = a < a1 ? topk_idx[a] : -1;
    const bool valid = e >= 0 && e < N;          // out-of-range experts: dropped
    MOE_CHECK(a >= a1 || valid, CK_SORT_EXPERT);
    const int key = valid ? e : (0x40000000 | lane);     // invalid lanes match nobody
    const uint32_t same = __match_any_sync(0xffffffffu, key);
    int32_t rank = 0;
    if (valid) rank = run[e] + __popc(same & lt_mask);
    __syncwarp();
    if (valid && (same & lt_mask) == 0) run[e] += __popc(same);   // group leader advances
    __syncwarp();
    if (a < a1) {
      const bool keep = valid && (capacity <= 0 || rank < capacity);
      int32_t row = -1;
      if (keep) {
        row = offsets[e] + rank;
        row_token[row] = int32_t(a / k);
      }
      token_row[a] = row;
    }
  }
}

// The whole counting sort in one block of 32 warps, for layers whose
// assignments (T*k) and per-warp expert counts fit in shared memory: the
// expert ids are staged as 16-bit values; warp w owns the contiguous range
// [w*L, (w+1)*L) of assignments.  Pass 1 counts per (warp, expert) with
// __match_any_sync and keeps each assignment's rank within its warp's range
// (16-bit, in shared memory); a per-expert scan over warps gives each warp's
// base rank; a scan over experts gives the padded group offsets; pass 2 adds
// the two ranks and writes rows, with no further warp-wide matching.  Same
// results as hist + scan + rank.
constexpr int kSortWarps = 32;

__global__ void __launch_bounds__(kSortWarps * 32)
    permute_sort_kernel(const int32_t* __restrict__ topk_idx, int T, int k, int N,
                        int64_t capacity, int has_shared, int32_t* __restrict__ counts,
                        int32_t* __restrict__ kept, int32_t* __restrict__ offsets,
                        int32_t* __restrict__ row_token, int32_t* __restrict__ token_row,
                        StatsArgs stats) {
  extern __shared__ int32_t sm[];
  pdl_launch_dependents();
  pdl_wait_previous();
  const int A = T * k;
  int32_t* cnt = sm;                              // [kSortWarps][N], then base ranks
  int32_t* off = cnt + kSortWarps * N;            // [N] group offsets
  int32_t* warp_tot = off + N;                    // [32], then kept [N], counts [N]
  int16_t* ids = reinterpret_cast<int16_t*>(warp_tot + 32 + 2 * N);   // [A]
  int16_t* lrank = ids + A;                       // [A] rank within the warp's range
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kSortWarps * N; i += blockDim.x) cnt[i] = 0;
  {
    // stage the expert ids: 16-byte loads, four in flight per thread
    auto clamp = [N](int e) {                    // out of range: dropped
      MOE_CHECK(e >= 0 && e < N, CK_SORT_EXPERT);
      return int16_t((e >= 0 && e < N) ? e : -1);
    };
    const int A4 = A / 4;
    const int4* src = reinterpret_cast<const int4*>(topk_idx);
    int i = threadIdx.x;
    for (; i + 3 * int(blockDim.x) < A4; i += 4 * blockDim.x) {
      int4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = __ldg(src + i + u * blockDim.x);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int a = 4 * (i + u * int(blockDim.x));
        ids[a] = clamp(v[u].x); ids[a + 1] = clamp(v[u].y);
        ids[a + 2] = clamp(v[u].z); ids[a + 3] = clamp(v[u].w);
      }
    }
    for (; i < A4; i += blockDim.x) {
      const int4 v = __ldg(src + i);
      const int a = 4 * i;
      ids[a] = clamp(v.x); ids[a + 1] = clamp(v.y); ids[a + 2] = clamp(v.z); ids[a + 3] = clamp(v.w);
    }
    for (int a = 4 * A4 + int(threadIdx.x); a < A; a += blockDim.x) ids[a] = clamp(topk_idx[a]);
  }
  __syncthreads();
  const int L = (A + kSortWarps - 1) / kSortWarps;
  const int a_begin = warp * L, a_end = min(A, a_begin + L);
  const uint32_t lt_mask = (1u << lane) - 1u;
  int32_t* my = cnt + warp * N;
  // pass 1: per-warp counts, and each assignment's rank among its expert's
  // assignments in the warp's range (the running count before this group of
  // 32 plus the equal lanes below it)
  for (int base = a_begin; base < a_end; base += 32) {
    const int a = base + lane;
    const int e = a < a_end ? ids[a] : -1;
    const int key = e >= 0 ? e : (0x40000000 | lane);
    const uint32_t same = __match_any_sync(0xffffffffu, key);
    const int32_t before = e >= 0 ? my[e] : 0;
    __syncwarp();
    if (e >= 0 && (same & lt_mask) == 0) my[e] += __popc(same);
    if (a < a_end) lrank[a] = int16_t(before + __popc(same & lt_mask));
    __syncwarp();
  }
  __syncthreads();
  // per expert: base rank of each warp (a warp-wide scan over the 32 warps'
  // counts, lane = warp index), totals, capacity; warp w takes experts w, w+32, ...
  for (int e = warp; e < N; e += kSortWarps) {
    const int32_t c = cnt[lane * N + e];
    int32_t inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
    cnt[lane * N + e] = inc - c;
    const int32_t run = __shfl_sync(0xffffffffu, inc, 31);
    if (lane == 0) {
      const int32_t kp = (capacity > 0 && int64_t(run) > capacity) ? int32_t(capacity) : run;
      counts[e] = run;
      kept[e] = kp;
      off[e] = kp;                                 // kept for now; offsets below
      warp_tot[32 + N + e] = run;                  // counts, for the statistics
    }
  }
  __syncthreads();
  // N <= blockDim: thread e holds expert e's padded size
  const int32_t padded = threadIdx.x < N ? int32_t(round_up(off[threadIdx.x], kGroupAlign)) : 0;
  // exclusive scan of padded sizes over experts (thread e holds expert e)
  int32_t incl = padded;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int32_t w = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += v;
    }
    warp_tot[lane] = w;
  }
  __syncthreads();
  const int32_t excl = incl - padded + (warp > 0 ? warp_tot[warp - 1] : 0);
  const int e_me = threadIdx.x;
  int32_t* kept_s = warp_tot + 32;                 // [N] kept, next to the ids' alignment pad
  if (e_me < N) {
    kept_s[e_me] = off[e_me];
    offsets[e_me] = excl;
  }
  __syncthreads();
  if (e_me < N) off[e_me] = excl;
  __syncthreads();
  // padding rows (-1): warp w takes experts w, w+32, ..., its lanes the rows
  for (int e = warp; e < N; e += kSortWarps) {
    const int32_t r0 = off[e] + kept_s[e], r1 = off[e] + int32_t(round_up(kept_s[e], kGroupAlign));
    for (int32_t r = r0 + lane; r < r1; r += 32) row_token[r] = -1;
  }
  if (e_me == N - 1) {
    offsets[N] = excl + padded;
    offsets[N + 1] = excl + padded + (has_shared ? int32_t(round_up(T, kGroupAlign)) : 0);
  }
  __syncthreads();
  // pass 2: rank = the warp's base rank for the expert (my[e] after the scan)
  // + the rank within the warp's range from pass 1
  for (int a = a_begin + lane; a < a_end; a += 32) {
    const int e = ids[a];
    int32_t row = -1;
    if (e >= 0) {
      const int32_t rank = my[e] + lrank[a];
      if (capacity <= 0 || rank < capacity) {
        row = off[e] + rank;
        row_token[row] = a / k;
      }
    }
    token_row[a] = row;
  }
  if (stats.prob_partials) {
    // the load statistics as well, once counts and kept are in memory
    __syncthreads();
    // counts and kept from shared memory (generic pointers), not read back from global
    block_load_stats(stats.prob_partials, stats.nblk, N, T, kept_s + N, kept_s,
                     stats.mean_prob, stats.balance, stats.dropped, stats.cv_squared);
  }
}

// Mid-size layers: the same counting sort in two launches over blocks of
// kMidThreads assignments (one per thread), so that it runs on several SMs.
//   mid_rank    : per block, each assignment's rank among its expert's
//                 assignments in the block (__match_any_sync within each warp,
//                 then a per-expert scan over the block's warps) and the
//                 block's per-expert counts
//   mid_scatter : every block sums the counts of all blocks (totals, capacity,
//                 padded group offsets) and of the blocks before it (its base
//                 ranks), then writes its assignments' rows; block 0 also
//                 writes counts, kept, offsets and the padding rows.  With
//                 statistics requested, one more block computes them from the
//                 same totals, beside the scatter.
// Ranks follow token-major assignment order, as in the other two paths.
constexpr int kMidThreads = kStatsThreads;
constexpr int kMidWarps = kMidThreads / 32;

__global__ void __launch_bounds__(kMidThreads)
    permute_mid_rank_kernel(const int32_t* __restrict__ topk_idx, int A, int N,
                            int32_t* __restrict__ block_counts, int32_t* __restrict__ lrank) {
  extern __shared__ int32_t wc[];                 // [kMidWarps][N] counts, then bases
  pdl_launch_dependents();
  pdl_wait_previous();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kMidWarps * N; i += kMidThreads) wc[i] = 0;
  __syncthreads();
  const int a = blockIdx.x * kMidThreads + threadIdx.x;
  const int e = a < A ? topk_idx[a] : -1;
  const bool valid = e >= 0 && e < N;             // out-of-range experts: dropped
  MOE_CHECK(a >= A || valid, CK_SORT_EXPERT);
  const int key = valid ? e : (0x40000000 | lane);
  const uint32_t same = __match_any_sync(0xffffffffu, key);
  const int r = __popc(same & ((1u << lane) - 1u));
  if (valid && r == 0) wc[warp * N + e] = __popc(same);   // one leader per expert and warp
  __syncthreads();
  for (int x = threadIdx.x; x < N; x += kMidThreads) {
    int32_t run = 0;
    for (int w = 0; w < kMidWarps; ++w) {
      const int32_t c = wc[w * N + x];
      wc[w * N + x] = run;
      run += c;
    }
    block_counts[int64_t(blockIdx.x) * N + x] = run;
  }
  __syncthreads();
  if (a < A) lrank[a] = valid ? wc[warp * N + e] + r : -1;
}

// N <= kMidThreads: thread e owns expert e.
__global__ void __launch_bounds__(kMidThreads)
    permute_mid_scatter_kernel(const int32_t* __restrict__ topk_idx,
                               const int32_t* __restrict__ lrank,
                               const int32_t* __restrict__ block_counts, int nblk, int T, int k,
                               int N, int64_t capacity, int has_shared,
                               int32_t* __restrict__ counts, int32_t* __restrict__ kept,
                               int32_t* __restrict__ offsets, int32_t* __restrict__ row_token,
                               int32_t* __restrict__ token_row, StatsArgs stats) {
  extern __shared__ int32_t sm[];
  int32_t* base = sm;                             // [N] this block's base rank per expert
  int32_t* kp = base + N;                         // [N] kept
  int32_t* off = kp + N;                          // [N] group offsets; the stats block: counts
  __shared__ int32_t warp_tot[kMidWarps];
  pdl_launch_dependents();
  pdl_wait_previous();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e_me = threadIdx.x;
  const bool stats_block = int(blockIdx.x) == nblk;
  int32_t tot = 0, mine = 0, kv = 0;
  if (e_me < N) {
    for (int b = 0; b < nblk; ++b) {
      const int32_t c = block_counts[int64_t(b) * N + e_me];
      if (b == int(blockIdx.x)) mine = tot;
      tot += c;
    }
    kv = (capacity > 0 && int64_t(tot) > capacity) ? int32_t(capacity) : tot;
    base[e_me] = mine;
    kp[e_me] = kv;
  }
  if (stats_block) {
    if (e_me < N) off[e_me] = tot;
    __syncthreads();
    // counts and kept from shared memory (generic pointers)
    block_load_stats(stats.prob_partials, stats.nblk, N, T, off, kp, stats.mean_prob,
                     stats.balance, stats.dropped, stats.cv_squared);
    return;
  }
  if (blockIdx.x == 0 && e_me < N) {
    counts[e_me] = tot;
    kept[e_me] = kv;
  }
  // exclusive scan of the padded sizes over experts
  const int32_t padded = e_me < N ? int32_t(round_up(kv, kGroupAlign)) : 0;
  int32_t incl = padded;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int32_t before = 0;
  for (int w = 0; w < warp; ++w) before += warp_tot[w];
  const int32_t excl = before + incl - padded;
  if (e_me < N) {
    off[e_me] = excl;
    if (blockIdx.x == 0) offsets[e_me] = excl;
  }
  if (blockIdx.x == 0 && e_me == N - 1) {
    offsets[N] = excl + padded;
    offsets[N + 1] = excl + padded + (has_shared ? int32_t(round_up(T, kGroupAlign)) : 0);
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    // padding rows (-1): warp w takes experts w, w + kMidWarps, ..., its lanes the rows
    for (int e = warp; e < N; e += kMidWarps) {
      const int32_t r0 = off[e] + kp[e], r1 = off[e] + int32_t(round_up(kp[e], kGroupAlign));
      for (int32_t r = r0 + lane; r < r1; r += 32) row_token[r] = -1;
    }
  }
  const int a = blockIdx.x * kMidThreads + threadIdx.x;
  if (a < T * k) {
    const int32_t lr = lrank[a];
    int32_t row = -1;
    if (lr >= 0) {
      const int e = topk_idx[a];
      const int32_t rank = base[e] + lr;
      if (capacity <= 0 || rank < capacity) {
        row = off[e] + rank;
        row_token[row] = a / k;
      }
    }
    token_row[a] = row;
  }
}

size_t sort_smem_bytes(const moe_config& c) {
  const int64_t A = c.T * c.top_k;
  return size_t(kSortWarps * c.n_experts + 3 * c.n_experts + 32) * 4 + size_t(A) * 4 + 16;
}

constexpr int kSortSmemMax = 190 * 1024;

// Above ~16K assignments the multi-block histogram path is faster.
bool single_block_sort_fits(const moe_config& c) {
  return c.n_experts <= kSortWarps * 32 && c.T * c.top_k <= 16384 &&
         sort_smem_bytes(c) <= size_t(kSortSmemMax);
}

// The two-launch path, from kMidMinAssign assignments up to kMidMaxBlocks
// blocks (every scatter block reads all blocks' counts): it spreads the sort
// over several SMs.  Its per-warp counts take kMidWarps * N ints of shared
// memory, at most the 48 KB a launch gets without opting in.
constexpr int64_t kMidMinAssign = 2048;
constexpr int64_t kMidMaxBlocks = 64;
constexpr int64_t kMidMaxExperts = 48 * 1024 / (kMidWarps * 4);

inline int64_t mid_blocks(const moe_config& c) {
  return ceil_div(c.T * c.top_k, kMidThreads);
}

bool mid_sort_used(const moe_config& c) {
  return c.n_experts <= kMidMaxExperts && c.T * c.top_k >= kMidMinAssign &&
         mid_blocks(c) <= kMidMaxBlocks;
}

// Lets permute_sort_kernel take up to kSortSmemMax of dynamic shared memory:
// set once per device and context rather than on every launch.
cudaError_t allow_sort_smem() {
  static std::mutex mu;
  static uint64_t done_ctx[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  const uint64_t ctx = context_id();
  if (ctx != 0 && done_ctx[dev] == ctx) return cudaSuccess;
  e = cudaFuncSetAttribute(permute_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSortSmemMax);
  if (e == cudaSuccess) done_ctx[dev] = context_id();
  return e;
}

template <typename T>
__global__ void __launch_bounds__(256)
    permute_copy_kernel(const T* __restrict__ x, int64_t d, int Ttok, int N,
                        const int32_t* __restrict__ offsets,
                        const int32_t* __restrict__ row_token, T* __restrict__ Xp,
                        int32_t* __restrict__ zero, int64_t n_zero, int64_t rows_max) {
  pdl_launch_dependents();
  pdl_wait_previous();
  // counters the next kernels count up from zero (the grouped FFN's split tiles)
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n_zero;
       i += int64_t(gridDim.x) * blockDim.x)
    zero[i] = 0;
  const int lane = threadIdx.x & 31;
  const int64_t routed_end = offsets[N], total = offsets[N + 1];
  if (blockIdx.x == 0 && threadIdx.x == 0) MOE_CHECK(total <= rows_max, CK_ROWS_TOTAL);
  const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
  constexpr int V = Vec16<T>::n;
  for (int64_t r = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); r < total;
       r += warps) {
    int64_t t;
    if (r < routed_end) {
      t = row_token[r];
    } else {
      t = r - routed_end;
      if (t >= Ttok) t = -1;
    }
    MOE_CHECK(t >= -1 && t < Ttok, CK_COPY_TOKEN);
    if (t < 0 || t >= Ttok) continue;             // padding row (or no such token)
    const uint4* src = reinterpret_cast<const uint4*>(x + t * d);
    uint4* dst = reinterpret_cast<uint4*>(Xp + r * d);
    const int64_t nv = d / V;
    int64_t i = lane;
    for (; i + 7 * 32 < nv; i += 8 * 32) {          // eight 16-byte loads in flight
      uint4 a[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) a[u] = __ldg(src + i + 32 * u);
#pragma unroll
      for (int u = 0; u < 8; ++u) dst[i + 32 * u] = a[u];
    }
    for (; i < nv; i += 32) dst[i] = __ldg(src + i);
  }
}

}  // namespace

size_t permute_scratch_bytes(const moe_config& c) {
  // the two-launch sort: [mid_blocks][N] counts, then [T * k] ranks
  if (mid_sort_used(c))
    return size_t(round_up(mid_blocks(c) * c.n_experts, 64) + c.T * c.top_k) * sizeof(int32_t);
  // the histogram path: per-block counts and bases
  const int64_t n = permute_blocks(c) * c.n_experts;
  return size_t(2 * round_up(n, 64)) * sizeof(int32_t);
}

namespace {

cudaError_t launch_copy(const moe_config& c, const void* x, const int32_t* offsets,
                        const int32_t* row_token, void* Xp, int64_t rows_max, cudaStream_t s,
                        int32_t* zero = nullptr, int64_t n_zero = 0) {
  if (rows_max <= 0) return cudaSuccess;
  const int N = int(c.n_experts), T = int(c.T);
  const int64_t want = ceil_div(rows_max, 8);
  const unsigned blocks = unsigned(want < 148 * 8 ? want : 148 * 8);
  if (!zero) n_zero = 0;
  if (c.dtype == MOE_F32)
    return launch_pdl(permute_copy_kernel<float>, dim3(blocks), dim3(256), 0, s,
                      static_cast<const float*>(x), c.d_model, T, N, offsets, row_token,
                      static_cast<float*>(Xp), zero, n_zero, rows_max);
  return launch_pdl(permute_copy_kernel<__nv_bfloat16>, dim3(blocks), dim3(256), 0, s,
                    static_cast<const __nv_bfloat16*>(x), c.d_model, T, N, offsets,
                    row_token, static_cast<__nv_bfloat16*>(Xp), zero, n_zero, rows_max);
}

}  // namespace

cudaError_t launch_row_copy(const moe_config& c, const void* x, const int32_t* offsets,
                            const int32_t* row_token, void* Xp, int64_t rows_max,
                            cudaStream_t s, int32_t* zero, int64_t n_zero) {
  return launch_copy(c, x, offsets, row_token, Xp, rows_max, s, zero, n_zero);
}

int permute_launch_count(const moe_config& c) {
  const int copy = moe::rows_max_for(c) > 0 ? 1 : 0;
  if (mid_sort_used(c)) return 2 + copy;
  if (single_block_sort_fits(c)) return 1 + copy;
  return (c.T > 0 ? 3 : 1) + copy;
}

bool permute_fuses_stats(const moe_config& c) {
  return mid_sort_used(c) || single_block_sort_fits(c);
}

cudaError_t launch_permute(const moe_config& c, const void* x, const int32_t* topk_idx,
                           int32_t* counts, int32_t* kept, int32_t* offsets,
                           int32_t* row_token, int32_t* token_row, void* Xp, void* scratch,
                           int64_t rows_max, cudaStream_t s, const StatsArgs* stats,
                           int32_t* zero, int64_t n_zero) {
  const int N = int(c.n_experts), k = int(c.top_k), T = int(c.T);
  const int nblk = int(permute_blocks(c));
  PermuteScratch p = carve(c, scratch);
  const size_t smemN = size_t(N) * sizeof(int32_t);
  cudaError_t e;
  if (mid_sort_used(c)) {
    const int A = T * k;
    const int mb = int(mid_blocks(c));
    int32_t* mcounts = static_cast<int32_t*>(scratch);
    int32_t* lrank = mcounts + round_up(int64_t(mb) * N, 64);
    e = launch_pdl(permute_mid_rank_kernel, dim3(mb), dim3(kMidThreads),
                   size_t(kMidWarps) * N * sizeof(int32_t), s, topk_idx, A, N, mcounts, lrank);
    if (e != cudaSuccess) return e;
    const StatsArgs none{};
    const bool with_stats = stats && stats->prob_partials;
    e = launch_pdl(permute_mid_scatter_kernel, dim3(mb + (with_stats ? 1 : 0)),
                   dim3(kMidThreads), size_t(3) * N * sizeof(int32_t), s,
                   static_cast<const int32_t*>(topk_idx), static_cast<const int32_t*>(lrank),
                   static_cast<const int32_t*>(mcounts), mb, T, k, N, c.capacity,
                   c.d_ff_shared > 0 ? 1 : 0, counts, kept, offsets, row_token, token_row,
                   with_stats ? *stats : none);
    if (e != cudaSuccess) return e;
    return launch_copy(c, x, offsets, row_token, Xp, rows_max, s, zero, n_zero);
  }
  if (single_block_sort_fits(c)) {
    const size_t smem = sort_smem_bytes(c);
    e = allow_sort_smem();
    if (e != cudaSuccess) return e;
    const StatsArgs none{};
    e = launch_pdl(permute_sort_kernel, dim3(1), dim3(kSortWarps * 32), smem, s, topk_idx, T, k,
                   N, c.capacity, c.d_ff_shared > 0 ? 1 : 0, counts, kept, offsets, row_token,
                   token_row, stats ? *stats : none);
    if (e != cudaSuccess) return e;
    return launch_copy(c, x, offsets, row_token, Xp, rows_max, s, zero, n_zero);
  }
  if (nblk > 0) {
    e = launch_pdl(permute_hist_kernel, dim3(nblk), dim3(256), smemN, s, topk_idx, T, k, N,
                   p.block_counts);
    if (e != cudaSuccess) return e;
  }
  e = launch_pdl(permute_scan_kernel, dim3(1), dim3(1024), 0, s, p.block_counts, nblk, N, T,
                 c.capacity, c.d_ff_shared > 0 ? 1 : 0, p.block_base, counts, kept, offsets,
                 row_token);
  if (e != cudaSuccess) return e;
  if (nblk > 0) {
    e = launch_pdl(permute_rank_kernel, dim3(nblk), dim3(32), smemN, s, topk_idx, T, k, N,
                   c.capacity, p.block_base, offsets, row_token, token_row);
    if (e != cudaSuccess) return e;
  }
  return launch_copy(c, x, offsets, row_token, Xp, rows_max, s, zero, n_zero);
}

}  // namespace moe

// ---- moe_permute_noalloc: the same step with its scratch in a fixed array ---------------
//
// For callers that cannot allocate device memory.  The per-block histograms
// and bases live in this file-scope array (1 MiB on every GPU that loads the
// library).  Host code must not pass the array's name to a kernel -- on the
// host it is only a stand-in symbol -- so each device's address is looked up
// once with cudaGetSymbolAddress, with that device current, and passed in.

static __device__ __align__(256) int32_t g_permute_static_scratch[MOE_PERMUTE_STATIC_SCRATCH_INTS];

namespace moe {
namespace {

constexpr int kMaxDevices = 64;
std::mutex g_static_scratch_mu;
void* g_static_scratch_addr[kMaxDevices] = {};
uint64_t g_static_scratch_ctx[kMaxDevices] = {};

// Device address of the array for the current device, looked up on the
// device's first use and again whenever the device's context has changed
// (for example after cudaDeviceReset), since the address belongs to one context.
cudaError_t static_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_static_scratch_mu);
  const uint64_t ctx = context_id();
  if (g_static_scratch_addr[dev] == nullptr || (ctx != 0 && ctx != g_static_scratch_ctx[dev])) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_permute_static_scratch);
    if (e != cudaSuccess) return e;
    g_static_scratch_addr[dev] = p;
    g_static_scratch_ctx[dev] = context_id();
  }
  *out = g_static_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_permute_noalloc(const moe_config* cfg, const void* x,
                                          const int32_t* topk_idx, int32_t* counts,
                                          int32_t* kept, int32_t* offsets, int32_t* row_token,
                                          int32_t* token_row, void* Xp, void* stream) {
  using namespace moe;
  moe_status st = validate_config(cfg);
  if (st != MOE_OK) return st;
  const void* ps[] = {x, topk_idx, counts, kept, offsets, row_token, token_row, Xp};
  for (const void* q : ps)
    if (!q || (reinterpret_cast<uintptr_t>(q) & 15u) != 0) return MOE_ERR_INVALID_ARG;
  if (permute_scratch_bytes(*cfg) > size_t(MOE_PERMUTE_STATIC_SCRATCH_INTS) * sizeof(int32_t))
    return MOE_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (static_scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  const cudaError_t e = launch_permute(*cfg, x, topk_idx, counts, kept, offsets, row_token,
                                       token_row, Xp, scratch, rows_max_for(*cfg),
                                       static_cast<cudaStream_t>(stream), nullptr, nullptr, 0);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

namespace moe {
MOE_CHECKS_UNIT(permute)
}  // namespace moe
