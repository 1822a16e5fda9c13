// bf16 expert FFN on the 5th-generation tensor cores (tcgen05 + TMEM, fed by
// TMA), sm_103a.
//
//   H  = act(Xp[group e] . W1[e]^T + b1[e])     (first Linear + activation)
//   Yp = H[group e] . W2[e]^T + b2[e]             (second Linear)
//
// per expert group e (botmartz.com "Mixture of Experts (MoE) and Mixtral",
// "Expert Routing": each expert is Linear(d_model, d_ff) -> GELU ->
// Linear(d_ff, d_model); codingnowai.in "Mixture of Experts", "Code": ReLU).
//
// One persistent kernel per Linear.  The output tiles of all groups form one
// list -- group by group, within a group the n-tiles outermost and the m-tiles
// innermost, so CTAs working at the same time share a weight tile in L2 --
// and CTA b takes tiles b, b + gridDim.x, ...  Roles inside a CTA:
//   warp 0      TMA producer: A tile [128 x 64] and B tile [BN x 64] per
//               k-block into a kStages-deep shared-memory ring (128B swizzle)
//   warp 1      allocates TMEM; one thread issues tcgen05.mma
//               (M=128, N=BN, K=16, bf16 x bf16 -> fp32) into one of two TMEM
//               accumulators and commits to the ring's "empty" barriers
//   warps 2-17  epilogue: tcgen05.ld the accumulator (four warps per TMEM
//               lane quarter, each a quarter of the columns), + bias,
//               activation, bf16, store the live rows; then free the
//               accumulator
// Double-buffered accumulators let the epilogue of one tile overlap the
// main loop of the next.  Every wait is bounded (a time limit, then the
// device status word records MOE_ERR_TIMEOUT and the CTA winds down).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <float.h>
#include <mutex>

#include "kernels.h"
#include "common.cuh"
#include "tc_common.cuh"

namespace moe {
namespace {

constexpr int BM = 128;                 // rows per tile = TMEM lanes
constexpr int BK = 64;                  // 64 bf16 = 128 B = one swizzle row
constexpr int kMaxGroups = 1025;        // 1024 routed + 1 shared

// Epilogues: + bias then bf16 (second Linear), + bias, GELU / ReLU then bf16
// (first Linear), + bias then fp32 (router scores).
enum { EPI_BIAS = 0, EPI_BIAS_GELU = 1, EPI_BIAS_RELU = 2, EPI_BIAS_F32 = 3,
       // backward dgrad on the CTA pair (weights as MN-major B): no bias; the
       // result times the activation's derivative at TcParams::pre, or as is
       EPI_DGRAD_GELU = 4, EPI_DGRAD_RELU = 5, EPI_DGRAD = 6,
       // router scores of 64 experts (one 64-wide tile per row): + bias, fp32
       // scores out, then the softmax, top-k and gates of each row and the
       // tile's column sums of p
       EPI_ROUTER_TOPK = 7 };
constexpr bool epi_is_dgrad(int e) { return e >= EPI_DGRAD_GELU && e <= EPI_DGRAD; }

// A kernel variant: output tile width BN, depth of the shared-memory ring,
// number of epilogue warps (a multiple of 4: one set per TMEM lane quarter).
// STAGED: the epilogue's bf16 stores go through shared memory (16-column
// pieces, warp_staged_store).
// EXTRA: more shared memory for the epilogue (the router's reductions).
template <int BN_, int STAGES_, int EPI_WARPS_, bool STAGED_ = true, int EXTRA_ = 0>
struct TileCfg {
  static constexpr int BN = BN_;
  static constexpr int STAGES = STAGES_;
  static constexpr int EPI_WARPS = EPI_WARPS_;
  static constexpr int THREADS = (2 + EPI_WARPS) * 32;
  static constexpr bool STAGED = STAGED_;
  static constexpr int STAGE_BYTES =
      (STAGED_ ? EPI_WARPS_ * staged_warp_bytes<16>() : 0) + EXTRA_;
};

template <int BN, int STAGES, int STAGE_BYTES = 0>
struct Layout {
  static constexpr int kABytes = BM * BK * 2;
  static constexpr int kBBytes = BN * BK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kA = 0;
  static constexpr int kB = STAGES * kABytes;
  static constexpr int kBar = kB + STAGES * kBBytes;        // full[S], empty[S], tfull[2], tempty[2], done
  static constexpr int kNumBars = 2 * STAGES + 5;
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kTileStart = (kAbort + 4 + 15) / 16 * 16;   // int32 [kMaxGroups + 1]
  static constexpr int kGroupOff = kTileStart + (kMaxGroups + 1) * 4;  // int32 [kMaxGroups]
  static constexpr int kStage = (kGroupOff + kMaxGroups * 4 + 127) / 128 * 128;
  static constexpr int kBytes = kStage + STAGE_BYTES;
  static constexpr int kAlloc = kBytes + 1024;              // room to align the base to 1 KB
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

struct TcParams {
  const int32_t* offsets;          // [n_groups + 1] first row of each group; nullptr:
                                   // one group of dense_rows rows starting at row 0
  const int32_t* kept;             // [n_routed] live rows of each routed group
  const __nv_bfloat16* pre;        // dgrad epilogues: the pre-activation [rows, Nd]
  // first Linear with an activation, staged tiles: also store the
  // pre-activation (bias added, before the activation) here, [rows, Nd]
  void* out_pre;
  const __nv_bfloat16* bias;       // [n_routed, Nd]
  const __nv_bfloat16* bias_s;     // [Nd] shared expert
  void* out;                       // [rows, Nd], bf16 (fp32 for EPI_BIAS_F32)
  int64_t Nd;
  int32_t n_routed;
  int32_t shared_rows;             // live rows of the shared group; 0 = none
  int32_t dense_rows;              // rows of the single group when offsets == nullptr
  int32_t num_kb;                  // K / BK
  int32_t* status;
  uint64_t wait_limit_ns;
  int64_t rows_total;              // rows of the grouped buffers (device checks; 0: unknown)
  // token-column tiles, stream-K (both nullptr: whole tiles): [kSkMaxCtas][nb][128]
  // fp32 partial accumulators and one counter per tile, 0 at launch
  float* sk_partials;
  int32_t* sk_counters;
  // token-column tiles: token columns per tile and depth of the ring
  int32_t sw_nb, sw_stages;
  // EPI_ROUTER_TOPK: [rows, k] experts and gates, [m-tiles, 64] column sums of p
  int32_t* topk_idx;
  float* topk_w;
  float* prob_rows;
  int32_t top_k, renorm;
};

// Epilogue of CW accumulator columns of one row: + bias, activation, store.
template <int EPI, int CW>
__device__ __forceinline__ void epilogue_store(const uint32_t (&r)[CW],
                                               const __nv_bfloat16* __restrict__ bias,
                                               void* out_row_col) {
  const uint4* bsrc = reinterpret_cast<const uint4*>(bias);
  if constexpr (EPI == EPI_BIAS_F32) {
    float4* dst = reinterpret_cast<float4*>(out_row_col);
#pragma unroll
    for (int v = 0; v < CW / 8; ++v) {
      const uint4 bv = __ldg(bsrc + v);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&bv);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float2 b0 = __bfloat1622float2(b2[2 * i]);
        const float2 b1 = __bfloat1622float2(b2[2 * i + 1]);
        dst[2 * v + i] = make_float4(__uint_as_float(r[8 * v + 4 * i]) + b0.x,
                                     __uint_as_float(r[8 * v + 4 * i + 1]) + b0.y,
                                     __uint_as_float(r[8 * v + 4 * i + 2]) + b1.x,
                                     __uint_as_float(r[8 * v + 4 * i + 3]) + b1.y);
      }
    }
  } else {
    uint4* dst = reinterpret_cast<uint4*>(out_row_col);
#pragma unroll
    for (int v = 0; v < CW / 8; ++v) {
      const uint4 bv = __ldg(bsrc + v);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&bv);
      uint4 o;
      __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 bf = __bfloat1622float2(b2[i]);
        float x0 = __uint_as_float(r[8 * v + 2 * i]) + bf.x;
        float x1 = __uint_as_float(r[8 * v + 2 * i + 1]) + bf.y;
        if (EPI == EPI_BIAS_GELU) { x0 = gelu_erf(x0); x1 = gelu_erf(x1); }
        if (EPI == EPI_BIAS_RELU) { x0 = fmaxf(x0, 0.f); x1 = fmaxf(x1, 0.f); }
        o2[i] = __floats2bfloat162_rn(x0, x1);
      }
      dst[v] = o;
    }
  }
}

// The bf16 epilogues as 16-byte words: + bias, activation, bf16 of CW columns.
template <int EPI, int CW>
__device__ __forceinline__ void epilogue_words(const uint32_t* r,
                                               const __nv_bfloat16* __restrict__ bias,
                                               uint4 (&w)[CW / 8]) {
  const uint4* bsrc = reinterpret_cast<const uint4*>(bias);
#pragma unroll
  for (int v = 0; v < CW / 8; ++v) {
    const uint4 bv = __ldg(bsrc + v);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&bv);
    __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&w[v]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 bf = __bfloat1622float2(b2[i]);
      float x0 = __uint_as_float(r[8 * v + 2 * i]) + bf.x;
      float x1 = __uint_as_float(r[8 * v + 2 * i + 1]) + bf.y;
      if (EPI == EPI_BIAS_GELU) { x0 = gelu_erf(x0); x1 = gelu_erf(x1); }
      if (EPI == EPI_BIAS_RELU) { x0 = fmaxf(x0, 0.f); x1 = fmaxf(x1, 0.f); }
      o2[i] = __floats2bfloat162_rn(x0, x1);
    }
  }
}

// The dgrad epilogues as 16-byte words: bf16(acc * act'(pre)) (or bf16(acc)),
// zeros for a padding row.
template <int EPI, int CW>
__device__ __forceinline__ void dgrad_words(const uint32_t* r, const __nv_bfloat16* pre,
                                            bool zero, uint4 (&w)[CW / 8]) {
#pragma unroll
  for (int v = 0; v < CW / 8; ++v) {
    if (zero) {
      w[v] = make_uint4(0, 0, 0, 0);
      continue;
    }
    float gr[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) gr[i] = 1.f;
    if (EPI != EPI_DGRAD) {
      const uint4 pv = __ldg(reinterpret_cast<const uint4*>(pre) + v);
      const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&pv);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 a = __bfloat1622float2(p2[i]);
        gr[2 * i] = EPI == EPI_DGRAD_GELU ? gelu_erf_grad(a.x) : (a.x > 0.f ? 1.f : 0.f);
        gr[2 * i + 1] = EPI == EPI_DGRAD_GELU ? gelu_erf_grad(a.y) : (a.y > 0.f ? 1.f : 0.f);
      }
    }
    __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&w[v]);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      o2[i] = __floats2bfloat162_rn(__uint_as_float(r[8 * v + 2 * i]) * gr[2 * i],
                                    __uint_as_float(r[8 * v + 2 * i + 1]) * gr[2 * i + 1]);
  }
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major.
template <int BN>
__host__ __device__ constexpr uint32_t idesc_bf16_f32() {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) |
         (uint32_t(BM >> 4) << 24);
}

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              const TcParams& p, volatile int* abort_flag) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(a, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > p.wait_limit_ns) {
        atomicCAS(p.status, MOE_OK, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

struct TileCoord {
  int g, m, n;
};

// Largest group g with tile_start[g] <= tile (non-empty by construction).
__device__ __forceinline__ TileCoord decode_tile(int tile, const int32_t* tile_start,
                                                 int n_groups, int ntiles) {
  int lo = 0, hi = n_groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  const int local = tile - tile_start[lo];
  const int mt = (tile_start[lo + 1] - tile_start[lo]) / ntiles;
  return TileCoord{lo, local % mt, local / mt};
}

__device__ __forceinline__ int32_t ld_acquire_gpu(const int32_t* p) {
  int32_t v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Stream-K over the token-column tiles.  A layer's token-column tiles are few
// and long (for a Mixtral-sized decode, 256 tiles of 224 k-blocks in the second
// Linear), so whole tiles per CTA leave the last wave of 148 CTAs partly idle.
// Instead every CTA takes an equal share of all tiles' k-blocks -- units
// [b * upc, (b + 1) * upc) of total_tiles * num_kb -- so each streams the same
// number of weight bytes.  A tile cut by share boundaries is finished by the
// CTA holding its first k-block: there the piece is the last of the CTA's
// share, while every other piece of the tile begins its CTA's share and is
// computed first.  Those CTAs write their fp32 partial accumulators to their
// slot and count themselves on the tile's counter; the finishing CTA waits
// for the count (bounded), adds the pieces to its own accumulator in k order
// (deterministic) and runs the epilogue.
constexpr int kSkMaxCtas = 256;

struct SegIter {
  int64_t u = 0, u1 = 0;
  int t, stride, total, nkb;
  bool sk;
  __device__ SegIter(bool sk_, int b, int G, int total_, int nkb_, int64_t upc)
      : t(b), stride(G), total(total_), nkb(nkb_), sk(sk_) {
    if (sk) {
      u = int64_t(b) * upc;
      const int64_t U = int64_t(total_) * nkb_;
      u1 = u + upc < U ? u + upc : U;
    }
  }
  // the next (tile, [kb0, kb1)) of this CTA
  __device__ bool next(int& tile, int& kb0, int& kb1) {
    if (sk) {
      if (u >= u1) return false;
      tile = int(u / nkb);
      kb0 = int(u - int64_t(tile) * nkb);
      const int64_t rest = u1 - u;
      kb1 = rest < int64_t(nkb - kb0) ? kb0 + int(rest) : nkb;
      u += kb1 - kb0;
      return true;
    }
    if (t >= total) return false;
    tile = t;
    kb0 = 0;
    kb1 = nkb;
    t += stride;
    return true;
  }
};

// Barrier of the epilogue warps only (named barrier 1).
__device__ __forceinline__ void epi_bar_sync(int threads = 128) {
  asm volatile("bar.sync 1, %0;" ::"r"(threads) : "memory");
}

// EPI_ROUTER_TOPK, run by the sixteen epilogue warps (CfgRouter): warp
// (part, q) holds TMEM lane quarter q (32 token rows, thread = row) and score
// columns [16 part, 16 part + 16), so that a row's 64 scores are spread over
// four threads and each warp's code is short.  Per row: the scores + bias,
// written as fp32; the maximum and the sum of exp(z - max) from the four
// parts' partials (added in part order); the top k -- each part selects its
// own k best (the larger score first, then the lower expert, as in the other
// router kernels), and part 0 merges the four lists in the same order -- and
// the gates; then the tile's column sums of p: a reduce-scatter across each
// warp's lanes (lane l ends with column 16 part + l / 2), the four quarters
// added in order, written as row m of p.prob_rows.  Rows past the live ones
// add 0.  `red` holds RouterRed.
constexpr int kRouterParts = 4;
constexpr int kRouterMaxK = 8;
struct RouterRed {
  float mx[kRouterParts][128];
  float sum[kRouterParts][128];
  float cand_v[kRouterParts][kRouterMaxK][128];
  uint8_t cand_e[kRouterParts][kRouterMaxK][128];
  float col[4][64];
};

__device__ __forceinline__ void router_topk_rows(const TcParams& p, uint32_t taddr,
                                                 const __nv_bfloat16* __restrict__ bias,
                                                 int row, bool valid, int m, int q, int part,
                                                 int lane, RouterRed* red, int epi_threads) {
  constexpr int NE = 64, NP = 16;
  const int c0 = part * NP;
  const int rl = q * 32 + lane;                  // row within the tile
  float z[NP];
  {
    uint32_t r[NP];
    tmem_ld_16cols(taddr + uint32_t(c0), r);
    const uint4* bsrc = reinterpret_cast<const uint4*>(bias + c0);
#pragma unroll
    for (int v = 0; v < NP / 8; ++v) {
      const uint4 bv = __ldg(bsrc + v);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&bv);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 bf = __bfloat1622float2(b2[i]);
        z[8 * v + 2 * i] = __uint_as_float(r[8 * v + 2 * i]) + bf.x;
        z[8 * v + 2 * i + 1] = __uint_as_float(r[8 * v + 2 * i + 1]) + bf.y;
      }
    }
  }
  if (valid) {
    float4* zo = reinterpret_cast<float4*>(static_cast<float*>(p.out) + int64_t(row) * NE + c0);
#pragma unroll
    for (int v = 0; v < NP / 4; ++v)
      zo[v] = make_float4(z[4 * v], z[4 * v + 1], z[4 * v + 2], z[4 * v + 3]);
  }
  float mp = -FLT_MAX;
#pragma unroll
  for (int i = 0; i < NP; ++i) mp = fmaxf(mp, z[i]);
  red->mx[part][rl] = mp;
  // this part's k best, in selection order
  const int k = p.top_k;
  uint32_t taken = 0;
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int be = 0xff;
#pragma unroll
    for (int i = 0; i < NP; ++i)
      if (!((taken >> i) & 1u) && (z[i] > bv || (z[i] == bv && c0 + i < be))) {
        bv = z[i];
        be = c0 + i;
      }
    if (be < NE) taken |= 1u << (be - c0);
    red->cand_v[part][j][rl] = bv;
    red->cand_e[part][j][rl] = uint8_t(be);
  }
  epi_bar_sync(epi_threads);
  const float mx = fmaxf(fmaxf(red->mx[0][rl], red->mx[1][rl]),
                         fmaxf(red->mx[2][rl], red->mx[3][rl]));
  float sp = 0.f;
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    z[i] = expf(z[i] - mx);                      // z now holds exp(z - max)
    sp += z[i];
  }
  red->sum[part][rl] = sp;
  epi_bar_sync(epi_threads);
  const float ssum = ((red->sum[0][rl] + red->sum[1][rl]) + red->sum[2][rl]) + red->sum[3][rl];
  const float inv = 1.0f / ssum;
  if (part == 0) {
    // merge the four parts' lists: k rounds over the list heads
    int h0 = 0, h1 = 0, h2 = 0, h3 = 0;
    float kept_sum = 0.f;
#pragma unroll 1
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int be = 0x7fffffff, bp = -1;
#pragma unroll
      for (int pp = 0; pp < kRouterParts; ++pp) {
        const int h = pp == 0 ? h0 : pp == 1 ? h1 : pp == 2 ? h2 : h3;
        if (h >= k) continue;
        const float v = red->cand_v[pp][h][rl];
        const int e = red->cand_e[pp][h][rl];
        if (v > bv || (v == bv && e < be)) {
          bv = v;
          be = e;
          bp = pp;
        }
      }
      h0 += bp == 0; h1 += bp == 1; h2 += bp == 2; h3 += bp == 3;
      const float g = expf(bv - mx);
      kept_sum += g;
      if (valid) {
        MOE_CHECK(be >= 0 && be < NE, CK_ROUTER_TOPK);
        p.topk_idx[int64_t(row) * k + j] = be;
        p.topk_w[int64_t(row) * k + j] = g;      // unnormalised for now
      }
    }
    if (valid) {
      const float scale = p.renorm ? 1.0f / kept_sum : inv;
#pragma unroll 1
      for (int j = 0; j < k; ++j) p.topk_w[int64_t(row) * k + j] *= scale;
    }
  }
  // column sums of p over the tile's rows: reduce-scatter across the lanes
#pragma unroll
  for (int i = 0; i < NP; ++i) z[i] = valid ? z[i] * inv : 0.f;
#pragma unroll
  for (int step = 0; step < 4; ++step) {
    const int o = 16 >> step;
    const int S = NP >> step;                    // values still held per lane
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < S / 2; ++i) {
      const float send = upper ? z[i] : z[i + S / 2];
      const float keep = upper ? z[i + S / 2] : z[i];
      z[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  z[0] += __shfl_xor_sync(0xffffffffu, z[0], 1);
  if ((lane & 1) == 0) red->col[q][c0 + (lane >> 1)] = z[0];
  epi_bar_sync(epi_threads);
  if (part == 0) {
    const int e = q * 32 + lane;
    if (e < NE)
      p.prob_rows[int64_t(m) * NE + e] =
          ((red->col[0][e] + red->col[1][e]) + red->col[2][e]) + red->col[3][e];
  }
  epi_bar_sync(epi_threads);                     // red is read before the next tile
}

template <class CFG, int EPI, int MINB>
__global__ void __launch_bounds__(CFG::THREADS, MINB)
    tc_grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmBs, const TcParams p) {
  constexpr int BN = CFG::BN;
  constexpr int kStages = CFG::STAGES;
  constexpr int kEpiWarps = CFG::EPI_WARPS;
  using L = Layout<BN, kStages, CFG::STAGE_BYTES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = bars + 2 * kStages + 2;
  uint64_t* done = bars + 2 * kStages + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  int32_t* tile_start = reinterpret_cast<int32_t*>(smem + L::kTileStart);
  int32_t* grp_off = reinterpret_cast<int32_t*>(smem + L::kGroupOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_groups = p.offsets ? p.n_routed + (p.shared_rows > 0 ? 1 : 0) : 1;
  const int ntiles = int(p.Nd / BN);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kEpiWarps);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(2 * BN));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // the next launch may start once this CTA holds its TMEM; global memory is
  // touched only after the previous kernel has completed
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait_previous();
  if (warp == 2) {
    // tile_start[g] = sum over earlier groups of m-tiles x n-tiles (warp scan)
    int32_t carry = 0;
    for (int base = 0; base < n_groups; base += 32) {
      const int g = base + lane;
      int32_t live = 0, off = 0;
      if (g < n_groups) {
        if (p.offsets) {
          off = p.offsets[g];
          live = g < p.n_routed ? p.kept[g] : p.shared_rows;
        } else {
          live = p.dense_rows;
        }
        grp_off[g] = off;
      }
      const int32_t tiles = int32_t((live + BM - 1) / BM) * ntiles;
      int32_t incl = tiles;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (g < n_groups) tile_start[g] = carry + incl - tiles;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) tile_start[n_groups] = carry;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = tile_start[n_groups];

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int last_parity[kStages];
#pragma unroll
      for (int s = 0; s < kStages; ++s) last_parity[s] = -1;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        const TileCoord tc = decode_tile(tile, tile_start, n_groups, ntiles);
        const int row0 = grp_off[tc.g] + tc.m * BM;
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!wait_or_abort(&empty[stage], phase ^ 1u, p, abort_flag)) { ok = false; break; }
          const uint32_t fb = smem_u32(&full[stage]);
          mbar_arrive_expect_tx(&full[stage], L::kStageBytes);
          tma_load_2d(&tmA, smem_u32(smem + L::kA + stage * L::kABytes), fb, kb * BK, row0);
          if (tc.g < p.n_routed)
            tma_load_3d(&tmB, smem_u32(smem + L::kB + stage * L::kBBytes), fb, kb * BK,
                        tc.n * BN, tc.g);
          else
            tma_load_2d(&tmBs, smem_u32(smem + L::kB + stage * L::kBBytes), fb, kb * BK,
                        tc.n * BN);
          last_parity[stage] = int(phase);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        // wind down: let copies already in flight land before the CTA exits
        for (int s = 0; s < kStages; ++s)
          if (last_parity[s] >= 0) {
            const uint32_t a = smem_u32(&full[s]);
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(a, uint32_t(last_parity[s])) &&
                   global_timer_ns() - t0 < p.wait_limit_ns) {
            }
          }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32<BN>();
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        if (!wait_or_abort(&tempty[acc], acc_phase ^ 1u, p, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!wait_or_abort(&full[stage], phase, p, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint64_t ad = sdesc_sw128(smem_u32(smem + L::kA + stage * L::kABytes));
          const uint64_t bd = sdesc_sw128(smem_u32(smem + L::kB + stage * L::kBBytes));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)   // +32 bytes along K per step
            tc_mma(d_tmem, ad + uint64_t(2 * kk), bd + uint64_t(2 * kk), idesc,
                   (kb | kk) != 0 ? 1u : 0u);
          tc_commit(smem_u32(&empty[stage]));
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(smem_u32(&tfull[acc]));
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      // every MMA issued by this thread has completed once `done` flips
      tc_commit(smem_u32(done));
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(smem_u32(done), 0) && global_timer_ns() - t0 < p.wait_limit_ns) {
      }
    }
  } else {
    // ---------------- epilogue ----------------
    const int q = warp & 3;                      // TMEM lane quarter of this warp
    const int part = (warp - 2) >> 2;            // which share of the tile's columns
    constexpr int kCols = BN / (kEpiWarps / 4);
    constexpr int CW = kCols < 32 ? kCols : 32;  // columns per tcgen05.ld
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      const TileCoord tc = decode_tile(tile, tile_start, n_groups, ntiles);
      bool ok = true;
      if (lane == 0) ok = wait_or_abort(&tfull[acc], acc_phase, p, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      tc_fence_after();
      const bool routed = tc.g < p.n_routed;
      const int live = p.offsets ? (routed ? p.kept[tc.g] : p.shared_rows) : p.dense_rows;
      if (warp == 2 && lane == 0)
        MOE_CHECK(p.rows_total == 0 || int64_t(grp_off[tc.g]) + live <= p.rows_total,
                  CK_GEMM_ROWS);
      const int row_in_group = tc.m * BM + q * 32 + lane;
      const bool valid = row_in_group < live;
      const int64_t out_row = int64_t(grp_off[tc.g]) + row_in_group;
      const __nv_bfloat16* bias = routed ? p.bias + int64_t(tc.g) * p.Nd : p.bias_s;
      constexpr int kOutBytes = EPI == EPI_BIAS_F32 ? 4 : 2;
      constexpr bool kStaged = CFG::STAGED && EPI != EPI_BIAS_F32;
      if constexpr (EPI == EPI_ROUTER_TOPK) {
        static_assert(kEpiWarps == 4 * kRouterParts && BN == 64, "router epilogue layout");
        router_topk_rows(p, tmem_base + (uint32_t(q * 32) << 16) + acc * BN, bias,
                         row_in_group, valid, tc.m, q, part, lane,
                         reinterpret_cast<RouterRed*>(smem + L::kStage), kEpiWarps * 32);
      } else
#pragma unroll 1
      for (int c = part * kCols; c < (part + 1) * kCols; c += CW) {
        uint32_t r[CW];
        tmem_ld_cols<CW>(tmem_base + (uint32_t(q * 32) << 16) + acc * BN + c, r);
        const int64_t col = int64_t(tc.n) * BN + c;
        if constexpr (kStaged) {
          uint8_t* stg = smem + L::kStage + (warp - 2) * staged_warp_bytes<16>();
          const int row_base = tc.m * BM + q * 32;
          __nv_bfloat16* out0 = static_cast<__nv_bfloat16*>(p.out) +
                                (int64_t(grp_off[tc.g]) + row_base) * p.Nd + col;
#pragma unroll
          for (int h = 0; h < CW / 16; ++h) {
            uint4 w[2];
            epilogue_words<EPI, 16>(r + 16 * h, bias + col + 16 * h, w);
            warp_staged_store<16>(w, stg, lane, out0 + 16 * h, p.Nd, live - row_base);
            if (EPI != EPI_BIAS && p.out_pre) {
              epilogue_words<EPI_BIAS, 16>(r + 16 * h, bias + col + 16 * h, w);
              warp_staged_store<16>(w, stg, lane,
                                    static_cast<__nv_bfloat16*>(p.out_pre) +
                                        (out0 - static_cast<__nv_bfloat16*>(p.out)) + 16 * h,
                                    p.Nd, live - row_base);
            }
          }
        } else if (valid) {
          epilogue_store<EPI, CW>(r, bias + col,
                                  static_cast<uint8_t*>(p.out) +
                                      (out_row * p.Nd + col) * kOutBytes);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(2 * BN));
  }
}

// ---- CTA-pair variant (tcgen05 cta_group::2) ---------------------------------------------
//
// A 256 x BN output tile is computed by a cluster of two CTAs on two SMs.
// Each CTA TMA-loads its own 128 rows of A and its half of the BN rows of B,
// so each SM's shared memory holds (and its tensor core reads) half of B: per
// k-block a CTA moves 32 KB through shared memory instead of 48 KB for the
// same tensor work, which is what lets the MMA run near its peak rate.  The
// even CTA of the pair issues the M=256 MMAs (cta_group::2); accumulator
// rows 0-127 land in its TMEM, rows 128-255 in the odd CTA's.  Barriers: the
// even CTA's "full" barrier counts both CTAs' arrivals and bytes; MMA commits
// are multicast to both CTAs' "empty" and "accumulator full" barriers; both
// CTAs' epilogue warps arrive on the even CTA's "accumulator empty" barrier.

template <int BN, int STAGES, int STAGE_BYTES = 0>
struct Layout2 {
  static constexpr int kABytes = 128 * BK * 2;          // this CTA's 128 rows of A
  static constexpr int kBBytes = (BN / 2) * BK * 2;     // this CTA's half of B
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kA = 0;
  static constexpr int kB = STAGES * kABytes;
  static constexpr int kBar = kB + STAGES * kBBytes;
  static constexpr int kNumBars = 2 * STAGES + 5;
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kTileStart = (kAbort + 4 + 15) / 16 * 16;
  static constexpr int kGroupOff = kTileStart + (kMaxGroups + 1) * 4;
  static constexpr int kStage = (kGroupOff + kMaxGroups * 4 + 127) / 128 * 128;
  static constexpr int kBytes = kStage + STAGE_BYTES;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t nclusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx_cluster(uint32_t bar_cluster, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cluster.b64 _, [%0], %1;" ::"r"(
                   bar_cluster),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

__device__ __forceinline__ void tma2_load_2d(const CUtensorMap* map, uint32_t dst, uint32_t bar,
                                             int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tma2_load_3d(const CUtensorMap* map, uint32_t dst, uint32_t bar,
                                             int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__device__ __forceinline__ void tc2_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// Arrives on the barrier at the same offset in both CTAs of the pair once all
// MMAs issued so far by this thread have completed.
__device__ __forceinline__ void tc2_commit_both(uint32_t bar) {
  const uint16_t mask = 0x3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

template <int BN>
__host__ __device__ constexpr uint32_t idesc2_bf16_f32() {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) |
         (uint32_t(256 >> 4) << 24);
}

template <class CFG, int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(CFG::THREADS, 1)
    tc2_grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmBs, const TcParams p) {
  constexpr int BN = CFG::BN;
  constexpr int kStages = CFG::STAGES;
  constexpr int kEpiWarps = CFG::EPI_WARPS;
  constexpr int BM2 = 256;
  using L = Layout2<BN, kStages, CFG::STAGE_BYTES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* full = bars;                       // used in CTA 0: both CTAs' loads
  uint64_t* empty = bars + kStages;            // per CTA: its ring slot is free
  uint64_t* tfull = bars + 2 * kStages;        // per CTA: accumulator ready
  uint64_t* tempty = bars + 2 * kStages + 2;   // used in CTA 0: both epilogues done
  uint64_t* done = bars + 2 * kStages + 4;     // CTA 0: all MMAs complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  int32_t* tile_start = reinterpret_cast<int32_t*>(smem + L::kTileStart);
  int32_t* grp_off = reinterpret_cast<int32_t*>(smem + L::kGroupOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int pair = int(cluster_id_x()), npairs = int(nclusters_x());
  const int n_groups = p.offsets ? p.n_routed + (p.shared_rows > 0 ? 1 : 0) : 1;
  const int ntiles = int(p.Nd / BN);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 2);                  // one arrival per CTA, with its bytes
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * kEpiWarps);    // every epilogue warp of both CTAs
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(2 * BN));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait_previous();
  if (warp == 2) {
    int32_t carry = 0;
    for (int base = 0; base < n_groups; base += 32) {
      const int g = base + lane;
      int32_t live = 0, off = 0;
      if (g < n_groups) {
        if (p.offsets) {
          off = p.offsets[g];
          live = g < p.n_routed ? p.kept[g] : p.shared_rows;
        } else {
          live = p.dense_rows;
        }
        grp_off[g] = off;
      }
      const int32_t tiles = int32_t((live + BM2 - 1) / BM2) * ntiles;
      int32_t incl = tiles;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (g < n_groups) tile_start[g] = carry + incl - tiles;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) tile_start[n_groups] = carry;
  }
  tc_fence_before();
  cluster_sync_all();                          // barriers of both CTAs are initialised
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = tile_start[n_groups];

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < total_tiles; tile += npairs) {
        const TileCoord tc = decode_tile(tile, tile_start, n_groups, ntiles);
        const int row0 = grp_off[tc.g] + tc.m * BM2 + int(rank) * 128;
        const int col0 = tc.n * BN + int(rank) * (BN / 2);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!wait_or_abort(&empty[stage], phase ^ 1u, p, abort_flag)) { ok = false; break; }
          const uint32_t fb = peer_addr(smem_u32(&full[stage]), 0);
          mbar_arrive_expect_tx_cluster(fb, L::kStageBytes);
          tma2_load_2d(&tmA, smem_u32(smem + L::kA + stage * L::kABytes), fb, kb * BK, row0);
          if constexpr (epi_is_dgrad(EPI)) {
            // the weight as stored, [K, Nd]: this CTA's BN / 2 columns as
            // 64-column boxes of 64 K-rows (MN-major)
            const uint32_t b_dst = smem_u32(smem + L::kB + stage * L::kBBytes);
#pragma unroll
            for (int c = 0; c < BN / 128; ++c) {
              if (tc.g < p.n_routed)
                tma2_load_3d(&tmB, b_dst + c * 8192, fb, col0 + 64 * c, kb * BK, tc.g);
              else
                tma2_load_2d(&tmBs, b_dst + c * 8192, fb, col0 + 64 * c, kb * BK);
            }
          } else if (tc.g < p.n_routed) {
            tma2_load_3d(&tmB, smem_u32(smem + L::kB + stage * L::kBBytes), fb, kb * BK, col0,
                         tc.g);
          } else {
            tma2_load_2d(&tmBs, smem_u32(smem + L::kB + stage * L::kBBytes), fb, kb * BK, col0);
          }
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (CTA 0 of the pair) ----------------
    if (lane == 0 && rank == 0) {
      // dgrad: B MN-major ("transpose B", bit 16)
      constexpr uint32_t idesc = idesc2_bf16_f32<BN>() | (epi_is_dgrad(EPI) ? (1u << 16) : 0u);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < total_tiles; tile += npairs) {
        if (!wait_or_abort(&tempty[acc], acc_phase ^ 1u, p, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!wait_or_abort(&full[stage], phase, p, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint64_t ad = sdesc_sw128(smem_u32(smem + L::kA + stage * L::kABytes));
          const uint32_t b_s = smem_u32(smem + L::kB + stage * L::kBBytes);
          const uint64_t bd = sdesc_sw128(b_s);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // MN-major B (dgrad): 64-column chunks 8 KB apart, +2 K groups per step
            const uint64_t bk = epi_is_dgrad(EPI) ? sdesc_mn_sw128(b_s + kk * 2048, 8192)
                                                  : bd + uint64_t(2 * kk);
            tc2_mma(d_tmem, ad + uint64_t(2 * kk), bk, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          tc2_commit_both(smem_u32(&empty[stage]));
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc2_commit_both(smem_u32(&tfull[acc]));
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      asm volatile(
          "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
              smem_u32(done))
          : "memory");
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(smem_u32(done), 0) && global_timer_ns() - t0 < p.wait_limit_ns) {
      }
    }
  } else {
    // ---------------- epilogue (both CTAs) ----------------
    const int q = warp & 3;
    const int part = (warp - 2) >> 2;
    constexpr int kCols = BN / (kEpiWarps / 4);
    constexpr int CW = kCols < 32 ? kCols : 32;
    const uint32_t tempty0 = peer_addr(smem_u32(&tempty[0]), 0);
    const uint32_t tempty1 = peer_addr(smem_u32(&tempty[1]), 0);
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = pair; tile < total_tiles; tile += npairs) {
      const TileCoord tc = decode_tile(tile, tile_start, n_groups, ntiles);
      bool ok = true;
      if (lane == 0) ok = wait_or_abort(&tfull[acc], acc_phase, p, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      tc_fence_after();
      const bool routed = tc.g < p.n_routed;
      const int live = p.offsets ? (routed ? p.kept[tc.g] : p.shared_rows) : p.dense_rows;
      if (warp == 2 && lane == 0)
        MOE_CHECK(p.rows_total == 0 || int64_t(grp_off[tc.g]) + live <= p.rows_total,
                  CK_GEMM_ROWS);
      const int row_in_group = tc.m * BM2 + int(rank) * 128 + q * 32 + lane;
      const bool valid = row_in_group < live;
      const int64_t out_row = int64_t(grp_off[tc.g]) + row_in_group;
      const __nv_bfloat16* bias = routed ? p.bias + int64_t(tc.g) * p.Nd : p.bias_s;
      constexpr int kOutBytes = EPI == EPI_BIAS_F32 ? 4 : 2;
      constexpr bool kStaged = CFG::STAGED && EPI != EPI_BIAS_F32;
#pragma unroll 1
      for (int c = part * kCols; c < (part + 1) * kCols; c += CW) {
        uint32_t r[CW];
        tmem_ld_cols<CW>(tmem_base + (uint32_t(q * 32) << 16) + acc * BN + c, r);
        const int64_t col = int64_t(tc.n) * BN + c;
        if constexpr (epi_is_dgrad(EPI)) {
          // live rows get the result, the group's padding rows (up to its
          // 128-row boundary, which a 256-row tile may pass) zeros
          uint8_t* stg = smem + L::kStage + (warp - 2) * staged_warp_bytes<16>();
          const int row_base = tc.m * BM2 + int(rank) * 128 + q * 32;
          const int padded = (live + 127) / 128 * 128;
          __nv_bfloat16* out0 = static_cast<__nv_bfloat16*>(p.out) +
                                (int64_t(grp_off[tc.g]) + row_base) * p.Nd + col;
          const __nv_bfloat16* pre_row = p.pre + out_row * p.Nd + col;
#pragma unroll
          for (int h = 0; h < CW / 16; ++h) {
            uint4 w[2];
            dgrad_words<EPI, 16>(r + 16 * h, pre_row + 16 * h, !valid, w);
            warp_staged_store<16>(w, stg, lane, out0 + 16 * h, p.Nd, padded - row_base);
          }
        } else if constexpr (kStaged) {
          uint8_t* stg = smem + L::kStage + (warp - 2) * staged_warp_bytes<16>();
          const int row_base = tc.m * BM2 + int(rank) * 128 + q * 32;
          __nv_bfloat16* out0 = static_cast<__nv_bfloat16*>(p.out) +
                                (int64_t(grp_off[tc.g]) + row_base) * p.Nd + col;
#pragma unroll
          for (int h = 0; h < CW / 16; ++h) {
            uint4 w[2];
            epilogue_words<EPI, 16>(r + 16 * h, bias + col + 16 * h, w);
            warp_staged_store<16>(w, stg, lane, out0 + 16 * h, p.Nd, live - row_base);
            if (EPI != EPI_BIAS && p.out_pre) {
              epilogue_words<EPI_BIAS, 16>(r + 16 * h, bias + col + 16 * h, w);
              warp_staged_store<16>(w, stg, lane,
                                    static_cast<__nv_bfloat16*>(p.out_pre) +
                                        (out0 - static_cast<__nv_bfloat16*>(p.out)) + 16 * h,
                                    p.Nd, live - row_base);
            }
          }
        } else if (valid) {
          epilogue_store<EPI, CW>(r, bias + col,
                                  static_cast<uint8_t*>(p.out) +
                                      (out_row * p.Nd + col) * kOutBytes);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc ? tempty1 : tempty0);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncwarp();
  cluster_sync_all();       // every remote arrive and every MMA of the pair has landed
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(2 * BN));
  }
}

// ---- token-column variant: the weights as the 128-row MMA operand ------------------------
//
// When an expert sees few tokens -- decoding, or a layer whose capacity caps
// every group at a few hundred rows -- a 128-row activation tile is mostly
// padding, and a weight tile is streamed once per 128-row m-tile of its group.
// Here the roles swap: each MMA takes 128 rows of the expert's weight matrix
// as its M=128 operand and up to nb of the group's token rows as its N operand
// (nb = 16, or a multiple of 32 up to 256).  The accumulator holds out^T for
// 128 output features x nb tokens; each epilogue thread owns one feature and
// writes it for every live token, 32 (or 16) tokens at a time.  Per k-block a
// CTA moves 16 KB of weights and nb x 128 B of activations; when nb covers the
// largest group, every weight byte is read once.

// Shared-memory layout of the token-column kernel for nb token columns and a
// ring of `stages` stages (1 KB-aligned base).
struct LayoutSw {
  int nb, stages;
  __host__ __device__ constexpr int w_bytes() const { return 128 * BK * 2; }
  __host__ __device__ constexpr int x_bytes() const { return nb * BK * 2; }
  __host__ __device__ constexpr int stage_bytes() const { return w_bytes() + x_bytes(); }
  __host__ __device__ constexpr int x_off() const { return stages * w_bytes(); }
  __host__ __device__ constexpr int bar_off() const { return x_off() + stages * x_bytes(); }
  __host__ __device__ constexpr int num_bars() const { return 2 * stages + 5; }
  __host__ __device__ constexpr int tmem_slot() const { return bar_off() + num_bars() * 8; }
  __host__ __device__ constexpr int abort_off() const { return tmem_slot() + 4; }
  __host__ __device__ constexpr int sk_last() const { return abort_off() + 4; }  // finishes the tile
  __host__ __device__ constexpr int sk_stop() const { return sk_last() + 4; }    // a warp gave up
  __host__ __device__ constexpr int tile_start() const { return (sk_stop() + 4 + 15) / 16 * 16; }
  __host__ __device__ constexpr int group_off() const { return tile_start() + (kMaxGroups + 1) * 4; }
  __host__ __device__ constexpr int alloc() const { return group_off() + kMaxGroups * 4 + 1024; }
  // TMEM columns: two accumulators of nb columns, a power of two >= 32
  __host__ __device__ constexpr uint32_t tmem_cols() const {
    return 2 * nb <= 32 ? 32u : 2 * nb <= 64 ? 64u : 2 * nb <= 128 ? 128u : 2 * nb <= 256 ? 256u : 512u;
  }
};
constexpr int kSwapMaxStages = 10;
constexpr int kSmemBudget = 227 * 1024;

__host__ __device__ constexpr uint32_t idesc_swap_bf16_f32(int nb) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(nb >> 3) << 17) |
         (uint32_t(128 >> 4) << 24);
}

// One chunk of CW token columns (tokens c0 .. c0 + CW - 1 of the tile) of a
// feature: + bias, activation, bf16 store of the live rows.
template <int EPI, int CW>
__device__ __forceinline__ void swap_store_chunk(const float (&v)[CW], float b, int c0,
                                                 int rows_left, __nv_bfloat16* out_col,
                                                 int64_t ld) {
#pragma unroll
  for (int i = 0; i < CW; ++i) {
    if (c0 + i < rows_left) {
      float o = v[i] + b;
      if (EPI == EPI_BIAS_GELU) o = gelu_erf(o);
      if (EPI == EPI_BIAS_RELU) o = fmaxf(o, 0.f);
      out_col[int64_t(c0 + i) * ld] = __float2bfloat16_rn(o);
    }
  }
}

// NBT: 16 for the 16-column decode tiles; 0 for p.sw_nb columns (a multiple
// of 32), handled 32 at a time.
template <int NBT, int EPI>
__global__ void __launch_bounds__(6 * 32, 1)
    tc_swap_gemm_kernel(const __grid_constant__ CUtensorMap tmW,
                        const __grid_constant__ CUtensorMap tmWs,
                        const __grid_constant__ CUtensorMap tmX, const TcParams p) {
  constexpr int kEpiWarps = 4;
  constexpr int kFeat = 128;                   // output features per tile
  constexpr int CW = NBT == 16 ? 16 : 32;      // token columns per epilogue chunk
  const int nb = NBT > 0 ? NBT : p.sw_nb;
  const int stages = p.sw_stages;
  const LayoutSw L{nb, stages};
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bar_off());
  uint64_t* full = bars;
  uint64_t* empty = bars + stages;
  uint64_t* tfull = bars + 2 * stages;
  uint64_t* tempty = bars + 2 * stages + 2;
  uint64_t* done = bars + 2 * stages + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.tmem_slot());
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.abort_off());
  int32_t* tile_start = reinterpret_cast<int32_t*>(smem + L.tile_start());
  int32_t* grp_off = reinterpret_cast<int32_t*>(smem + L.group_off());
  const uint32_t tmem_cols = L.tmem_cols();
  const int stage_bytes = L.stage_bytes();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_groups = p.n_routed + (p.shared_rows > 0 ? 1 : 0);
  const int ntiles = int(p.Nd / kFeat);

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kEpiWarps);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    *reinterpret_cast<volatile int*>(smem + L.sk_stop()) = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(tmem_cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // the next launch may start once this CTA holds its TMEM; global memory is
  // touched only after the previous kernel has completed
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait_previous();
  if (warp == 2) {
    int32_t carry = 0;
    for (int base = 0; base < n_groups; base += 32) {
      const int g = base + lane;
      int32_t live = 0, off = 0;
      if (g < n_groups) {
        off = p.offsets[g];
        live = g < p.n_routed ? p.kept[g] : p.shared_rows;
        grp_off[g] = off;
      }
      const int32_t tiles = int32_t((live + nb - 1) / nb) * ntiles;
      int32_t incl = tiles;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (g < n_groups) tile_start[g] = carry + incl - tiles;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) tile_start[n_groups] = carry;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = tile_start[n_groups];
  const bool sk = p.sk_counters != nullptr;
  const int64_t units = int64_t(total_tiles) * p.num_kb;
  const int64_t upc = sk ? (units + gridDim.x - 1) / gridDim.x : 0;   // units per CTA

  if (warp == 0) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int64_t issued = 0;
      bool ok = true;
      SegIter it(sk, blockIdx.x, gridDim.x, total_tiles, p.num_kb, upc);
      int tile, kb0, kb1;
      while (ok && it.next(tile, kb0, kb1)) {
        const TileCoord tc = decode_tile(tile, tile_start, n_groups, ntiles);
        const int r0 = grp_off[tc.g] + tc.m * nb;
        const int f0 = tc.n * kFeat;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_or_abort(&empty[stage], phase ^ 1u, p, abort_flag)) { ok = false; break; }
          const uint32_t fb = smem_u32(&full[stage]);
          mbar_arrive_expect_tx(&full[stage], uint32_t(stage_bytes));
          if (tc.g < p.n_routed)
            tma_load_3d(&tmW, smem_u32(smem + stage * L.w_bytes()), fb, kb * BK, f0, tc.g);
          else
            tma_load_2d(&tmWs, smem_u32(smem + stage * L.w_bytes()), fb, kb * BK, f0);
          tma_load_2d(&tmX, smem_u32(smem + L.x_off() + stage * L.x_bytes()), fb, kb * BK, r0);
          ++issued;
          if (++stage == uint32_t(stages)) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        // let the copies in flight land before the CTA exits: stage s was last
        // filled by load number i (the largest i < issued with i % stages == s),
        // whose completion is phase (i / stages) & 1 of full[s]
        for (int s = 0; s < stages; ++s) {
          if (issued <= s) continue;
          const int64_t i = s + (issued - 1 - s) / stages * stages;
          const uint32_t a = smem_u32(&full[s]);
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(a, uint32_t((i / stages) & 1)) &&
                 global_timer_ns() - t0 < p.wait_limit_ns) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_swap_bf16_f32(nb);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      SegIter it(sk, blockIdx.x, gridDim.x, total_tiles, p.num_kb, upc);
      int tile, kb0, kb1;
      while (ok && it.next(tile, kb0, kb1)) {
        if (!wait_or_abort(&tempty[acc], acc_phase ^ 1u, p, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * uint32_t(nb);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_or_abort(&full[stage], phase, p, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint64_t wd = sdesc_sw128(smem_u32(smem + stage * L.w_bytes()));
          const uint64_t xd = sdesc_sw128(smem_u32(smem + L.x_off() + stage * L.x_bytes()));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc_mma(d_tmem, wd + uint64_t(2 * kk), xd + uint64_t(2 * kk), idesc,
                   (kb != kb0 || kk != 0) ? 1u : 0u);
          tc_commit(smem_u32(&empty[stage]));
          if (++stage == uint32_t(stages)) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(smem_u32(&tfull[acc]));
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      tc_commit(smem_u32(done));
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(smem_u32(done), 0) && global_timer_ns() - t0 < p.wait_limit_ns) {
      }
    }
  } else {
    // epilogue: warps 2-5, one TMEM lane quarter each; thread = one feature.
    // Stream-K: a piece that does not hold its tile's first k-block is
    // published to this CTA's partial slot (it always starts the CTA's share)
    // and counted on the tile's counter.  The CTA that holds the first
    // k-block -- the last piece of its share, so the other pieces, which
    // began their CTAs' shares, are long done -- waits for that count, adds
    // the other pieces to its own accumulator in k order and stores the tile.
    const int q = warp & 3;
    const int fl = q * 32 + lane;                  // feature within the tile
    volatile int* sk_stop = reinterpret_cast<volatile int*>(smem + L.sk_stop());
    const int chunks = nb / CW;
    const int64_t slot_floats = int64_t(nb) * kFeat;
    uint32_t acc = 0, acc_phase = 0;
    SegIter it(sk, blockIdx.x, gridDim.x, total_tiles, p.num_kb, upc);
    int tile, kb0, kb1;
    while (it.next(tile, kb0, kb1)) {
      const TileCoord tc = decode_tile(tile, tile_start, n_groups, ntiles);
      bool ok = true;
      if (lane == 0) ok = wait_or_abort(&tfull[acc], acc_phase, p, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      const bool whole = kb0 == 0 && kb1 == p.num_kb;
      const bool head = !whole && kb0 == 0;        // this CTA finishes the tile
      const int64_t t0 = int64_t(tile) * p.num_kb;
      const int c_first = sk ? int(t0 / upc) : 0;
      const int c_last = sk ? int((t0 + p.num_kb - 1) / upc) : 0;
      if (sk) {
        // the head waits until the tile's other pieces are published
        if (ok && head && warp == 2 && lane == 0) {
          const int want = c_last - c_first;
          int32_t* cnt = p.sk_counters + tile;
          const uint64_t w0 = global_timer_ns();
          for (uint32_t it2 = 0; ld_acquire_gpu(cnt) < want; ++it2) {
            if ((it2 & 63u) == 63u && (*abort_flag || global_timer_ns() - w0 > p.wait_limit_ns)) {
              atomicCAS(p.status, MOE_OK, MOE_ERR_TIMEOUT);
              *abort_flag = 1;
              ok = false;
              break;
            }
          }
          if (ok) *reinterpret_cast<volatile int32_t*>(cnt) = 0;   // ready for the next call
        }
        // the four epilogue warps stop together, whichever of them gave up
        if (!ok && lane == 0) *sk_stop = 1;
        epi_bar_sync();
        ok = *sk_stop == 0;
        epi_bar_sync();                            // every warp has read the flag
      }
      if (!ok) break;
      tc_fence_after();
      if (head) __threadfence();                   // the other pieces are visible
      const bool routed = tc.g < p.n_routed;
      const int live = routed ? p.kept[tc.g] : p.shared_rows;
      if (warp == 2 && lane == 0)
        MOE_CHECK(p.rows_total == 0 || int64_t(grp_off[tc.g]) + live <= p.rows_total,
                  CK_GEMM_ROWS);
      const int feat = tc.n * kFeat + fl;
      const __nv_bfloat16* bias = routed ? p.bias + int64_t(tc.g) * p.Nd : p.bias_s;
      const float b = __bfloat162float(bias[feat]);
      const int rows_left = live - tc.m * nb;      // live token rows of this tile
      __nv_bfloat16* out_col = static_cast<__nv_bfloat16*>(p.out) +
                               (int64_t(grp_off[tc.g]) + int64_t(tc.m) * nb) * p.Nd + feat;
      const uint32_t tacc = tmem_base + (uint32_t(q * 32) << 16) + acc * uint32_t(nb);
      const bool publish = !whole && !head;
      float* mine = publish ? p.sk_partials + int64_t(blockIdx.x) * slot_floats : nullptr;
      for (int c = 0; c < chunks; ++c) {
        uint32_t r[CW];
        tmem_ld_cols<CW>(tacc + uint32_t(c * CW), r);
        if (c == chunks - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[acc]);   // the accumulator is read
        }
        float v[CW];
#pragma unroll
        for (int i = 0; i < CW; ++i) v[i] = __uint_as_float(r[i]);
        if (publish) {
#pragma unroll
          for (int i = 0; i < CW; ++i) __stcg(mine + (c * CW + i) * kFeat + fl, v[i]);
          continue;
        }
        if (head) {
          // the other pieces in k order, two at a time
          int cta = c_first + 1;
          for (; cta + 1 <= c_last; cta += 2) {
            const float* pa = p.sk_partials + int64_t(cta) * slot_floats + (c * CW) * kFeat + fl;
            const float* pb = pa + slot_floats;
            float a[CW], a2[CW];
#pragma unroll
            for (int i = 0; i < CW; ++i) {
              a[i] = __ldcg(pa + i * kFeat);
              a2[i] = __ldcg(pb + i * kFeat);
            }
#pragma unroll
            for (int i = 0; i < CW; ++i) v[i] = (v[i] + a[i]) + a2[i];
          }
          if (cta <= c_last) {
            const float* pa = p.sk_partials + int64_t(cta) * slot_floats + (c * CW) * kFeat + fl;
#pragma unroll
            for (int i = 0; i < CW; ++i) v[i] += __ldcg(pa + i * kFeat);
          }
        }
        swap_store_chunk<EPI, CW>(v, b, c * CW, rows_left, out_col, p.Nd);
      }
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
      if (!publish) continue;
      // count the piece once all four warps' stores are visible
      __threadfence();
      epi_bar_sync();
      if (warp == 2 && lane == 0) atomicAdd(p.sk_counters + tile, 1);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(tmem_cols));
  }
}

// ---- host side -----------------------------------------------------------------------

// bf16 tensor [outer, inner] (or [z, outer, inner]) read in boxes of
// [box_outer, 64] with 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t z,
              uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {inner, outer, z};
  const cuuint64_t strides[2] = {inner * 2, inner * outer * 2};
  const cuuint32_t box[3] = {uint32_t(BK), box_outer, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const cuuint32_t rank = z > 0 ? 3 : 2;
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <class CFG, int EPI>
cudaError_t launch_tc(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& Bs,
                      const TcParams& p, int grid, cudaStream_t s) {
  constexpr int smem = Layout<CFG::BN, CFG::STAGES, CFG::STAGE_BYTES>::kAlloc;
  constexpr int minb = smem <= 110 * 1024 ? 2 : 1;    // two CTAs per SM when they fit
  auto kern = tc_grouped_gemm_kernel<CFG, EPI, minb>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(CFG::THREADS), smem, s, A, B, Bs, p);
}

template <class CFG>
cudaError_t launch_epi(int epi, const CUtensorMap& A, const CUtensorMap& B,
                       const CUtensorMap& Bs, const TcParams& p, int grid, cudaStream_t s) {
  if (epi == EPI_BIAS_F32) return launch_tc<CFG, EPI_BIAS_F32>(A, B, Bs, p, grid, s);
  if (epi == EPI_BIAS_GELU) return launch_tc<CFG, EPI_BIAS_GELU>(A, B, Bs, p, grid, s);
  if (epi == EPI_BIAS_RELU) return launch_tc<CFG, EPI_BIAS_RELU>(A, B, Bs, p, grid, s);
  return launch_tc<CFG, EPI_BIAS>(A, B, Bs, p, grid, s);
}

// The kernel variants this library instantiates.
enum TileChoice {
  TILE_256 = 0, TILE_128 = 1, TILE_64 = 2, TILE_128_2CTA = 3, TILE_256_PAIR = 4, NUM_TILES
};
using Cfg256 = TileCfg<256, 4, 16>;        // one CTA per SM, 192 KB ring
using Cfg128 = TileCfg<128, 4, 16>;
using Cfg64 = TileCfg<64, 6, 16>;
using Cfg128x2 = TileCfg<128, 3, 8, false>;  // two CTAs per SM, 96 KB ring each
using Cfg256Pair = TileCfg<256, 6, 16>;    // CTA pair, 256 x 256 tiles, 6 x 32 KB ring per CTA
// router with the top-k epilogue: four warps per TMEM lane quarter, a row's
// 64 scores split over four threads (router_topk_rows)
using CfgRouter = TileCfg<64, 6, 16, false, int(sizeof(RouterRed))>;

int tile_bn(int choice) {
  switch (choice) {
    case TILE_256: case TILE_256_PAIR: return 256;
    case TILE_64: return 64;
    default: return 128;
  }
}

int tile_rows(int choice) { return choice == TILE_256_PAIR ? 256 : BM; }
int tile_ctas_per_sm(int choice) { return choice == TILE_128_2CTA ? 2 : 1; }

template <class CFG, int EPI>
cudaError_t launch_pair(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& Bs,
                        const TcParams& p, int64_t tiles, int num_sms, cudaStream_t s) {
  constexpr int smem = Layout2<CFG::BN, CFG::STAGES, CFG::STAGE_BYTES>::kAlloc;
  auto kern = tc2_grouped_gemm_kernel<CFG, EPI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // CTA pairs that can be resident at once (pairs sit on two SMs of one GPC)
  static int max_pairs[64] = {};
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (max_pairs[dev] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(num_sms & ~1));
    cfg.blockDim = dim3(CFG::THREADS);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    max_pairs[dev] = n > 0 ? n : 1;
  }
  const int64_t pairs = tiles < max_pairs[dev] ? tiles : max_pairs[dev];
  if (pairs <= 0) return cudaSuccess;
  return launch_pdl(kern, dim3(unsigned(2 * pairs)), dim3(CFG::THREADS), smem, s, A, B, Bs, p);
}

cudaError_t launch_choice(int choice, int epi, const CUtensorMap& A, const CUtensorMap& B,
                          const CUtensorMap& Bs, const TcParams& p, int64_t max_tiles,
                          int num_sms, cudaStream_t s) {
  if (choice == TILE_256_PAIR) {
    if (epi == EPI_BIAS_GELU)
      return launch_pair<Cfg256Pair, EPI_BIAS_GELU>(A, B, Bs, p, max_tiles, num_sms, s);
    if (epi == EPI_BIAS_RELU)
      return launch_pair<Cfg256Pair, EPI_BIAS_RELU>(A, B, Bs, p, max_tiles, num_sms, s);
    return launch_pair<Cfg256Pair, EPI_BIAS>(A, B, Bs, p, max_tiles, num_sms, s);
  }
  const int64_t slots = int64_t(num_sms) * tile_ctas_per_sm(choice);
  const int grid = int(max_tiles < slots ? max_tiles : slots);
  if (grid <= 0) return cudaSuccess;
  switch (choice) {
    case TILE_256: return launch_epi<Cfg256>(epi, A, B, Bs, p, grid, s);
    case TILE_128: return launch_epi<Cfg128>(epi, A, B, Bs, p, grid, s);
    case TILE_64: return launch_epi<Cfg64>(epi, A, B, Bs, p, grid, s);
    default: return launch_epi<Cfg128x2>(epi, A, B, Bs, p, grid, s);
  }
}

// Tile variant for one grouped Linear with output width Nd, reduction length
// K and rows_per_group rows in an average expert group: CTA-pair 256 x 256
// tiles when the groups fill them and K is long enough to amortise the pair's
// synchronisation (half the shared-memory traffic per MMA); otherwise the
// widest single-CTA tile that divides Nd.
int pick_tile(int64_t Nd, int64_t rows_per_group, int64_t K) {
  if (Nd % 256 == 0 && rows_per_group >= 256 && K >= 2048) return TILE_256_PAIR;
  if (Nd % 256 == 0) return TILE_256;
  if (Nd % 128 == 0) return TILE_128;
  return TILE_64;
}

// Deepest ring of the token-column kernel that fits the shared memory.
int swap_stages(int nb) {
  int st = kSwapMaxStages;
  while (st > 2 && LayoutSw{nb, st}.alloc() > kSmemBudget) --st;
  return st;
}

template <int NBT, int EPI>
cudaError_t launch_swap_epi(const CUtensorMap& W, const CUtensorMap& Ws, const CUtensorMap& X,
                            const TcParams& p, int grid, cudaStream_t s) {
  const int smem = LayoutSw{p.sw_nb, p.sw_stages}.alloc();
  auto kern = tc_swap_gemm_kernel<NBT, EPI>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(6 * 32), smem, s, W, Ws, X, p);
}

template <int NBT>
cudaError_t launch_swap(int epi, const CUtensorMap& W, const CUtensorMap& Ws,
                        const CUtensorMap& X, const TcParams& p, int grid, cudaStream_t s) {
  if (epi == EPI_BIAS_GELU) return launch_swap_epi<NBT, EPI_BIAS_GELU>(W, Ws, X, p, grid, s);
  if (epi == EPI_BIAS_RELU) return launch_swap_epi<NBT, EPI_BIAS_RELU>(W, Ws, X, p, grid, s);
  return launch_swap_epi<NBT, EPI_BIAS>(W, Ws, X, p, grid, s);
}

// Token columns per tile of the token-column variant (0: the regular tiles):
// 16 or 32 when an average group holds a few rows (decoding).  (Wider
// token-column tiles -- a capacity-capped layer's groups as single column
// tiles of up to 256 tokens -- measured slower than the regular tiles on the
// Switch-sized layer, 45 vs 28 us for its first Linear, and are not used.)
int swap_rows(int64_t Nd, int64_t rows_per_group, int epi) {
  if (epi == EPI_BIAS_F32 || Nd % 128 != 0) return 0;
  if (rows_per_group <= 8) return 16;
  if (rows_per_group <= 24) return 32;
  return 0;
}

// How one grouped Linear runs: the decode tiles (nb token columns, stream-K
// when moe_forward's workspace holds its scratch: `forward`) or a tile family,
// and a bound on its tiles (the size of its stream-K counters).
struct LinearPlan {
  int nb = 0;              // token-column tiles: token columns; 0: regular tiles
  int choice = TILE_256;   // regular tiles: TileChoice
  bool sk = false;
  int64_t max_tiles = 0;
};

LinearPlan plan_linear(const moe_config& c, int64_t K, int64_t Nd, int epi, int64_t routed_rows,
                       bool forward) {
  LinearPlan pl;
  const int64_t groups = c.n_experts + (c.d_ff_shared > 0 ? 1 : 0);
  const int64_t routed = routed_rows > 0 ? routed_rows : c.T * c.top_k;
  const int64_t rows = routed + (c.d_ff_shared > 0 ? c.T : 0);
  pl.nb = swap_rows(Nd, rows / groups, epi);
  if (pl.nb > 0) {
    pl.sk = forward;
    pl.max_tiles = (ceil_div(rows, pl.nb) + groups) * (Nd / 128);
    return pl;
  }
  pl.choice = pick_tile(Nd, rows / groups, K);
  pl.max_tiles = (ceil_div(rows_max_for(c), tile_rows(pl.choice)) + groups) *
                 (Nd / tile_bn(pl.choice));
  return pl;
}

LinearPlan plan_forward_linear(const moe_config& c, int linear) {
  const int64_t K = linear == 1 ? c.d_model : c.d_ff;
  const int64_t Nd = linear == 1 ? c.d_ff : c.d_model;
  const int epi = linear == 2 ? EPI_BIAS
                              : (c.act == MOE_ACT_RELU ? EPI_BIAS_RELU : EPI_BIAS_GELU);
  return plan_linear(c, K, Nd, epi, 0, true);
}

// One grouped Linear: out[group g] = epi(A[group g] . W[g]^T + bias[g]).
// out_pre: with an activation epilogue, also store the pre-activation there
// (only on the staged tile families; see linear_saves_pre).
// sk_counters: the decode tiles run stream-K with these counters (all 0) and
// g.sk_partials; nullptr: whole tiles per CTA.
cudaError_t grouped_linear(const moe_config& c, const GroupedFfnArgs& g, const void* A,
                           const void* W, const void* Ws, const void* bias,
                           const void* bias_s, void* out, int64_t K, int64_t Nd, int epi,
                           cudaStream_t s, void* out_pre = nullptr,
                           int32_t* sk_counters = nullptr) {
  const int64_t groups = c.n_experts + (c.d_ff_shared > 0 ? 1 : 0);
  const bool forward = sk_counters != nullptr && g.sk_partials != nullptr;
  const LinearPlan pl = plan_linear(c, K, Nd, epi, g.routed_rows, forward);
  const int nb = pl.nb;
  if (nb > 0) {
    // decode: weights as the MMA's 128-row operand, tokens as its NB columns
    CUtensorMap mW, mWs, mX;
    if (!make_map(&mW, W, uint64_t(K), uint64_t(Nd), uint64_t(c.n_experts), 128))
      return cudaErrorInvalidValue;
    if (c.d_ff_shared > 0) {
      if (!make_map(&mWs, Ws, uint64_t(K), uint64_t(Nd), 0, 128)) return cudaErrorInvalidValue;
    } else {
      mWs = mW;
    }
    if (!make_map(&mX, A, uint64_t(K), uint64_t(g.rows_max), 0, uint32_t(nb)))
      return cudaErrorInvalidValue;
    TcParams p{};
    p.offsets = g.offsets;
    p.kept = g.kept;
    p.bias = static_cast<const __nv_bfloat16*>(bias);
    p.bias_s = static_cast<const __nv_bfloat16*>(bias_s);
    p.out = out;
    p.Nd = Nd;
    p.n_routed = int32_t(c.n_experts);
    p.shared_rows = c.d_ff_shared > 0 ? int32_t(c.T) : 0;
    p.num_kb = int32_t(K / BK);
    p.status = g.status;
    p.wait_limit_ns = g.wait_limit_ns;
    p.rows_total = g.rows_max;
    const int64_t max_tiles = pl.max_tiles;
    int grid = int(max_tiles < g.num_sms ? max_tiles : g.num_sms);
    if (pl.sk) {
      // stream-K: every CTA takes an equal share of the k-blocks
      p.sk_partials = g.sk_partials;
      p.sk_counters = sk_counters;
      grid = g.num_sms < kSkMaxCtas ? g.num_sms : kSkMaxCtas;
    }
    p.sw_nb = nb;
    p.sw_stages = swap_stages(nb);
    return nb == 16 ? launch_swap<16>(epi, mW, mWs, mX, p, grid, s)
                    : launch_swap<0>(epi, mW, mWs, mX, p, grid, s);
  }
  const int choice = pl.choice;
  const int bn = tile_bn(choice);
  // the CTA pair loads half of each B tile per CTA
  const uint32_t b_box = uint32_t(choice == TILE_256_PAIR ? bn / 2 : bn);
  const int64_t N = c.n_experts;
  CUtensorMap mA, mB, mBs;
  if (!make_map(&mA, A, uint64_t(K), uint64_t(g.rows_max), 0, BM)) return cudaErrorInvalidValue;
  if (!make_map(&mB, W, uint64_t(K), uint64_t(Nd), uint64_t(N), b_box))
    return cudaErrorInvalidValue;
  if (c.d_ff_shared > 0) {
    if (!make_map(&mBs, Ws, uint64_t(K), uint64_t(Nd), 0, b_box))
      return cudaErrorInvalidValue;
  } else {
    mBs = mB;
  }
  TcParams p{};
  p.offsets = g.offsets;
  p.kept = g.kept;
  p.bias = static_cast<const __nv_bfloat16*>(bias);
  p.bias_s = static_cast<const __nv_bfloat16*>(bias_s);
  p.out = out;
  p.Nd = Nd;
  p.n_routed = int32_t(N);
  p.shared_rows = c.d_ff_shared > 0 ? int32_t(c.T) : 0;
  p.num_kb = int32_t(K / BK);
  p.status = g.status;
  p.wait_limit_ns = g.wait_limit_ns;
  p.out_pre = out_pre;
  p.rows_total = g.rows_max;
  // upper bound on the tiles (every group may add one partial m-tile)
  const int64_t max_tiles =
      (ceil_div(g.rows_max, tile_rows(choice)) + groups) * (Nd / bn);
  return launch_choice(choice, epi, mA, mB, mBs, p, max_tiles, g.num_sms, s);
}

}  // namespace

cudaError_t launch_grouped_linear_bf16(const moe_config& c, const GroupedFfnArgs& g,
                                       const void* A, const void* W, const void* Ws,
                                       const void* bias, const void* bias_s, void* out,
                                       int64_t K, int64_t Nd, cudaStream_t s) {
  if (g.rows_max == 0) return cudaSuccess;
  return grouped_linear(c, g, A, W, Ws, bias, bias_s, out, K, Nd, EPI_BIAS, s);
}

bool bwd_dgrad_on_pair(const moe_config& c, int64_t K, int64_t Nd) {
  const int64_t groups = c.n_experts + (c.d_ff_shared > 0 ? 1 : 0);
  const int64_t rows = c.T * c.top_k + (c.d_ff_shared > 0 ? c.T : 0);
  return pick_tile(Nd, rows / groups, K) == TILE_256_PAIR;
}

cudaError_t launch_bwd_dgrad_pair(const moe_config& c, const BwdGemmArgs& g, const void* dOut,
                                  const void* W, const void* Ws, int64_t K, int64_t Nd,
                                  int act, const void* pre, void* out, cudaStream_t s) {
  const int64_t N = c.n_experts;
  CUtensorMap mA, mB, mBs;
  // A = dOut [rows, K] K-major; B = the weight as stored [N, K, Nd], MN-major boxes
  if (!make_map(&mA, dOut, uint64_t(K), uint64_t(g.rows_max), 0, BM))
    return cudaErrorInvalidValue;
  if (!make_map(&mB, W, uint64_t(Nd), uint64_t(K), uint64_t(N), BK))
    return cudaErrorInvalidValue;
  if (c.d_ff_shared > 0) {
    if (!make_map(&mBs, Ws, uint64_t(Nd), uint64_t(K), 0, BK)) return cudaErrorInvalidValue;
  } else {
    mBs = mB;
  }
  TcParams p{};
  p.offsets = g.offsets;
  p.kept = g.kept;
  p.pre = static_cast<const __nv_bfloat16*>(pre);
  p.out = out;
  p.Nd = Nd;
  p.n_routed = int32_t(N);
  p.shared_rows = c.d_ff_shared > 0 ? int32_t(c.T) : 0;
  p.num_kb = int32_t(K / BK);
  p.status = g.status;
  p.wait_limit_ns = g.wait_limit_ns;
  const int64_t groups = N + (c.d_ff_shared > 0 ? 1 : 0);
  const int64_t max_tiles = (ceil_div(g.rows_max, 256) + groups) * (Nd / 256);
  if (act < 0)
    return launch_pair<Cfg256Pair, EPI_DGRAD>(mA, mB, mBs, p, max_tiles, g.num_sms, s);
  if (act == MOE_ACT_RELU)
    return launch_pair<Cfg256Pair, EPI_DGRAD_RELU>(mA, mB, mBs, p, max_tiles, g.num_sms, s);
  return launch_pair<Cfg256Pair, EPI_DGRAD_GELU>(mA, mB, mBs, p, max_tiles, g.num_sms, s);
}

// Whether the first Linear's epilogue can also store its pre-activation: the
// staged single-CTA and CTA-pair tiles can, the decode (swap) tiles and the
// two-CTAs-per-SM tiles cannot.
bool linear_saves_pre(const moe_config& c) {
  const int epi1 = c.act == MOE_ACT_RELU ? EPI_BIAS_RELU : EPI_BIAS_GELU;
  const int64_t groups = c.n_experts + (c.d_ff_shared > 0 ? 1 : 0);
  const int64_t rows = c.T * c.top_k + (c.d_ff_shared > 0 ? c.T : 0);
  return swap_rows(c.d_ff, rows / groups, epi1) == 0 &&
         pick_tile(c.d_ff, rows / groups, c.d_model) != TILE_128_2CTA;
}

int64_t sk_counter_ints(const moe_config& c, int linear) {
  if (c.dtype == MOE_F32) return 0;
  const LinearPlan pl = plan_forward_linear(c, linear);
  return pl.sk ? pl.max_tiles : 0;
}

size_t sk_partial_bytes(const moe_config& c) {
  if (c.dtype == MOE_F32) return 0;
  size_t slot = 0;                       // fp32 partial accumulator of one tile
  for (int linear = 1; linear <= 2; ++linear) {
    const LinearPlan pl = plan_forward_linear(c, linear);
    if (!pl.sk) continue;
    const size_t b = size_t(pl.nb) * 128 * sizeof(float);   // token-column tiles only
    if (b > slot) slot = b;
  }
  return size_t(kSkMaxCtas) * slot;
}

cudaError_t launch_grouped_ffn_bf16(const moe_config& c, const GroupedFfnArgs& g,
                                    cudaStream_t s) {
  if (g.rows_max == 0) return cudaSuccess;
  const int epi1 = c.act == MOE_ACT_RELU ? EPI_BIAS_RELU : EPI_BIAS_GELU;
  // the pre-activation for a later backward: from the epilogue, or else by a
  // second pass of the first Linear without its activation
  const bool in_epi = g.pre_out && linear_saves_pre(c);
  int32_t* sk1 = nullptr;
  int32_t* sk2 = nullptr;
  if (g.sk_counters && g.sk_partials) {
    const int64_t n1 = sk_counter_ints(c, 1);
    if (n1 > 0) sk1 = g.sk_counters;
    if (sk_counter_ints(c, 2) > 0) sk2 = g.sk_counters + n1;
  }
  cudaError_t e = grouped_linear(c, g, g.Xp, g.w->W1, g.w->W1s, g.w->b1, g.w->b1s, g.H,
                                 c.d_model, c.d_ff, epi1, s, in_epi ? g.pre_out : nullptr,
                                 sk1);
  if (e == cudaSuccess && g.pre_out && !in_epi)
    e = grouped_linear(c, g, g.Xp, g.w->W1, g.w->W1s, g.w->b1, g.w->b1s, g.pre_out, c.d_model,
                       c.d_ff, EPI_BIAS, s);
  if (e == cudaSuccess) e = record_event(g.mid_event, s);
  if (e != cudaSuccess) return e;
  return grouped_linear(c, g, g.H, g.w->W2, g.w->W2s, g.w->b2, g.w->b2s, g.Yp, c.d_ff,
                        c.d_model, EPI_BIAS, s, nullptr, sk2);
}

// Name of the kernel (and tile) one grouped Linear of moe_forward launches,
// chosen by the same rules as grouped_linear (linear 1: Xp -> H, 2: H -> Yp).
const char* grouped_linear_kernel_name(const moe_config& c, int linear, int64_t routed_rows) {
  if (c.dtype == MOE_F32) return "simt_gemm_kernel (fp32 CUDA cores)";
  const int64_t K = linear == 1 ? c.d_model : c.d_ff;
  const int64_t Nd = linear == 1 ? c.d_ff : c.d_model;
  const int epi = linear == 2 ? EPI_BIAS
                              : (c.act == MOE_ACT_RELU ? EPI_BIAS_RELU : EPI_BIAS_GELU);
  const LinearPlan pl = plan_linear(c, K, Nd, epi, routed_rows, true);
  if (pl.nb == 16) return "tc_swap_gemm_kernel (128 weight rows x 16 tokens, stream-K)";
  if (pl.nb == 32) return "tc_swap_gemm_kernel (128 weight rows x 32 tokens, stream-K)";
  switch (pl.choice) {
    case TILE_256_PAIR: return "tc2_grouped_gemm_kernel (256 x 256 on a CTA pair)";
    case TILE_256: return "tc_grouped_gemm_kernel (128 x 256)";
    case TILE_128: return "tc_grouped_gemm_kernel (128 x 128)";
    case TILE_64: return "tc_grouped_gemm_kernel (128 x 64)";
    default: return "tc_grouped_gemm_kernel (128 x 128, two CTAs per SM)";
  }
}

// Router scores z = x . W_g^T + b_g (fp32) as one dense group on the tensor
// cores: bf16 products are exact in fp32, so only the summation order differs
// from a CUDA-core dot product.  N % 64 == 0; 64-wide tiles give ceil(T/128)
// * N/64 tiles to spread over the SMs.
cudaError_t launch_router_logits_tc(const moe_config& c, const void* x, const void* W_g,
                                    const void* b_g, float* logits, int num_sms,
                                    int32_t* status, uint64_t wait_limit_ns, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  constexpr int bn = 64;
  CUtensorMap mA, mB;
  if (!make_map(&mA, x, uint64_t(c.d_model), uint64_t(c.T), 0, BM)) return cudaErrorInvalidValue;
  if (!make_map(&mB, W_g, uint64_t(c.d_model), uint64_t(c.n_experts), 1, bn))
    return cudaErrorInvalidValue;
  TcParams p{};
  p.offsets = nullptr;
  p.kept = nullptr;
  p.bias = static_cast<const __nv_bfloat16*>(b_g);
  p.bias_s = nullptr;
  p.out = logits;
  p.Nd = c.n_experts;
  p.n_routed = 1;
  p.shared_rows = 0;
  p.dense_rows = int32_t(c.T);
  p.num_kb = int32_t(c.d_model / BK);
  p.status = status;
  p.wait_limit_ns = wait_limit_ns;
  const int64_t tiles = ceil_div(c.T, BM) * (c.n_experts / bn);
  const int grid = int(tiles < num_sms ? tiles : num_sms);
  return launch_tc<Cfg64, EPI_BIAS_F32>(mA, mB, mB, p, grid, s);
}

// The same GEMM for 64 experts with the softmax, top-k and gates in its
// epilogue (router_topk_rows): one 64-wide tile holds a row's every score.
// prob_rows [ceil(T/128), 64]: column sums of p per 128-row tile.
cudaError_t launch_router_topk_tc(const moe_config& c, const void* x, const void* W_g,
                                  const void* b_g, float* logits, int32_t* topk_idx,
                                  float* topk_w, float* prob_rows, int num_sms,
                                  int32_t* status, uint64_t wait_limit_ns, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  if (c.n_experts != 64 || c.top_k < 1 || c.top_k > 8) return cudaErrorInvalidValue;
  constexpr int bn = 64;
  CUtensorMap mA, mB;
  if (!make_map(&mA, x, uint64_t(c.d_model), uint64_t(c.T), 0, BM)) return cudaErrorInvalidValue;
  if (!make_map(&mB, W_g, uint64_t(c.d_model), uint64_t(c.n_experts), 1, bn))
    return cudaErrorInvalidValue;
  TcParams p{};
  p.bias = static_cast<const __nv_bfloat16*>(b_g);
  p.out = logits;
  p.Nd = c.n_experts;
  p.n_routed = 1;
  p.dense_rows = int32_t(c.T);
  p.num_kb = int32_t(c.d_model / BK);
  p.status = status;
  p.wait_limit_ns = wait_limit_ns;
  p.topk_idx = topk_idx;
  p.topk_w = topk_w;
  p.prob_rows = prob_rows;
  p.top_k = int32_t(c.top_k);
  p.renorm = c.renormalize ? 1 : 0;
  const int64_t tiles = ceil_div(c.T, BM);
  const int grid = int(tiles < num_sms ? tiles : num_sms);
  return launch_tc<CfgRouter, EPI_ROUTER_TOPK>(mA, mB, mB, p, grid, s);
}

MOE_CHECKS_UNIT(grouped_ffn)

}  // namespace moe
