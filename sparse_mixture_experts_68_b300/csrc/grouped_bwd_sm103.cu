// Backward of the bf16 grouped expert FFN on the tcgen05 tensor cores (the
// chain rule through botmartz.com "Mixture of Experts (MoE) and Mixtral",
// "Expert Routing": Linear -> GELU / ReLU -> Linear per expert, for the
// training loss of "Load Balancing: The Hidden Challenge").  Per expert group
// e with rows R (its kept tokens), given dO = d loss / d Yp:
//
//   dA   = (dO . W2[e]) * act'(A1)     dgrad of the second Linear, times the
//                                      activation's derivative at the saved
//                                      pre-activation A1 = Xp W1[e]^T + b1[e]
//   dXp  = dA . W1[e]                  dgrad of the first Linear
//   dW2[e] = dO^T . H,  dW1[e] = dA^T . Xp     wgrads (K = the group's rows)
//
// One kernel, two modes, on the same warp roles, ring and double-buffered
// TMEM accumulator as the forward kernel:
//   DGRAD  tiles of 128 rows x BN columns per group, K fixed.  A (dO or dA)
//          is K-major as in the forward.  B is the weight in its stored
//          layout, [K, Nd] with Nd contiguous: an MN-major operand, loaded as
//          BN/64 boxes of 64 columns x 64 K-rows and described to the MMA
//          with the "transpose B" bit.  No transposed weight copy is made.
//   WGRAD  per group a dense [Md, Nd] output, K = the group's rows (0 rows:
//          the tile is written as zeros).  A and B are both activations
//          [rows, M] / [rows, N], i.e. MN-major, read the same way.
// MN-major 128-byte-swizzle operands: 64-element MN chunks of 64 K-rows x
// 128 B (8 KB) side by side (leading byte offset 8 KB), 8-row K groups 1 KB
// apart (stride byte offset); one MMA of K = 16 spans two K groups, so the
// next MMA starts 2 KB further on.
// The DGRAD epilogue writes zeros into a group's padding rows (up to its
// 128-row boundary), so the WGRAD of the same rows sees exact zeros there.
#include "kernels.h"
#include "tc_common.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kMaxGroups = 1025;

enum { MODE_DGRAD = 0, MODE_WGRAD = 1 };
enum { BEPI_STORE = 0, BEPI_DGELU = 1, BEPI_DRELU = 2 };

// Output staging (WGRAD): each epilogue warp's 32 rows x BN/4 columns of
// bf16, laid out as the tensor store's box with the swizzle matching its row
// width (BN/4 * 2 = 128, 64 or 32 bytes): the 16-byte chunk c of row r sits
// at chunk c ^ (r / (128 / width)) mod (width / 16), so that a warp writing
// one chunk of 32 rows (lane = row) hits every bank once per quarter warp.
template <int BN>
__host__ __device__ constexpr int stage_warp_bytes() {
  return 32 * (BN / 4) * 2;
}

template <int BN, int STAGES, int STAGE_BYTES = 0>
struct BwdLayout {
  static constexpr int kABytes = BM * BK * 2;
  static constexpr int kBBytes = BN * BK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kA = 0;
  static constexpr int kB = STAGES * kABytes;
  static constexpr int kBar = kB + STAGES * kBBytes;   // full[S], empty[S], tfull[2], tempty[2], done
  static constexpr int kNumBars = 2 * STAGES + 5;
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kTileStart = (kAbort + 4 + 15) / 16 * 16;     // [kMaxGroups + 1]
  static constexpr int kGroupOff = kTileStart + (kMaxGroups + 1) * 4;  // [kMaxGroups]
  static constexpr int kGroupLive = kGroupOff + kMaxGroups * 4;        // [kMaxGroups]
  static constexpr int kStage = (kGroupLive + kMaxGroups * 4 + 1023) / 1024 * 1024;
  static constexpr int kBytes = kStage + STAGE_BYTES;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

struct BwdParams {
  const int32_t* offsets;       // [n_groups + 1]
  const int32_t* kept;          // [n_routed]
  int32_t n_routed;
  int32_t shared_rows;          // rows of the shared group (0: none)
  int32_t Md;                   // WGRAD: output rows per group
  int32_t num_kb;               // DGRAD: K / 64
  int64_t Nd;                   // output columns
  void* out;                    // DGRAD [rows, Nd]; WGRAD [n_routed, Md, Nd]
  void* out_s;                  // WGRAD: shared expert's [Md, Nd]
  const __nv_bfloat16* pre;     // DGRAD with an activation: A1 [rows, Nd]
  int32_t* status;
  uint64_t wait_limit_ns;
};

// kind::f16, D fp32, A and B bf16; bit 15: A MN-major, bit 16: B MN-major.
template <int BN, int MODE>
__host__ __device__ constexpr uint32_t idesc_bwd() {
  return (1u << 4) | (1u << 7) | (1u << 10) | (MODE == MODE_WGRAD ? (1u << 15) : 0u) |
         (1u << 16) | (uint32_t(BN >> 3) << 17) | (uint32_t(BM >> 4) << 24);
}

__device__ __forceinline__ bool bwd_wait(uint64_t* bar, uint32_t parity, const BwdParams& p,
                                         volatile int* abort_flag) {
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

struct BwdTile {
  int g, m, n;
};

__device__ __forceinline__ BwdTile bwd_decode(int tile, const int32_t* tile_start, int n_groups,
                                              int ntiles) {
  int lo = 0, hi = n_groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  const int local = tile - tile_start[lo];
  const int mt = (tile_start[lo + 1] - tile_start[lo]) / ntiles;
  return BwdTile{lo, local % mt, local / mt};
}

template <int MODE>
__device__ __forceinline__ int tile_kb(const BwdParams& p, int live) {
  return MODE == MODE_DGRAD ? p.num_kb : (live + BK - 1) / BK;
}

template <int BN, int STAGES, int MODE, int EPI>
__global__ void __launch_bounds__(18 * 32, 1)
    tc_bwd_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmBs,
                       const __grid_constant__ CUtensorMap tmO,
                       const __grid_constant__ CUtensorMap tmOs, const BwdParams p) {
  constexpr int kEpiWarps = 16;
  // the wgrads write whole weight-sized outputs: each epilogue warp puts its
  // 32 x BN/4 piece of a tile into shared memory and one lane hands it to a
  // tensor store (tmO: [n_routed, Md, Nd], tmOs: the shared expert's [Md, Nd])
  constexpr bool kStaged = MODE == MODE_WGRAD;
  constexpr int kWarpStage = stage_warp_bytes<BN>();
  using L = BwdLayout<BN, STAGES, kStaged ? kEpiWarps * kWarpStage : 0>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = bars + 2 * STAGES + 2;
  uint64_t* done = bars + 2 * STAGES + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  int32_t* tile_start = reinterpret_cast<int32_t*>(smem + L::kTileStart);
  int32_t* grp_off = reinterpret_cast<int32_t*>(smem + L::kGroupOff);
  int32_t* grp_live = reinterpret_cast<int32_t*>(smem + L::kGroupLive);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_groups = p.n_routed + (p.shared_rows > 0 ? 1 : 0);
  const int ntiles = int(p.Nd / BN);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
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
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait_previous();
  if (warp == 2) {
    // tiles per group: DGRAD ceil(live / 128) x ntiles, WGRAD ceil(Md / 128) x ntiles
    int32_t carry = 0;
    for (int base = 0; base < n_groups; base += 32) {
      const int g = base + lane;
      int32_t live = 0;
      if (g < n_groups) {
        live = g < p.n_routed ? p.kept[g] : p.shared_rows;
        grp_off[g] = p.offsets[g];
        grp_live[g] = live;
      }
      const int32_t mrows = MODE == MODE_DGRAD ? live : (g < n_groups ? p.Md : 0);
      const int32_t tiles = int32_t((mrows + BM - 1) / BM) * ntiles;
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
      int last_parity[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) last_parity[s] = -1;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        const BwdTile tc = bwd_decode(tile, tile_start, n_groups, ntiles);
        const int nkb = tile_kb<MODE>(p, grp_live[tc.g]);
        const int off = grp_off[tc.g];
        for (int kb = 0; kb < nkb; ++kb) {
          if (!bwd_wait(&empty[stage], phase ^ 1u, p, abort_flag)) { ok = false; break; }
          const uint32_t fb = smem_u32(&full[stage]);
          const uint32_t a_dst = smem_u32(smem + L::kA + stage * L::kABytes);
          const uint32_t b_dst = smem_u32(smem + L::kB + stage * L::kBBytes);
          mbar_arrive_expect_tx(&full[stage], L::kStageBytes);
          if (MODE == MODE_DGRAD) {
            tma_load_2d(&tmA, a_dst, fb, kb * BK, off + tc.m * BM);
#pragma unroll
            for (int c = 0; c < BN / 64; ++c) {
              if (tc.g < p.n_routed)
                tma_load_3d(&tmB, b_dst + c * 8192, fb, tc.n * BN + 64 * c, kb * BK, tc.g);
              else
                tma_load_2d(&tmBs, b_dst + c * 8192, fb, tc.n * BN + 64 * c, kb * BK);
            }
          } else {
            const int r = off + kb * BK;
#pragma unroll
            for (int c = 0; c < BM / 64; ++c)
              tma_load_2d(&tmA, a_dst + c * 8192, fb, tc.m * BM + 64 * c, r);
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)
              tma_load_2d(&tmB, b_dst + c * 8192, fb, tc.n * BN + 64 * c, r);
          }
          last_parity[stage] = int(phase);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        for (int s = 0; s < STAGES; ++s)
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
    // WGRAD: a group's last K block issues only the 16-row K steps that hold
    // live rows; the rows past the live ones inside the last of those steps
    // are the group's padding rows, which the caller zeroes (up to the next
    // multiple of 16).  A K block never reaches into the next group: groups
    // start on 128-row boundaries.
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bwd<BN, MODE>();
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        const BwdTile tc = bwd_decode(tile, tile_start, n_groups, ntiles);
        const int live = grp_live[tc.g];
        const int nkb = tile_kb<MODE>(p, live);
        if (!bwd_wait(&tempty[acc], acc_phase ^ 1u, p, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!bwd_wait(&full[stage], phase, p, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_s = smem_u32(smem + L::kA + stage * L::kABytes);
          const uint32_t b_s = smem_u32(smem + L::kB + stage * L::kBBytes);
          const int rem = live - kb * BK;
          const int ksteps = MODE == MODE_WGRAD && rem < BK ? (rem + 15) / 16 : BK / 16;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            if (kk < ksteps) {
              // K-major A: +32 bytes per K step; MN-major operands: +2 K groups
              const uint64_t ad = MODE == MODE_DGRAD ? sdesc_sw128(a_s) + uint64_t(2 * kk)
                                                     : sdesc_mn_sw128(a_s + kk * 2048, 8192);
              const uint64_t bd = sdesc_mn_sw128(b_s + kk * 2048, 8192);
              tc_mma(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
            }
          }
          tc_commit(smem_u32(&empty[stage]));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
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
    // ---------------- epilogue ----------------
    const int q = warp & 3;
    const int part = (warp - 2) >> 2;
    constexpr int kCols = BN / (kEpiWarps / 4);
    constexpr int CW = kCols < 32 ? kCols : 32;
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      const BwdTile tc = bwd_decode(tile, tile_start, n_groups, ntiles);
      bool ok = true;
      if (lane == 0) ok = bwd_wait(&tfull[acc], acc_phase, p, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      tc_fence_after();
      const int live = grp_live[tc.g];
      const bool has_acc = tile_kb<MODE>(p, live) > 0;
      const int row = tc.m * BM + q * 32 + lane;
      __nv_bfloat16* dst_row;
      const __nv_bfloat16* pre_row = nullptr;
      bool store, zero;
      if (MODE == MODE_DGRAD) {
        // live rows get the result, the group's padding rows zeros
        const int64_t out_row = int64_t(grp_off[tc.g]) + row;
        dst_row = static_cast<__nv_bfloat16*>(p.out) + out_row * p.Nd;
        if (EPI != BEPI_STORE) pre_row = p.pre + out_row * p.Nd;
        store = true;
        zero = row >= live;
      } else {
        __nv_bfloat16* base = tc.g < p.n_routed
                                  ? static_cast<__nv_bfloat16*>(p.out) +
                                        int64_t(tc.g) * p.Md * p.Nd
                                  : static_cast<__nv_bfloat16*>(p.out_s);
        dst_row = base + int64_t(row) * p.Nd;
        store = row < p.Md;
        zero = !has_acc;
      }
      if constexpr (kStaged) {
        // wait until this warp's previous tensor store has read its staging
        uint8_t* stg = smem + L::kStage + (warp - 2) * kWarpStage;
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
        constexpr int kRowBytes = kCols * 2;           // 128, 64 or 32
        constexpr int kChunks = kRowBytes / 16;
        const int swz = (lane / (128 / kRowBytes)) % kChunks;
#pragma unroll
        for (int c = 0; c < kCols; c += CW) {
          uint32_t r[CW];
          tmem_ld_cols<CW>(tmem_base + (uint32_t(q * 32) << 16) + acc * BN + part * kCols + c,
                           r);
          if (c + CW == kCols) {                       // the accumulator is free again
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
          }
#pragma unroll
          for (int v = 0; v < CW / 8; ++v) {
            uint4 o;
            __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              o2[i] = zero ? __floats2bfloat162_rn(0.f, 0.f)
                           : __floats2bfloat162_rn(__uint_as_float(r[8 * v + 2 * i]),
                                                   __uint_as_float(r[8 * v + 2 * i + 1]));
            const int ch = (c / 8 + v) ^ swz;
            *reinterpret_cast<uint4*>(stg + lane * kRowBytes + ch * 16) = o;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        const int row0 = tc.m * BM + q * 32;
        if (lane == 0 && row0 < p.Md) {
          const int x = tc.n * BN + part * kCols;
          if (tc.g < p.n_routed) tma_store_3d(&tmO, smem_u32(stg), x, row0, tc.g);
          else tma_store_2d(&tmOs, smem_u32(stg), x, row0);
          bulk_commit();
        }
      } else {
#pragma unroll 1
        for (int c = part * kCols; c < (part + 1) * kCols; c += CW) {
          uint32_t r[CW];
          tmem_ld_cols<CW>(tmem_base + (uint32_t(q * 32) << 16) + acc * BN + c, r);
          if (store) {
            const int64_t col = int64_t(tc.n) * BN + c;
            uint4* dst = reinterpret_cast<uint4*>(dst_row + col);
#pragma unroll
            for (int v = 0; v < CW / 8; ++v) {
              uint4 o;
              __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&o);
              if (zero) {
                o = make_uint4(0, 0, 0, 0);
              } else {
                float gr[8];
                if (EPI != BEPI_STORE) {
                  const uint4 pv = __ldg(reinterpret_cast<const uint4*>(pre_row + col) + v);
                  const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&pv);
#pragma unroll
                  for (int i = 0; i < 4; ++i) {
                    const float2 a = __bfloat1622float2(p2[i]);
                    gr[2 * i] = EPI == BEPI_DGELU ? gelu_erf_grad(a.x) : (a.x > 0.f ? 1.f : 0.f);
                    gr[2 * i + 1] =
                        EPI == BEPI_DGELU ? gelu_erf_grad(a.y) : (a.y > 0.f ? 1.f : 0.f);
                  }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  float x0 = __uint_as_float(r[8 * v + 2 * i]);
                  float x1 = __uint_as_float(r[8 * v + 2 * i + 1]);
                  if (EPI != BEPI_STORE) {
                    x0 *= gr[2 * i];
                    x1 *= gr[2 * i + 1];
                  }
                  o2[i] = __floats2bfloat162_rn(x0, x1);
                }
              }
              dst[v] = o;
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
      }
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    // the tensor stores complete before the block's shared memory goes away
    if (kStaged && lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(2 * BN));
  }
}

// bf16 tensor [outer, inner] (or [z, outer, inner]) in boxes of
// [box_outer, box_inner] (box_inner = 64, 32 or 16: a 128-, 64- or 32-byte
// swizzle, the row width).
bool bwd_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t z,
             uint32_t box_outer, uint32_t box_inner = BK) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {inner, outer, z};
  const cuuint64_t strides[2] = {inner * 2, inner * outer * 2};
  const cuuint32_t box[3] = {box_inner, box_outer, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const cuuint32_t rank = z > 0 ? 3 : 2;
  const CUtensorMapSwizzle sw = box_inner == 64   ? CU_TENSOR_MAP_SWIZZLE_128B
                                : box_inner == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                  : CU_TENSOR_MAP_SWIZZLE_32B;
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int MODE, int EPI>
cudaError_t launch_bwd(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& Bs,
                       const CUtensorMap& O, const CUtensorMap& Os, const BwdParams& p,
                       int64_t max_tiles, int num_sms, cudaStream_t s) {
  // the wgrads trade a ring stage for their store staging
  constexpr int STAGES = MODE == MODE_WGRAD ? 3 : 4;
  constexpr int smem =
      BwdLayout<BN, STAGES, MODE == MODE_WGRAD ? 16 * stage_warp_bytes<BN>() : 0>::kAlloc;
  auto kern = tc_bwd_gemm_kernel<BN, STAGES, MODE, EPI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = int(max_tiles < num_sms ? (max_tiles > 0 ? max_tiles : 1) : num_sms);
  return launch_pdl(kern, dim3(grid), dim3(18 * 32), smem, s, A, B, Bs, O, Os, p);
}

// O, Os: the wgrads' output maps (DGRAD ignores them)
template <int MODE, int EPI>
cudaError_t launch_bwd_bn(int bn, const CUtensorMap& A, const CUtensorMap& B,
                          const CUtensorMap& Bs, const CUtensorMap& O, const CUtensorMap& Os,
                          const BwdParams& p, int64_t max_tiles, int num_sms, cudaStream_t s) {
  if (bn == 256) return launch_bwd<256, MODE, EPI>(A, B, Bs, O, Os, p, max_tiles, num_sms, s);
  if (bn == 128) return launch_bwd<128, MODE, EPI>(A, B, Bs, O, Os, p, max_tiles, num_sms, s);
  return launch_bwd<64, MODE, EPI>(A, B, Bs, O, Os, p, max_tiles, num_sms, s);
}

int bwd_bn(int64_t Nd) { return Nd % 256 == 0 ? 256 : (Nd % 128 == 0 ? 128 : 64); }

}  // namespace

// dOut [rows, K] . W[e] ([K, Nd] stored, per expert) -> out [rows, Nd], times
// act'(pre) when act >= 0; padding rows of each group written as zeros.
cudaError_t launch_bwd_dgrad(const moe_config& c, const BwdGemmArgs& g, const void* dOut,
                             const void* W, const void* Ws, int64_t K, int64_t Nd, int act,
                             const void* pre, void* out, cudaStream_t s) {
  if (bwd_dgrad_on_pair(c, K, Nd))
    return launch_bwd_dgrad_pair(c, g, dOut, W, Ws, K, Nd, act, pre, out, s);
  CUtensorMap mA, mB, mBs;
  const int bn = bwd_bn(Nd);
  if (!bwd_map(&mA, dOut, uint64_t(K), uint64_t(g.rows_max), 0, BM)) return cudaErrorInvalidValue;
  if (!bwd_map(&mB, W, uint64_t(Nd), uint64_t(K), uint64_t(c.n_experts), BK))
    return cudaErrorInvalidValue;
  if (c.d_ff_shared > 0) {
    if (!bwd_map(&mBs, Ws, uint64_t(Nd), uint64_t(K), 0, BK)) return cudaErrorInvalidValue;
  } else {
    mBs = mB;
  }
  BwdParams p{};
  p.offsets = g.offsets;
  p.kept = g.kept;
  p.n_routed = int32_t(c.n_experts);
  p.shared_rows = c.d_ff_shared > 0 ? int32_t(c.T) : 0;
  p.num_kb = int32_t(K / BK);
  p.Nd = Nd;
  p.out = out;
  p.pre = static_cast<const __nv_bfloat16*>(pre);
  p.status = g.status;
  p.wait_limit_ns = g.wait_limit_ns;
  const int64_t groups = c.n_experts + (c.d_ff_shared > 0 ? 1 : 0);
  const int64_t max_tiles = ((g.rows_max + BM - 1) / BM + groups) * (Nd / bn);
  if (act < 0)
    return launch_bwd_bn<MODE_DGRAD, BEPI_STORE>(bn, mA, mB, mBs, mA, mA, p, max_tiles,
                                                 g.num_sms, s);
  if (act == MOE_ACT_RELU)
    return launch_bwd_bn<MODE_DGRAD, BEPI_DRELU>(bn, mA, mB, mBs, mA, mA, p, max_tiles,
                                                 g.num_sms, s);
  return launch_bwd_bn<MODE_DGRAD, BEPI_DGELU>(bn, mA, mB, mBs, mA, mA, p, max_tiles,
                                               g.num_sms, s);
}

// out[e] = L[group e]^T . R[group e]: L [rows, Md], R [rows, Nd] -> [Md, Nd]
// per routed expert (out), the shared expert's into out_s.
cudaError_t launch_bwd_wgrad(const moe_config& c, const BwdGemmArgs& g, const void* Lm,
                             int64_t Md, const void* Rm, int64_t Nd, void* out, void* out_s,
                             cudaStream_t s) {
  CUtensorMap mA, mB, mO, mOs;
  const int bn = bwd_bn(Nd);
  if (!bwd_map(&mA, Lm, uint64_t(Md), uint64_t(g.rows_max), 0, BK)) return cudaErrorInvalidValue;
  if (!bwd_map(&mB, Rm, uint64_t(Nd), uint64_t(g.rows_max), 0, BK)) return cudaErrorInvalidValue;
  // outputs: boxes of 32 rows x bn/4 columns, one per epilogue warp and tile
  if (!bwd_map(&mO, out, uint64_t(Nd), uint64_t(Md), uint64_t(c.n_experts), 32,
               uint32_t(bn / 4)))
    return cudaErrorInvalidValue;
  if (c.d_ff_shared > 0) {
    if (!bwd_map(&mOs, out_s, uint64_t(Nd), uint64_t(Md), 0, 32, uint32_t(bn / 4)))
      return cudaErrorInvalidValue;
  } else {
    mOs = mO;
  }
  BwdParams p{};
  p.offsets = g.offsets;
  p.kept = g.kept;
  p.n_routed = int32_t(c.n_experts);
  p.shared_rows = c.d_ff_shared > 0 ? int32_t(c.T) : 0;
  p.Md = int32_t(Md);
  p.Nd = Nd;
  p.out = out;
  p.out_s = out_s;
  p.status = g.status;
  p.wait_limit_ns = g.wait_limit_ns;
  const int64_t groups = c.n_experts + (c.d_ff_shared > 0 ? 1 : 0);
  const int64_t max_tiles = groups * ((Md + BM - 1) / BM) * (Nd / bn);
  return launch_bwd_bn<MODE_WGRAD, BEPI_STORE>(bn, mA, mB, mB, mO, mOs, p, max_tiles, g.num_sms,
                                               s);
}

MOE_CHECKS_UNIT(grouped_bwd)

}  // namespace moe
