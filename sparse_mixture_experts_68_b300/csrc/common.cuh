// Shared device helpers of libmoe: element types, vector loads, the device
// status word and bounded waits on shared-memory barriers.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

constexpr int kGroupAlign = MOE_GROUP_ALIGN;

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// ---- element conversion ----------------------------------------------------

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// 16-byte vectors: 4 floats or 8 bf16.
template <typename T> struct Vec16;
template <> struct Vec16<float> {
  static constexpr int n = 4;
  __device__ __forceinline__ static void load(const float* p, float* o) {
    float4 v = *reinterpret_cast<const float4*>(p);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
  __device__ __forceinline__ static void store(float* p, const float* o) {
    *reinterpret_cast<float4*>(p) = make_float4(o[0], o[1], o[2], o[3]);
  }
};
template <> struct Vec16<__nv_bfloat16> {
  static constexpr int n = 8;
  __device__ __forceinline__ static void load(const __nv_bfloat16* p, float* o) {
    uint4 v = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(h[i]);
      o[2 * i] = f.x; o[2 * i + 1] = f.y;
    }
  }
  __device__ __forceinline__ static void store(__nv_bfloat16* p, const float* o) {
    uint4 v;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
    *reinterpret_cast<uint4*>(p) = v;
  }
};

// ---- activations -------------------------------------------------------------

// The hardware's approximate reciprocal and base-2 exponential (relative
// errors of a few fp32 ulps), one special-function instruction each.
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// erf by Abramowitz & Stegun, "Handbook of Mathematical Functions", formula
// 7.1.26: erf(z) = 1 - t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-z^2),
// t = 1 / (1 + p z) for z >= 0, odd in z; absolute error <= 1.5e-7, below
// fp32 resolution near 1 and far below the bf16 the hidden layer is stored in.
constexpr float kAsP = 0.3275911f;
constexpr float kAsA1 = 0.254829592f, kAsA2 = -0.284496736f, kAsA3 = 1.421413741f,
                kAsA4 = -1.453152027f, kAsA5 = 1.061405429f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRsqrt2 = 0.70710678118654752440f;

__device__ __forceinline__ float erf_as7126(float z) {
  const float a = fabsf(z);
  const float t = rcp_approx(fmaf(kAsP, a, 1.0f));
  float poly = fmaf(t, kAsA5, kAsA4);
  poly = fmaf(t, poly, kAsA3);
  poly = fmaf(t, poly, kAsA2);
  poly = fmaf(t, poly, kAsA1);
  const float r = 1.0f - t * poly * ex2_approx(-a * a * kLog2e);
  return copysignf(r, z);
}

// GELU with the exact (erf) form: 0.5 v (1 + erf(v / sqrt(2))).  With the
// erf above and q = t P(t) exp(-v^2 / 2) / 2 (z = |v| / sqrt(2)), this is
// v - v q for v >= 0 and v q for v < 0: the halving is folded into the
// coefficients and the sign into the last select.
__device__ __forceinline__ float gelu_erf(float v) {
  const float t = rcp_approx(fmaf(kAsP * kRsqrt2, fabsf(v), 1.0f));
  float q = fmaf(t, 0.5f * kAsA5, 0.5f * kAsA4);
  q = fmaf(t, q, 0.5f * kAsA3);
  q = fmaf(t, q, 0.5f * kAsA2);
  q = fmaf(t, q, 0.5f * kAsA1);
  const float e = ex2_approx(v * v * (-0.5f * kLog2e));
  const float r = v * (t * q * e);
  return v < 0.0f ? r : v - r;
}
// d GELU / d v = Phi(v) + v phi(v): the normal CDF (from the erf above) plus
// v times the normal density exp(-v^2 / 2) / sqrt(2 pi).
__device__ __forceinline__ float gelu_erf_grad(float v) {
  return 0.5f * (1.0f + erf_as7126(v * kRsqrt2)) +
         v * 0.39894228040143267794f * ex2_approx(v * v * (-0.5f * kLog2e));
}
__device__ __forceinline__ float apply_act(float v, int act) {
  return act == MOE_ACT_RELU ? fmaxf(v, 0.0f) : gelu_erf(v);
}

// ---- programmatic dependent launch ----------------------------------------------
// Every kernel of the layer lets the next launch start at once (its blocks can
// then run their local set-up on SMs this kernel frees) and waits for the
// previous kernel to complete -- with its memory visible -- before its first
// global-memory access.  Both are no-ops when the launch had no programmatic
// dependency.

__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait_previous() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---- shared-memory barriers with a time limit ---------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits until the barrier phase with the given parity has completed, or
// until limit_ns has passed; then records MOE_ERR_TIMEOUT in *status (the
// library's device status word) and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns, int32_t* status) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(a, parity)) return true;
    if ((it & 63u) == 0 && global_timer_ns() - t0 > limit_ns) {
      atomicCAS(status, MOE_OK, MOE_ERR_TIMEOUT);
      return false;
    }
  }
}

// ---- optional device-side checks (a build with -DMOE_CHECKS) ----------------
//
// MOE_CHECK(cond, site) guards an index before the access it controls.  In a
// checks build a failed check counts itself in its translation unit's record
// and the first one also records the site, the source line and the block;
// nothing traps, and the kernel carries on (the accesses stay bounded as in
// the ordinary build).  moe_checks_read gathers and clears every unit's
// record.  In the ordinary build the checks compile to nothing.
struct CheckRecord {
  int32_t fails, site, line, block;
};

enum CheckSite {
  CK_ROUTER_TOPK = 1,    // a selected expert outside [0, N)
  CK_SORT_EXPERT = 2,    // an expert id outside [0, N) reached the permutation
  CK_COPY_TOKEN = 3,     // a grouped row names a token outside [-1, T)
  CK_ROWS_TOTAL = 4,     // the grouped layout ends past rows_max
  CK_COMBINE_ROW = 5,    // a kept slot's row lies outside the routed groups
  CK_GEMM_ROWS = 6,      // a grouped Linear's group reaches past rows_max
  CK_EC_PICK = 7,        // an expert-choice pick outside [0, T)
};

#ifdef MOE_CHECKS
static __device__ CheckRecord g_tu_checks = {0, 0, 0, 0};

static __device__ __noinline__ void check_fail(int site, int line) {
  if (atomicAdd(&g_tu_checks.fails, 1) == 0) {
    g_tu_checks.site = site;
    g_tu_checks.line = line;
    g_tu_checks.block = int32_t(blockIdx.x);
  }
}
#define MOE_CHECK(cond, site)                                   \
  do {                                                          \
    if (!(cond)) ::moe::check_fail(int(site), __LINE__);        \
  } while (0)

// Host side: this unit's record (then cleared when `clear`).
inline cudaError_t read_tu_checks(CheckRecord* out, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_tu_checks, sizeof(CheckRecord));
  if (e == cudaSuccess && clear) {
    const CheckRecord zero = {0, 0, 0, 0};
    e = cudaMemcpyToSymbol(g_tu_checks, &zero, sizeof(CheckRecord));
  }
  return e;
}
#else
#define MOE_CHECK(cond, site) \
  do {                        \
  } while (0)
inline cudaError_t read_tu_checks(CheckRecord* out, bool) {
  *out = CheckRecord{0, 0, 0, 0};
  return cudaSuccess;
}
#endif

// Defines checks_read_<unit>(), the reader of one translation unit's record.
#define MOE_CHECKS_UNIT(unit)                                              \
  cudaError_t checks_read_##unit(::moe::CheckRecord* out, bool clear) {    \
    return ::moe::read_tu_checks(out, clear);                              \
  }

}  // namespace moe
