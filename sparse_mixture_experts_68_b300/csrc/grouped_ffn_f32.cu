// fp32 expert FFN on CUDA cores: H = act(Xp . W1[e]^T + b1[e]),
// Yp = H . W2[e]^T + b2[e] per expert group (botmartz.com "Mixture of Experts
// (MoE) and Mixtral", "Expert Routing": Linear -> GELU -> Linear;
// codingnowai.in "Mixture of Experts", "Code": Linear -> ReLU -> Linear).
// The fp32 layer keeps full fp32 products and sums (tf32 tensor-core inputs
// would round the operands to 11 bits).
#include "kernels.h"
#include "simt_gemm.cuh"

namespace moe {

cudaError_t launch_grouped_ffn_f32(const moe_config& c, const GroupedFfnArgs& g,
                                   cudaStream_t s) {
  if (g.rows_max == 0) return cudaSuccess;
  SimtGemmArgs a{};
  a.offsets = g.offsets;
  a.kept = g.kept;
  a.n_routed = int32_t(c.n_experts);
  a.shared_rows = c.d_ff_shared > 0 ? int32_t(c.T) : 0;
  a.act = c.act;
  // first Linear: [rows, d] x [d_ff, d]^T
  a.A = g.Xp; a.B = g.w->W1; a.Bs = g.w->W1s; a.bias = g.w->b1; a.bias_s = g.w->b1s;
  a.C = g.H; a.K = c.d_model; a.Nc = c.d_ff;
  // the pre-activation for a later backward, from the same epilogue
  a.C_pre = g.pre_out;
  cudaError_t e = launch_simt_gemm<float, float>(a, g.rows_max, g.num_sms, s);
  a.C_pre = nullptr;
  if (e == cudaSuccess) e = record_event(g.mid_event, s);
  if (e != cudaSuccess) return e;
  // second Linear: [rows, d_ff] x [d, d_ff]^T
  a.act = -1;
  a.A = g.H; a.B = g.w->W2; a.Bs = g.w->W2s; a.bias = g.w->b2; a.bias_s = g.w->b2s;
  a.C = g.Yp; a.K = c.d_ff; a.Nc = c.d_model;
  return launch_simt_gemm<float, float>(a, g.rows_max, g.num_sms, s);
}

// ---- backward on CUDA cores (fp32 layers) ----------------------------------------------

// out = A W^T + b per group, no activation (the recomputed pre-activation)
cudaError_t launch_grouped_linear_f32(const moe_config& c, const BwdGemmArgs& g, const void* A,
                                      const void* W, const void* Ws, const void* bias,
                                      const void* bias_s, void* out, int64_t K, int64_t Nd,
                                      cudaStream_t s) {
  if (g.rows_max == 0) return cudaSuccess;
  SimtGemmArgs a{};
  a.offsets = g.offsets;
  a.kept = g.kept;
  a.n_routed = int32_t(c.n_experts);
  a.shared_rows = c.d_ff_shared > 0 ? int32_t(c.T) : 0;
  a.act = -1;
  a.A = A; a.B = W; a.Bs = Ws; a.bias = bias; a.bias_s = bias_s;
  a.C = out; a.K = K; a.Nc = Nd;
  return launch_simt_gemm<float, float>(a, g.rows_max, g.num_sms, s);
}

// out = dOut W[e] per group (the weight as stored, [K, Nd]), times act'(pre)
// when act >= 0
cudaError_t launch_bwd_dgrad_f32(const moe_config& c, const BwdGemmArgs& g, const void* dOut,
                                 const void* W, const void* Ws, int64_t K, int64_t Nd, int act,
                                 const void* pre, void* out, cudaStream_t s) {
  if (g.rows_max == 0) return cudaSuccess;
  SimtGemmArgs a{};
  a.offsets = g.offsets;
  a.kept = g.kept;
  a.n_routed = int32_t(c.n_experts);
  a.shared_rows = c.d_ff_shared > 0 ? int32_t(c.T) : 0;
  a.act = -1;
  a.b_kn = 1;
  a.dact = act;
  a.pre = act >= 0 ? pre : nullptr;
  a.A = dOut; a.B = W; a.Bs = Ws;
  a.C = out; a.K = K; a.Nc = Nd;
  return launch_simt_gemm<float, float>(a, g.rows_max, g.num_sms, s);
}

// out[e] = L[group e]^T R[group e] per group ([Md, Nd]; the shared one in out_s)
cudaError_t launch_bwd_wgrad_f32(const moe_config& c, const BwdGemmArgs& g, const void* Lm,
                                 int64_t Md, const void* Rm, int64_t Nd, void* out, void* out_s,
                                 cudaStream_t s) {
  SimtWgradArgs a{};
  a.L = Lm; a.R = Rm; a.C = out; a.Cs = out_s; a.Md = Md; a.Nd = Nd;
  a.offsets = g.offsets;
  a.kept = g.kept;
  a.n_routed = int32_t(c.n_experts);
  a.shared_rows = c.d_ff_shared > 0 ? int32_t(c.T) : 0;
  const unsigned groups = unsigned(c.n_experts + (c.d_ff_shared > 0 ? 1 : 0));
  // 128 x 128 tiles when they still give about two blocks per SM, else 64 x 64
  const int64_t want = 2 * int64_t(g.num_sms > 0 ? g.num_sms : 148);
  if (ceil_div(Nd, 128) * ceil_div(Md, 128) * groups >= want)
    return launch_pdl(simt_wgrad_kernel<float, 128, 128>,
                      dim3(unsigned(ceil_div(Nd, 128)), unsigned(ceil_div(Md, 128)), groups),
                      dim3(kSimtThreads), 0, s, a);
  return launch_pdl(simt_wgrad_kernel<float, 64, 64>,
                    dim3(unsigned(ceil_div(Nd, 64)), unsigned(ceil_div(Md, 64)), groups),
                    dim3(kSimtThreads), 0, s, a);
}

MOE_CHECKS_UNIT(grouped_ffn_f32)

}  // namespace moe
