// k_route.cu -- K1: fused RMSNorm + router logits (top-k runs in the align kernels).
//
// RMSNorm ("4 · La fusion de noyaux", §4.2 "Réduction + élémentaire"; "CuTeDSL
// chez Perplexity", "Norme QK"): one warp per token row, 128-bit loads of 8
// bf16 per lane, fp32 sum of squares reduced by an xor butterfly of warp
// shuffles, h = bf16((x * rstd) * g) with rstd = 1/sqrt(mean + eps).
//
// Router: l_e = sum_j h_j Wr[e,j] (+ b_e) in fp32.  Every dot product (and
// the sum of squares) is taken in one fixed order so that the routing
// decision is reproducible bit for bit:
//   chunk c = elements [8c, 8c+8) belongs to lane c mod 32; a lane runs over
//   its chunks in increasing c, one fused multiply-add per element in
//   increasing index, from +0; the 32 lane sums are combined by
//   v += shfl_xor(v, off) for off = 16, 8, 4, 2, 1.
// All roundings are explicit (__fmaf_rn, __fadd_rn, __fmul_rn, __fdiv_rn,
// __fsqrt_rn), so the compiler cannot contract or reorder them.
#include <cuda_bf16.h>

#include <cfloat>
#include <climits>

#include "launch_config.cuh"
#include "moe_kernels.cuh"
#include "pdl.cuh"
#include "route_tile.cuh"

namespace moe {
namespace {

// grid = (ceil(T / TT), ceil(E / experts_per_cta)), block = 256, dyn smem = TT*H*2.
template <int TT, int TE, bool PAIRED = false>
__global__ void __launch_bounds__(rt::kRouteWarps * 32, (TT >= 8) ? 2 : 1)
    norm_router_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ g,
                       const float* __restrict__ w_router, const float* __restrict__ bias, int T, int H, int E,
                       float eps, int experts_per_cta, uint16_t* __restrict__ h_out, float* __restrict__ logits,
                       int32_t* __restrict__ err) {
  extern __shared__ uint4 h_s[];  // [TT][H/8]
  const int t0 = blockIdx.x * TT;
  const int e0 = blockIdx.y * experts_per_cta;
  // The router rows this CTA will need and the norm gain do not depend on the
  // previous kernel: start pulling them into L2 now, so that their DRAM
  // latency overlaps the RMSNorm below.
  rt::route_prefetch(w_router, g, H, e0, min(E, e0 + experts_per_cta));
  pdl_wait();
  pdl_launch_dependents();
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x < 4) err[threadIdx.x] = 0;
  rt::norm_router_tile<TT, TE, true, PAIRED>(x, g, w_router, bias, T, H, E, eps, t0, e0, experts_per_cta,
                                             blockIdx.y == 0, h_out, logits, h_s);
}

template <int TT, int TE, bool PAIRED = false>
cudaError_t launch_nr(const uint16_t* x, const uint16_t* g, const float* wr, const float* bias, int T, int H, int E,
                      float eps, uint16_t* h, float* logits, int32_t* err, int num_sms, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(TT) * H * 2;
  static PerDevice config;  // the attribute is per device
  const cudaError_t ce = config.get([](int&) {
    return cudaFuncSetAttribute(norm_router_kernel<TT, TE, PAIRED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                200 * 1024);
  });
  if (ce != cudaSuccess) return ce;
  const int tiles = (T + TT - 1) / TT;
  const int group = rt::kRouteWarps * TE;
  // fewer token tiles than SMs: one expert group per CTA spreads the work
  // (and the router weights) over the SMs; otherwise a CTA takes all experts
  // so that its tokens are normalised once
  int epc = group;
  if (tiles >= num_sms) epc = (E + group - 1) / group * group;
  dim3 grid(tiles, (E + epc - 1) / epc);
  return launch_pdl(norm_router_kernel<TT, TE, PAIRED>, grid, dim3(rt::kRouteWarps * 32), smem, stream, x, g, wr,
                    bias, T, H, E, eps, epc, h, logits, err);
}

}  // namespace

cudaError_t launch_norm_router(const uint16_t* x, const uint16_t* g, const float* w_router, const float* bias,
                               int T, int H, int E, float eps, uint16_t* h, float* logits, int32_t* err,
                               int num_sms, cudaStream_t stream) {
  if (T <= 3) return launch_nr<1, 1>(x, g, w_router, bias, T, H, E, eps, h, logits, err, num_sms, stream);
  if (T <= 64) return launch_nr<4, 1>(x, g, w_router, bias, T, H, E, eps, h, logits, err, num_sms, stream);
  if (H > 8192)
    return launch_nr<4, 2>(x, g, w_router, bias, T, H, E, eps, h, logits, err, num_sms, stream);
  // Large batches with rows up to 4096: 14-token tiles (two CTAs of 112 KB
  // per SM) cover T = 4096 in 293 CTAs, one wave over 152 SMs x 2, where
  // 8-token tiles need 1.7 waves; the tokens go in pairs through the paired
  // FMA.  Only once the 14-token tiles alone fill the SMs: with fewer tiles
  // the expert groups are split over CTAs, and the 8-token tiles do that
  // better.
  if (H <= 4096 && (T + 13) / 14 >= num_sms)
    return launch_nr<14, 4, true>(x, g, w_router, bias, T, H, E, eps, h, logits, err, num_sms, stream);
  return launch_nr<8, 4>(x, g, w_router, bias, T, H, E, eps, h, logits, err, num_sms, stream);
}

}  // namespace moe
