// topk.cuh -- one warp selects a token's top-k experts and their softmax weights.
#pragma once

#include <cfloat>
#include <climits>
#include <cstdint>

namespace moe {

// Warp-cooperative (all 32 lanes call it with the same arguments).
// l[E] (E <= 32 * VPL): the token's fp32 logits; VPL = values per lane.  Writes ids[k] (largest logit
// first; equal logits: lower expert index first) and w[k]: the softmax over
// all E taken at the selected experts, or over the selected ones only
// (renormalised) when renorm != 0.  k <= 32.  The logits are read with
// L2-coherent loads, so they may have been written earlier in the same kernel.
template <int VPL>
__device__ __forceinline__ void topk_softmax_warp(const float* l, int E, int k, int renorm, int32_t* ids,
                                                  float* w) {
  constexpr unsigned kAll = 0xFFFFFFFFu;
  const int lane = threadIdx.x & 31;
  float v[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? __ldcg(l + e) : -FLT_MAX;
  }
  uint32_t taken = 0;
  float my_v = 0.0f;  // lane j keeps the j-th selection
  int my_e = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int be = INT_MAX;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < be))) {
        bv = v[i];
        be = e;
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const float ov = __shfl_xor_sync(kAll, bv, off);
      const int oe = __shfl_xor_sync(kAll, be, off);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == j) {
      my_v = bv;
      my_e = be;
    }
  }
  const float m = __shfl_sync(kAll, my_v, 0);  // the largest logit
  float s = 0.0f;
  if (renorm) {
    s = (lane < k) ? expf(my_v - m) : 0.0f;
  } else {
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (lane + 32 * i < E) s += expf(v[i] - m);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(kAll, s, off);
  if (lane < k) {
    ids[lane] = my_e;
    w[lane] = expf(my_v - m) / s;
  }
}

// values per lane for E experts, rounded up to a power of two
__host__ __device__ inline int topk_vpl(int E) {
  const int need = (E + 31) / 32;
  int v = 1;
  while (v < need) v <<= 1;
  return v;
}

}  // namespace moe
