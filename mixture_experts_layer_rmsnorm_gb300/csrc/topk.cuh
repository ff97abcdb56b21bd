// topk.cuh -- one warp selects a token's top-k experts and their softmax weights.
#pragma once

#include <cfloat>
#include <climits>
#include <cstdint>

namespace moe {

// Order-preserving key of a logit for unsigned comparison: larger value ->
// larger key; -0 and +0 share a key; 0 is kept for "not a candidate" (NaN,
// an expert already taken, a lane past E), so NaN is never selected.
__device__ __forceinline__ uint32_t topk_key(float v) {
  if (v != v) return 0u;
  if (v == 0.0f) v = 0.0f;  // -0 -> +0: equal logits tie on the expert index
  const uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);  // -inf -> 0x007FFFFF > 0
}

// Warp-cooperative (all 32 lanes call it with the same arguments).
// l[E] (E <= 32 * VPL): the token's fp32 logits; VPL = values per lane.  Writes ids[k] (largest logit
// first; equal logits: lower expert index first) and w[k]: the softmax over
// all E taken at the selected experts, or over the selected ones only
// (renormalised) when renorm != 0.  k <= 32.  The logits are read with
// L2-coherent loads, so they may have been written earlier in the same kernel.
// ids_s: optional second copy of ids (e.g. in shared memory).  Each selection
// is a warp max of keys, then a warp min of the expert index among the lanes
// holding that key (two redux.sync).  A step with no candidate left selects
// expert INT_MAX (reported by the align as an id out of range).
template <int VPL>
__device__ __forceinline__ void topk_softmax_warp(const float* l, int E, int k, int renorm, int32_t* ids,
                                                  float* w, int32_t* ids_s = nullptr) {
  constexpr unsigned kAll = 0xFFFFFFFFu;
  const int lane = threadIdx.x & 31;
  float v[VPL];
  uint32_t key[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? __ldcg(l + e) : -FLT_MAX;
    key[i] = (e < E) ? topk_key(v[i]) : 0u;
  }
  float my_v = 0.0f;  // lane j keeps the j-th selection
  int my_e = 0;
  for (int j = 0; j < k; ++j) {
    // this lane's best candidate: largest key, lowest expert index on ties
    uint32_t bk = 0u;
    int bi = 0;
    float bv = -INFINITY;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (key[i] > bk) {
        bk = key[i];
        bi = i;
        bv = v[i];
      }
    const uint32_t mk = __reduce_max_sync(kAll, bk);
    const uint32_t cand = (mk != 0u && bk == mk) ? static_cast<uint32_t>(lane + 32 * bi) : 0xFFFFFFFFu;
    const uint32_t be = __reduce_min_sync(kAll, cand);
    int sel = INT_MAX;
    float sv = -INFINITY;
    if (mk != 0u) {
      sel = static_cast<int>(be);
      if ((sel & 31) == lane) {
#pragma unroll
        for (int i = 0; i < VPL; ++i)
          if (i == (sel >> 5)) key[i] = 0u;  // taken
      }
    }
    sv = __shfl_sync(kAll, bv, sel & 31);  // the selected lane's own best is the selection
    if (mk == 0u) sv = -INFINITY;
    if (lane == j) {
      my_v = sv;
      my_e = sel;
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
    if (ids_s) ids_s[lane] = my_e;
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
