// align_core.cuh -- the expert align of one CTA: counts, padded offsets,
// work-unit prefix sums and the stable permutation (sorted_ids / slot_of).
//
// "CuTeDSL chez Perplexity", MoE dispatch / combine, "Local": count the
// tokens routed to each expert and give each routed token a unique index in
// its expert's (optionally padded) list.  The pages hand out the indices with
// atomic counters; here the list of expert e holds the flat routing indices
// i = t*k + j with ids[i] == e in increasing i (warp match/popc ranks plus a
// per-warp prefix in shared memory), so the permutation is the same on every
// run.  Each list is padded to a multiple of `pad` rows with the sentinel N.
#pragma once

#include <cstdint>

#include "block_scan.cuh"

namespace moe {

// NT threads (E <= NT) call it together.  id_at(i) returns ids[i] (0 <= i < N).
// Shared scratch: cnt[E], cursor[E], wbase[E][NT/32], scan_tmp[3 * 33], *bad.
// Outputs may live in shared or global memory; unit_off1/2 may be null (a
// table is only written when its bn > 0).  Returns false, having written no
// output, when an id lies outside [0, E) (the result is uniform over the CTA).
template <int NT, typename IdAt>
__device__ bool align_core(IdAt id_at, int N, int E, int pad, int bn1, int tiles1, int bn2, int tiles2, int* cnt,
                           int* cursor, int* wbase, int* scan_tmp, int* bad, int32_t* counts, int32_t* offsets,
                           int32_t* sorted_ids, int32_t* slot_of, int32_t* unit_off1, int32_t* unit_off2) {
  constexpr int kWarps = NT / 32;
  constexpr unsigned kFull = 0xFFFFFFFFu;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) *bad = 0;
  for (int e = tid; e < E; e += NT) cnt[e] = 0;
  __syncthreads();
  for (int i = tid; i < N; i += NT) {
    const int e = id_at(i);
    if (e < 0 || e >= E)
      *bad = 1;
    else
      atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  if (*bad) return false;

  // padded sizes, offsets and work-unit prefix sums (thread e = expert e)
  {
    const int e = tid;
    const int c = (e < E) ? cnt[e] : 0;
    const int p = (c + pad - 1) / pad * pad;
    const int u1 = (bn1 > 0) ? (p + bn1 - 1) / bn1 * tiles1 : 0;
    const int u2 = (bn2 > 0) ? (p + bn2 - 1) / bn2 * tiles2 : 0;
    const int v3[3] = {p, u1, u2};
    int pre[3], tot[3];
    block_exclusive_scan3<NT>(v3, scan_tmp, pre, tot);
    const int off = pre[0], o1 = pre[1], o2 = pre[2];
    const int tot_p = tot[0], tot_u1 = tot[1], tot_u2 = tot[2];
    if (e < E) {
      counts[e] = c;
      offsets[e] = off;
      cursor[e] = off;
      if (bn1 > 0) unit_off1[e] = o1;
      if (bn2 > 0) unit_off2[e] = o2;
      for (int q = off + c; q < off + p; ++q) sorted_ids[q] = N;  // padding rows
    }
    if (tid == 0) {
      offsets[E] = tot_p;
      if (bn1 > 0) unit_off1[E] = tot_u1;
      if (bn2 > 0) unit_off2[E] = tot_u2;
    }
  }
  __syncthreads();

  // stable ranks, NT routing entries per round
  for (int base = 0; base < N; base += NT) {
    const int i = base + tid;
    const bool valid = i < N;
    const int e = valid ? id_at(i) : -1;
    const unsigned same = __match_any_sync(kFull, e);
    const int rank = __popc(same & ((1u << lane) - 1u));
    for (int q = tid; q < kWarps * E; q += NT) wbase[q] = 0;
    __syncthreads();
    if (valid && rank == 0) wbase[e * kWarps + warp] = __popc(same);
    __syncthreads();
    // per expert, an exclusive scan over the warps' counts (one warp per
    // expert, lane w = warp w), offset by the expert's cursor
    for (int ex = warp; ex < E; ex += kWarps) {
      const int c = (lane < kWarps) ? wbase[ex * kWarps + lane] : 0;
      int inc = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(kFull, inc, off);
        if (lane >= off) inc += o;
      }
      const int cur = cursor[ex];
      if (lane < kWarps) wbase[ex * kWarps + lane] = cur + inc - c;
      __syncwarp();
      if (lane == 31) cursor[ex] = cur + inc;
    }
    __syncthreads();
    if (valid) {
      const int pos = wbase[e * kWarps + warp] + rank;
      sorted_ids[pos] = i;
      slot_of[i] = pos;
    }
    __syncthreads();
  }
  return true;
}

}  // namespace moe
