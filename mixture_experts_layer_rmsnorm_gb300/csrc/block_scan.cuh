// block_scan.cuh -- block-wide exclusive prefix sums of ints held one per thread.
#pragma once

namespace moe {

// Three independent exclusive scans over a block of exactly NT threads (NT a
// multiple of 32, at most 1024) in one pass: one set of barriers for all three.
// `tmp` is 3 * 33 ints of shared memory.  v[i] in; prefix[i] (this thread's
// exclusive prefix) and total[i] (the block total) out.  Contains
// __syncthreads(): all threads must call.
template <int NT>
__device__ __forceinline__ void block_exclusive_scan3(const int (&v)[3], int* tmp, int (&prefix)[3], int (&total)[3]) {
  static_assert(NT % 32 == 0 && NT <= 1024, "block size");
  constexpr int kWarps = NT / 32;
  constexpr unsigned kAll = 0xFFFFFFFFu;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc[3] = {v[0], v[1], v[2]};
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      const int o = __shfl_up_sync(kAll, inc[q], off);
      if (lane >= off) inc[q] += o;
    }
  }
  if (lane == 31)
#pragma unroll
    for (int q = 0; q < 3; ++q) tmp[q * 33 + warp] = inc[q];
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      const int w = (lane < kWarps) ? tmp[q * 33 + lane] : 0;
      int winc = w;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(kAll, winc, off);
        if (lane >= off) winc += o;
      }
      tmp[q * 33 + lane] = winc - w;  // exclusive prefix of warp totals
      if (lane == 31) tmp[q * 33 + 32] = winc;
    }
  }
  __syncthreads();
#pragma unroll
  for (int q = 0; q < 3; ++q) {
    prefix[q] = tmp[q * 33 + warp] + inc[q] - v[q];
    total[q] = tmp[q * 33 + 32];
  }
  __syncthreads();
}

}  // namespace moe
