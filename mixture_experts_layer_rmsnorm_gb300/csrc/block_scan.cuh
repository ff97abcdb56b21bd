// block_scan.cuh -- block-wide exclusive prefix sum of one int per thread.
#pragma once

namespace moe {

// Exclusive scan over a block of exactly NT threads (NT a multiple of 32, at
// most 1024).  `tmp` is 33 ints of shared memory.  Returns this thread's
// exclusive prefix; *total receives the block total.  Contains
// __syncthreads(): all threads must call.
template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int v, int* tmp, int* total) {
  static_assert(NT % 32 == 0 && NT <= 1024, "block size");
  constexpr int kWarps = NT / 32;
  constexpr unsigned kAll = 0xFFFFFFFFu;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(kAll, inc, off);
    if (lane >= off) inc += o;
  }
  if (lane == 31) tmp[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int w = (lane < kWarps) ? tmp[lane] : 0;
    int winc = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(kAll, winc, off);
      if (lane >= off) winc += o;
    }
    tmp[lane] = winc - w;  // exclusive prefix of warp totals
    if (lane == 31) tmp[32] = winc;
  }
  __syncthreads();
  const int r = tmp[warp] + inc - v;
  *total = tmp[32];
  __syncthreads();
  return r;
}

__device__ __forceinline__ int block_exclusive_scan_1024(int v, int* tmp, int* total) {
  return block_exclusive_scan<1024>(v, tmp, total);
}

}  // namespace moe
