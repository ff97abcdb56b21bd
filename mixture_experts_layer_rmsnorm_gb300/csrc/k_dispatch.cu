// k_dispatch.cu -- K2 expert align, K3 gather into padded per-expert rows,
// K6 top-k weighted combine.
//
// Dispatch and combine follow "CuTeDSL chez Perplexity", MoE dispatch /
// combine, "Local": count the tokens routed to each expert, give each routed
// token a unique index in its expert's list, copy the tokens into optionally
// padded per-expert buffers for the MoE GEMM, and after the GEMMs accumulate
// each token's expert outputs in registers with its routing weights.
//
// The pages hand out list slots with atomic counters, which makes the order
// inside a list depend on timing.  Here slots follow the flat routing index
// t*k + j in increasing order, found with warp match/popc ranks and a
// per-warp prefix in shared memory, so the permutation is the same on every
// run.
#include <cuda_bf16.h>

#include "align_core.cuh"
#include "launch_config.cuh"
#include "moe_kernels.cuh"
#include "pdl.cuh"
#include "topk.cuh"

namespace moe {
namespace {

// One CTA of NT threads: 1024, or 256 for a handful of tokens (one warp per
// token still covers them in one round, and the block's barriers are
// cheaper).  Dynamic shared memory: cnt[E], cursor[E], wbase[E][NT/32]
// (ints), and ids_s[N] in the fused form.  With FUSED_TOPK the CTA first
// selects the top-k experts of all T tokens from the logits (one warp per
// token; used for small T, where a separate launch costs more than the work),
// keeps a copy of the ids in shared memory and aligns from it.  Otherwise the
// routing ids are read with L2-coherent loads.
template <int FUSED_VPL, int NT>  // FUSED_VPL 0: ids given; else top-k first, with FUSED_VPL logits per lane
__global__ void __launch_bounds__(NT)
    align_kernel(const float* __restrict__ logits, int T, int k, int renorm, float* __restrict__ topk_w,
                 int32_t* ids, int N, int E, int pad, int bn1, int tiles1, int bn2, int tiles2,
                 int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_ids,
                 int32_t* __restrict__ slot_of, int32_t* __restrict__ unit_off1, int32_t* __restrict__ unit_off2,
                 int32_t* __restrict__ err, int32_t* __restrict__ flags, int n_flags) {
  constexpr int kAlignThreads = NT, kAlignWarps = NT / 32;
  extern __shared__ int sm[];
  int* cnt = sm;                 // [E]
  int* cursor = sm + E;          // [E]
  int* wbase = sm + 2 * E;       // [E][NT / 32]
  int* ids_s = wbase + kAlignWarps * E;  // [N], fused form only
  __shared__ int scan_tmp[3 * 33];
  __shared__ int bad;
  const int tid = threadIdx.x, warp = tid >> 5;
  pdl_wait();
  pdl_launch_dependents();
  for (int i = tid; i < n_flags; i += kAlignThreads) flags[i] = 0;
  if constexpr (FUSED_VPL > 0) {
    for (int t = warp; t < T; t += kAlignWarps)
      topk_softmax_warp<FUSED_VPL>(logits + static_cast<size_t>(t) * E, E, k, renorm,
                                   ids + static_cast<size_t>(t) * k, topk_w + static_cast<size_t>(t) * k,
                                   ids_s + static_cast<size_t>(t) * k);
    __syncthreads();
  }

  const bool ok = align_core<kAlignThreads>(
      [&](int i) { return FUSED_VPL > 0 ? ids_s[i] : __ldcg(ids + i); }, N, E, pad, bn1, tiles1, bn2, tiles2, cnt,
      cursor, wbase, scan_tmp, &bad, counts, offsets, sorted_ids, slot_of, unit_off1, unit_off2);
  if (!ok) {
    if (tid == 0) {
      err[1] = kKernAlign;
      err[0] = kErrDevice;
    }
    // leave an empty, consistent routing behind: no rows, no units, and every
    // routed token pointing at row 0 (so the combine stays in bounds)
    for (int e = tid; e <= E; e += kAlignThreads) {
      offsets[e] = 0;
      if (unit_off1) unit_off1[e] = 0;
      if (unit_off2) unit_off2[e] = 0;
      if (e < E) counts[e] = 0;
    }
    for (int i = tid; i < N; i += kAlignThreads) slot_of[i] = 0;
  }
}

// One warp per padded row; 8 rows per block of 256 threads.  Padding rows
// are not written: each feeds only its own MMA column, whose results are
// never read.  The grid also zeroes clear[0, n_clear).
__global__ void __launch_bounds__(256) gather_kernel(const uint16_t* __restrict__ h, const int32_t* __restrict__ sorted_ids,
                                                     const int32_t* __restrict__ offsets, int E, int N, int k, int H,
                                                     int64_t P_max, uint16_t* __restrict__ xg,
                                                     int32_t* __restrict__ clear, int64_t n_clear) {
  pdl_wait();
  pdl_launch_dependents();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x; i < n_clear;
       i += static_cast<int64_t>(gridDim.x) * 256)
    clear[i] = 0;
  const int64_t p = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (p >= P_max || p >= offsets[E]) return;
  const int src = sorted_ids[p];
  if (src >= N || src < 0) return;  // padding row
  const int nch = H >> 3;
  uint4* dst = reinterpret_cast<uint4*>(xg + p * H);
  const uint4* s = reinterpret_cast<const uint4*>(h + static_cast<int64_t>(src / k) * H);
#pragma unroll 4
  for (int c = lane; c < nch; c += 32) dst[c] = __ldg(s + c);
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  const uint32_t hh = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return l | (hh << 16);
}

// Block (t, s) covers token t's output chunks [s * cpb, (s + 1) * cpb) of 8
// features; each thread owns 8 consecutive outputs (128-bit loads and stores)
// and accumulates over the k routed rows in order j = 0..k-1.  A token's slots
// and weights come from the align, at least two launches back, so they are
// read before the wait for the down GEMM (see pdl.cuh).
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ rows, const int32_t* __restrict__ slot_of,
                                                      const float* __restrict__ w, int T, int H, int k, int cpb,
                                                      uint16_t* __restrict__ y) {
  __shared__ int s_slot[32];
  __shared__ float s_w[32];
  const int t = blockIdx.x;
  if (threadIdx.x < k) {
    s_slot[threadIdx.x] = slot_of[static_cast<int64_t>(t) * k + threadIdx.x];
    s_w[threadIdx.x] = w[static_cast<int64_t>(t) * k + threadIdx.x];
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();
  const int nch = H >> 3;
  const int c_end = min(nch, static_cast<int>(blockIdx.y + 1) * cpb);
  for (int c = static_cast<int>(blockIdx.y) * cpb + threadIdx.x; c < c_end; c += blockDim.x) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    // up to 8 routed rows' loads in flight, then accumulated in j order
    for (int j0 = 0; j0 < k; j0 += 8) {
      uint4 v[8];
      float wj[8];
#pragma unroll
      for (int d = 0; d < 8; ++d) {
        if (j0 + d < k) {
          wj[d] = s_w[j0 + d];
          v[d] = __ldg(reinterpret_cast<const uint4*>(rows + static_cast<int64_t>(s_slot[j0 + d]) * H) + c);
        }
      }
#pragma unroll
      for (int d = 0; d < 8; ++d) {
        if (j0 + d < k) {
          float f[8];
          unpack8(v[d], f);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj[d], f[i], acc[i]);
        }
      }
    }
    uint4 o;
    o.x = pack2_bf16(acc[0], acc[1]);
    o.y = pack2_bf16(acc[2], acc[3]);
    o.z = pack2_bf16(acc[4], acc[5]);
    o.w = pack2_bf16(acc[6], acc[7]);
    reinterpret_cast<uint4*>(y + static_cast<int64_t>(t) * H)[c] = o;
  }
}

}  // namespace

template <int VPL, int NT>
cudaError_t launch_align_nt(const float* logits, int T, int k, int renorm, int32_t* topk_ids, float* topk_w, int N,
                            int E, int pad, int bn1, int tiles1, int bn2, int tiles2, int32_t* counts,
                            int32_t* offsets, int32_t* sorted_ids, int32_t* slot_of, int32_t* unit_off1,
                            int32_t* unit_off2, int32_t* err, int32_t* flags, int n_flags, cudaStream_t stream) {
  const size_t smem = (static_cast<size_t>(2 + NT / 32) * E + (VPL > 0 ? N : 0)) * sizeof(int);
  static PerDevice config;
  const cudaError_t e = config.get([](int&) {
    return cudaFuncSetAttribute(align_kernel<VPL, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
  });
  if (e != cudaSuccess) return e;
  return launch_pdl(align_kernel<VPL, NT>, dim3(1), dim3(NT), smem, stream, logits, T, k, renorm, topk_w, topk_ids, N,
                    E, pad, bn1, tiles1, bn2, tiles2, counts, offsets, sorted_ids, slot_of, unit_off1, unit_off2, err,
                    flags, n_flags);
}

// 256 threads for up to 8 tokens and 256 experts (one warp per token covers
// the top-k in one round, one thread per expert the align's scans, and the
// block's barriers are cheaper than with 1024), else 1024
template <int VPL>
cudaError_t launch_align_t(const float* logits, int T, int k, int renorm, int32_t* topk_ids, float* topk_w, int N,
                           int E, int pad, int bn1, int tiles1, int bn2, int tiles2, int32_t* counts, int32_t* offsets,
                           int32_t* sorted_ids, int32_t* slot_of, int32_t* unit_off1, int32_t* unit_off2,
                           int32_t* err, int32_t* flags, int n_flags, cudaStream_t stream) {
  if (VPL > 0 && T <= 8 && E <= 256)
    return launch_align_nt<VPL, 256>(logits, T, k, renorm, topk_ids, topk_w, N, E, pad, bn1, tiles1, bn2, tiles2,
                                     counts, offsets, sorted_ids, slot_of, unit_off1, unit_off2, err, flags, n_flags,
                                     stream);
  return launch_align_nt<VPL, 1024>(logits, T, k, renorm, topk_ids, topk_w, N, E, pad, bn1, tiles1, bn2, tiles2,
                                    counts, offsets, sorted_ids, slot_of, unit_off1, unit_off2, err, flags, n_flags,
                                    stream);
}


bool align_fuses_topk(int T, int E) { return T <= kFusedTopkMaxT && E <= kFusedTopkMaxE; }

cudaError_t launch_align(const float* logits, int T, int k, int renorm, int32_t* topk_ids, float* topk_w, int N,
                         int E, int pad, int bn1, int tiles1, int bn2, int tiles2, int32_t* counts, int32_t* offsets,
                         int32_t* sorted_ids, int32_t* slot_of, int32_t* unit_off1, int32_t* unit_off2, int32_t* err,
                         int32_t* flags, int n_flags, cudaStream_t stream) {
#define MOE_ALIGN_ARGS logits, T, k, renorm, topk_ids, topk_w, N, E, pad, bn1, tiles1, bn2, tiles2, counts, offsets, \
                       sorted_ids, slot_of, unit_off1, unit_off2, err, flags, n_flags, stream
  if (!align_fuses_topk(T, E)) return launch_align_t<0>(MOE_ALIGN_ARGS);
  switch (topk_vpl(E)) {
    case 1: return launch_align_t<1>(MOE_ALIGN_ARGS);
    case 2: return launch_align_t<2>(MOE_ALIGN_ARGS);
    case 4: return launch_align_t<4>(MOE_ALIGN_ARGS);
    default: return launch_align_t<8>(MOE_ALIGN_ARGS);
  }
#undef MOE_ALIGN_ARGS
}


cudaError_t launch_gather(const uint16_t* h, const int32_t* sorted_ids, const int32_t* offsets, int E, int N, int k,
                          int H, int64_t P_max, uint16_t* xg, int32_t* clear, int64_t n_clear, cudaStream_t stream) {
  const int64_t blocks = (P_max + 7) / 8;
  if (blocks == 0) return cudaSuccess;
  return launch_pdl(gather_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, h, sorted_ids, offsets, E,
                    N, k, H, P_max, xg, clear, n_clear);
}

cudaError_t launch_combine(const uint16_t* out_rows, const int32_t* slot_of, const float* topk_w, int T, int H, int k,
                           uint16_t* y, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int nch = H / 8;
  // few tokens: each token's row split over CTAs of 64 threads, one chunk of
  // 8 outputs per thread (the row loads of a thread are one round trip);
  // many tokens: one CTA of up to 256 threads per token
  int threads, cpb;
  if (T < 256) {
    threads = nch >= 64 ? 64 : (nch + 31) / 32 * 32;
    cpb = threads;
  } else {
    threads = nch >= 256 ? 256 : (nch + 31) / 32 * 32;
    cpb = nch;
  }
  const dim3 grid(T, (nch + cpb - 1) / cpb);
  return launch_pdl(combine_kernel, grid, dim3(threads), 0, stream, out_rows, slot_of, topk_w, T, H, k, cpb, y);
}

}  // namespace moe
