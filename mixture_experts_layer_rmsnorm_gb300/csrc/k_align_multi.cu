// k_align_multi.cu -- K1b + K2 over many CTAs, for large token counts.
//
// Same result as the single-CTA align (counts per expert, lists padded to
// `pad` rows, slots in increasing flat index t*k + j inside each list), split
// into three launches so that it scales with T ("CuTeDSL chez Perplexity",
// MoE dispatch/combine: the prefill dispatch assigns indices with local
// counters first and then combines them across blocks in global memory):
//   count   one CTA per 32 tokens: top-k + softmax of its tokens, then the
//           CTA's count per expert -> blk_counts[b][e]
//   scan    one CTA: totals, padded offsets, work-unit prefix sums, and each
//           CTA's base row per expert blk_base[b][e] (a prefix over b)
//   scatter one CTA per 32 tokens again: stable ranks of its entries (warp
//           match / popc + per-warp prefix), written to sorted_ids / slot_of
// Every step is deterministic.
#include "block_scan.cuh"
#include "moe_kernels.cuh"
#include "pdl.cuh"
#include "topk.cuh"

namespace moe {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int VPL>
__global__ void __launch_bounds__(kThreads)
    align_count_kernel(const float* __restrict__ logits, int T, int k, int renorm, int32_t* ids,
                       float* __restrict__ topk_w, int E, int32_t* __restrict__ blk_counts,
                       int32_t* __restrict__ flags, int n_flags, int32_t* __restrict__ err) {
  extern __shared__ int cnt[];  // [E]
  __shared__ int bad;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int b = blockIdx.x;
  const int t0 = b * kAlignTokPerBlk;
  const int t1 = min(T, t0 + kAlignTokPerBlk);
  pdl_wait();
  pdl_launch_dependents();
  if (b == 0)
    for (int i = tid; i < n_flags; i += kThreads) flags[i] = 0;
  if (tid == 0) bad = 0;
  for (int e = tid; e < E; e += kThreads) cnt[e] = 0;
  for (int t = t0 + warp; t < t1; t += kWarps)
    topk_softmax_warp<VPL>(logits + static_cast<size_t>(t) * E, E, k, renorm, ids + static_cast<size_t>(t) * k,
                           topk_w + static_cast<size_t>(t) * k);
  __syncthreads();
  for (int i = t0 * k + tid; i < t1 * k; i += kThreads) {
    int e = __ldcg(ids + i);
    if (e < 0 || e >= E) {  // only from non-finite logits: keep the routing in bounds, report it
      bad = 1;
      e = 0;
      ids[i] = 0;
    }
    atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  for (int e = tid; e < E; e += kThreads) blk_counts[static_cast<size_t>(b) * E + e] = cnt[e];
  if (tid == 0 && bad) {
    err[1] = kKernAlign;
    err[0] = kErrDevice;
  }
}

// One CTA of 1024 threads, thread e = expert e (E <= 1024).  The per-block
// counts are read once, by all threads together, into shared memory when they
// fit (kScanStageInts); each thread then walks its expert's column there
// instead of making nblk dependent trips to L2.
constexpr int kScanStageInts = 11264;  // 44 KB: with the static scan buffer, under the 48 KB default
__global__ void __launch_bounds__(1024)
    align_scan_kernel(const int32_t* __restrict__ blk_counts, int nblk, int E, int pad, int bn1, int tiles1, int bn2,
                      int tiles2, int N, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                      int32_t* __restrict__ unit_off1, int32_t* __restrict__ unit_off2,
                      int32_t* __restrict__ blk_base, int32_t* __restrict__ sorted_ids) {
  __shared__ int scan_tmp[3 * 33];
  extern __shared__ int staged[];  // [nblk][E] when nblk * E <= kScanStageInts
  pdl_wait();
  pdl_launch_dependents();
  const int n_counts = nblk * E;
  const bool stage = n_counts <= kScanStageInts;
  if (stage)
    for (int i = threadIdx.x; i < n_counts; i += 1024) staged[i] = __ldcg(blk_counts + i);
  __syncthreads();
  const int32_t* bc = stage ? staged : blk_counts;
  const int e = threadIdx.x;
  int c = 0;
  if (e < E)
    for (int b = 0; b < nblk; ++b) c += bc[static_cast<size_t>(b) * E + e];
  const int p = (c + pad - 1) / pad * pad;
  const int u1 = (bn1 > 0) ? (p + bn1 - 1) / bn1 * tiles1 : 0;
  const int u2 = (bn2 > 0) ? (p + bn2 - 1) / bn2 * tiles2 : 0;
  const int v3[3] = {p, u1, u2};
  int pre[3], tot[3];
  block_exclusive_scan3<1024>(v3, scan_tmp, pre, tot);
  const int off = pre[0], o1 = pre[1], o2 = pre[2];
  const int tot_p = tot[0], tot_u1 = tot[1], tot_u2 = tot[2];
  if (e < E) {
    counts[e] = c;
    offsets[e] = off;
    if (unit_off1) unit_off1[e] = o1;
    if (unit_off2) unit_off2[e] = o2;
    int run = off;
    for (int b = 0; b < nblk; ++b) {
      blk_base[static_cast<size_t>(b) * E + e] = run;
      run += bc[static_cast<size_t>(b) * E + e];
    }
    for (int q = off + c; q < off + p; ++q) sorted_ids[q] = N;  // padding rows
  }
  if (threadIdx.x == 0) {
    offsets[E] = tot_p;
    if (unit_off1) unit_off1[E] = tot_u1;
    if (unit_off2) unit_off2[E] = tot_u2;
  }
}

// Dynamic shared memory: cursor[E], wbase[E][kWarps] (ints).
__global__ void __launch_bounds__(kThreads)
    align_scatter_kernel(const int32_t* __restrict__ ids, int T, int k, int E, const int32_t* __restrict__ blk_base,
                         int32_t* __restrict__ sorted_ids, int32_t* __restrict__ slot_of) {
  extern __shared__ int sm[];
  int* cursor = sm;
  int* wbase = sm + E;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  const int i0 = b * kAlignTokPerBlk * k;
  const int i1 = min(T, (b + 1) * kAlignTokPerBlk) * k;
  pdl_wait();
  pdl_launch_dependents();
  for (int e = tid; e < E; e += kThreads) cursor[e] = blk_base[static_cast<size_t>(b) * E + e];
  __syncthreads();
  for (int base = i0; base < i1; base += kThreads) {
    const int i = base + tid;
    const bool valid = i < i1;
    const int e = valid ? ids[i] : -1;
    const unsigned same = __match_any_sync(kFull, e);
    const int rank = __popc(same & ((1u << lane) - 1u));
    for (int q = tid; q < kWarps * E; q += kThreads) wbase[q] = 0;
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
}

template <int VPL>
cudaError_t launch_count(dim3 grid, size_t smem, cudaStream_t stream, const float* logits, int T, int k, int renorm,
                         int32_t* ids, float* topk_w, int E, int32_t* blk_counts, int32_t* flags, int n_flags,
                         int32_t* err) {
  return launch_pdl(align_count_kernel<VPL>, grid, dim3(kThreads), smem, stream, logits, T, k, renorm, ids, topk_w, E,
                    blk_counts, flags, n_flags, err);
}

}  // namespace

int align_multi_blocks(int T) { return (T + kAlignTokPerBlk - 1) / kAlignTokPerBlk; }

cudaError_t launch_align_multi(const float* logits, int T, int k, int renorm, int32_t* topk_ids, float* topk_w, int E,
                               int pad, int bn1, int tiles1, int bn2, int tiles2, int32_t* counts, int32_t* offsets,
                               int32_t* sorted_ids, int32_t* slot_of, int32_t* unit_off1, int32_t* unit_off2,
                               int32_t* blk_counts, int32_t* blk_base, int32_t* err, int32_t* flags, int n_flags,
                               cudaStream_t stream, void* count_done_event) {
  const int nblk = align_multi_blocks(T);
  const dim3 grid(nblk);
  const size_t smem_count = static_cast<size_t>(E) * sizeof(int);
  cudaError_t st;
  switch (topk_vpl(E)) {
    case 1: st = launch_count<1>(grid, smem_count, stream, logits, T, k, renorm, topk_ids, topk_w, E, blk_counts, flags, n_flags, err); break;
    case 2: st = launch_count<2>(grid, smem_count, stream, logits, T, k, renorm, topk_ids, topk_w, E, blk_counts, flags, n_flags, err); break;
    case 4: st = launch_count<4>(grid, smem_count, stream, logits, T, k, renorm, topk_ids, topk_w, E, blk_counts, flags, n_flags, err); break;
    case 8: st = launch_count<8>(grid, smem_count, stream, logits, T, k, renorm, topk_ids, topk_w, E, blk_counts, flags, n_flags, err); break;
    case 16: st = launch_count<16>(grid, smem_count, stream, logits, T, k, renorm, topk_ids, topk_w, E, blk_counts, flags, n_flags, err); break;
    default: st = launch_count<32>(grid, smem_count, stream, logits, T, k, renorm, topk_ids, topk_w, E, blk_counts, flags, n_flags, err); break;
  }
  if (st != cudaSuccess) return st;
  if (count_done_event) {
    st = cudaEventRecord(static_cast<cudaEvent_t>(count_done_event), stream);
    if (st != cudaSuccess) return st;
  }
  const size_t smem_scan =
      static_cast<size_t>(nblk) * E <= kScanStageInts ? static_cast<size_t>(nblk) * E * sizeof(int) : 0;
  st = launch_pdl(align_scan_kernel, dim3(1), dim3(1024), smem_scan, stream, blk_counts, nblk, E, pad, bn1, tiles1,
                  bn2, tiles2, T * k, counts, offsets, unit_off1, unit_off2, blk_base, sorted_ids);
  if (st != cudaSuccess) return st;
  const size_t smem_scatter = static_cast<size_t>(1 + kWarps) * E * sizeof(int);
  return launch_pdl(align_scatter_kernel, grid, dim3(kThreads), smem_scatter, stream, topk_ids, T, k, E, blk_base,
                    sorted_ids, slot_of);
}

}  // namespace moe
