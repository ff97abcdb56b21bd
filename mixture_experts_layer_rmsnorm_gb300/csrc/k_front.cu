// k_front.cu -- the decode front end in one launch: RMSNorm + router logits,
// top-k + expert align, and the gather of the routed token rows, run by one
// thread-block cluster.
//
// In decode the layer's weights can only start to stream once the routing is
// known, so the kernels before the first expert GEMM are pure latency.  The
// pages run the decode dispatch as one kernel with a grid-wide barrier
// ("CuTeDSL chez Perplexity", "Synchronisation de la grille"; "Pré-remplir et
// décoder la spécialisation").  Here the grid is a single cluster, whose
// hardware barrier needs no counters in memory:
//   1. each CTA takes router work items (a tile of tokens x a group of
//      experts): RMSNorm of the tile's tokens, their logits for the group;
//      h and the logits go to global memory
//   2. cluster barrier (release / acquire: every CTA's h and logits are
//      visible to all)
//   3. every CTA runs top-k + softmax and the align of all tokens in its own
//      shared memory (the same deterministic result in each); CTA 0 publishes
//      the routing tables
//   4. each CTA copies its share of the routed rows h[t] -> xg[slot].  Padding
//      rows of xg are not written: they only feed MMA columns whose results are
//      never stored or read.  (One token: no copy; the gate/up GEMM reads h.)
// The arithmetic is that of the router kernel and the align kernels (same
// device functions), so h, the logits, the ids and the permutation are the
// same bits as on the multi-launch path.
#include <cuda_bf16.h>

#include "align_core.cuh"
#include "launch_config.cuh"
#include "moe_kernels.cuh"
#include "pdl.cuh"
#include "route_tile.cuh"
#include "tc_ptx.cuh"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int kFrontThreads = rt::kRouteWarps * 32;  // 256
constexpr int kFrontWarps = kFrontThreads / 32;

// shared memory of the align phase (ints), for N routed entries, E experts
__host__ __device__ inline size_t front_align_ints(int N, int E) {
  const int p_cap = N + (kPadRows - 1) * E;
  return static_cast<size_t>(2 * N)                 // ids, weights
         + 2 * E + kFrontWarps * E                  // cnt, cursor, wbase
         + E + 3 * (E + 1)                          // counts, offsets, two unit tables
         + p_cap + N                                // sorted_ids, slot_of
         + 3 * 33 + 1;                              // scan scratch, error flag
}

template <int TT, int TE, int VPL>
__global__ void __launch_bounds__(kFrontThreads, 1) front_kernel(const __grid_constant__ FrontArgs a) {
  extern __shared__ __align__(16) uint8_t fsm[];
  const int C = gridDim.x;   // the grid is one cluster
  const int c = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int N = a.T * a.k;

  for (int it = c; it < a.n_items; it += C) {
    const int e0 = (it % a.groups) * a.experts_per_item;
    rt::route_prefetch(a.w_router, a.g, a.H, e0, min(a.E, e0 + a.experts_per_item));
  }
  pdl_wait();
  pdl_launch_dependents();
  if (c == 0 && tid < 4) a.err[tid] = 0;
  for (int i = c * kFrontThreads + tid; i < a.n_flags; i += C * kFrontThreads) a.flags[i] = 0;
  for (int i = c * kFrontThreads + tid; i < a.n_combine_cnt; i += C * kFrontThreads) a.combine_cnt[i] = 0;

  // ---- 1. norm + logits of this CTA's work items
  uint4* h_s = reinterpret_cast<uint4*>(fsm);
  for (int it = c; it < a.n_items; it += C) {
    const int tt = it / a.groups, eg = it % a.groups;
    rt::norm_router_tile<TT, TE, false>(a.x, a.g, a.w_router, a.bias, a.T, a.H, a.E, a.eps, tt * TT,
                                 eg * a.experts_per_item, a.experts_per_item, eg == 0, a.h, a.logits, h_s);
    __syncthreads();  // h_s is reused by the next item
  }

  // ---- 2. every CTA's h rows and logits are visible cluster-wide after this
  ptx::cluster_sync();

  // ---- 3. top-k + align of all tokens, in this CTA's shared memory
  int* s = reinterpret_cast<int*>(fsm);
  const int E = a.E;
  const int p_cap = N + (kPadRows - 1) * E;
  int32_t* s_ids = s;
  float* s_w = reinterpret_cast<float*>(s_ids + N);
  int* cnt = reinterpret_cast<int*>(s_w + N);
  int* cursor = cnt + E;
  int* wbase = cursor + E;
  int32_t* s_counts = wbase + kFrontWarps * E;
  int32_t* s_offsets = s_counts + E;
  int32_t* s_unit1 = s_offsets + (E + 1);
  int32_t* s_unit2 = s_unit1 + (E + 1);
  int32_t* s_sorted = s_unit2 + (E + 1);
  int32_t* s_slot = s_sorted + p_cap;
  int* scan_tmp = s_slot + N;
  int* bad = scan_tmp + 3 * 33;

  for (int t = warp; t < a.T; t += kFrontWarps)
    topk_softmax_warp<VPL>(a.logits + static_cast<size_t>(t) * E, E, a.k, a.renorm, s_ids + t * a.k,
                           s_w + t * a.k);
  __syncthreads();
  const bool ok = align_core<kFrontThreads>([&](int i) { return s_ids[i]; }, N, E, a.pad, a.bn1, a.tiles1, a.bn2,
                                            a.tiles2, cnt, cursor, wbase, scan_tmp, bad, s_counts, s_offsets,
                                            s_sorted, s_slot, s_unit1, s_unit2);
  if (!ok) {
    // only from non-finite logits: report it and leave an empty, consistent
    // routing behind (no rows, no units, every routed token at row 0)
    if (c == 0) {
      if (tid == 0) {
        a.err[1] = kKernAlign;
        a.err[0] = kErrDevice;
      }
      for (int e = tid; e <= E; e += kFrontThreads) {
        a.offsets[e] = 0;
        a.unit_off1[e] = 0;
        a.unit_off2[e] = 0;
        if (e < E) a.counts[e] = 0;
      }
      for (int i = tid; i < N; i += kFrontThreads) {
        a.slot_of[i] = 0;
        a.ids[i] = s_ids[i];
        a.topk_w[i] = s_w[i];
      }
    }
    return;
  }
  const int P = s_offsets[E];
  if (c == 0) {
    for (int i = tid; i < N; i += kFrontThreads) {
      a.ids[i] = s_ids[i];
      a.topk_w[i] = s_w[i];
      a.slot_of[i] = s_slot[i];
    }
    for (int e = tid; e <= E; e += kFrontThreads) {
      a.offsets[e] = s_offsets[e];
      a.unit_off1[e] = s_unit1[e];
      a.unit_off2[e] = s_unit2[e];
      if (e < E) a.counts[e] = s_counts[e];
    }
    for (int p = tid; p < P; p += kFrontThreads) a.sorted_ids[p] = s_sorted[p];
  }

  // ---- 4. gather: one warp per routed row, 128-bit copies
  if (a.skip_gather) return;
  const int nch = a.H >> 3;
  for (int i = c * kFrontWarps + warp; i < N; i += C * kFrontWarps) {
    const int p = s_slot[i];
    const uint4* src = reinterpret_cast<const uint4*>(a.h + static_cast<int64_t>(i / a.k) * a.H);
    uint4* dst = reinterpret_cast<uint4*>(a.xg + static_cast<int64_t>(p) * a.H);
#pragma unroll 4
    for (int q = lane; q < nch; q += 32) dst[q] = __ldcg(src + q);  // h was written in this kernel
  }
}

template <int TT, int TE, int VPL>
struct FrontLauncher {
  static size_t smem(const FrontArgs& a) {
    const size_t tile = static_cast<size_t>(TT) * a.H * 2;
    const size_t al = front_align_ints(a.T * a.k, a.E) * 4;
    return tile > al ? tile : al;
  }
  // Cluster size to use on the current device (16 when the device allows a
  // non-portable cluster of 16 of these CTAs, else 8), 0 if none fits.
  static int cluster_size() {
    static PerDevice config;  // the attributes and the cluster size, once per device
    int size = 0;
    const cudaError_t e = config.get([](int& found) -> cudaError_t {
      auto kernel = front_kernel<TT, TE, VPL>;
      found = 0;
      if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kFrontMaxSmem) != cudaSuccess ||
          cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return cudaErrorNotSupported;
      for (int want : {16, 8}) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(want);
        cfg.blockDim = dim3(kFrontThreads);
        cfg.dynamicSmemBytes = kFrontMaxSmem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = want;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) == cudaSuccess && n >= 1) {
          found = want;
          return cudaSuccess;
        }
        cudaGetLastError();  // a refused size leaves no sticky error
      }
      return cudaSuccess;  // no size fits: 0
    }, &size);
    return e == cudaSuccess ? size : 0;
  }
  static cudaError_t launch(FrontArgs a, cudaStream_t stream) {
    const int C = cluster_size();
    if (C == 0) return cudaErrorNotSupported;
    // work items: token tiles x expert groups, about one per CTA
    const int tiles = (a.T + TT - 1) / TT;
    const int groups = tiles >= C ? 1 : C / tiles;
    int epi = (a.E + groups - 1) / groups;
    epi = (epi + TE - 1) / TE * TE;
    a.experts_per_item = epi;
    a.groups = (a.E + epi - 1) / epi;
    a.n_items = tiles * a.groups;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C);
    cfg.blockDim = dim3(kFrontThreads);
    cfg.dynamicSmemBytes = smem(a);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, front_kernel<TT, TE, VPL>, a);
  }
};

template <int TT, int TE>
cudaError_t launch_front_tt(const FrontArgs& a, cudaStream_t stream) {
  switch (topk_vpl(a.E)) {
    case 1: return FrontLauncher<TT, TE, 1>::launch(a, stream);
    case 2: return FrontLauncher<TT, TE, 2>::launch(a, stream);
    case 4: return FrontLauncher<TT, TE, 4>::launch(a, stream);
    default: return FrontLauncher<TT, TE, 8>::launch(a, stream);
  }
}

}  // namespace

bool front_fits(int T, int H, int E, int k) {
  if (T < 1 || T > kFrontMaxT || E > kFrontMaxE || k > 32) return false;
  const int TT = T <= 3 ? 1 : 4;
  const size_t tile = static_cast<size_t>(TT) * H * 2;
  const size_t al = front_align_ints(T * k, E) * 4;
  if ((tile > al ? tile : al) > static_cast<size_t>(kFrontMaxSmem)) return false;
  return (T <= 3 ? FrontLauncher<1, 1, 8>::cluster_size() : FrontLauncher<4, 2, 8>::cluster_size()) > 0;
}

cudaError_t launch_front(const FrontArgs& a, cudaStream_t stream) {
  if (a.T <= 3) return launch_front_tt<1, 1>(a, stream);
  return launch_front_tt<4, 2>(a, stream);
}

}  // namespace moe
