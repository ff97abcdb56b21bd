// k_expert_gemm.cu -- K4 gate/up grouped GEMM with the SwiGLU epilogue and K5
// down grouped GEMM, on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// Mapping.  For every expert e the layer computes C[n_e, F] = X_e[n_e, K] W_e^T
// with X_e the e-th list of gathered token rows and W_e [F, K] the expert's
// weight.  The MMA's M dimension is fixed at 128 rows, while an expert often
// holds only a handful of tokens in decode.  So the weights take the M side:
// each work unit computes C^T tile = W_e[128 rows, K] * X_e[n tok, K]^T, the
// transposition trick of the fused-MoE article ("Swap-AB para la utilización
// de WGMMA", Fig. 1), re-done for tcgen05 (M = 128, N = tokens in
// multiples of 16 up to 256).  The same mapping serves prefill: a unit then
// covers 128 weight rows x up to 256 tokens.
//
// Gate/up: W13[e] holds W_gate^T in rows [0, I) and W_up^T in rows [I, 2I) (the
// concatenated (d x 2 d_ff) weight of "4 · La fusion de noyaux", §4.2
// "GEMM + GEMM").  A unit covers 64 features [i0, i0+64): its 128-row A tile
// interleaves them in groups of 16, gate rows i0+16g .. +15 then the matching
// up rows, for g = 0..3 (one 5-D TMA box over the [E][2][I/16][16][H] view of
// W13).  One MMA per K step then leaves, in the 32 TMEM lanes of epilogue warp
// g, gate(i0+16g+l) in lane l and up(i0+16g+l) in lane 16+l, so the warp pairs
// them with one shuffle and applies SiLU(gate) * up to the accumulators before
// the only store ("GEMM + épilogue", §4.2).
//
// Work split.  Units are dealt round-robin to the persistent CTAs, except in
// the decode tile plan (each weight tile read once, so no L2 reuse to keep),
// which splits stream-K: the U units x KB K-blocks form one list of
// iterations; CTA c (of G persistent CTAs) takes the contiguous range
// [c*W/G, (c+1)*W/G), W = U*KB, so every CTA streams the same number of
// weight bytes whatever the routing.  A range can start or end inside a
// unit: the CTA that holds a unit's first K-blocks finishes that unit, as
// the last work of its range; every later CTA that holds a part of the unit
// does that part first, writes the fp32 partial sums of its TMEM accumulator
// to a per-CTA slot in global memory and raises one flag per TMEM lane
// quarter.  The finishing CTA adds the partials of the following CTAs
// before its epilogue, so it never waits on work that has not started.
//
// Roles in a CTA of 192 threads (320 for block-scaled pairs and for the FP4
// layers' one-CTA units; persistent, one CTA per SM):
//   warp 0 lane 0   TMA producer: weight tiles [128 x 64] (one box) and token
//                   tiles of TOKBOX rows per box, 128-byte swizzle, into a
//                   STAGES-deep ring
//   warp 1          owns the TMEM allocation; lane 0 issues tcgen05.mma and
//                   tcgen05.commit (frees a ring slot / hands an accumulator
//                   buffer to the epilogue)
//   warps 2..5      epilogue: tcgen05.ld of their TMEM lane quarter, partial
//                   sums, SwiGLU or plain bf16 convert, global stores (warps
//                   2..9, two per quarter, for block-scaled pairs: their
//                   single accumulator buffer must drain quickly)
//   warps 6..9      FP4 layers, one-CTA units: scale warps, one per TMEM lane
//                   quarter, writing each stage's scale tiles into TMEM with
//                   tcgen05.st (elsewhere the MMA thread copies them with
//                   tcgen05.cp before its MMAs)
// Block-scaled operands (MX): E4M3 (MXFP8), E2M1 weights spread by the 4-bit
// TMA type to the E4M3 image (W4), packed E2M1 tokens too (A4, kind::mxf4, 256
// elements of K per stage) or NVFP4 (NV, kind::mxf4nvf4, E4M3 scales per 16
// and the fp32 tensor scales applied in the epilogue); scales in 512-byte tiles
// copied per stage into TMEM columns next to the accumulators.
// Two accumulator buffers in TMEM let the epilogue of one range segment
// overlap the MMAs of the next.  Every wait is bounded; a wait that runs out
// sets the workspace error word and the kernel winds down.
//
// CTA pairs (prefill tiles).  A cluster of two CTAs on one TPC works as one
// worker: a unit is weight tiles 2t (even CTA) and 2t+1 (odd CTA) x up to 256
// tokens.  The even CTA's thread issues tcgen05.mma.cta_group::2 (M = 256):
// each CTA supplies its 128 weight rows and half of the token tile from its
// own shared memory and receives its 128 rows of the accumulator in its own
// TMEM.  Both CTAs' TMA loads signal the even CTA's ring barrier; its MMA
// commits release the ring slot and hand over the accumulator in both CTAs;
// both CTAs' epilogue warps report a drained accumulator to the even CTA.
// Per SM a stage holds half the token bytes of a one-CTA unit of the same
// size, which leaves room for a 7-deep ring.
#include <cuda_bf16.h>

#include "launch_config.cuh"
#include "moe_kernels.cuh"
#include "bounded_wait.cuh"
#include "pdl.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace ptx;

constexpr int kTabMaxE = 256;
constexpr int kABytes = kWeightBoxRows * kBlockK * 2;  // 16 KB weight tile per stage
constexpr int kTokRowBytes = kBlockK * 2;              // 128 B per token row per stage

template <bool SWIGLU, int BN, int STAGES, int TOKBOX, bool PAIR, bool MX = false, bool W4 = false,
          bool A4 = false, bool NV = false, bool FUSED = false, bool GATHER = false>
struct GemmCfg {
  // a CTA pair splits the unit's tokens: each CTA holds half of the B tile
  static constexpr int kBBytes = (PAIR ? BN / 2 : BN) * kTokRowBytes;
  // MXFP8: one byte per element, so a 128-byte row holds 128 elements of K;
  // each stage also carries its scale tiles: 512 bytes for the 128 weight rows
  // and 512 per 128 token rows of the unit's token chunk (a CTA of a pair needs
  // the scales of all 256 tokens: the pair MMA reads them from its own TMEM)
  // A4 (the MXFP4 layer): tokens are packed E2M1 codes too, so a 128-byte row
  // holds 256 elements of K, a stage issues 4 kind::mxf4 MMAs of K = 64 and
  // carries two scale tiles (two 128-element chunks) per operand
  static constexpr int kKPerStage = A4 ? 256 : MX ? 128 : kBlockK;
  static constexpr int kBoxX = MX ? 128 : kBlockK;    // TMA x coordinate per stage (elements of the map's type)
  // scale tiles per operand per stage (a tile: 128 rows x 128 elements of K
  // with 32-element blocks, or x 64 elements with NVFP4's 16-element blocks)
  static constexpr int kChunks = NV ? 4 : A4 ? 2 : 1;
  // MXFP4 weights (W4): two E2M1 codes per byte in global memory; the TMA's
  // 16U4_ALIGN16B type spreads each 8 bytes (16 codes) over 16 bytes of shared
  // memory, so the tile's image and descriptors are those of an FP8 tile while
  // the barrier counts only the 64 data bytes per 128-element row
  static constexpr int kWTxBytes = (W4 && !A4) ? kABytes / 2 : kABytes;
  static constexpr int kSfTokTiles = MX ? (BN > 128 ? 2 : 1) : 0;  // 512-byte token scale tiles per chunk
  static constexpr int kSfTokBytes = kSfTokTiles * 512 * kChunks;
  static constexpr int kSfWBytes = MX ? 512 * kChunks : 0;
  static constexpr int kSfBytes = kSfWBytes + kSfTokBytes;
  static constexpr int kStageBytes = (kABytes + kBBytes + kSfBytes + 1023) / 1024 * 1024;
  static constexpr int kAccCols = BN;  // fp32 TMEM columns per accumulator buffer
  // accumulator buffers: two (the epilogue of one unit overlaps the MMAs of the
  // next); one for MXFP8 pairs, whose 256 columns leave no room for a second
  // next to the scale slots
  static constexpr int kSfColsPerStage = MX ? 32 : 0;
  static constexpr int kAccBufs = (2 * BN + STAGES * kSfColsPerStage <= 512) ? 2 : 1;
  // epilogue warps: 4 (one per TMEM lane quarter); 8 with a single accumulator
  // buffer (two per quarter, alternate 16-column groups), which halves the time
  // the MMAs of the next unit wait for it
  static constexpr int kEpiWarps = kAccBufs == 1 ? 8 : 4;
  // block-scaled one-CTA units with several scale tiles per operand and stage
  // (the MXFP4 and NVFP4 layers): four scale warps (one per TMEM lane quarter)
  // write each stage's scale tiles into TMEM with tcgen05.st, so that the
  // tensor pipe runs only MMAs (NVFP4 decode 1.21x, prefill 1.20x; with one
  // tile per stage, as in the MXFP8 layer, tcgen05.cp measured 2% faster; a CTA
  // pair keeps tcgen05.cp: its 8 epilogue warps and 168 registers leave no
  // room for 4 more warps)
  static constexpr int kScaleWarps = (MX && !PAIR && kChunks > 1) ? 4 : 0;
  // GATHER (bf16 gate/up GEMM, decode tile plan): two row warps copy the
  // stages' token rows from h (rows picked by sorted_ids) into the B tile
  // with cp.async, in place of a gather kernel and the token TMA
  static constexpr int kGatherWarps = GATHER ? 2 : 0;
  static constexpr int kThreads = 64 + 32 * (kEpiWarps + kScaleWarps + kGatherWarps);
  // TMEM columns of one stage's scales: weight scales at +0 (4 columns), token
  // scales at +16 (4 columns per 128 tokens); slots of 32 keep both addresses
  // 16-column aligned
  static constexpr int kSfCols = MX ? 32 : 0;
  static constexpr int kTmemNeed = kAccBufs * kAccCols + STAGES * kSfCols;
  static constexpr uint32_t kTmemCols = kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128
                                        : kTmemNeed <= 256 ? 256 : 512;
  static constexpr int kBarBytes = 512;
  // one-CTA plans keep a shared-memory copy of the routing tables (E <= kTabMaxE):
  // offsets and the unit prefix sums (of both GEMMs in the fused kernel)
  static constexpr int kTabBytes = PAIR ? 0 : (FUSED ? 3 : 2) * (kTabMaxE + 1) * 4;
  static constexpr size_t kSmemBytes = 1024 + static_cast<size_t>(STAGES) * kStageBytes + kBarBytes + kTabBytes;
  static_assert(BN % TOKBOX == 0 && TOKBOX % 16 == 0 && BN >= 16 && BN <= 256, "token tile");
  static_assert(!PAIR || (BN / 2) % TOKBOX == 0, "token boxes of a CTA pair");
  static_assert(!MX || (PAIR ? (BN == 256 || BN == 128) : (BN % 32 == 0 && BN <= 128)),
                "MXFP8 units: one CTA with 32..128 tokens, or a CTA pair with 128 or 256");
  static_assert(kAccBufs == 2 || (MX && PAIR), "a single accumulator buffer only for MXFP8 pairs");
  static_assert(!W4 || MX, "FP4 weights only with block-scaled tokens");
  static_assert(!A4 || W4, "FP4 tokens only with FP4 weights");
  static_assert(!NV || (A4 && !PAIR), "NVFP4: both operands E2M1, one-CTA units (TMEM columns of the scales)");
  static_assert(!FUSED || (SWIGLU && !PAIR && !MX && kEpiWarps == 4),
                "the fused gate/up -> down kernel: bf16, one-CTA units, four epilogue warps");
  static_assert(!GATHER || (SWIGLU && !PAIR && !MX && !FUSED && BN % 4 == 0),
                "row warps: the bf16 gate/up GEMM on one-CTA units");
  static_assert(!MX || (4 * kChunks <= 16 && 16 + 4 * kChunks * kSfTokTiles <= kSfCols),
                "scale columns of a stage: weight tiles from +0, token tiles from +16");
  static_assert(kStageBytes % 1024 == 0, "stage tiles must stay 1024-byte aligned");
  static_assert(kTmemNeed <= 512, "TMEM has 512 columns");
  static_assert((3 * STAGES + 7) * 8 + 32 <= kBarBytes, "barrier area");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
};

struct Unit {
  int e, tile, tok0, n;
};

// The waits of the kernel, as recorded in the error word's detail bits.
enum : int {
  kWaitRingSlotFree = 1,  // producer: a ring slot consumed by the MMAs
  kWaitAccFree = 2,       // MMA: an accumulator buffer drained by the epilogue
  kWaitRingSlotFull = 3,  // MMA: a ring slot's loads landed
  kWaitAccFull = 4,       // epilogue: an accumulator's MMAs complete
  kWaitPartials = 5,      // epilogue: a later CTA's stream-K partial sums
  kWaitCombine = 6,       // epilogue: the fused combine's rendezvous
  kWaitScales = 7,        // MMA: a stage's scales written to TMEM by the scale warps
  kWaitScaleLoads = 8,    // scale warps: a ring slot's loads landed
  kWaitActReady = 9       // fused kernel, producer: a gate/up unit's activation rows stored
};

// Work unit u -> expert (binary search in the unit prefix sums), weight tile
// and token chunk, chunk index fastest: the units that read the same weight
// tile are neighbours, so CTAs running side by side read it from DRAM once
// (with the tile index fastest, an expert's chunks fell into different waves
// of the persistent grid and prefill re-read ~60% of the weights), while the
// expert's few token chunks stay in L2 for all its tiles.
// The tables are read through generic pointers: a copy in shared memory, or
// global memory.
__device__ __forceinline__ Unit decode_unit(int u, const int32_t* unit_off, const int32_t* offsets, int E, int tiles,
                                            int bn) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (unit_off[mid] <= u)
      lo = mid;
    else
      hi = mid;
  }
  Unit r;
  r.e = lo;
  const int base = unit_off[lo];
  const int chunks = (unit_off[lo + 1] - base) / tiles;  // >= 1: u lies in this expert's range
  const int local = u - base;
  r.tile = local / chunks;
  const int chunk = local - r.tile * chunks;
  r.tok0 = offsets[lo] + chunk * bn;
  r.n = min(bn, offsets[lo + 1] - r.tok0);
  return r;
}

// The CTA's work, walked as segments: K-blocks [kb0, kb1) of unit u.
// Stream-K: a contiguous range of (unit, K-block) iterations.  Otherwise
// whole units u = cta, cta + ctas, ... (CTAs running side by side then work
// on neighbouring units, which share weight and token tiles in L2).
struct Range {
  int64_t it, end, W;
  int kblocks, units, step;
  bool stream_k;
  __device__ Range(int n_units, int kb, int cta, int ctas, bool sk)
      : kblocks(kb), units(n_units), step(ctas), stream_k(sk) {
    W = static_cast<int64_t>(n_units) * kb;
    if (sk) {
      it = W * cta / ctas;
      end = W * (cta + 1) / ctas;
    } else {
      it = cta;
      end = n_units;
    }
  }
  __device__ bool next(int& u, int& kb0, int& kb1) {
    if (it >= end) return false;
    if (!stream_k) {
      u = static_cast<int>(it);
      kb0 = 0;
      kb1 = kblocks;
      it += step;
      return true;
    }
    u = static_cast<int>(it / kblocks);
    kb0 = static_cast<int>(it - static_cast<int64_t>(u) * kblocks);
    const int64_t stop = kb0 + (end - it);
    kb1 = stop < kblocks ? static_cast<int>(stop) : kblocks;
    it += kb1 - kb0;
    return true;
  }
};

__device__ __forceinline__ int64_t range_start(int64_t W, int cta, int ctas) { return W * cta / ctas; }

// The segments of a CTA, tagged with their GEMM: its range of the gate/up
// GEMM (phase 0), then, in the fused kernel, its range of the down GEMM
// (phase 1), each split like a kernel of its own.
struct Work {
  Range r0, r1;
  int phase;
  __device__ Work(int units0, int kblocks0, int units1, int kblocks1, int cta, int ctas, bool sk)
      : r0(units0, kblocks0, cta, ctas, sk), r1(units1, kblocks1, cta, ctas, sk), phase(0) {}
  __device__ bool next(int& ph, int& u, int& kb0, int& kb1) {
    if (phase == 0) {
      if (r0.next(u, kb0, kb1)) {
        ph = 0;
        return true;
      }
      phase = 1;
    }
    if (r1.next(u, kb0, kb1)) {
      ph = 1;
      return true;
    }
    return false;
  }
  __device__ const Range& range(int ph) const { return ph ? r1 : r0; }
};

__device__ __forceinline__ uint16_t f2bf(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }

// The four epilogue warps meet: each warp's lane 0 arrives on `bar` (count 4)
// and every lane waits for the phase, bounded like every other wait.
// Warp-uniform result; false when the wait ran out or the CTA is aborting.
__device__ __forceinline__ bool epilogue_rendezvous(uint64_t* bar, uint32_t& phase, int lane,
                                                    const volatile int* abort) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
  const bool got = mbar_wait(bar, phase, kWaitTimeoutNs, abort);
  phase ^= 1u;
  return __all_sync(0xFFFFFFFFu, got);
}

// The top-k weighted combine of the down GEMM, for the unit whose output rows
// of weight tile `tile` (features [128 tile, +128)) this CTA has just stored:
// the combine moves into the GEMM's epilogue ("4 · La fusion de noyaux", §4.2
// "GEMM + épilogue"), ordered by one counter per piece of output (§4.2
// "GEMM + GEMM"), here per (tile, token); nothing ever waits on a counter.
// 1. Every epilogue thread fences its stores; the warps meet.
// 2. Thread r takes unit rows r, r + 128: a real row of token t counts one
//    arrival at combine_cnt[tile][t]; the arrival that makes it k marks the
//    row in `mask` (every other row of t in this tile is then stored and
//    visible: each was fenced before its own arrival).
// 3. The warps meet; 8 groups of 16 threads finish the marked rows' tokens
//    (group g: rows g, g + 8, ...), each thread 8 features:
//    y = bf16(sum_j w_j * out_j) over j = 0..k-1 in order
//    (fp32 fma from 0, the separate combine kernel's arithmetic), reading the
//    rows through L2.  4. The warps meet again before the mask is reused.
template <int BN>
__device__ __noinline__ bool combine_unit(const ExpertGemmArgs& a, const Unit& un, int tile, int row, int lane,
                                          uint64_t* bar, uint32_t& phase, uint32_t* mask, const volatile int* abort) {
  const int T = a.n_routed / a.top_k;
  __threadfence();
  if (!epilogue_rendezvous(bar, phase, lane, abort)) return false;
  int32_t* cnt = a.combine_cnt + static_cast<int64_t>(tile) * T;
  for (int i = row; i < un.n; i += 128) {
    const int sid = __ldg(a.sorted_ids + un.tok0 + i);
    if (sid < a.n_routed && atomicAdd(cnt + sid / a.top_k, 1) == a.top_k - 1) atomicOr(mask + (i >> 5), 1u << (i & 31));
  }
  __threadfence();
  if (!epilogue_rendezvous(bar, phase, lane, abort)) return false;
  const int grp = row >> 4, chunk = row & 15;  // 8 groups x 16 chunks of 8 features
  const int64_t col = static_cast<int64_t>(tile) * 128 + chunk * 8;
  for (int i = grp; i < un.n; i += 8) {
    if (!((mask[i >> 5] >> (i & 31)) & 1u)) continue;
    const int t = __ldg(a.sorted_ids + un.tok0 + i) / a.top_k;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
    for (int j0 = 0; j0 < a.top_k; j0 += 8) {
      uint4 v[8];
      float wj[8];
#pragma unroll
      for (int d = 0; d < 8; ++d) {
        if (j0 + d < a.top_k) {
          const int64_t r = static_cast<int64_t>(t) * a.top_k + j0 + d;
          wj[d] = __ldg(a.topk_w + r);
          v[d] = __ldcg(reinterpret_cast<const uint4*>(a.out + static_cast<int64_t>(__ldg(a.slot_of + r)) * a.n_out + col));
        }
      }
#pragma unroll
      for (int d = 0; d < 8; ++d) {
        if (j0 + d < a.top_k) {
          const uint32_t wv[4] = {v[d].x, v[d].y, v[d].z, v[d].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc[2 * e] = fmaf(wj[d], __uint_as_float(wv[e] << 16), acc[2 * e]);
            acc[2 * e + 1] = fmaf(wj[d], __uint_as_float(wv[e] & 0xFFFF0000u), acc[2 * e + 1]);
          }
        }
      }
    }
    uint4 o;
    o.x = static_cast<uint32_t>(f2bf(acc[0])) | (static_cast<uint32_t>(f2bf(acc[1])) << 16);
    o.y = static_cast<uint32_t>(f2bf(acc[2])) | (static_cast<uint32_t>(f2bf(acc[3])) << 16);
    o.z = static_cast<uint32_t>(f2bf(acc[4])) | (static_cast<uint32_t>(f2bf(acc[5])) << 16);
    o.w = static_cast<uint32_t>(f2bf(acc[6])) | (static_cast<uint32_t>(f2bf(acc[7])) << 16);
    *reinterpret_cast<uint4*>(a.y + static_cast<int64_t>(t) * a.n_out + col) = o;
  }
  if (!epilogue_rendezvous(bar, phase, lane, abort)) return false;
  if (row < BN / 32) mask[row] = 0;  // cleared before any thread marks rows of the next unit (next rendezvous)
  return true;
}

// FUSED: the gate/up GEMM (args, tm_w, tm_x) and then the down GEMM (args2;
// tm_sw maps W2, tm_sx the activations) in one persistent launch.  KTAIL
// (packed E2M1 operands, 256 elements of K per stage): K ends half way into
// the last stage; its own instance, so that whole-stage shapes keep
// compile-time scale sizes and MMA counts.
template <bool SWIGLU, int BN, int STAGES, int TOKBOX, bool PAIR, bool MX = false, bool W4 = false,
          bool A4 = false, bool NV = false, bool FUSED = false, bool KTAIL = false, bool GATHER = false>
__global__ void __launch_bounds__(GemmCfg<SWIGLU, BN, STAGES, TOKBOX, PAIR, MX, W4, A4, NV, FUSED, GATHER>::kThreads, 1)
    expert_gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                       const __grid_constant__ CUtensorMap tm_sw, const __grid_constant__ CUtensorMap tm_sx,
                       const __grid_constant__ ExpertGemmArgs args, const __grid_constant__ ExpertGemmArgs args2) {
  using C = GemmCfg<SWIGLU, BN, STAGES, TOKBOX, PAIR, MX, W4, A4, NV, FUSED, GATHER>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * C::kStageBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint64_t* cbar = done + 2;                                       // the epilogue warps' rendezvous (fused combine)
  uint32_t* cmask = reinterpret_cast<uint32_t*>(cbar + 1);         // [8]: unit rows that complete a token
  uint64_t* sfull = reinterpret_cast<uint64_t*>(cmask + 8);        // [STAGES]: a stage's scales are in TMEM
  int32_t* tab = reinterpret_cast<int32_t*>(smem + STAGES * C::kStageBytes + C::kBarBytes);  // [2 or 3][kTabMaxE+1]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kern = SWIGLU ? kKernGemm1 : kKernGemm2;
  // CTA pair (cluster of 2): rank 0 issues the MMAs for both; the pair takes
  // work as one worker
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int worker = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int workers = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  // The routing tables come from a kernel at least two launches back, which
  // has completed (see pdl.cuh); only the token / activation rows written by
  // the immediately preceding kernel need the producer's pdl_wait below.
  // After the single-launch front end the tables come from the previous
  // kernel itself: then every thread waits for it first.
  if (args.tables_from_parent) pdl_wait();
  const int32_t* t_unit = args.unit_off;
  const int32_t* t_off = args.offsets;
  const int32_t* t_unit2 = args2.unit_off;  // fused kernel: the down GEMM's units
  if (!PAIR && args.E <= kTabMaxE) {
    for (int i = threadIdx.x; i <= args.E; i += C::kThreads) {
      tab[i] = __ldcg(args.unit_off + i);
      tab[kTabMaxE + 1 + i] = __ldcg(args.offsets + i);
      if (FUSED) tab[2 * (kTabMaxE + 1) + i] = __ldcg(args2.unit_off + i);
    }
    t_unit = tab;
    t_off = tab + kTabMaxE + 1;  // visible to all threads after the barrier below
    if (FUSED) t_unit2 = tab + 2 * (kTabMaxE + 1);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], GATHER ? 2 : 1);  // the producer's arrival (with the TMA bytes) [+ the row warp's]
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], (PAIR ? 2 : 1) * C::kEpiWarps);  // the epilogue warps (of both CTAs of a pair)
    }
    mbar_init(done, 1);
    mbar_init(cbar, 4);  // one arrival per epilogue warp
    for (int st = 0; st < STAGES; ++st) mbar_init(&sfull[st], C::kScaleWarps > 0 ? C::kScaleWarps : 1);
    for (int i = 0; i < 8; ++i) cmask[i] = 0;
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(tmem_slot, C::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, C::kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if (PAIR)
    cluster_sync();  // the peer's barriers are initialised before any remote signal
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int total_units = t_unit[args.E];
  // stages along K; with packed E2M1 operands (256 elements of K per stage)
  // K may end half way into the last stage: its box reads zero codes past K,
  // and only its valid scale tiles are loaded and its valid MMAs issued
  const int kblocks = (args.K + C::kKPerStage - 1) / C::kKPerStage;
  const int total_units2 = FUSED ? t_unit2[args.E] : 0;
  const int kblocks2 = FUSED ? args2.K / C::kKPerStage : 1;
  // block-scaled GEMMs: scale tiles per 128-row group along K (one per
  // kKPerStage / kChunks elements), and the valid ones in stage kb
  const int sf_tiles_k = args.K / (C::kKPerStage / C::kChunks);
  // scale tiles of the last stage when K ends half way into it (KTAIL)
  const int sf_tail = sf_tiles_k % C::kChunks;
  auto tail_stage = [&](int kb) { return KTAIL && kb == kblocks - 1; };
  const int ctas = workers;
  // per phase (the fused kernel: 0 gate/up, 1 down), the arguments read per
  // segment, stage or output chunk, held in registers: a reference to one of
  // the two parameter structs chosen at run time would turn each of these
  // reads into a generic load from the parameter space
  struct PhaseArgs {
    uint16_t* out;
    float* partials;
    int32_t* flags;
    int n_out, tiles, w_rows;
  };
  const PhaseArgs pa0{args.out, args.partials, args.flags, args.n_out, args.tiles_per_expert, args.w_rows_per_expert};
  const PhaseArgs pa1 = FUSED ? PhaseArgs{args2.out, args2.partials, args2.flags, args2.n_out, args2.tiles_per_expert,
                                          args2.w_rows_per_expert}
                              : pa0;
  auto phase_args = [&](int ph) { return (FUSED && ph) ? pa1 : pa0; };  // a copy, in registers
  auto unit_tab = [&](int ph) { return (FUSED && ph) ? t_unit2 : t_unit; };
  auto is_swiglu = [&](int ph) { return FUSED ? ph == 0 : SWIGLU; };
  const bool tok_from_h = args.tokens_from_h != 0;
  int32_t* const ready = args.ready;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      prefetch_tensormap(&tm_w);
      prefetch_tensormap(&tm_x);
      if (FUSED) {
        prefetch_tensormap(&tm_sw);
        prefetch_tensormap(&tm_sx);
      }
      // A weight tile is read by every token chunk of its expert: streamed once
      // (evict first) when the expert's tokens fit one chunk, kept (evict last)
      // when more chunks will read it.  Token tiles are re-read by every
      // weight tile of their expert.
      const uint64_t pol_stream = policy_evict_first();
      const uint64_t pol_keep = policy_evict_last();
      const uint64_t pol_x = pol_keep;
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      int where = kWaitRingSlotFree;  // the wait that ran out
      // The token (or activation) loads of the stages wait until their rows
      // exist: the gate/up GEMM's token rows until the previous kernel has
      // completed (pdl_wait), so the first ring-full of stages gets its weight
      // tiles at once and its token rows after (then all at once).  In the
      // fused kernel they wait in a FIFO, a down-GEMM stage's activation rows
      // until every gate/up unit of the same expert and token chunk has
      // counted the stores of its four epilogue warps (one counter per chunk,
      // checked once per segment: a poll per stage, an L2 round trip, would
      // hold the producer back).  The other instances keep the plain scheme:
      // the FIFO's code, inlined at every call site, makes these large
      // kernels measurably slower.
      bool deps_ready = false;
      int n_pend = 0, pend_head = 0;
      int pend_stage[STAGES] = {}, pend_kb[STAGES] = {}, pend_tok0[STAGES] = {}, pend_rows[STAGES] = {},
          pend_chunk[STAGES] = {};
      int pend_ready[STAGES] = {};  // fused kernel: the token chunk a down-GEMM stage awaits, or -1
      int chunk_seen_ready = -1;  // the last chunk found complete
      const int chunk_need = C::kEpiWarps * pa0.tiles;
      // a CTA pair signals every load on the even CTA's full barrier
      const uint32_t full_cl = PAIR ? mapa_shared(smem_u32(full), 0) : 0u;
      auto load_2d = [&](void* dst, const CUtensorMap* map, int st, int c0, int c1, uint64_t pol) {
        if (PAIR)
          tma_load_2d_pair(dst, map, full_cl + 8u * st, c0, c1, pol);
        else
          tma_load_2d(dst, map, &full[st], c0, c1, pol);
      };
      // gate/up A tile: box {64 K, 16 rows, gate+up, 4 groups, 1 expert}
      auto load_gate_up = [&](void* dst, int st, int kb, int tile, int e, uint64_t pol) {
        if (PAIR)
          tma_load_5d_pair(dst, &tm_w, full_cl + 8u * st, kb * C::kBoxX, 0, 0, tile * 4, e, pol);
        else
          tma_load_5d(dst, &tm_w, &full[st], kb * C::kBoxX, 0, 0, tile * 4, e, pol);
      };
      // chunk: the unit's token chunk (MXFP8 token scales are stored per chunk)
      auto load_tokens = [&](int st, int kb, int tok0, int rows, int chunk) {
        if (GATHER) return;  // the row warps copy them
        uint8_t* sb = smem + st * C::kStageBytes + kABytes;
        const int row0 = tok_from_h ? 0 : tok0;  // one token: its row of h, then zeros
        for (int r = 0; r < rows; r += TOKBOX)
          load_2d(sb + r * kTokRowBytes, &tm_x, st, kb * C::kBoxX, row0 + r, pol_x);
        if (MX && PAIR) {
          // the 512-byte scale tiles of the whole token chunk (one per 128 tokens
          // and 128-element K chunk; tile (h, c) at 512 (c G + h)), in each CTA
          // (tensor map tm_sx: one tile = a box of 2 rows x 256 bytes)
          constexpr int G = C::kSfTokTiles;
          for (int c = 0; c < (tail_stage(kb) ? sf_tail : C::kChunks); ++c)
            for (int h = 0; h < G; ++h)
              load_2d(sb + C::kBBytes + C::kSfWBytes + 512 * (c * G + h), &tm_sx, st, 0,
                      2 * ((G * chunk + h) * sf_tiles_k + kb * C::kChunks + c), pol_x);
        } else if (MX) {  // one tile per K chunk, the chunks of a stage adjacent
          const uint8_t* src = args.x_scales + (static_cast<size_t>(chunk) * sf_tiles_k + kb * C::kChunks) * 512;
          if (!tail_stage(kb))
            bulk_load(sb + C::kBBytes + C::kSfWBytes, src, 512 * C::kChunks, &full[st], pol_x);
          else
            bulk_load(sb + C::kBBytes + C::kSfWBytes, src, 512 * sf_tail, &full[st], pol_x);
        }
      };
      // fused kernel: a down-GEMM stage's activation rows (written by this
      // kernel's gate/up epilogues through the generic proxy, read here by TMA
      // after head_ready's acquire and proxy fence)
      auto load_act = [&](int st, int kb, int tok0, int rows) {
        uint8_t* sb = smem + st * C::kStageBytes + kABytes;
        for (int r = 0; r < rows; r += TOKBOX) tma_load_2d(sb + r * kTokRowBytes, &tm_sx, &full[st], kb * C::kBoxX,
                                                           tok0 + r, pol_x);
      };
      auto resolve_deps = [&]() {
        pdl_wait();
        pdl_launch_dependents();
        deps_ready = true;
      };
      auto issue_head = [&]() {
        const int i = pend_head;
        if (FUSED && pend_ready[i] >= 0)
          load_act(pend_stage[i], pend_kb[i], pend_tok0[i], pend_rows[i]);
        else
          load_tokens(pend_stage[i], pend_kb[i], pend_tok0[i], pend_rows[i], pend_chunk[i]);
        pend_head = pend_head + 1 == STAGES ? 0 : pend_head + 1;
        --n_pend;
      };
      // whether the FIFO head's rows exist: polled, or waited for (bounded)
      auto head_ready = [&](bool wait) -> bool {
        const int r = pend_ready[pend_head];
        if (!deps_ready) {
          if (!wait && !(FUSED && r >= 0)) return false;
          resolve_deps();
        }
        if (!FUSED || r < 0 || r == chunk_seen_ready) return true;
        if (ld_acquire(ready + r) < chunk_need) {
          if (!wait) return false;
          const uint64_t t0 = globaltimer_ns();
          // (up to one producer per SM polls the same few counters: a slow
          // poll keeps them from crowding the L2 slices the weights stream through)
          while (ld_acquire(ready + r) < chunk_need) {
            if (*abort_flag || globaltimer_ns() - t0 > kWaitTimeoutNs) return false;
            __nanosleep(1000);
          }
        }
        fence_proxy_async_global();  // the TMA reads that follow see what the acquire saw
        chunk_seen_ready = r;
        return true;
      };
      Work rg(total_units, kblocks, total_units2, kblocks2, worker, ctas, args.stream_k != 0);
      int ph, u, kb0, kb1;
      while (ok && rg.next(ph, u, kb0, kb1)) {
        const PhaseArgs A = phase_args(ph);
        const bool sw = is_swiglu(ph);
        const Unit un = decode_unit(u, unit_tab(ph), t_off, args.E, A.tiles, BN);
        // a pair's unit: weight tiles 2t (even CTA) and 2t+1; the MMA's N
        // tokens split in halves, the first half in the even CTA
        const int tile = PAIR ? 2 * un.tile + static_cast<int>(rank) : un.tile;
        const int n_mma = PAIR ? (un.n + 31) / 32 * 32 : un.n;
        const int half = PAIR ? n_mma / 2 : n_mma;
        const int tok_first = un.tok0 + static_cast<int>(rank) * half;
        const int wrow = un.e * A.w_rows + tile * (sw ? kGateUpTileFeat : kDownTileFeat);
        const int tok_rows = (half + TOKBOX - 1) / TOKBOX * TOKBOX;  // whole boxes; rows past n are unused
        const bool reused = t_off[un.e + 1] - t_off[un.e] > BN;
        const uint64_t pol_w = reused ? pol_keep : pol_stream;
        // per CTA (both of a pair); scale bytes of a full stage: C::kSfBytes
        const uint32_t bytes_base = C::kWTxBytes + (GATHER ? 0 : tok_rows * kTokRowBytes);
        const int chunk = MX ? t_unit[un.e] / pa0.tiles + (un.tok0 - t_off[un.e]) / BN : 0;
        // fused kernel, down GEMM: the token chunk (expert, rows [tok0, tok0 + BN))
        // whose activation rows this unit reads, numbered over all experts
        const int rd_chunk = (FUSED && ph == 1) ? t_unit[un.e] / pa0.tiles + (un.tok0 - t_off[un.e]) / BN
                                                : -1;
        if (FUSED && ph == 1 && rd_chunk != chunk_seen_ready) {
          // a down-GEMM segment starts its weight stream only once its chunk's
          // activation rows are complete: streamed earlier, the W2 tiles compete
          // for DRAM with the gate/up phase's last loads, which every CTA's
          // readiness waits for
          while (n_pend > 0) {
            if (!head_ready(true)) {
              ok = false;
              where = kWaitActReady;
              break;
            }
            issue_head();
          }
          if (ok) {
            pend_ready[pend_head] = rd_chunk;  // an empty FIFO's head slot: ask for this chunk
            if (!head_ready(true)) {
              ok = false;
              where = kWaitActReady;
            }
          }
          if (!ok) break;
        }
        for (int kb = kb0; kb < kb1; ++kb) {
          if (FUSED && n_pend == STAGES) {  // the slot about to be refilled still waits for its token rows
            if (!head_ready(true)) {
              ok = false;
              where = kWaitActReady;
              break;
            }
            do {  // it, and every later one whose rows now exist too
              issue_head();
            } while (n_pend > 0 && head_ready(false));
          }
          if (!mbar_wait(&empty[stage], phase ^ 1u, kWaitTimeoutNs, abort_flag)) {
            ok = false;
            where = kWaitRingSlotFree;
            break;
          }
          uint8_t* sa = smem + stage * C::kStageBytes;
          const uint32_t bytes =
              bytes_base + (tail_stage(kb) ? static_cast<uint32_t>(sf_tail) * 512u * (1u + C::kSfTokTiles)
                                           : static_cast<uint32_t>(C::kSfBytes));
          if (!PAIR)
            mbar_arrive_expect_tx(&full[stage], bytes);
          else if (leader)
            mbar_arrive_expect_tx(&full[stage], 2 * bytes);  // both CTAs' loads
          if (sw) {  // 16 gate rows, the matching 16 up rows, x 4
            load_gate_up(sa, stage, kb, tile, un.e, pol_w);
          } else {
            load_2d(sa, FUSED ? &tm_sw : &tm_w, stage, kb * C::kBoxX, wrow, pol_w);
          }
          if (MX) {  // the weight tile's scales (static: loaded before the parent kernel ends)
            const int wtiles = PAIR ? 2 * pa0.tiles : pa0.tiles;  // 128-row tiles per expert
            const int64_t wt = static_cast<int64_t>(un.e * wtiles + tile) * sf_tiles_k + kb * C::kChunks;
            if (PAIR) {
              for (int c = 0; c < (tail_stage(kb) ? sf_tail : C::kChunks); ++c)
                load_2d(sa + kABytes + C::kBBytes + 512 * c, &tm_sw, stage, 0, static_cast<int>(2 * (wt + c)), pol_w);
            } else {
              bulk_load(sa + kABytes + C::kBBytes, args.w_scales + static_cast<size_t>(wt) * 512,
                        512 * (tail_stage(kb) ? sf_tail : C::kChunks), &full[stage], pol_w);
            }
          }
          if constexpr (!FUSED) {
            // only the first ring-full of stages waits for the parent kernel;
            // once it has completed, every pending load goes out at once
            if (deps_ready) {
              load_tokens(stage, kb, tok_first, tok_rows, chunk);
            } else {
              pend_stage[n_pend] = stage;
              pend_kb[n_pend] = kb;
              pend_tok0[n_pend] = tok_first;
              pend_rows[n_pend] = tok_rows;
              pend_chunk[n_pend] = chunk;
              if (++n_pend == STAGES) {
                resolve_deps();
                for (int i = 0; i < n_pend; ++i)
                  load_tokens(pend_stage[i], pend_kb[i], pend_tok0[i], pend_rows[i], pend_chunk[i]);
                n_pend = 0;
              }
            }
          } else if (n_pend == 0 && deps_ready && (rd_chunk < 0 || rd_chunk == chunk_seen_ready)) {
            // the rows exist and nothing waits ahead of them: load them now
            if (rd_chunk >= 0)
              load_act(stage, kb, tok_first, tok_rows);
            else
              load_tokens(stage, kb, tok_first, tok_rows, chunk);
          } else {
            const int slot = pend_head + n_pend < STAGES ? pend_head + n_pend : pend_head + n_pend - STAGES;
            pend_stage[slot] = stage;
            pend_kb[slot] = kb;
            pend_tok0[slot] = tok_first;
            pend_rows[slot] = tok_rows;
            pend_chunk[slot] = chunk;
            pend_ready[slot] = rd_chunk;
            ++n_pend;
            while (n_pend > 0 && head_ready(false)) issue_head();
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // the token loads still waiting (fewer iterations than stages, or the
      // last ones); after a wait that ran out they are issued all the same
      // (the call reports the timeout), so that every stage's loads land
      if constexpr (!FUSED) {
        if (!deps_ready) resolve_deps();
        for (int i = 0; i < n_pend; ++i)
          load_tokens(pend_stage[i], pend_kb[i], pend_tok0[i], pend_rows[i], pend_chunk[i]);
        n_pend = 0;
      } else {
        while (n_pend > 0) {
          if (ok && !head_ready(true)) {
            ok = false;
            where = kWaitActReady;
          }
          if (!deps_ready) resolve_deps();
          issue_head();
        }
      }
      if (!deps_ready) resolve_deps();
      if (!ok) raise_timeout(args.err, abort_flag, kern, where);
      // every load this thread issued must have landed before the CTA exits
      // (the odd CTA of a pair sees that through the release of its stages:
      // the pair's MMA ran on them, so they had landed)
      for (int s = 0; s < STAGES; ++s) {
        if (issued <= s) break;
        const uint32_t par = (s < stage) ? phase : (phase ^ 1u);
        int dummy = 0;
        mbar_wait(PAIR && !leader ? &empty[s] : &full[s], par, kWaitTimeoutNs, &dummy);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- MMA issuer (the even CTA of a pair issues for both)
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      int where = 0;  // the wait that ran out
      Work rg(total_units, kblocks, total_units2, kblocks2, worker, ctas, args.stream_k != 0);
      int ph, u, kb0, kb1;
      while (ok && rg.next(ph, u, kb0, kb1)) {
        const Unit un = decode_unit(u, unit_tab(ph), t_off, args.E, phase_args(ph).tiles, BN);
        const bool free_acc = PAIR ? mbar_wait_cluster(&tempty[acc], acc_phase ^ 1u, kWaitTimeoutNs, abort_flag)
                                   : mbar_wait(&tempty[acc], acc_phase ^ 1u, kWaitTimeoutNs, abort_flag);
        if (!free_acc) {
          ok = false;
          where = kWaitAccFree;
          break;
        }
        tc_fence_after();
        const int n_mma = PAIR ? (un.n + 31) / 32 * 32 : un.n;
        const uint32_t idesc = idesc_bf16_f32(PAIR ? 256 : 128, static_cast<uint32_t>(n_mma));
        const uint32_t d_acc = tmem_base + static_cast<uint32_t>(acc * C::kAccCols);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, kWaitTimeoutNs, abort_flag)) {
            ok = false;
            where = kWaitRingSlotFull;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * C::kStageBytes);
          const uint32_t sb = sa + kABytes;
          if (MX) {
            // this stage's scales into its TMEM columns, then 4 MMAs of K = 32
            // (a pair: each CTA's own tiles into its own TMEM, by one copy)
            const uint32_t sf_t =
                tmem_base + static_cast<uint32_t>(C::kAccBufs * C::kAccCols + stage * C::kSfCols);
            const uint32_t sf_s = sb + C::kBBytes;
            const uint32_t sfb_t = sf_t + 16;
            // weight tile of chunk c -> columns +4c; token tile (h, c) -> +16 + 4 (c G + h)
            // (tokens 128h .. 128h+127 of chunk c)
            constexpr int G = C::kSfTokTiles;
            if (C::kScaleWarps > 0) {  // written by the scale warps
              if (!mbar_wait(&sfull[stage], phase, kWaitTimeoutNs, abort_flag)) {
                ok = false;
                where = kWaitScales;
                break;
              }
              tc_fence_after();
            }
#pragma unroll
            for (int c = 0; c < C::kChunks * (C::kScaleWarps == 0); ++c) {
              if (PAIR)
                tmem_cp_32x128b_x4_pair(sf_t + 4 * c, sf_s + 512 * c);
              else
                tmem_cp_32x128b_x4(sf_t + 4 * c, sf_s + 512 * c);
#pragma unroll
              for (int h = 0; h < G; ++h) {
                const uint32_t src = sf_s + C::kSfWBytes + 512 * (c * G + h);
                if (PAIR)
                  tmem_cp_32x128b_x4_pair(sfb_t + 4 * (c * G + h), src);
                else
                  tmem_cp_32x128b_x4(sfb_t + 4 * (c * G + h), src);
              }
            }
            // MMAs over K in the stage: 4, fewer in a KTAIL instance's last stage
            // (past K its scales were not loaded)
            const int n_k = tail_stage(kb) ? 4 * sf_tail / C::kChunks : 4;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              if (k >= n_k) break;
              const uint32_t accum = (kb > kb0 || k > 0) ? 1u : 0u;
              const uint64_t ad = sdesc_kmajor_sw128(sa + k * 32), bd = sdesc_kmajor_sw128(sb + k * 32);
              if (NV) {  // MMA k: K elements 64k .. 64k+63 = tile k, its 4 scales one word
                const uint32_t id = idesc_nvf4(128, static_cast<uint32_t>(n_mma));
                mma_nvf4_ss(d_acc, ad, bd, id, sf_t + 4 * k, sfb_t + 4 * k, accum);
              } else if (A4) {  // MMA k: K elements 64k .. 64k+63 = chunk k/2, blocks 2 (k&1), +1
                const uint32_t c = static_cast<uint32_t>(k >> 1), sid = 2u * static_cast<uint32_t>(k & 1);
                const uint32_t id = idesc_mxf4(PAIR ? 256 : 128, static_cast<uint32_t>(n_mma), sid, sid);
                if (PAIR)
                  mma_mxf4_ss_pair(d_acc, ad, bd, id, sf_t + 4 * c, sfb_t + 4 * G * c, accum);
                else
                  mma_mxf4_ss(d_acc, ad, bd, id, sf_t + 4 * c, sfb_t + 4 * G * c, accum);
              } else {
                const uint32_t id =
                    idesc_mxf8(PAIR ? 256 : 128, static_cast<uint32_t>(n_mma), k, k, W4 ? kFmtE2M1 : 0);
                if (PAIR)
                  mma_mxf8_ss_pair(d_acc, ad, bd, id, sf_t, sfb_t, accum);
                else
                  mma_mxf8_ss(d_acc, ad, bd, id, sf_t, sfb_t, accum);
              }
            }
          } else {
#pragma unroll
            for (int k = 0; k < kBlockK / 16; ++k) {
              const uint32_t accum = (kb > kb0 || k > 0) ? 1u : 0u;  // each segment starts a fresh sum
              if (PAIR)
                mma_bf16_ss_pair(d_acc, sdesc_kmajor_sw128(sa + k * 32), sdesc_kmajor_sw128(sb + k * 32), idesc,
                                 accum);
              else
                mma_bf16_ss(d_acc, sdesc_kmajor_sw128(sa + k * 32), sdesc_kmajor_sw128(sb + k * 32), idesc, accum);
            }
          }
          if (PAIR)
            mma_commit_pair_mc(&empty[stage], 0x3);  // frees the stage in both CTAs
          else
            mma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (PAIR)
          mma_commit_pair_mc(&tfull[acc], 0x3);
        else
          mma_commit(&tfull[acc]);
        if (++acc == C::kAccBufs) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) raise_timeout(args.err, abort_flag, kern, where);
      // all MMAs this thread issued have finished before TMEM is released
      if (PAIR)
        mma_commit_pair(done);
      else
        mma_commit(done);
      int dummy = 0;
      mbar_wait(done, 0, kWaitTimeoutNs, &dummy);
    }
  } else if (GATHER && warp >= 2 + C::kEpiWarps) {
    if constexpr (GATHER) {
      // ---------------- row warps: a stage's token rows of the unit, copied
      // from h into the B tile in the layout a 128-byte swizzled TMA box gives
      // (row r at r * 128, its 16-byte piece p at p ^ (r mod 8)).  The stages
      // go round-robin to the row warps (stage iteration i to warp i mod 2);
      // in a warp, lane takes piece (lane mod 8) of rows lane / 8 + 4 j.
      // Padding rows (sorted_ids past the routed rows) are left as they are:
      // they feed MMA columns whose outputs are dropped.  A warp signals a
      // stage once it has issued its next one: cp.async.wait_group, a proxy
      // fence (generic writes -> the MMAs' async-proxy reads), then one
      // arrival on the stage's full barrier.
      constexpr int kPasses = BN / 4;
      const int gw = warp - (2 + C::kEpiWarps);
      const int rsub = lane >> 3, piece = lane & 7;
      pdl_wait();  // sorted_ids come from the previous kernel
      const uint64_t pol_rows = policy_evict_last();  // each row is read by every weight tile of its expert
      const int32_t* sorted = args.sorted_ids;
      const char* hsrc = reinterpret_cast<const char*>(args.h_rows) + piece * 16;
      const size_t row_bytes = static_cast<size_t>(args.K) * 2;
      auto signal = [&](int st) {
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[st]);
      };
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int pending = -1;  // this warp's last stage copied, not yet signalled
      int64_t iter = 0;  // stage iterations of the CTA so far
      Range rg(total_units, kblocks, worker, ctas, args.stream_k != 0);
      int u, kb0, kb1;
      while (ok && rg.next(u, kb0, kb1)) {
        const int first_mine = static_cast<int>((C::kGatherWarps - iter % C::kGatherWarps + gw) % C::kGatherWarps);
        iter += kb1 - kb0;
        if (kb0 + first_mine >= kb1) {  // none of this segment's stages is this warp's
          for (int kb = kb0; kb < kb1; ++kb)
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          continue;
        }
        const Unit un = decode_unit(u, t_unit, t_off, args.E, pa0.tiles, BN);
        int src[kPasses];  // h row of each of this lane's rows, or -1
#pragma unroll
        for (int j = 0; j < kPasses; ++j) {
          const int r = rsub + 4 * j;
          int t = -1;
          if (r < un.n) {
            const int id = __ldg(sorted + un.tok0 + r);
            if (id >= 0 && id < args.n_routed) t = id / args.top_k;
          }
          src[j] = t;
        }
        for (int kb = kb0; kb < kb1; ++kb) {
          if ((kb - kb0) % C::kGatherWarps == first_mine) {
            const bool got = mbar_wait(&empty[stage], phase ^ 1u, kWaitTimeoutNs, abort_flag);
            if (!__all_sync(0xFFFFFFFFu, got)) {
              ok = false;
              break;
            }
            const uint32_t sb = smem_u32(smem + stage * C::kStageBytes + kABytes);
            const char* col = hsrc + static_cast<size_t>(kb) * (C::kBoxX * 2);
#pragma unroll
            for (int j = 0; j < kPasses; ++j) {
              const int r = rsub + 4 * j;
              if (src[j] >= 0)
                cp_async_16(sb + static_cast<uint32_t>(r * kTokRowBytes + ((piece ^ (r & 7)) << 4)),
                            col + static_cast<size_t>(src[j]) * row_bytes, pol_rows);
            }
            cp_async_commit();
            if (pending >= 0) {
              cp_async_wait<1>();
              signal(pending);
            }
            pending = stage;
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      cp_async_wait<0>();
      if (pending >= 0) signal(pending);
      if (!ok && lane == 0) raise_timeout(args.err, abort_flag, kern, kWaitRingSlotFree);
    }
  } else if (warp >= 2 + C::kEpiWarps) {
    // ---------------- scale warps (block-scaled one-CTA units): per stage, the
    // 16 bytes of each scale tile's row (lane & 31) into this warp's TMEM lane
    // quarter, columns as the MMA reads them (the image a 32x128b.warpx4 copy
    // of the tile gives), then one arrival on sfull[stage]
    if constexpr (C::kScaleWarps > 0) {
      const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
      constexpr int G = C::kSfTokTiles;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      Range rg(total_units, kblocks, worker, ctas, args.stream_k != 0);
      int u, kb0, kb1;
      while (ok && rg.next(u, kb0, kb1)) {
        for (int kb = kb0; kb < kb1; ++kb) {
          const bool got = mbar_wait(&full[stage], phase, kWaitTimeoutNs, abort_flag);
          if (!__all_sync(0xFFFFFFFFu, got)) {  // warp-uniform: tcgen05.st needs every lane
            ok = false;
            break;
          }
          const uint8_t* sf_s = smem + stage * C::kStageBytes + kABytes + C::kBBytes;
          const uint32_t sf_t =
              tmem_base + static_cast<uint32_t>(C::kAccBufs * C::kAccCols + stage * C::kSfCols) + lane_base;
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c) {
            tmem_st_32x32b_x4(sf_t + 4 * c, *reinterpret_cast<const uint4*>(sf_s + 512 * c + lane * 16));
#pragma unroll
            for (int h = 0; h < G; ++h)
              tmem_st_32x32b_x4(sf_t + 16 + 4 * (c * G + h),
                                *reinterpret_cast<const uint4*>(sf_s + C::kSfWBytes + 512 * (c * G + h) + lane * 16));
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sfull[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && lane == 0) raise_timeout(args.err, abort_flag, kern, kWaitScaleLoads);
    }
  } else {
    // ---------------- epilogue: warps 2.., TMEM lane quarter = warp % 4; with
    // 8 epilogue warps, group egrp of the two warps of a quarter takes the
    // 16-column groups egrp, egrp + 2, ... (no stream-K then: large plan only)
    const int q = warp & 3;
    const int egrp = (warp - 2) >> 2;
    const int c_first = 16 * egrp, c_step = 16 * (C::kEpiWarps / 4);
    const int row = q * 32 + lane;  // this thread's TMEM lane = A-tile row
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    int where = 0;  // the wait that ran out
    // gate/up: warp quarter q holds features +16q .. +16q+15, gate in lanes
    // 0..15 and up in lanes 16..31
    const bool lo = lane < 16;
    uint32_t cbar_phase = 0;  // uses of the combine rendezvous so far, mod 2
    const uint32_t tempty_cl = PAIR ? mapa_shared(smem_u32(tempty), 0) : 0u;
    Work rg(total_units, kblocks, total_units2, kblocks2, worker, ctas, args.stream_k != 0);
    int ph, u, kb0, kb1;
    while (ok && rg.next(ph, u, kb0, kb1)) {
      const PhaseArgs A = phase_args(ph);
      const bool sw = is_swiglu(ph);
      const int kb_total = ph ? kblocks2 : kblocks;
      const int64_t W = rg.range(ph).W;
      // this CTA's partial-sum slot of this GEMM: [BN columns][128 rows] fp32
      float* my_slot = A.partials + static_cast<int64_t>(blockIdx.x) * BN * 128;
      const Unit un = decode_unit(u, unit_tab(ph), t_off, args.E, A.tiles, BN);
      // warp-uniform outcome: tcgen05.ld below must be executed by all 32 lanes
      const bool got = mbar_wait(&tfull[acc], acc_phase, kWaitTimeoutNs, abort_flag);
      if (!__all_sync(0xFFFFFFFFu, got)) {
        ok = false;
        where = kWaitAccFull;
        break;
      }
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * C::kAccCols);
      // hand the accumulator buffer back to the MMA thread (the even CTA's, for a pair)
      bool released = false;
      auto release_acc = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (PAIR)
            mbar_arrive_cluster(tempty_cl + 8u * acc);  // the even CTA's MMA waits for both CTAs
          else
            mbar_arrive(&tempty[acc]);
        }
      };

      if (kb0 > 0) {
        // a later part of a unit started by an earlier CTA: hand over the partial sums
        for (int c0 = c_first; c0 < un.n; c0 += c_step) {
          uint32_t ra[16];
          tmem_ld_32x32b_x16(t_row + c0, ra);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) __stcg(my_slot + (c0 + j) * 128 + row, __uint_as_float(ra[j]));
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release(A.flags + blockIdx.x * 4 + q, 1);
      } else {
        // this CTA finishes the unit: the CTAs after it whose (non-empty)
        // ranges start inside the unit hold its later K-blocks and have
        // written their partial sums as their first work
        const int64_t unit_end = static_cast<int64_t>(u + 1) * kb_total;
        int c_last = blockIdx.x;  // producers are the CTAs in (blockIdx.x, c_last] with non-empty ranges
        if (kb1 < kb_total)
          while (c_last + 1 < ctas && range_start(W, c_last + 1, ctas) < unit_end) ++c_last;
        const int feat_base =
            (PAIR ? 2 * un.tile + static_cast<int>(rank) : un.tile) * (sw ? kGateUpTileFeat : kDownTileFeat);
        // SwiGLU (gate/up GEMM) or plain convert of one 16-column group, and its stores
        auto emit_chunk = [&](int c0, float (&v)[16]) {
          if (NV) {  // NVFP4 tensor scales: the expert matrix's times each token row's
            const float gw = __ldg(args.w_gscale + un.e);
            const float* gx = args.x_gscale + un.tok0 + c0;
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __fmul_rn(v[j], __fmul_rn(gw, __ldcg(gx + j)));
          }
          if (!sw) {
            uint16_t* out = A.out + static_cast<int64_t>(un.tok0 + c0) * A.n_out + feat_base + row;
#pragma unroll
            for (int j = 0; j < 16; ++j) out[static_cast<int64_t>(j) * A.n_out] = f2bf(v[j]);
          } else {
            // lanes l and l+16 swap half of their columns: lane l keeps the
            // gate values of columns 0..7 and receives the matching up values,
            // lane l+16 keeps the up values of columns 8..15 and receives the
            // gate values; each then finishes 8 outputs
            float a[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float mine = lo ? v[j] : v[j + 8];
              const float other = __shfl_xor_sync(0xFFFFFFFFu, lo ? v[j + 8] : v[j], 16);
              const float g = lo ? mine : other;
              const float up = lo ? other : mine;
              a[j] = __fdividef(g, 1.0f + __expf(-g)) * up;  // SiLU(gate) * up
            }
            const int feat = feat_base + q * 16 + (lane & 15);
            uint16_t* out = A.out + static_cast<int64_t>(un.tok0 + c0 + (lo ? 0 : 8)) * A.n_out + feat;
#pragma unroll
            for (int j = 0; j < 8; ++j) out[static_cast<int64_t>(j) * A.n_out] = f2bf(a[j]);
          }
        };
        if constexpr (C::kAccBufs == 1) {
          // a single accumulator buffer (MXFP8 pairs: no stream-K): all of this
          // warp's columns to registers, hand the buffer back to the MMAs, then
          // the math and the stores
          constexpr int kMine = BN / 16 / (C::kEpiWarps / 4);
          uint32_t ra[kMine][16];
#pragma unroll
          for (int i = 0; i < kMine; ++i)
            if (c_first + i * c_step < un.n) tmem_ld_32x32b_x16(t_row + c_first + i * c_step, ra[i]);
          tmem_ld_wait();
          release_acc();
          released = true;
#pragma unroll
          for (int i = 0; i < kMine; ++i) {
            if (c_first + i * c_step >= un.n) break;
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(ra[i][j]);
            emit_chunk(c_first + i * c_step, v);
          }
        } else {
          for (int c0 = c_first; c0 < un.n && ok; c0 += c_step) {
            uint32_t ra[16];
            tmem_ld_32x32b_x16(t_row + c0, ra);
            tmem_ld_wait();
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(ra[j]);
            bool good = true;
            for (int c = blockIdx.x + 1; c <= c_last; ++c) {
              if (range_start(W, c, ctas) == range_start(W, c + 1, ctas)) continue;  // empty range
              if (c0 == c_first && !wait_flag(A.flags + c * 4 + q, abort_flag, kWaitTimeoutNs)) {
                good = false;
                break;
              }
              const float* slot = A.partials + static_cast<int64_t>(c) * BN * 128;
#pragma unroll
              for (int j = 0; j < 16; ++j) v[j] += __ldcg(slot + (c0 + j) * 128 + row);
            }
            if (!__all_sync(0xFFFFFFFFu, good)) {  // warp-uniform: the shuffles below need every lane
              ok = false;
              where = kWaitPartials;
              break;
            }
            emit_chunk(c0, v);
          }
          // the partial-sum flags read here are cleared for the next launch
          if (ok && lane == 0)
            for (int c = blockIdx.x + 1; c <= c_last; ++c) A.flags[c * 4 + q] = 0;
        }
        // fused kernel: the unit's activation rows of this lane quarter are
        // stored; count this warp in its token chunk's counter (the down
        // GEMM's producers wait for four per weight tile, then order their TMA
        // reads after that acquire with a proxy fence)
        if (FUSED && ph == 0 && ok) {
          __threadfence();
          __syncwarp();
          if (lane == 0)
            red_release_add(ready + t_unit[un.e] / pa0.tiles + (un.tok0 - t_off[un.e]) / BN, 1);
        }
      }
      if (!ok) break;
      if (!released) release_acc();
      if (++acc == C::kAccBufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
      if (!SWIGLU && !FUSED && kb0 == 0 && args.fuse_combine && C::kEpiWarps == 4) {
        const int tile = PAIR ? 2 * un.tile + static_cast<int>(rank) : un.tile;
        ok = combine_unit<BN>(args, un, tile, row, lane, cbar, cbar_phase, cmask, abort_flag);
        if (!ok) {
          where = kWaitCombine;
          break;
        }
      }
    }
    if (!ok && lane == 0) raise_timeout(args.err, abort_flag, kern, where);
  }

  __syncthreads();
  // a pair keeps both CTAs (their shared memory, barriers and TMEM, which the
  // pair's MMAs and signals reach) until both are done
  if (PAIR) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, C::kTmemCols);
    else
      tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// tsw / tsx: the scale maps of MXFP8 pairs, or the fused kernel's W2 and
// activation maps; a2: the fused kernel's down GEMM.
template <bool SWIGLU, int BN, int STAGES, int TOKBOX, bool PAIR, bool MX = false, bool W4 = false,
          bool A4 = false, bool NV = false, bool FUSED = false, bool KTAIL = false, bool GATHER = false>
cudaError_t launch_expert_gemm(const CUtensorMap& tw, const CUtensorMap& tx, const ExpertGemmArgs& a, int num_sms,
                               cudaStream_t stream, const CUtensorMap* tsw = nullptr,
                               const CUtensorMap* tsx = nullptr, const ExpertGemmArgs* a2 = nullptr) {
  static const CUtensorMap kNoMap = {};  // unused map arguments
  using C = GemmCfg<SWIGLU, BN, STAGES, TOKBOX, PAIR, MX, W4, A4, NV, FUSED, GATHER>;
  auto kernel = expert_gemm_kernel<SWIGLU, BN, STAGES, TOKBOX, PAIR, MX, W4, A4, NV, FUSED, KTAIL, GATHER>;
  static PerDevice config;  // the smem attribute, and the CTA pairs that fit on the device at once
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = PAIR ? 2 : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  int max_pairs = 0;
  cudaError_t e = config.get(
      [&](int& pairs) -> cudaError_t {
        cudaError_t ce =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::kSmemBytes));
        if (ce != cudaSuccess || !PAIR) return ce;
        cudaLaunchConfig_t q = cfg;
        q.gridDim = dim3(2 * (kMaxGemmCtas / 2));
        q.attrs = attr + 1;
        q.numAttrs = 1;
        int n = 0;
        ce = cudaOccupancyMaxActiveClusters(&n, kernel, &q);
        if (ce != cudaSuccess) return ce;
        if (n <= 0) return cudaErrorInvalidConfiguration;
        pairs = n;
        return cudaSuccess;
      },
      &max_pairs);
  if (e != cudaSuccess) return e;
  int grid;
  if (PAIR) {
    const int pairs = max_pairs < kMaxGemmCtas / 2 ? max_pairs : kMaxGemmCtas / 2;
    grid = 2 * pairs;
  } else {
    grid = num_sms < kMaxGemmCtas ? num_sms : kMaxGemmCtas;
  }
  cfg.gridDim = dim3(grid);
  cfg.attrs = attr;
  cfg.numAttrs = PAIR ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, tw, tx, tsw ? *tsw : kNoMap, tsx ? *tsx : kNoMap, a, a2 ? *a2 : a);
}

// Two tile plans by the expected tokens per expert (T*top_k/E):
//   small (<= 16): 32-token units, deep weight pipelines, stream-K (decode);
//   large (> 16) : units of up to 256 tokens (the MMA's N follows the chunk's
//                  rows) and 128-row token boxes, on CTA pairs (M = 256 MMAs,
//                  each CTA loads half of the token tile) when the expert's
//                  weight tiles come in pairs.
// Between 16 and 64 rows per expert a one-CTA plan of 64-token units was
// slower than the large plan except under uniform routing at 32 rows per
// expert (by 1-2%): 17% slower under skewed routing, where the hot experts'
// weight tiles were streamed once per 64-token chunk, and 36% slower at 64
// rows per expert.
constexpr int kGateUpBn[2] = {32, 256}, kGateUpStages[2] = {10, 4};  // stages of 20 / 48 KB
constexpr int kDownBn[2] = {32, 256}, kDownStages[2] = {10, 4};      // stages of 20 / 48 KB
constexpr int kPairStages[2] = {7, 7};  // gate/up, down: stages of 32 KB
// token rows per TMA box: small units hold few tokens (16-row boxes waste
// nothing); large units hold up to 256 (128-row boxes: 8x fewer TMA requests)
constexpr int kTokBox[2] = {16, 128};

// MXFP8 plans: one CTA per unit of 32 tokens (10 stages of 22 KB) or, in
// the large plan, 128 tokens (6 of 33 KB; TMEM: two 128-column
// accumulators + 6 x 32 scale columns); prefill on CTA pairs when the weight
// tiles come in pairs: 256-token units, 6 stages of 34 KB per CTA (one
// 256-column accumulator + 6 x 32 scale columns)
constexpr int kMxBn[2] = {32, 128}, kMxStages[2] = {10, 6};
constexpr int kMxPairBn = 256;                              // tokens per pair unit (128: two accumulators)
constexpr int kMxPairStages = kMxPairBn == 256 ? 6 : 8;     // 34 KB / 25 KB stages per CTA
constexpr int kMxPairTokBox = kMxPairBn / 2;                // each CTA loads half of the unit's tokens

// The block-scaled GEMMs of one tile plan; W4: E2M1 weight codes; A4: E2M1
// token codes too (kind::mxf4).
// KTAIL: the MXFP4 layer's instances for K an odd multiple of 128 (its
// stages cover 256 elements of K)
template <bool SWIGLU, bool W4, bool A4 = false, bool KTAIL = false>
cudaError_t launch_mx_k(const CUtensorMap& tw, const CUtensorMap& tx, const CUtensorMap& tsw,
                        const CUtensorMap& tsx, const ExpertGemmArgs& a, GemmPlan plan, int num_sms,
                        cudaStream_t stream) {
  switch (plan) {
    case GemmPlan::kSmall:
      return launch_expert_gemm<SWIGLU, kMxBn[0], kMxStages[0], kTokBox[0], false, true, W4, A4, false, false, KTAIL>(
          tw, tx, a, num_sms, stream);
    default:
      if (a.pair)
        return launch_expert_gemm<SWIGLU, kMxPairBn, kMxPairStages, kMxPairTokBox, true, true, W4, A4, false, false,
                                  KTAIL>(tw, tx, a, num_sms, stream, &tsw, &tsx);
      return launch_expert_gemm<SWIGLU, kMxBn[1], kMxStages[1], kTokBox[1], false, true, W4, A4, false, false, KTAIL>(
          tw, tx, a, num_sms, stream);
  }
}

template <bool SWIGLU, bool W4, bool A4 = false>
cudaError_t launch_mx(const CUtensorMap& tw, const CUtensorMap& tx, const CUtensorMap& tsw, const CUtensorMap& tsx,
                      const ExpertGemmArgs& a, GemmPlan plan, int num_sms, cudaStream_t stream) {
  if (A4 && a.K % 256 != 0) return launch_mx_k<SWIGLU, W4, A4, true>(tw, tx, tsw, tsx, a, plan, num_sms, stream);
  return launch_mx_k<SWIGLU, W4, A4, false>(tw, tx, tsw, tsx, a, plan, num_sms, stream);
}

// NVFP4 plans: one CTA per unit of 32 / 128 tokens, 9 / 6 stages of 24 / 36 KB
// (4 KB of scale tiles per stage)
constexpr int kNvStages[2] = {9, 6};

template <bool SWIGLU, bool KTAIL>
cudaError_t launch_nv_k(const CUtensorMap& tw, const CUtensorMap& tx, const ExpertGemmArgs& a, GemmPlan plan,
                        int num_sms, cudaStream_t stream) {
  switch (plan) {
    case GemmPlan::kSmall:
      return launch_expert_gemm<SWIGLU, kMxBn[0], kNvStages[0], kTokBox[0], false, true, true, true, true, false,
                                KTAIL>(tw, tx, a, num_sms, stream);
    default:
      return launch_expert_gemm<SWIGLU, kMxBn[1], kNvStages[1], kTokBox[1], false, true, true, true, true, false,
                                KTAIL>(tw, tx, a, num_sms, stream);
  }
}

template <bool SWIGLU>
cudaError_t launch_nv(const CUtensorMap& tw, const CUtensorMap& tx, const ExpertGemmArgs& a, GemmPlan plan,
                      int num_sms, cudaStream_t stream) {
  if (a.K % 256 != 0) return launch_nv_k<SWIGLU, true>(tw, tx, a, plan, num_sms, stream);
  return launch_nv_k<SWIGLU, false>(tw, tx, a, plan, num_sms, stream);
}

}  // namespace

cudaError_t launch_gemm_gate_up_mx(const CUtensorMap& tm_w13, const CUtensorMap& tm_x, const CUtensorMap& tm_sw,
                                   const CUtensorMap& tm_sx, const ExpertGemmArgs& a, GemmPlan plan, int num_sms,
                                   cudaStream_t stream, MxKind kind) {
  switch (kind) {
    case MxKind::kW4A8:
      return launch_mx<true, true>(tm_w13, tm_x, tm_sw, tm_sx, a, plan, num_sms, stream);
    case MxKind::kW4A4:
      return launch_mx<true, true, true>(tm_w13, tm_x, tm_sw, tm_sx, a, plan, num_sms, stream);
    case MxKind::kNV4:
      return launch_nv<true>(tm_w13, tm_x, a, plan, num_sms, stream);
    default:
      return launch_mx<true, false>(tm_w13, tm_x, tm_sw, tm_sx, a, plan, num_sms, stream);
  }
}

cudaError_t launch_gemm_down_mx(const CUtensorMap& tm_w2, const CUtensorMap& tm_act, const CUtensorMap& tm_sw,
                                const CUtensorMap& tm_sx, const ExpertGemmArgs& a, GemmPlan plan, int num_sms,
                                cudaStream_t stream, MxKind kind) {
  switch (kind) {
    case MxKind::kW4A8:
      return launch_mx<false, true>(tm_w2, tm_act, tm_sw, tm_sx, a, plan, num_sms, stream);
    case MxKind::kW4A4:
      return launch_mx<false, true, true>(tm_w2, tm_act, tm_sw, tm_sx, a, plan, num_sms, stream);
    case MxKind::kNV4:
      return launch_nv<false>(tm_w2, tm_act, a, plan, num_sms, stream);
    default:
      return launch_mx<false, false>(tm_w2, tm_act, tm_sw, tm_sx, a, plan, num_sms, stream);
  }
}

int gemm_bn_mx(GemmPlan plan, bool pair) { return pair ? kMxPairBn : kMxBn[static_cast<int>(plan)]; }
int gemm_tok_box_rows_mx(GemmPlan plan, bool pair) { return pair ? kMxPairTokBox : kTokBox[static_cast<int>(plan)]; }

int gemm_gate_up_bn(GemmPlan plan) { return kGateUpBn[static_cast<int>(plan)]; }
int gemm_down_bn(GemmPlan plan) { return kDownBn[static_cast<int>(plan)]; }
int gemm_tok_box_rows(GemmPlan plan) { return kTokBox[static_cast<int>(plan)]; }
bool gemm_uses_pairs(GemmPlan plan, int tiles) { return plan == GemmPlan::kLarge && tiles % 2 == 0; }
int gemm_unit_tiles(GemmPlan plan, int tiles) { return gemm_uses_pairs(plan, tiles) ? tiles / 2 : tiles; }
// The block-scaled layers take CTA pairs only above 64 rows per expert: with
// thinner token chunks the per-stage scale copies of a pair's MMA thread, not
// the weight stream, set the pace (the MXFP4 layer at 32 rows per expert: 19%
// slower on pairs than on one-CTA units).
bool gemm_uses_pairs_mx(GemmPlan plan, int tiles, int64_t T, int64_t top_k, int64_t E) {
  return gemm_uses_pairs(plan, tiles) && T * top_k > 64 * E;
}

cudaError_t launch_gemm_gate_up(const CUtensorMap& tm_w13, const CUtensorMap& tm_x, const ExpertGemmArgs& a,
                                GemmPlan plan, int num_sms, cudaStream_t stream) {
  switch (plan) {
    case GemmPlan::kSmall:
      if (a.h_rows)  // token rows fetched from h by the row warps
        return launch_expert_gemm<true, kGateUpBn[0], kGateUpStages[0], kTokBox[0], false, false, false, false, false,
                                  false, false, true>(tm_w13, tm_x, a, num_sms, stream);
      return launch_expert_gemm<true, kGateUpBn[0], kGateUpStages[0], kTokBox[0], false>(tm_w13, tm_x, a, num_sms,
                                                                                          stream);
    default:
      if (a.pair)
        return launch_expert_gemm<true, kGateUpBn[1], kPairStages[0], kTokBox[1], true>(tm_w13, tm_x, a, num_sms,
                                                                                      stream);
      return launch_expert_gemm<true, kGateUpBn[1], kGateUpStages[1], kTokBox[1], false>(tm_w13, tm_x, a, num_sms,
                                                                                          stream);
  }
}

cudaError_t launch_gemm_fused_mlp(const CUtensorMap& tm_w13, const CUtensorMap& tm_x, const CUtensorMap& tm_w2,
                                  const CUtensorMap& tm_act, const ExpertGemmArgs& a1, const ExpertGemmArgs& a2,
                                  int num_sms, cudaStream_t stream) {
  return launch_expert_gemm<true, kGateUpBn[0], kGateUpStages[0], kTokBox[0], false, false, false, false, false, true>(
      tm_w13, tm_x, a1, num_sms, stream, &tm_w2, &tm_act, &a2);
}

cudaError_t launch_gemm_down(const CUtensorMap& tm_w2, const CUtensorMap& tm_act, const ExpertGemmArgs& a,
                             GemmPlan plan, int num_sms, cudaStream_t stream) {
  switch (plan) {
    case GemmPlan::kSmall:
      return launch_expert_gemm<false, kDownBn[0], kDownStages[0], kTokBox[0], false>(tm_w2, tm_act, a, num_sms,
                                                                                       stream);
    default:
      if (a.pair)
        return launch_expert_gemm<false, kDownBn[1], kPairStages[1], kTokBox[1], true>(tm_w2, tm_act, a, num_sms,
                                                                                     stream);
      return launch_expert_gemm<false, kDownBn[1], kDownStages[1], kTokBox[1], false>(tm_w2, tm_act, a, num_sms,
                                                                                       stream);
  }
}

}  // namespace moe
