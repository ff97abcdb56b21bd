// moe_kernels.cuh -- launchers of the layer's kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace moe {

// error word codes (match moe_status) and kernel ids written with them
enum : int32_t { kErrTimeout = 5, kErrDevice = 6 };
enum : int32_t { kKernNormRouter = 1, kKernTopk = 2, kKernAlign = 3, kKernGather = 4, kKernGemm1 = 5,
                 kKernGemm2 = 6, kKernCombine = 7 };

// rows of padding granularity of each expert's list in the expert GEMMs
constexpr int kPadRows = 16;
// bounded device waits give up after this long
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

// K1: RMSNorm of every token + fp32 router logits (canonical summation order).
// Writes h[T,H] bf16 and logits[T,E] fp32; clears the error word.
cudaError_t launch_norm_router(const uint16_t* x, const uint16_t* g, const float* w_router, const float* bias,
                               int T, int H, int E, float eps, uint16_t* h, float* logits, int32_t* err,
                               int num_sms, cudaStream_t stream);

// K2: deterministic align: counts, padded offsets, sorted_ids, slot_of and the
// prefix sums of work units of the two expert GEMMs (units per expert =
// ceil(P_e / bn) * tiles; bn = 0 skips that table).  When
// align_fuses_topk(T, E), the same single CTA first runs K1b for all T tokens
// (topk_ids / topk_w from the logits) and K1b must not be launched.
// It also clears n_flags ints at `flags` (the expert GEMMs' stream-K flags).
cudaError_t launch_align(const float* logits, int T, int k, int renorm, int32_t* topk_ids, float* topk_w, int N,
                         int E, int pad, int bn1, int tiles1, int bn2, int tiles2, int32_t* counts, int32_t* offsets,
                         int32_t* sorted_ids, int32_t* slot_of, int32_t* unit_off1, int32_t* unit_off2, int32_t* err,
                         int32_t* flags, int n_flags, cudaStream_t stream);
constexpr int kFusedTopkMaxT = 256;
constexpr int kFusedTopkMaxE = 256;
bool align_fuses_topk(int T, int E);

// K1b + K2 for the other shapes, over many CTAs (three launches: count with
// top-k, scan, scatter).  blk_counts / blk_base: align_multi_blocks(T) * E
// ints of scratch each.  count_done_event (a cudaEvent_t, or null) is recorded
// after the first of the three kernels.
constexpr int kAlignTokPerBlk = 32;
int align_multi_blocks(int T);
cudaError_t launch_align_multi(const float* logits, int T, int k, int renorm, int32_t* topk_ids, float* topk_w, int E,
                               int pad, int bn1, int tiles1, int bn2, int tiles2, int32_t* counts, int32_t* offsets,
                               int32_t* sorted_ids, int32_t* slot_of, int32_t* unit_off1, int32_t* unit_off2,
                               int32_t* blk_counts, int32_t* blk_base, int32_t* err, int32_t* flags, int n_flags,
                               cudaStream_t stream, void* count_done_event);

// K3: xg[p,:] = h[sorted_ids[p] / k, :] for real rows, zeros for padding rows.
cudaError_t launch_gather(const uint16_t* h, const int32_t* sorted_ids, const int32_t* offsets, int E, int N,
                          int k, int H, int64_t P_max, uint16_t* xg, cudaStream_t stream);

// K4 / K5: grouped expert GEMMs on tcgen05.  Weights are the MMA's A operand
// (128 weight rows per tile), the tokens of one expert its B operand.
struct ExpertGemmArgs {
  const int32_t* offsets;   // [E+1] padded row offsets
  const int32_t* unit_off;  // [E+1] prefix sums of work units
  int E;
  int K;                    // reduction length
  int tiles_per_expert;     // output features / 128
  int w_rows_per_expert;    // 2I (gate/up) or H (down)
  int up_offset;            // I for gate/up, unused for down
  int n_out;                // output row length (I or H)
  uint16_t* out;            // [P_max, n_out] bf16
  int32_t* err;
  float* partials;          // stream-K partial sums: [kMaxGemmCtas][BN][128] fp32
  int32_t* flags;           // [kMaxGemmCtas * 4], zero on entry; left zero on exit
  int stream_k;             // 1: equal K-block ranges per CTA; 0: whole units round-robin
  int pair;                 // 1: CTA pairs, a unit = weight tiles 2t and 2t+1 (large plan only)
};
// persistent GEMM grid: min(SM count, kMaxGemmCtas) CTAs
constexpr int kMaxGemmCtas = 256;

// tile plan of the expert GEMMs, by the expected tokens per expert
enum class GemmPlan { kSmall = 0, kMid = 1, kLarge = 2 };
inline GemmPlan choose_plan(int64_t T, int64_t top_k, int64_t E) {
  const int64_t tk = T * top_k;
  if (tk <= 16 * E) return GemmPlan::kSmall;
  if (tk <= 64 * E) return GemmPlan::kMid;
  return GemmPlan::kLarge;
}

// Encodes nothing itself: the tensor maps are built by the caller.
cudaError_t launch_gemm_gate_up(const CUtensorMap& tm_w13, const CUtensorMap& tm_x, const ExpertGemmArgs& a,
                                GemmPlan plan, int num_sms, cudaStream_t stream);
cudaError_t launch_gemm_down(const CUtensorMap& tm_w2, const CUtensorMap& tm_act, const ExpertGemmArgs& a,
                             GemmPlan plan, int num_sms, cudaStream_t stream);
// Whether a GEMM with `tiles` weight tiles per expert runs on CTA pairs, and
// the tiles per expert its work-unit table counts (pairs of tiles then).
bool gemm_uses_pairs(GemmPlan plan, int tiles);
int gemm_unit_tiles(GemmPlan plan, int tiles);
// token rows per unit (B-operand width) and rows per TMA box of the token tile
int gemm_gate_up_bn(GemmPlan plan);
int gemm_down_bn(GemmPlan plan);
int gemm_tok_box_rows(GemmPlan plan);
constexpr int kWeightBoxRows = 128;  // A-operand rows of one unit (one MMA's M)
constexpr int kGateUpTileFeat = 64;  // gate/up unit: 64 gate rows stacked on the matching 64 up rows
constexpr int kDownTileFeat = 128;   // down unit: 128 rows of W2
constexpr int kBlockK = 64;

// Launch with programmatic dependent launch allowed: the kernel may be
// scheduled while the previous kernel in the stream is finishing; it must
// execute griddepcontrol.wait (pdl_wait) before touching global memory that
// earlier stream work reads or writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// K6: y[t,:] = bf16(sum_j topk_w[t,j] * out_rows[slot_of[t*k+j], :]).
cudaError_t launch_combine(const uint16_t* out_rows, const int32_t* slot_of, const float* topk_w, int T, int H,
                           int k, uint16_t* y, cudaStream_t stream);

}  // namespace moe
