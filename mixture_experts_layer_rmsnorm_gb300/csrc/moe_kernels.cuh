// moe_kernels.cuh -- launchers of the layer's kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace moe {

// error word codes (match moe_status) and kernel ids written with them
enum : int32_t { kErrTimeout = 5, kErrDevice = 6 };
enum : int32_t { kKernNormRouter = 1, kKernTopk = 2, kKernAlign = 3, kKernGather = 4, kKernGemm1 = 5,
                 kKernGemm2 = 6, kKernCombine = 7, kKernSelfTest = 8 };

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

// K1 + K1b + K2 + K3 for decode batches in one launch of one thread-block
// cluster (k_front.cu): same outputs as launch_norm_router, launch_align and
// launch_gather, except that padding rows of xg are left unwritten.
constexpr int kFrontMaxT = 64;
constexpr int kFrontMaxE = 256;
constexpr int kFrontMaxSmem = 136 * 1024;
struct FrontArgs {
  const uint16_t* x;
  const uint16_t* g;
  const float* w_router;
  const float* bias;
  int T, H, E, k, renorm;
  float eps;
  int pad, bn1, tiles1, bn2, tiles2;  // align padding and the GEMMs' work-unit tables
  uint16_t* h;
  float* logits;
  int32_t* ids;
  float* topk_w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* sorted_ids;
  int32_t* slot_of;
  int32_t* unit_off1;
  int32_t* unit_off2;
  int32_t* err;
  int32_t* flags;  // the expert GEMMs' stream-K flags: zeroed
  int n_flags;
  int32_t* combine_cnt;  // the down GEMM's combine arrival counters: zeroed
  int n_combine_cnt;
  uint16_t* xg;
  int skip_gather;  // 1: no gather (one token: the gate/up GEMM reads h itself)
  // set by the launcher: router work items = token tiles x expert groups
  int n_items, groups, experts_per_item;
};
// Whether the shape takes the single-launch front end on the current device.
bool front_fits(int T, int H, int E, int k);
cudaError_t launch_front(const FrontArgs& a, cudaStream_t stream);

// K3: xg[p,:] = h[sorted_ids[p] / k, :] for real rows, zeros for padding rows;
// also zeroes clear[0, n_clear) (the down GEMM's combine arrival counters).
cudaError_t launch_gather(const uint16_t* h, const int32_t* sorted_ids, const int32_t* offsets, int E, int N,
                          int k, int H, int64_t P_max, uint16_t* xg, int32_t* clear, int64_t n_clear,
                          cudaStream_t stream);

// K4 / K5: grouped expert GEMMs on tcgen05.  Weights are the MMA's A operand
// (128 weight rows per tile), the tokens of one expert its B operand.  The
// gate/up GEMM reads W13 through a 5-D tensor map (64 features per tile:
// 16 gate rows, the matching 16 up rows, x 4); the down GEMM reads W2 through
// a 2-D map of 128-row boxes.
struct ExpertGemmArgs {
  const int32_t* offsets;   // [E+1] padded row offsets
  const int32_t* unit_off;  // [E+1] prefix sums of work units
  int E;
  int K;                    // reduction length
  int tiles_per_expert;     // output features / 128
  int w_rows_per_expert;    // weight rows per expert of the down GEMM's 2-D map (H)
  int n_out;                // output row length (I or H)
  uint16_t* out;            // [P_max, n_out] bf16
  int32_t* err;
  float* partials;          // stream-K partial sums: [kMaxGemmCtas][BN][128] fp32
  int32_t* flags;           // [kMaxGemmCtas * 4], zero on entry; left zero on exit
  int stream_k;             // 1: equal K-block ranges per CTA; 0: whole units round-robin
  int pair;                 // 1: CTA pairs, a unit = weight tiles 2t and 2t+1 (large plan only)
  int tables_from_parent;   // 1: the routing tables come from the previous kernel (wait before reading)
  int tokens_from_h;        // 1 (one token, gate/up GEMM): tm_x maps h itself; every unit's token rows start
                            // at h row 0 (rows past T are read as zeros)
  int32_t* ready;           // fused gate/up -> down kernel: per token chunk, the gate/up epilogue warps that
                            // have stored their activation rows of it (zero on entry)
  const uint16_t* h_rows;   // gate/up GEMM of the decode tile plan: non-null = no gathered copy; the kernel's
                            // row warps fetch each unit's token rows from h [T, K] through sorted_ids (then
                            // also set: sorted_ids, top_k, n_routed)
  const uint8_t* w_scales;  // MXFP8 GEMMs: weight scales (512-byte tiles per 128 rows x 128 of K)
  const uint8_t* x_scales;  // MXFP8 GEMMs: token scales, one 512-byte tile per token chunk and 128 of K
  const float* w_gscale;    // NVFP4 GEMMs: fp32 tensor scale per expert matrix [E]
  const float* x_gscale;    // NVFP4 GEMMs: fp32 tensor scale per token row
  // Down GEMM with the top-k weighted combine in its epilogue (fuse_combine = 1):
  // a unit that has stored its output rows of a 128-feature tile counts one
  // arrival per real row at combine_cnt[tile * T + t]; the arrival that
  // completes token t's k rows writes y[t, tile] = bf16(sum_j topk_w[t,j] *
  // out[slot_of[t*k+j], tile]) in j order, from the bf16 rows, with the
  // arithmetic of the separate combine kernel.
  int fuse_combine;
  int32_t* combine_cnt;       // [n_out / 128][T] ints, zero on entry
  const int32_t* sorted_ids;  // [P] flat routing index t*k+j of each row; >= n_routed: padding
  const int32_t* slot_of;     // [T*k] row of each routed token
  const float* topk_w;        // [T*k]
  uint16_t* y;                // [T, n_out] bf16
  int top_k;
  int n_routed;               // T*k
};
// persistent GEMM grid: min(SM count, kMaxGemmCtas) CTAs
constexpr int kMaxGemmCtas = 256;

// tile plan of the expert GEMMs, by the expected tokens per expert
enum class GemmPlan { kSmall = 0, kLarge = 1 };
inline GemmPlan choose_plan(int64_t T, int64_t top_k, int64_t E) {
  return T * top_k <= 16 * E ? GemmPlan::kSmall : GemmPlan::kLarge;
}

// Whether an entry point that asks for both expert GEMMs in one launch
// (launch_gemm_fused_mlp) gets it: the small tile plan only.
inline bool fused_mlp_fits(GemmPlan plan) { return plan == GemmPlan::kSmall; }

// Whether the gate/up GEMM of a bf16 layer call reads its token tiles from h
// (one token: no gather), given the entry point's options (the fused combine
// keeps the gather, which zeroes its counters).
inline bool tokens_from_h(int T, bool fused_combine) { return T == 1 && !fused_combine; }
// Above one token on the decode tile plan, the gate/up GEMM copies its token
// rows from h itself (no gather kernel) unless a fused combine needs the
// gather's counter reset.
inline bool gate_up_gathers_rows(int T, GemmPlan plan, bool fused_combine) {
  return T > 1 && plan == GemmPlan::kSmall && !fused_combine;
}

// Encodes nothing itself: the tensor maps are built by the caller.
cudaError_t launch_gemm_gate_up(const CUtensorMap& tm_w13, const CUtensorMap& tm_x, const ExpertGemmArgs& a,
                                GemmPlan plan, int num_sms, cudaStream_t stream);
cudaError_t launch_gemm_down(const CUtensorMap& tm_w2, const CUtensorMap& tm_act, const ExpertGemmArgs& a,
                             GemmPlan plan, int num_sms, cudaStream_t stream);
// Both GEMMs of the small tile plan in one persistent launch ("4 · La fusion
// de noyaux", §4.2 "GEMM + GEMM" and §4.6): every CTA runs its stream-K range
// of the gate/up GEMM (a1), then its range of the down GEMM (a2); a down-GEMM
// unit's activation rows are loaded once every gate/up unit of its expert and
// token chunk has counted its four epilogue warps in a1.ready[chunk] (chunks
// numbered over all experts).  a1.ready: >= fused_mlp_ready_ints ints, zero
// on entry.
cudaError_t launch_gemm_fused_mlp(const CUtensorMap& tm_w13, const CUtensorMap& tm_x, const CUtensorMap& tm_w2,
                                  const CUtensorMap& tm_act, const ExpertGemmArgs& a1, const ExpertGemmArgs& a2,
                                  int num_sms, cudaStream_t stream);
// token chunks of the small plan at most: P_max rows in lists of >= 16 rows
inline int64_t fused_mlp_ready_ints(int64_t P_max) { return (P_max + 15) / 16; }
// Whether a GEMM with `tiles` weight tiles per expert runs on CTA pairs, and
// the tiles per expert its work-unit table counts (pairs of tiles then).
bool gemm_uses_pairs(GemmPlan plan, int tiles);
int gemm_unit_tiles(GemmPlan plan, int tiles);
bool gemm_uses_pairs_mx(GemmPlan plan, int tiles, int64_t T, int64_t top_k, int64_t E);  // block-scaled layers
// The same GEMMs on MXFP8 operands (block-scaled tcgen05 MMA):
// gemm_bn_mx(plan, a.pair) tokens per unit, on CTA pairs in the large plan when
// a.pair is set (weight tiles in pairs).  tm_sw / tm_sx map the weight and
// token scales as [tiles * 2][256] bytes (one 512-byte tile = a box of 2 rows);
// only the pair instances read them (the others load tiles from a.w_scales /
// a.x_scales directly).  tm_x maps E4M3 codes (one byte per element); tm_w
// E4M3 codes too, or for kW4A8 E2M1 codes (two per byte, a 16U4_ALIGN16B map
// with the same boxes); a.w_scales / a.x_scales hold the E8M0 scales.
// The operand formats of the block-scaled GEMMs: E4M3 x E4M3, E2M1 weights x
// E4M3 tokens (both kind::mxf8f6f4), E2M1 x E2M1 (kind::mxf4; tm_w and tm_x
// then map the packed code bytes, 256 elements of K per stage); NVFP4 on both
// (kind::mxf4nvf4, E4M3 scales per 16 elements, one-CTA units only, the fp32
// tensor scales a.w_gscale[e] * a.x_gscale[row] applied in the epilogue).
enum class MxKind { kW8A8, kW4A8, kW4A4, kNV4 };
cudaError_t launch_gemm_gate_up_mx(const CUtensorMap& tm_w13, const CUtensorMap& tm_x, const CUtensorMap& tm_sw,
                                   const CUtensorMap& tm_sx, const ExpertGemmArgs& a, GemmPlan plan, int num_sms,
                                   cudaStream_t stream, MxKind kind = MxKind::kW8A8);
cudaError_t launch_gemm_down_mx(const CUtensorMap& tm_w2, const CUtensorMap& tm_act, const CUtensorMap& tm_sw,
                                const CUtensorMap& tm_sx, const ExpertGemmArgs& a, GemmPlan plan, int num_sms,
                                cudaStream_t stream, MxKind kind = MxKind::kW8A8);
// rows of padding granularity of each expert's list for the MXFP8 GEMMs (a
// token scale group is 32 rows)
constexpr int kPadRowsMx = 32;
// token rows per unit (B-operand width) and rows per TMA box of the token tile
int gemm_gate_up_bn(GemmPlan plan);
int gemm_bn_mx(GemmPlan plan, bool pair);  // token rows per unit of an MXFP8 GEMM (pair: on CTA pairs)
int gemm_tok_box_rows_mx(GemmPlan plan, bool pair);  // token rows per TMA box of that GEMM
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

// MXFP8 quantization (k_mx_quant.cu): E4M3 codes [rows, K] in the rows'
// layout, E8M0 scales in the block-scaled MMA's tile layout (512 bytes per
// 128-row group and 128-element chunk of K).  K and rows: multiples of 128.
cudaError_t launch_mx_quantize_rows(const uint16_t* src, int64_t rows, int K, uint8_t* codes, uint8_t* scales,
                                    cudaStream_t stream);
cudaError_t launch_mx_quantize_w13(const uint16_t* w13, int E, int H, int I, uint8_t* codes, uint8_t* scales,
                                   cudaStream_t stream);
// MXFP4 weights: the same scale layout, E2M1 codes two per byte ([rows, K/2]
// bytes, element 2i in the low nibble of byte i), exponent floor(log2 amax) - 2
cudaError_t launch_mx4_quantize_rows(const uint16_t* src, int64_t rows, int K, uint8_t* codes, uint8_t* scales,
                                     cudaStream_t stream);
cudaError_t launch_mx4_quantize_w13(const uint16_t* w13, int E, int H, int I, uint8_t* codes, uint8_t* scales,
                                    cudaStream_t stream);
// token rows (gathered inputs / activations below offsets[E]): scales grouped
// by the GEMMs' token chunks (bn rows of an expert, chunk unit_off[e]/tiles + c)
cudaError_t launch_mx_gather(const uint16_t* h, const int32_t* sorted_ids, const int32_t* offsets,
                             const int32_t* unit_off, int tiles, int bn, int E, int N, int k, int H, int64_t rows,
                             uint8_t* codes, uint8_t* scales, cudaStream_t stream);
cudaError_t launch_mx_quantize_act(const uint16_t* act, int64_t rows, int K, const int32_t* offsets,
                                   const int32_t* unit_off, int tiles, int bn, int E, uint8_t* codes, uint8_t* scales,
                                   cudaStream_t stream);
// the MXFP4 layer's token rows and activations: E2M1 codes two per byte
// ([rows, K/2] bytes), scales as above
cudaError_t launch_mx4_gather(const uint16_t* h, const int32_t* sorted_ids, const int32_t* offsets,
                              const int32_t* unit_off, int tiles, int bn, int E, int N, int k, int H, int64_t rows,
                              uint8_t* codes, uint8_t* scales, cudaStream_t stream);
cudaError_t launch_mx4_quantize_act(const uint16_t* act, int64_t rows, int K, const int32_t* offsets,
                                    const int32_t* unit_off, int tiles, int bn, int E, uint8_t* codes,
                                    uint8_t* scales, cudaStream_t stream);
// NVFP4 (k_mx_quant.cu): E2M1 codes two per byte, E4M3 scales per 16 elements
// in 512-byte tiles per 128 rows and 64 elements of K, fp32 tensor scales.
// Weights: the absolute maximum per expert matrix (rows_per_tensor rows) into
// amax[] (launch_nv4_weight_amax), the codes and scales from it, then amax[]
// turned into the tensor scales in place (launch_nv4_global).  Token rows and
// activations: one tensor scale per row, written to g_rows[row].
cudaError_t launch_nv4_weight_amax(const uint16_t* src, int64_t rows, int K, int64_t rows_per_tensor, float* amax,
                                   int n_tensors, cudaStream_t stream);
cudaError_t launch_nv4_global(float* amax_to_g, int n, cudaStream_t stream);
cudaError_t launch_nv4_quantize_rows(const uint16_t* src, int64_t rows, int K, int64_t rows_per_tensor,
                                     const float* tensor_amax, uint8_t* codes, uint8_t* scales, cudaStream_t stream);
cudaError_t launch_nv4_quantize_w13(const uint16_t* w13, int E, int H, int I, const float* tensor_amax,
                                    uint8_t* codes, uint8_t* scales, cudaStream_t stream);
cudaError_t launch_nv4_gather(const uint16_t* h, const int32_t* sorted_ids, const int32_t* offsets,
                              const int32_t* unit_off, int tiles, int bn, int E, int N, int k, int H, int64_t rows,
                              uint8_t* codes, uint8_t* scales, float* g_rows, cudaStream_t stream);
cudaError_t launch_nv4_quantize_act(const uint16_t* act, int64_t rows, int K, const int32_t* offsets,
                                    const int32_t* unit_off, int tiles, int bn, int E, uint8_t* codes,
                                    uint8_t* scales, float* g_rows, cudaStream_t stream);
inline size_t nv4_scale_bytes(int64_t rows, int64_t K) { return static_cast<size_t>(rows / 128) * (K / 64) * 512; }
inline size_t mx_scale_bytes(int64_t rows, int64_t K) { return static_cast<size_t>(rows / 128) * (K / 128) * 512; }

// QK-norm of q[T, Hq, D] and k[T, Hk, D] in place (k_qk_norm.cu); D = 64, 128 or 256.
cudaError_t launch_qk_norm(uint16_t* q, uint16_t* k, const uint16_t* q_weight, const uint16_t* k_weight, int64_t T,
                           int Hq, int Hk, int D, float weight_bias, float eps, cudaStream_t stream);

// Self-test of the bounded waits: one kernel whose two waits (an mbarrier
// phase, a global flag) run out after timeout_ns and report MOE_ERR_TIMEOUT
// with kernel id kKernSelfTest in the error word at `err` (>= 64 bytes).
cudaError_t launch_selftest_wait(int32_t* err, uint64_t timeout_ns, cudaStream_t stream);

// K6: y[t,:] = bf16(sum_j topk_w[t,j] * out_rows[slot_of[t*k+j], :]).
cudaError_t launch_combine(const uint16_t* out_rows, const int32_t* slot_of, const float* topk_w, int T, int H,
                           int k, uint16_t* y, cudaStream_t stream);

}  // namespace moe
