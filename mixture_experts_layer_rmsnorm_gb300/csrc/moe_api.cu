// moe_api.cu -- the C ABI declared in include/moe.h: argument checks, the
// workspace layout, TMA tensor maps, the decode / prefill plan and the launch
// sequence K1 -> K1b -> K2 -> K3 -> K4 -> K5 -> K6 on the caller's stream.
//
// Plan ("CuTeDSL chez Perplexity", "Pré-remplir et décoder la
// spécialisation": kernels are split into prefill and decode variants by
// token count, hidden size and dtype).  The expected tokens per expert
// T*top_k/E picks the expert-GEMM tiles: <= 16 small (32 tokens per unit,
// deepest weight pipelines), <= 64 mid (64 tokens per unit), above that the
// prefill tiles (128 / 256 tokens per unit).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/moe.h"
#include "moe_forward_impl.h"
#include "moe_kernels.cuh"

namespace {

using moe::GemmPlan;

constexpr size_t kAlign = 256;
constexpr int kMaxDebugPad = 256;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Layout {
  size_t err, h, logits, ids, w, counts, offsets, unit1, unit2, sorted, slot, flags, ccnt, blk_counts, blk_base,
      partials, xg, act, out, xs, aq, as, gx, ga, total;
  int64_t n_ccnt;      // combine arrival counters of the down GEMM: [H / 128][T]
  int64_t n_flags;     // ints at `flags` cleared by the align: stream-K flags, then (small tile plan) the
                       // fused gate/up -> down kernel's per-chunk completion counters
  int64_t P_max;       // padded rows: 16-row padding (bf16), 32-row padding rounded to 128 (MXFP8)
  int64_t sorted_cap;  // sorted_ids entries (room for debug padding up to 256)
};

// stream-K flags: [2 GEMMs][kMaxGemmCtas][4 lane quarters]
constexpr int kGemmFlagInts = 2 * moe::kMaxGemmCtas * 4;

// stream-K partial sums of one GEMM: per CTA a [BN][128] fp32 slot
size_t partial_slots_bytes(const moe_shape& s) {
  return static_cast<size_t>(moe::kMaxGemmCtas) * moe::gemm_gate_up_bn(moe::choose_plan(s.T, s.top_k, s.E)) * 128 * 4;
}

// mx: the MXFP8 layer (token rows padded to 32 per expert; xg holds E4M3
// codes, plus token and activation scales and activation codes).
Layout make_layout(const moe_shape& s, bool mx = false) {
  Layout L{};
  const int64_t T = s.T, H = s.H, I = s.I, E = s.E, k = s.top_k;
  L.P_max = mx ? (T * k + E * (moe::kPadRowsMx - 1) + 127) / 128 * 128 : T * k + E * (moe::kPadRows - 1);
  L.sorted_cap = T * k + E * (kMaxDebugPad - 1);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t r = off;
    off = align_up(off + bytes, kAlign);
    return r;
  };
  L.err = take(64);
  L.h = take(static_cast<size_t>(T * H * 2));
  L.logits = take(static_cast<size_t>(T * E * 4));
  L.ids = take(static_cast<size_t>(T * k * 4));
  L.w = take(static_cast<size_t>(T * k * 4));
  L.counts = take(static_cast<size_t>(E * 4));
  L.offsets = take(static_cast<size_t>((E + 1) * 4));
  L.unit1 = take(static_cast<size_t>((E + 1) * 4));
  L.unit2 = take(static_cast<size_t>((E + 1) * 4));
  L.sorted = take(static_cast<size_t>(L.sorted_cap * 4));
  L.slot = take(static_cast<size_t>(T * k * 4));
  // stream-K flags and partial sums of the expert GEMMs (slot = BN x 128 fp32 per CTA)
  const bool small = moe::choose_plan(T, k, E) == moe::GemmPlan::kSmall;
  L.n_flags = kGemmFlagInts + (small && !mx ? moe::fused_mlp_ready_ints(L.P_max) : 0);
  L.flags = take(static_cast<size_t>(L.n_flags) * 4);
  L.n_ccnt = (H / 128) * T;
  L.ccnt = take(static_cast<size_t>(L.n_ccnt) * 4);
  // per-block counts / bases of the multi-CTA align
  L.blk_counts = take(static_cast<size_t>((T + moe::kAlignTokPerBlk - 1) / moe::kAlignTokPerBlk) * E * 4);
  L.blk_base = take(static_cast<size_t>((T + moe::kAlignTokPerBlk - 1) / moe::kAlignTokPerBlk) * E * 4);
  L.partials = take(2 * partial_slots_bytes(s));
  L.xg = take(static_cast<size_t>(L.P_max * H * 2));
  L.act = take(static_cast<size_t>(L.P_max * I * 2));
  L.out = take(static_cast<size_t>(L.P_max * H * 2));
  if (mx) {  // token scales per token chunk: at most P_max / 32 chunks (each >= 32 rows)
    L.xs = take(static_cast<size_t>(L.P_max / 32) * 2 * (H / 128) * 512);
    L.aq = take(static_cast<size_t>(L.P_max * I));
    L.as = take(static_cast<size_t>(L.P_max / 32) * 2 * (I / 128) * 512);
    // NVFP4: fp32 tensor scale of each gathered token row and activation row
    // (its token scales, one 512-byte tile per <= 128 rows and 64 of K, fit xs / as)
    L.gx = take(static_cast<size_t>(L.P_max) * 4);
    L.ga = take(static_cast<size_t>(L.P_max) * 4);
  }
  L.total = off;
  return L;
}

moe_status check_shape(const moe_shape* s) {
  if (!s) return MOE_ERR_INVALID_ARG;
  if (s->T < 0 || s->H <= 0 || s->I <= 0 || s->E <= 0 || s->top_k <= 0 || s->top_k > s->E)
    return MOE_ERR_INVALID_ARG;
  if (!(s->eps >= 0.0f) || !std::isfinite(s->eps)) return MOE_ERR_INVALID_ARG;
  // H: 128 output features per down-GEMM weight tile; I: 64 features per
  // gate/up unit and 64 elements of K per down-GEMM stage; H <= 16384: the
  // router keeps its tokens' h rows in shared memory; top_k <= 32: one lane
  // of the selecting warp per selected expert
  if (s->H % 128 != 0 || s->I % 64 != 0 || s->H > 16384 || s->I > 16384 || s->E > 1024 || s->top_k > 32)
    return MOE_ERR_UNSUPPORTED;
  // 32-bit row indices inside the kernels
  const int64_t rows = static_cast<int64_t>(s->T) * s->top_k + static_cast<int64_t>(s->E) * (kMaxDebugPad - 1);
  if (rows >= (int64_t(1) << 30)) return MOE_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(s->E) * 2 * s->I >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// The block-scaled layers: scale tiles cover 128 elements of K (and a
// block-scaled GEMM stage at least 128), so I must be a multiple of 128 too.
moe_status check_shape_mx(const moe_shape* s) {
  const moe_status st = check_shape(s);
  if (st != MOE_OK) return st;
  return s->I % 128 != 0 ? MOE_ERR_UNSUPPORTED : MOE_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 row-major [rows, inner] tensor, boxes of 64 x box_rows, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(moe::kBlockK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// W13 [E][2I][H] bf16 viewed as [E][2][I/16][16][H] (innermost last in the
// names, first in the dims below): one box of {64, 16, 2, 4, 1} is a 128-row
// gate/up tile whose 16-row groups alternate gate rows and the matching up rows.
bool make_map_gate_up(CUtensorMap* m, const void* w13, uint64_t H, uint64_t I, uint64_t E) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[5] = {H, 16, 2, I / 16, E};
  cuuint64_t strides[4] = {H * 2, I * H * 2, 16 * H * 2, 2 * I * H * 2};
  cuuint32_t box[5] = {static_cast<cuuint32_t>(moe::kBlockK), 16, 2, moe::kGateUpTileFeat / 16, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(w13), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// E4M3 codes [rows, inner] (one byte per element), boxes of 128 x box_rows.
bool make_map_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MXFP8 scale tiles (512 bytes each) viewed as [2 * n_tiles][256] bytes: tile
// i is the box of 2 rows at row 2i (no swizzle: its bytes land in order).
bool make_map_scales(CUtensorMap* m, const void* base, uint64_t n_tiles) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {256, 2 * n_tiles};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {256, 2};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// W13 codes viewed as [E][2][I/16][16][H] like the bf16 map: boxes of 128 x 16 x 2 x 4 x 1.
bool make_map_gate_up_u8(CUtensorMap* m, const void* w13c, uint64_t H, uint64_t I, uint64_t E) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[5] = {H, 16, 2, I / 16, E};
  cuuint64_t strides[4] = {H, I * H, 16 * H, 2 * I * H};
  cuuint32_t box[5] = {128, 16, 2, moe::kGateUpTileFeat / 16, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void*>(w13c), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// E2M1 codes [rows, inner], two per byte (inner / 2 bytes per row), boxes of
// 128 x box_rows; 16U4_ALIGN16B spreads each 8 code bytes over 16 bytes of
// shared memory, so a box lands as the image of an E4M3 box of the same shape.
// inner: a multiple of 128 (the type's rule; the row stride is then a multiple
// of 32 bytes); base: 32-byte aligned.
bool make_map_u4(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner / 2};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// W13 E2M1 codes viewed as [E][2][I/16][16][H] like the bf16 map (dimensions
// in elements, strides in bytes of the packed codes).
bool make_map_gate_up_u4(CUtensorMap* m, const void* w13c, uint64_t H, uint64_t I, uint64_t E) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[5] = {H, 16, 2, I / 16, E};
  cuuint64_t strides[4] = {H / 2, I * H / 2, 16 * H / 2, 2 * I * H / 2};
  cuuint32_t box[5] = {128, 16, 2, moe::kGateUpTileFeat / 16, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 5, const_cast<void*>(w13c), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms_of_current_device() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 0 || dev >= 64) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

moe_status check_inputs(const moe_shape* s, const void* x, const void* g, const float* wr, const float* bias,
                        void* ws, size_t ws_bytes, bool mx = false) {
  if (!x || !g || !wr || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(g, 16) || !aligned(wr, 16) || (bias && !aligned(bias, 4)) || !aligned(ws, kAlign))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < make_layout(*s, mx).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

// K1 + K1b + K2 with the given padding; unit tables only when bn1/bn2 > 0.
moe_status run_front(const moe_shape& s, const Layout& L, const moe_bf16* x, const moe_bf16* g, const float* wr,
                     const float* bias, int pad, int bn1, int utiles1, int bn2, int utiles2, void* ws,
                     cudaStream_t st, int num_sms) {
  int32_t* err = at<int32_t>(ws, L.err);
  if (moe::launch_norm_router(x, g, wr, bias, s.T, s.H, s.E, s.eps, at<uint16_t>(ws, L.h), at<float>(ws, L.logits),
                              err, num_sms, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  cudaError_t ce;
  if (moe::align_fuses_topk(s.T, s.E))
    ce = moe::launch_align(at<float>(ws, L.logits), s.T, s.top_k, s.renormalize, at<int32_t>(ws, L.ids),
                           at<float>(ws, L.w), s.T * s.top_k, s.E, pad, bn1, utiles1, bn2,
                           utiles2, at<int32_t>(ws, L.counts), at<int32_t>(ws, L.offsets),
                           at<int32_t>(ws, L.sorted), at<int32_t>(ws, L.slot),
                           bn1 > 0 ? at<int32_t>(ws, L.unit1) : nullptr, bn2 > 0 ? at<int32_t>(ws, L.unit2) : nullptr,
                           err, at<int32_t>(ws, L.flags), static_cast<int>(L.n_flags), st);
  else
    ce = moe::launch_align_multi(at<float>(ws, L.logits), s.T, s.top_k, s.renormalize, at<int32_t>(ws, L.ids),
                                 at<float>(ws, L.w), s.E, pad, bn1, utiles1, bn2,
                                 utiles2, at<int32_t>(ws, L.counts), at<int32_t>(ws, L.offsets),
                                 at<int32_t>(ws, L.sorted), at<int32_t>(ws, L.slot),
                                 bn1 > 0 ? at<int32_t>(ws, L.unit1) : nullptr,
                                 bn2 > 0 ? at<int32_t>(ws, L.unit2) : nullptr, at<int32_t>(ws, L.blk_counts),
                                 at<int32_t>(ws, L.blk_base), err, at<int32_t>(ws, L.flags), static_cast<int>(L.n_flags), st,
                                 nullptr);
  if (ce != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_workspace_size(const moe_shape* shape, size_t* bytes) {
  const moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = make_layout(*shape).total;
  return MOE_OK;
}

moe_status moe_kernels_per_call_of(const moe_shape* shape, int32_t call, int32_t* count) {
  const moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (!count || call < MOE_CALL_FORWARD || call > MOE_CALL_FORWARD_FUSED_MLP) return MOE_ERR_INVALID_ARG;
  const moe_shape& s = *shape;
  if (s.T == 0) {
    *count = 0;
    return MOE_OK;
  }
  // router, top-k + align (1 kernel, or 3), gather, the two GEMMs, combine
  const int front = 1 + (moe::align_fuses_topk(s.T, s.E) ? 1 : 3) + 1;
  if (call == MOE_CALL_FORWARD_FUSED_MLP && !moe::fused_mlp_fits(moe::choose_plan(s.T, s.top_k, s.E)))
    return MOE_ERR_UNSUPPORTED;
  // no gather for one token, nor (moe_forward) when the decode-plan gate/up
  // GEMM reads the rows of h itself
  const int one_token = moe::tokens_from_h(s.T, false) ? 1 : 0;
  const int rows_from_h = moe::gate_up_gathers_rows(s.T, moe::choose_plan(s.T, s.top_k, s.E), false) ? 1 : 0;
  if (call == MOE_CALL_FORWARD)
    *count = front + 3 - one_token - rows_from_h;
  else if (call == MOE_CALL_FORWARD_FUSED_MLP)
    *count = front + 2 - one_token;  // both GEMMs in one launch
  else if (call == MOE_CALL_FORWARD_FUSED_FRONT)
    *count = 1 + 3;
  else if (call == MOE_CALL_FORWARD_MX || call == MOE_CALL_FORWARD_MXFP4 || call == MOE_CALL_FORWARD_MXFP4A4 ||
           call == MOE_CALL_FORWARD_NVFP4)
    *count = front + 4;  // + the activation quantize between the GEMMs
  else
    *count = front + 2;  // the combine runs inside the down GEMM
  return MOE_OK;
}

moe_status moe_kernels_per_call(const moe_shape* shape, int32_t* count) {
  return moe_kernels_per_call_of(shape, MOE_CALL_FORWARD, count);
}

moe_status moe_workspace_views(const moe_shape* shape, void* workspace, size_t workspace_bytes, moe_views* v) {
  const moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (!workspace || !v) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(*shape);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
  v->error_word = at<void>(workspace, L.err);
  v->h = at<void>(workspace, L.h);
  v->logits = at<void>(workspace, L.logits);
  v->topk_ids = at<void>(workspace, L.ids);
  v->topk_w = at<void>(workspace, L.w);
  v->counts = at<void>(workspace, L.counts);
  v->offsets = at<void>(workspace, L.offsets);
  v->sorted_ids = at<void>(workspace, L.sorted);
  v->slot_of = at<void>(workspace, L.slot);
  v->xg = at<void>(workspace, L.xg);
  v->act = at<void>(workspace, L.act);
  v->out_rows = at<void>(workspace, L.out);
  v->P_max = L.P_max;
  return MOE_OK;
}

}  // extern "C"

namespace moe {

// The down GEMM's arguments for the top-k weighted combine in its epilogue.
void set_fused_combine(moe::ExpertGemmArgs& a, const moe_shape& s, const Layout& L, void* workspace, moe_bf16* y) {
  a.fuse_combine = 1;
  a.combine_cnt = at<int32_t>(workspace, L.ccnt);
  a.sorted_ids = at<int32_t>(workspace, L.sorted);
  a.slot_of = at<int32_t>(workspace, L.slot);
  a.topk_w = at<float>(workspace, L.w);
  a.y = reinterpret_cast<uint16_t*>(y);
  a.top_k = s.top_k;
  a.n_routed = s.T * s.top_k;
}

// The forward pass; when `events` is given, events[0] is recorded before the
// first kernel and events[i] after the i-th of the seven kernels.
moe_status forward_impl(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm, const float* w_router,
                        const float* router_bias, const moe_bf16* w13, const moe_bf16* w2, moe_bf16* y,
                        void* workspace, size_t workspace_bytes, moe_stream_t stream, void* const* events,
                        bool single_launch_front, bool fused_combine, bool fused_mlp) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  const moe_shape& s = *shape;
  if (s.T == 0) return MOE_OK;  // nothing to compute; no pointer is touched
  st = check_inputs(shape, x, g_norm, w_router, router_bias, workspace, workspace_bytes);
  if (st != MOE_OK) return st;
  if (!w13 || !w2 || !y || !aligned(w13, 16) || !aligned(w2, 16) || !aligned(y, 16)) return MOE_ERR_INVALID_ARG;
  if (fused_mlp && (fused_combine || !moe::fused_mlp_fits(moe::choose_plan(s.T, s.top_k, s.E))))
    return MOE_ERR_UNSUPPORTED;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const int num_sms = num_sms_of_current_device();
  if (num_sms <= 0) return MOE_ERR_CUDA;
  if (single_launch_front && !moe::front_fits(s.T, s.H, s.E, s.top_k)) return MOE_ERR_UNSUPPORTED;
  const Layout L = make_layout(s);
  const GemmPlan plan = moe::choose_plan(s.T, s.top_k, s.E);
  const int bn1 = moe::gemm_gate_up_bn(plan), bn2 = moe::gemm_down_bn(plan);
  // work-unit tables count weight tiles, or pairs of them for CTA-pair GEMMs
  const int tiles1 = s.I / moe::kGateUpTileFeat, tiles2 = s.H / moe::kDownTileFeat;
  const int utiles1 = moe::gemm_unit_tiles(plan, tiles1), utiles2 = moe::gemm_unit_tiles(plan, tiles2);
  auto mark = [&](int i) {
    return !events || cudaEventRecord(static_cast<cudaEvent_t>(events[i]), cs) == cudaSuccess;
  };

  // One token: every expert's list is that token's row of h (padded to 16
  // rows), so the gate/up GEMM reads its token tiles straight from h, rows
  // past T reading as zeros, and no gather runs.
  const bool tokens_from_h = moe::tokens_from_h(s.T, fused_combine);
  // More tokens on the decode tile plan: the gate/up GEMM copies each unit's
  // token rows from h itself (its row warps read sorted_ids); no gather runs.
  const bool rows_from_h = !single_launch_front && !fused_mlp && moe::gate_up_gathers_rows(s.T, plan, fused_combine);
  CUtensorMap tm_w13, tm_xg, tm_w2, tm_act;
  if (!make_map_gate_up(&tm_w13, w13, s.H, s.I, s.E) ||
      !(tokens_from_h ? make_map(&tm_xg, at<void>(workspace, L.h), s.H, s.T, moe::gemm_tok_box_rows(plan))
                      : make_map(&tm_xg, at<void>(workspace, L.xg), s.H, L.P_max, moe::gemm_tok_box_rows(plan))) ||
      !make_map(&tm_w2, w2, s.I, static_cast<uint64_t>(s.E) * s.H, moe::kWeightBoxRows) ||
      !make_map(&tm_act, at<void>(workspace, L.act), s.I, L.P_max, moe::gemm_tok_box_rows(plan)))
    return MOE_ERR_CUDA;

  int32_t* err = at<int32_t>(workspace, L.err);
  if (!mark(0)) return MOE_ERR_CUDA;
  const int N = s.T * s.top_k;
  // norm, router, top-k, align and gather in one launch (when asked for)
  const bool front = single_launch_front;
  if (front) {
    moe::FrontArgs fa{};
    fa.x = x;
    fa.g = g_norm;
    fa.w_router = w_router;
    fa.bias = router_bias;
    fa.T = s.T;
    fa.H = s.H;
    fa.E = s.E;
    fa.k = s.top_k;
    fa.renorm = s.renormalize;
    fa.eps = s.eps;
    fa.pad = moe::kPadRows;
    fa.bn1 = bn1;
    fa.tiles1 = utiles1;
    fa.bn2 = bn2;
    fa.tiles2 = utiles2;
    fa.h = at<uint16_t>(workspace, L.h);
    fa.logits = at<float>(workspace, L.logits);
    fa.ids = at<int32_t>(workspace, L.ids);
    fa.topk_w = at<float>(workspace, L.w);
    fa.counts = at<int32_t>(workspace, L.counts);
    fa.offsets = at<int32_t>(workspace, L.offsets);
    fa.sorted_ids = at<int32_t>(workspace, L.sorted);
    fa.slot_of = at<int32_t>(workspace, L.slot);
    fa.unit_off1 = at<int32_t>(workspace, L.unit1);
    fa.unit_off2 = at<int32_t>(workspace, L.unit2);
    fa.err = err;
    fa.flags = at<int32_t>(workspace, L.flags);
    fa.n_flags = static_cast<int>(L.n_flags);
    fa.combine_cnt = at<int32_t>(workspace, L.ccnt);
    fa.n_combine_cnt = fused_combine ? static_cast<int>(L.n_ccnt) : 0;
    fa.xg = at<uint16_t>(workspace, L.xg);
    fa.skip_gather = tokens_from_h;
    if (moe::launch_front(fa, cs) != cudaSuccess || !mark(1) || !mark(2) || !mark(3) || !mark(4))
      return MOE_ERR_CUDA;
  } else {
    if (moe::launch_norm_router(x, g_norm, w_router, router_bias, s.T, s.H, s.E, s.eps,
                                at<uint16_t>(workspace, L.h), at<float>(workspace, L.logits), err, num_sms,
                                cs) != cudaSuccess ||
        !mark(1))
      return MOE_ERR_CUDA;
    // small T and E: top-k and align in one single-CTA kernel (events[2] then
    // follows events[1] at once); otherwise three multi-CTA kernels: top-k with
    // per-block counts (ends at events[2]), scan and scatter (end at events[3])
    cudaError_t ce;
    if (moe::align_fuses_topk(s.T, s.E)) {
      if (!mark(2)) return MOE_ERR_CUDA;
      ce = moe::launch_align(at<float>(workspace, L.logits), s.T, s.top_k, s.renormalize,
                             at<int32_t>(workspace, L.ids), at<float>(workspace, L.w), N, s.E, moe::kPadRows, bn1,
                             utiles1, bn2, utiles2, at<int32_t>(workspace, L.counts),
                             at<int32_t>(workspace, L.offsets), at<int32_t>(workspace, L.sorted),
                             at<int32_t>(workspace, L.slot), at<int32_t>(workspace, L.unit1),
                             at<int32_t>(workspace, L.unit2), err, at<int32_t>(workspace, L.flags),
                             static_cast<int>(L.n_flags),
                             cs);
    } else {
      ce = moe::launch_align_multi(at<float>(workspace, L.logits), s.T, s.top_k, s.renormalize,
                                   at<int32_t>(workspace, L.ids), at<float>(workspace, L.w), s.E, moe::kPadRows, bn1,
                                   utiles1, bn2, utiles2, at<int32_t>(workspace, L.counts),
                                   at<int32_t>(workspace, L.offsets), at<int32_t>(workspace, L.sorted),
                                   at<int32_t>(workspace, L.slot), at<int32_t>(workspace, L.unit1),
                                   at<int32_t>(workspace, L.unit2), at<int32_t>(workspace, L.blk_counts),
                                   at<int32_t>(workspace, L.blk_base), err, at<int32_t>(workspace, L.flags),
                                   static_cast<int>(L.n_flags), cs, events ? events[2] : nullptr);
    }
    if (ce != cudaSuccess || !mark(3)) return MOE_ERR_CUDA;
    if (!tokens_from_h && !rows_from_h &&
        moe::launch_gather(at<uint16_t>(workspace, L.h), at<int32_t>(workspace, L.sorted),
                           at<int32_t>(workspace, L.offsets), s.E, N, s.top_k, s.H, L.P_max,
                           at<uint16_t>(workspace, L.xg), at<int32_t>(workspace, L.ccnt),
                           fused_combine ? L.n_ccnt : 0, cs) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (!mark(4)) return MOE_ERR_CUDA;
  }

  moe::ExpertGemmArgs a1{};
  a1.offsets = at<int32_t>(workspace, L.offsets);
  a1.unit_off = at<int32_t>(workspace, L.unit1);
  a1.E = s.E;
  a1.K = s.H;
  a1.tiles_per_expert = utiles1;
  a1.w_rows_per_expert = 2 * s.I;
  a1.n_out = s.I;
  a1.out = at<uint16_t>(workspace, L.act);
  a1.err = err;
  a1.partials = at<float>(workspace, L.partials);
  a1.flags = at<int32_t>(workspace, L.flags);
  a1.stream_k = plan == GemmPlan::kSmall;
  a1.pair = moe::gemm_uses_pairs(plan, tiles1);
  a1.tables_from_parent = front || tokens_from_h || rows_from_h;  // the align is then the GEMM's parent
  a1.tokens_from_h = tokens_from_h;
  if (rows_from_h) {
    a1.h_rows = at<uint16_t>(workspace, L.h);
    a1.sorted_ids = at<int32_t>(workspace, L.sorted);
    a1.top_k = s.top_k;
    a1.n_routed = N;
  }
  a1.ready = at<int32_t>(workspace, L.flags) + kGemmFlagInts;

  moe::ExpertGemmArgs a2{};
  a2.offsets = at<int32_t>(workspace, L.offsets);
  a2.unit_off = at<int32_t>(workspace, L.unit2);
  a2.E = s.E;
  a2.K = s.I;
  a2.tiles_per_expert = utiles2;
  a2.w_rows_per_expert = s.H;
  a2.n_out = s.H;
  a2.out = at<uint16_t>(workspace, L.out);
  a2.err = err;
  a2.partials = at<float>(workspace, L.partials + partial_slots_bytes(s));  // own slots and flags: the
  a2.flags = at<int32_t>(workspace, L.flags) + moe::kMaxGemmCtas * 4;        // two GEMMs may overlap
  a2.stream_k = plan == GemmPlan::kSmall;
  a2.pair = moe::gemm_uses_pairs(plan, tiles2);
  if (fused_combine) set_fused_combine(a2, s, L, workspace, y);


  if (fused_mlp) {
    // both GEMMs in one launch (events[6] then follows events[5] at once)
    if (moe::launch_gemm_fused_mlp(tm_w13, tm_xg, tm_w2, tm_act, a1, a2, num_sms, cs) != cudaSuccess || !mark(5) ||
        !mark(6))
      return MOE_ERR_CUDA;
  } else {
    if (moe::launch_gemm_gate_up(tm_w13, tm_xg, a1, plan, num_sms, cs) != cudaSuccess || !mark(5))
      return MOE_ERR_CUDA;
    if (moe::launch_gemm_down(tm_w2, tm_act, a2, plan, num_sms, cs) != cudaSuccess || !mark(6))
      return MOE_ERR_CUDA;
  }

  if (!fused_combine &&
      moe::launch_combine(at<uint16_t>(workspace, L.out), at<int32_t>(workspace, L.slot), at<float>(workspace, L.w),
                          s.T, s.H, s.top_k, y, cs) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (!mark(7)) return MOE_ERR_CUDA;
  return MOE_OK;
}

// The block-scaled layers: the bf16 layer's routing, then quantized token
// rows and weights in block-scaled tcgen05 GEMMs.  kind: MXFP8 weights and
// tokens (kW8A8), MXFP4 weights with MXFP8 tokens (kW4A8), or MXFP4 weights
// and tokens (kW4A4: packed codes, 256 elements of K per GEMM stage; H or I
// an odd multiple of 128 ends half way into a GEMM's last stage).
moe_status forward_mx_impl(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm, const float* w_router,
                           const float* router_bias, const uint8_t* w13c, const uint8_t* w13s, const uint8_t* w2c,
                           const uint8_t* w2s, moe_bf16* y, void* workspace, size_t workspace_bytes,
                           moe_stream_t stream, void* const* events, MxKind kind = MxKind::kW8A8,
                           const float* w13g = nullptr, const float* w2g = nullptr) {
  moe_status st = check_shape_mx(shape);
  if (st != MOE_OK) return st;
  const moe_shape& s = *shape;
  if (s.T == 0) return MOE_OK;
  const GemmPlan plan = moe::choose_plan(s.T, s.top_k, s.E);
  if (s.E > 256) return MOE_ERR_UNSUPPORTED;
  const bool fp4 = kind != MxKind::kW8A8, nv = kind == MxKind::kNV4;
  const bool a4 = kind == MxKind::kW4A4 || nv;  // packed E2M1 token codes too
  if (nv && (!w13g || !w2g || !aligned(w13g, 4) || !aligned(w2g, 4))) return MOE_ERR_INVALID_ARG;
  st = check_inputs(shape, x, g_norm, w_router, router_bias, workspace, workspace_bytes, true);
  if (st != MOE_OK) return st;
  const size_t code_align = fp4 ? 32 : 16;  // the 4-bit tensor maps want 32-byte bases (one rule for both layers)
  if (!w13c || !w13s || !w2c || !w2s || !y || !aligned(w13c, code_align) || !aligned(w13s, 16) ||
      !aligned(w2c, code_align) || !aligned(w2s, 16) || !aligned(y, 16))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const int num_sms = num_sms_of_current_device();
  if (num_sms <= 0) return MOE_ERR_CUDA;
  const Layout L = make_layout(s, true);
  const int tiles1 = s.I / moe::kGateUpTileFeat, tiles2 = s.H / moe::kDownTileFeat;
  // dense prefill: CTA pairs where the weight tiles come in pairs (256-token units)
  // (NVFP4: one CTA per unit in every plan; its scale tiles take the TMEM a pair's accumulator needs)
  const bool pair1 = !nv && moe::gemm_uses_pairs_mx(plan, tiles1, s.T, s.top_k, s.E);
  const bool pair2 = !nv && moe::gemm_uses_pairs_mx(plan, tiles2, s.T, s.top_k, s.E);
  const int bn1 = moe::gemm_bn_mx(plan, pair1), bn2 = moe::gemm_bn_mx(plan, pair2);
  const int utiles1 = pair1 ? tiles1 / 2 : tiles1, utiles2 = pair2 ? tiles2 / 2 : tiles2;
  auto mark = [&](int i) {
    return !events || cudaEventRecord(static_cast<cudaEvent_t>(events[i]), cs) == cudaSuccess;
  };
  const uint64_t n_tok_tiles1 = static_cast<uint64_t>(L.P_max / 32) * 2 * (s.H / 128);
  const uint64_t n_tok_tiles2 = static_cast<uint64_t>(L.P_max / 32) * 2 * (s.I / 128);
  CUtensorMap tm_w13, tm_xq, tm_w2, tm_aq, tm_s13, tm_sxq, tm_s2, tm_saq;
  // kW4A8: 4-bit weight maps (the TMA spreads the codes to the E4M3 image);
  // kW4A4: byte maps over the packed codes (H / 2 and I / 2 bytes per row)
  const uint64_t kx1 = a4 ? s.H / 2 : s.H, kx2 = a4 ? s.I / 2 : s.I;
  const bool maps_w = kind == MxKind::kW4A8
                          ? make_map_gate_up_u4(&tm_w13, w13c, s.H, s.I, s.E) &&
                                make_map_u4(&tm_w2, w2c, s.I, static_cast<uint64_t>(s.E) * s.H, moe::kWeightBoxRows)
                          : make_map_gate_up_u8(&tm_w13, w13c, kx1, s.I, s.E) &&
                                make_map_u8(&tm_w2, w2c, kx2, static_cast<uint64_t>(s.E) * s.H, moe::kWeightBoxRows);
  if (!maps_w ||
      !make_map_u8(&tm_xq, at<void>(workspace, L.xg), kx1, L.P_max, moe::gemm_tok_box_rows_mx(plan, pair1)) ||
      !make_map_u8(&tm_aq, at<void>(workspace, L.aq), kx2, L.P_max, moe::gemm_tok_box_rows_mx(plan, pair2)) ||
      !make_map_scales(&tm_s13, w13s, static_cast<uint64_t>(s.E) * (2 * s.I / 128) * (s.H / 128)) ||
      !make_map_scales(&tm_sxq, at<void>(workspace, L.xs), n_tok_tiles1) ||
      !make_map_scales(&tm_s2, w2s, static_cast<uint64_t>(s.E) * (s.H / 128) * (s.I / 128)) ||
      !make_map_scales(&tm_saq, at<void>(workspace, L.as), n_tok_tiles2))
    return MOE_ERR_CUDA;
  int32_t* err = at<int32_t>(workspace, L.err);
  if (!mark(0)) return MOE_ERR_CUDA;
  st = run_front(s, L, x, g_norm, w_router, router_bias, moe::kPadRowsMx, bn1, utiles1, bn2, utiles2, workspace, cs,
                 num_sms);
  if (st != MOE_OK) return st;
  if (!mark(1) || !mark(2) || !mark(3)) return MOE_ERR_CUDA;
  const int N = s.T * s.top_k;
  cudaError_t ge;
  if (nv) {
    ge = moe::launch_nv4_gather(at<uint16_t>(workspace, L.h), at<int32_t>(workspace, L.sorted),
                                at<int32_t>(workspace, L.offsets), at<int32_t>(workspace, L.unit1), utiles1, bn1, s.E,
                                N, s.top_k, s.H, L.P_max, at<uint8_t>(workspace, L.xg), at<uint8_t>(workspace, L.xs),
                                at<float>(workspace, L.gx), cs);
  } else {
    auto gather = a4 ? moe::launch_mx4_gather : moe::launch_mx_gather;
    ge = gather(at<uint16_t>(workspace, L.h), at<int32_t>(workspace, L.sorted), at<int32_t>(workspace, L.offsets),
                at<int32_t>(workspace, L.unit1), utiles1, bn1, s.E, N, s.top_k, s.H, L.P_max,
                at<uint8_t>(workspace, L.xg), at<uint8_t>(workspace, L.xs), cs);
  }
  if (ge != cudaSuccess || !mark(4)) return MOE_ERR_CUDA;

  moe::ExpertGemmArgs a1{};
  a1.offsets = at<int32_t>(workspace, L.offsets);
  a1.unit_off = at<int32_t>(workspace, L.unit1);
  a1.E = s.E;
  a1.K = s.H;
  a1.tiles_per_expert = utiles1;
  a1.w_rows_per_expert = 2 * s.I;
  a1.n_out = s.I;
  a1.out = at<uint16_t>(workspace, L.act);
  a1.err = err;
  a1.partials = at<float>(workspace, L.partials);
  a1.flags = at<int32_t>(workspace, L.flags);
  a1.stream_k = plan == GemmPlan::kSmall;
  a1.pair = pair1;
  a1.w_scales = w13s;
  a1.x_scales = at<uint8_t>(workspace, L.xs);
  a1.w_gscale = w13g;
  a1.x_gscale = nv ? at<float>(workspace, L.gx) : nullptr;
  if (moe::launch_gemm_gate_up_mx(tm_w13, tm_xq, tm_s13, tm_sxq, a1, plan, num_sms, cs, kind) != cudaSuccess ||
      !mark(5))
    return MOE_ERR_CUDA;
  // the activations (bf16) -> MXFP8, rows below offsets[E], their scales in
  // the down GEMM's token chunks
  if (nv) {
    ge = moe::launch_nv4_quantize_act(at<uint16_t>(workspace, L.act), L.P_max, s.I, at<int32_t>(workspace, L.offsets),
                                      at<int32_t>(workspace, L.unit2), utiles2, bn2, s.E, at<uint8_t>(workspace, L.aq),
                                      at<uint8_t>(workspace, L.as), at<float>(workspace, L.ga), cs);
  } else {
    auto quantize_act = a4 ? moe::launch_mx4_quantize_act : moe::launch_mx_quantize_act;
    ge = quantize_act(at<uint16_t>(workspace, L.act), L.P_max, s.I, at<int32_t>(workspace, L.offsets),
                      at<int32_t>(workspace, L.unit2), utiles2, bn2, s.E, at<uint8_t>(workspace, L.aq),
                      at<uint8_t>(workspace, L.as), cs);
  }
  if (ge != cudaSuccess) return MOE_ERR_CUDA;
  moe::ExpertGemmArgs a2{};
  a2.offsets = at<int32_t>(workspace, L.offsets);
  a2.unit_off = at<int32_t>(workspace, L.unit2);
  a2.E = s.E;
  a2.K = s.I;
  a2.tiles_per_expert = utiles2;
  a2.w_rows_per_expert = s.H;
  a2.n_out = s.H;
  a2.out = at<uint16_t>(workspace, L.out);
  a2.err = err;
  a2.partials = at<float>(workspace, L.partials + partial_slots_bytes(s));
  a2.flags = at<int32_t>(workspace, L.flags) + moe::kMaxGemmCtas * 4;
  a2.stream_k = plan == GemmPlan::kSmall;
  a2.pair = pair2;
  a2.w_scales = w2s;
  a2.x_scales = at<uint8_t>(workspace, L.as);
  a2.w_gscale = w2g;
  a2.x_gscale = nv ? at<float>(workspace, L.ga) : nullptr;
  if (moe::launch_gemm_down_mx(tm_w2, tm_aq, tm_s2, tm_saq, a2, plan, num_sms, cs, kind) != cudaSuccess || !mark(6))
    return MOE_ERR_CUDA;
  if (moe::launch_combine(at<uint16_t>(workspace, L.out), at<int32_t>(workspace, L.slot), at<float>(workspace, L.w),
                          s.T, s.H, s.top_k, y, cs) != cudaSuccess ||
      !mark(7))
    return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace moe

extern "C" {

moe_status moe_mx_weight_sizes(const moe_shape* shape, size_t* w13_codes, size_t* w13_scales, size_t* w2_codes,
                               size_t* w2_scales) {
  const moe_status st = check_shape_mx(shape);
  if (st != MOE_OK) return st;
  if (!w13_codes || !w13_scales || !w2_codes || !w2_scales) return MOE_ERR_INVALID_ARG;
  const int64_t E = shape->E, H = shape->H, I = shape->I;
  *w13_codes = static_cast<size_t>(E * 2 * I * H);
  *w13_scales = moe::mx_scale_bytes(E * 2 * I, H);
  *w2_codes = static_cast<size_t>(E * H * I);
  *w2_scales = moe::mx_scale_bytes(E * H, I);
  return MOE_OK;
}

moe_status moe_mx_quantize_weights(const moe_shape* shape, const moe_bf16* w13, const moe_bf16* w2, uint8_t* w13_codes,
                                   uint8_t* w13_scales, uint8_t* w2_codes, uint8_t* w2_scales, moe_stream_t stream) {
  const moe_status st = check_shape_mx(shape);
  if (st != MOE_OK) return st;
  if (!w13 || !w2 || !w13_codes || !w13_scales || !w2_codes || !w2_scales || !aligned(w13, 16) || !aligned(w2, 16) ||
      !aligned(w13_codes, 16) || !aligned(w13_scales, 16) || !aligned(w2_codes, 16) || !aligned(w2_scales, 16))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const moe_shape& s = *shape;
  if (moe::launch_mx_quantize_w13(w13, s.E, s.H, s.I, w13_codes, w13_scales, cs) != cudaSuccess ||
      moe::launch_mx_quantize_rows(w2, static_cast<int64_t>(s.E) * s.H, s.I, w2_codes, w2_scales, cs) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_mxfp4_weight_sizes(const moe_shape* shape, size_t* w13_codes, size_t* w13_scales, size_t* w2_codes,
                                  size_t* w2_scales) {
  const moe_status st = moe_mx_weight_sizes(shape, w13_codes, w13_scales, w2_codes, w2_scales);
  if (st != MOE_OK) return st;
  *w13_codes /= 2;  // two E2M1 codes per byte
  *w2_codes /= 2;
  return MOE_OK;
}

moe_status moe_mxfp4_quantize_weights(const moe_shape* shape, const moe_bf16* w13, const moe_bf16* w2,
                                      uint8_t* w13_codes, uint8_t* w13_scales, uint8_t* w2_codes, uint8_t* w2_scales,
                                      moe_stream_t stream) {
  const moe_status st = check_shape_mx(shape);
  if (st != MOE_OK) return st;
  if (!w13 || !w2 || !w13_codes || !w13_scales || !w2_codes || !w2_scales || !aligned(w13, 16) || !aligned(w2, 16) ||
      !aligned(w13_codes, 32) || !aligned(w13_scales, 16) || !aligned(w2_codes, 32) || !aligned(w2_scales, 16))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const moe_shape& s = *shape;
  if (moe::launch_mx4_quantize_w13(w13, s.E, s.H, s.I, w13_codes, w13_scales, cs) != cudaSuccess ||
      moe::launch_mx4_quantize_rows(w2, static_cast<int64_t>(s.E) * s.H, s.I, w2_codes, w2_scales, cs) !=
          cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_nvfp4_weight_sizes(const moe_shape* shape, size_t* w13_codes, size_t* w13_scales, size_t* w2_codes,
                                  size_t* w2_scales) {
  const moe_status st = check_shape_mx(shape);
  if (st != MOE_OK) return st;
  if (!w13_codes || !w13_scales || !w2_codes || !w2_scales) return MOE_ERR_INVALID_ARG;
  const int64_t E = shape->E, H = shape->H, I = shape->I;
  *w13_codes = static_cast<size_t>(E * 2 * I * H / 2);
  *w13_scales = moe::nv4_scale_bytes(E * 2 * I, H);
  *w2_codes = static_cast<size_t>(E * H * I / 2);
  *w2_scales = moe::nv4_scale_bytes(E * H, I);
  return MOE_OK;
}

moe_status moe_nvfp4_quantize_weights(const moe_shape* shape, const moe_bf16* w13, const moe_bf16* w2,
                                      uint8_t* w13_codes, uint8_t* w13_scales, float* w13_gscale, uint8_t* w2_codes,
                                      uint8_t* w2_scales, float* w2_gscale, moe_stream_t stream) {
  const moe_status st = check_shape_mx(shape);
  if (st != MOE_OK) return st;
  if (!w13 || !w2 || !w13_codes || !w13_scales || !w13_gscale || !w2_codes || !w2_scales || !w2_gscale ||
      !aligned(w13, 16) || !aligned(w2, 16) || !aligned(w13_codes, 32) || !aligned(w13_scales, 16) ||
      !aligned(w2_codes, 32) || !aligned(w2_scales, 16) || !aligned(w13_gscale, 4) || !aligned(w2_gscale, 4))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const moe_shape& s = *shape;
  const int64_t r13 = static_cast<int64_t>(s.E) * 2 * s.I, r2 = static_cast<int64_t>(s.E) * s.H;
  // the tensor-scale arrays hold each expert matrix's absolute maximum until
  // the codes are written, then its tensor scale
  if (moe::launch_nv4_weight_amax(w13, r13, s.H, 2 * s.I, w13_gscale, s.E, cs) != cudaSuccess ||
      moe::launch_nv4_weight_amax(w2, r2, s.I, s.H, w2_gscale, s.E, cs) != cudaSuccess ||
      moe::launch_nv4_quantize_w13(w13, s.E, s.H, s.I, w13_gscale, w13_codes, w13_scales, cs) != cudaSuccess ||
      moe::launch_nv4_quantize_rows(w2, r2, s.I, s.H, w2_gscale, w2_codes, w2_scales, cs) != cudaSuccess ||
      moe::launch_nv4_global(w13_gscale, s.E, cs) != cudaSuccess ||
      moe::launch_nv4_global(w2_gscale, s.E, cs) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_workspace_size_mx(const moe_shape* shape, size_t* bytes) {
  const moe_status st = check_shape_mx(shape);
  if (st != MOE_OK) return st;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = make_layout(*shape, true).total;
  return MOE_OK;
}

moe_status moe_workspace_views_mx(const moe_shape* shape, void* workspace, size_t workspace_bytes, moe_views* v,
                                  moe_mx_views* mv) {
  const moe_status st = check_shape_mx(shape);
  if (st != MOE_OK) return st;
  if (!workspace || !v || !mv) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(*shape, true);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
  v->error_word = at<void>(workspace, L.err);
  v->h = at<void>(workspace, L.h);
  v->logits = at<void>(workspace, L.logits);
  v->topk_ids = at<void>(workspace, L.ids);
  v->topk_w = at<void>(workspace, L.w);
  v->counts = at<void>(workspace, L.counts);
  v->offsets = at<void>(workspace, L.offsets);
  v->sorted_ids = at<void>(workspace, L.sorted);
  v->slot_of = at<void>(workspace, L.slot);
  v->xg = at<void>(workspace, L.xg);
  v->act = at<void>(workspace, L.act);
  v->out_rows = at<void>(workspace, L.out);
  v->P_max = L.P_max;
  mv->x_codes = at<void>(workspace, L.xg);
  mv->x_scales = at<void>(workspace, L.xs);
  mv->act_codes = at<void>(workspace, L.aq);
  mv->act_scales = at<void>(workspace, L.as);
  const moe_shape& s = *shape;
  const GemmPlan plan = moe::choose_plan(s.T, s.top_k, s.E);
  const int tiles1 = s.I / moe::kGateUpTileFeat, tiles2 = s.H / moe::kDownTileFeat;
  mv->x_chunk_rows = moe::gemm_bn_mx(plan, moe::gemm_uses_pairs_mx(plan, tiles1, s.T, s.top_k, s.E));
  mv->act_chunk_rows = moe::gemm_bn_mx(plan, moe::gemm_uses_pairs_mx(plan, tiles2, s.T, s.top_k, s.E));
  mv->x_gscale = at<void>(workspace, L.gx);
  mv->act_gscale = at<void>(workspace, L.ga);
  mv->nv_chunk_rows = moe::gemm_bn_mx(plan, false);
  return MOE_OK;
}

moe_status moe_forward_mx(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm, const float* w_router,
                          const float* router_bias, const uint8_t* w13_codes, const uint8_t* w13_scales,
                          const uint8_t* w2_codes, const uint8_t* w2_scales, moe_bf16* y, void* workspace,
                          size_t workspace_bytes, moe_stream_t stream, void* const* events, int32_t n_events) {
  if (events) {
    if (n_events < MOE_NUM_KERNELS + 1) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i <= MOE_NUM_KERNELS; ++i)
      if (!events[i]) return MOE_ERR_INVALID_ARG;
  }
  return moe::forward_mx_impl(shape, x, g_norm, w_router, router_bias, w13_codes, w13_scales, w2_codes, w2_scales, y,
                              workspace, workspace_bytes, stream, events);
}

moe_status moe_forward_mxfp4(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm,
                             const float* w_router, const float* router_bias, const uint8_t* w13_codes,
                             const uint8_t* w13_scales, const uint8_t* w2_codes, const uint8_t* w2_scales,
                             moe_bf16* y, void* workspace, size_t workspace_bytes, moe_stream_t stream,
                             void* const* events, int32_t n_events) {
  if (events) {
    if (n_events < MOE_NUM_KERNELS + 1) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i <= MOE_NUM_KERNELS; ++i)
      if (!events[i]) return MOE_ERR_INVALID_ARG;
  }
  return moe::forward_mx_impl(shape, x, g_norm, w_router, router_bias, w13_codes, w13_scales, w2_codes, w2_scales, y,
                              workspace, workspace_bytes, stream, events, moe::MxKind::kW4A8);
}

moe_status moe_forward_mxfp4a4(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm,
                               const float* w_router, const float* router_bias, const uint8_t* w13_codes,
                               const uint8_t* w13_scales, const uint8_t* w2_codes, const uint8_t* w2_scales,
                               moe_bf16* y, void* workspace, size_t workspace_bytes, moe_stream_t stream,
                               void* const* events, int32_t n_events) {
  if (events) {
    if (n_events < MOE_NUM_KERNELS + 1) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i <= MOE_NUM_KERNELS; ++i)
      if (!events[i]) return MOE_ERR_INVALID_ARG;
  }
  return moe::forward_mx_impl(shape, x, g_norm, w_router, router_bias, w13_codes, w13_scales, w2_codes, w2_scales, y,
                              workspace, workspace_bytes, stream, events, moe::MxKind::kW4A4);
}

moe_status moe_forward_nvfp4(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm,
                             const float* w_router, const float* router_bias, const uint8_t* w13_codes,
                             const uint8_t* w13_scales, const float* w13_gscale, const uint8_t* w2_codes,
                             const uint8_t* w2_scales, const float* w2_gscale, moe_bf16* y, void* workspace,
                             size_t workspace_bytes, moe_stream_t stream, void* const* events, int32_t n_events) {
  if (events) {
    if (n_events < MOE_NUM_KERNELS + 1) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i <= MOE_NUM_KERNELS; ++i)
      if (!events[i]) return MOE_ERR_INVALID_ARG;
  }
  return moe::forward_mx_impl(shape, x, g_norm, w_router, router_bias, w13_codes, w13_scales, w2_codes, w2_scales, y,
                              workspace, workspace_bytes, stream, events, moe::MxKind::kNV4, w13_gscale, w2_gscale);
}

moe_status moe_forward(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm, const float* w_router,
                       const float* router_bias, const moe_bf16* w13, const moe_bf16* w2, moe_bf16* y,
                       void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  return moe::forward_impl(shape, x, g_norm, w_router, router_bias, w13, w2, y, workspace, workspace_bytes, stream,
                           nullptr);
}

moe_status moe_forward_events(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm,
                              const float* w_router, const float* router_bias, const moe_bf16* w13, const moe_bf16* w2,
                              moe_bf16* y, void* workspace, size_t workspace_bytes, moe_stream_t stream,
                              void* const* events, int32_t n_events) {
  if (!events || n_events < MOE_NUM_KERNELS + 1) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i <= MOE_NUM_KERNELS; ++i)
    if (!events[i]) return MOE_ERR_INVALID_ARG;
  return moe::forward_impl(shape, x, g_norm, w_router, router_bias, w13, w2, y, workspace, workspace_bytes, stream,
                           events);
}

moe_status moe_forward_fused_front(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm,
                                   const float* w_router, const float* router_bias, const moe_bf16* w13,
                                   const moe_bf16* w2, moe_bf16* y, void* workspace, size_t workspace_bytes,
                                   moe_stream_t stream, void* const* events, int32_t n_events) {
  if (events) {
    if (n_events < MOE_NUM_KERNELS + 1) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i <= MOE_NUM_KERNELS; ++i)
      if (!events[i]) return MOE_ERR_INVALID_ARG;
  }
  return moe::forward_impl(shape, x, g_norm, w_router, router_bias, w13, w2, y, workspace, workspace_bytes, stream,
                           events, true);
}

moe_status moe_forward_fused_mlp(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm,
                                 const float* w_router, const float* router_bias, const moe_bf16* w13,
                                 const moe_bf16* w2, moe_bf16* y, void* workspace, size_t workspace_bytes,
                                 moe_stream_t stream, void* const* events, int32_t n_events) {
  if (events) {
    if (n_events < MOE_NUM_KERNELS + 1) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i <= MOE_NUM_KERNELS; ++i)
      if (!events[i]) return MOE_ERR_INVALID_ARG;
  }
  return moe::forward_impl(shape, x, g_norm, w_router, router_bias, w13, w2, y, workspace, workspace_bytes, stream,
                           events, false, false, true);
}

moe_status moe_forward_fused_combine(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm,
                                     const float* w_router, const float* router_bias, const moe_bf16* w13,
                                     const moe_bf16* w2, moe_bf16* y, void* workspace, size_t workspace_bytes,
                                     moe_stream_t stream, void* const* events, int32_t n_events) {
  if (events) {
    if (n_events < MOE_NUM_KERNELS + 1) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i <= MOE_NUM_KERNELS; ++i)
      if (!events[i]) return MOE_ERR_INVALID_ARG;
  }
  return moe::forward_impl(shape, x, g_norm, w_router, router_bias, w13, w2, y, workspace, workspace_bytes, stream,
                           events, false, true);
}

moe_status moe_route_debug(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm, const float* w_router,
                           const float* router_bias, int32_t pad_rows, int32_t* topk_ids, float* topk_w,
                           int32_t* expert_offsets, int32_t* sorted_ids, int64_t sorted_capacity, void* workspace,
                           size_t workspace_bytes, moe_stream_t stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  st = check_inputs(shape, x, g_norm, w_router, router_bias, workspace, workspace_bytes);
  if (st != MOE_OK) return st;
  if (pad_rows < 1 || pad_rows > kMaxDebugPad) return MOE_ERR_INVALID_ARG;
  if (!topk_ids || !topk_w || !expert_offsets || !sorted_ids) return MOE_ERR_INVALID_ARG;
  const moe_shape& s = *shape;
  const int64_t need = static_cast<int64_t>(s.T) * s.top_k + static_cast<int64_t>(s.E) * (pad_rows - 1);
  if (sorted_capacity < need) return MOE_ERR_INVALID_ARG;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const Layout L = make_layout(s);
  if (s.T == 0) {
    // an empty routing: every list is empty
    if (cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (s.E + 1), cs) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  const int num_sms = num_sms_of_current_device();
  if (num_sms <= 0) return MOE_ERR_CUDA;
  st = run_front(s, L, x, g_norm, w_router, router_bias, pad_rows, 0, 1, 0, 1, workspace, cs, num_sms);
  if (st != MOE_OK) return st;
  const size_t tk = static_cast<size_t>(s.T) * s.top_k;
  if (cudaMemcpyAsync(topk_ids, at<void>(workspace, L.ids), tk * 4, cudaMemcpyDeviceToDevice, cs) != cudaSuccess ||
      cudaMemcpyAsync(topk_w, at<void>(workspace, L.w), tk * 4, cudaMemcpyDeviceToDevice, cs) != cudaSuccess ||
      cudaMemcpyAsync(expert_offsets, at<void>(workspace, L.offsets), (s.E + 1) * 4, cudaMemcpyDeviceToDevice, cs) !=
          cudaSuccess ||
      cudaMemcpyAsync(sorted_ids, at<void>(workspace, L.sorted), static_cast<size_t>(need) * 4,
                      cudaMemcpyDeviceToDevice, cs) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_device_status(const void* workspace, size_t workspace_bytes, moe_stream_t stream, int32_t* detail) {
  if (!workspace || workspace_bytes < 64) return MOE_ERR_INVALID_ARG;
  int32_t w[4] = {0, 0, 0, 0};
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(w, workspace, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (detail) std::memcpy(detail, w, sizeof(w));
  if (w[0] == moe::kErrTimeout) return MOE_ERR_TIMEOUT;
  if (w[0] == moe::kErrDevice) return MOE_ERR_DEVICE;
  return MOE_OK;
}

moe_status moe_qk_norm(int64_t T, int32_t Hq, int32_t Hk, int32_t D, moe_bf16* q, moe_bf16* k,
                       const moe_bf16* q_weight, const moe_bf16* k_weight, float weight_bias, float eps,
                       moe_stream_t stream) {
  if (T < 0 || Hq < 0 || Hk < 0 || (D != 64 && D != 128 && D != 256)) return MOE_ERR_INVALID_ARG;
  if (!(eps >= 0.0f) || !std::isfinite(eps) || !std::isfinite(weight_bias)) return MOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(Hq) + Hk > (1 << 20) || T * (static_cast<int64_t>(Hq) + Hk) >= (int64_t(1) << 31))
    return MOE_ERR_UNSUPPORTED;
  if (T == 0 || Hq + Hk == 0) return MOE_OK;
  if (Hq > 0 && (!q || !q_weight || !aligned(q, 16) || !aligned(q_weight, 16))) return MOE_ERR_INVALID_ARG;
  if (Hk > 0 && (!k || !k_weight || !aligned(k, 16) || !aligned(k_weight, 16))) return MOE_ERR_INVALID_ARG;
  if (moe::launch_qk_norm(q, k, q_weight, k_weight, T, Hq, Hk, D, weight_bias, eps,
                          reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_selftest_wait_timeout(void* workspace, size_t workspace_bytes, int64_t timeout_ns,
                                     moe_stream_t stream) {
  if (!workspace || workspace_bytes < 64 || !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
  if (timeout_ns <= 0 || timeout_ns > 1000000000) return MOE_ERR_INVALID_ARG;
  if (moe::launch_selftest_wait(static_cast<int32_t*>(workspace), static_cast<uint64_t>(timeout_ns),
                                reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

const char* moe_status_string(moe_status status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (null pointer, misaligned pointer or bad shape value)";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape (H a multiple of 128, I of 64 (128 for block-scaled layers), both up to 16384; E <= 1024; top_k <= 32)";
    case MOE_ERR_WORKSPACE: return "workspace smaller than moe_workspace_size()";
    case MOE_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case MOE_ERR_TIMEOUT: return "a bounded device-side wait ran out";
    case MOE_ERR_DEVICE: return "the device found invalid data (expert index out of range)";
  }
  return "unknown status";
}

}  // extern "C"
