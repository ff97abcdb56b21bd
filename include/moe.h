/*
 * moe.h -- C ABI of the fused MoE layer forward on one GB300 (sm_103a).
 *
 * One call runs the whole layer on the GPU:
 *   RMSNorm -> router GEMV + top-k softmax -> expert align (histogram,
 *   prefix sum, padded permutation) -> gather -> gate/up grouped GEMM with a
 *   SwiGLU epilogue -> down grouped GEMM -> top-k weighted combine.
 *
 * Definitions the calls implement:
 *   RMSNorm      h_j = bf16( x_j / sqrt(mean_i x_i^2 + eps) * g_j ), fp32
 *                accumulation -- "4 · La fusion de noyaux", §4.2
 *                "Réduction + élémentaire"; eps inside the square root and
 *                the cast back to the input type as in "CuTeDSL chez
 *                Perplexity", section "Norme QK".
 *   Router       fp32 logits l_e = sum_j h_j Wr[e,j] (+ b_e); the top_k
 *                largest (ties to the lower expert index), weights =
 *                softmax over all E taken at the selected experts, divided
 *                by their sum when renormalize != 0.
 *   Dispatch     per-expert counts, a unique slot per routed token in its
 *                expert's list, lists copied into padded per-expert buffers
 *                -- "CuTeDSL chez Perplexity", MoE dispatch/combine, "Local".
 *   Experts      SwiGLU(x) = (SiLU(x W_gate) (.) (x W_up)) W_down with gate
 *                and up in one concatenated weight -- "4 · La fusion de
 *                noyaux", §4.2 "GEMM + GEMM"; SiLU(gate)*up is applied to
 *                the accumulators before the only store ("GEMM + épilogue").
 *   Combine      y_t = bf16( sum_j w_tj * o_tj ) -- "CuTeDSL chez
 *                Perplexity", MoE dispatch/combine, "Local".
 *
 * Conventions for every call:
 *   - bf16 tensors are passed as raw bfloat16 bits (moe_bf16).
 *   - All tensor pointers are DEVICE pointers of the current CUDA device,
 *     row-major and contiguous, 16-byte aligned; the workspace is 256-byte
 *     aligned.  The caller owns every buffer; the library allocates no
 *     device memory on any call.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default
 *     stream).  Outputs are valid once the stream has reached the end of
 *     the call.  Inputs are never modified.
 *   - A call can be captured into a CUDA graph (stream capture on `stream`)
 *     and replayed: it makes no host synchronisation and no allocation, and
 *     it reads the pointed-to data when the kernels run.  The shape, the
 *     pointers and the tensor maps built from them are fixed at capture;
 *     new inputs go into the same buffers between replays.  Make one call
 *     outside capture first on each device (it sets per-device kernel
 *     attributes, which are not stream work).  A replay gives the same bits
 *     as the direct call.
 *   - Argument and shape errors are reported synchronously, before anything
 *     is enqueued.  A failed launch returns MOE_ERR_CUDA.  Errors found on
 *     the device (a routing index out of range, a bounded wait that ran out)
 *     are written to an error word at the start of the workspace and are
 *     returned by moe_device_status().
 *   - The library keeps no state between calls except per-device kernel
 *     attributes set once; it is reentrant as long as concurrent calls use
 *     different workspaces.  One exception: moe_forward_static_scratch keeps
 *     its scratch in one device array per GPU that every call of it on that
 *     GPU shares (and caches that array's address), so its callers must
 *     serialise their calls although they pass no workspace.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* raw bfloat16 bits */
typedef uint16_t moe_bf16;
/* a cudaStream_t */
typedef struct CUstream_st* moe_stream_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null pointer, bad alignment, bad shape value */
  MOE_ERR_UNSUPPORTED = 2, /* a shape outside the supported set (see moe_shape) */
  MOE_ERR_WORKSPACE = 3,   /* workspace smaller than moe_workspace_size() */
  MOE_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
  MOE_ERR_TIMEOUT = 5,     /* a device-side bounded wait ran out (reported by moe_device_status) */
  MOE_ERR_DEVICE = 6       /* the device found bad data, e.g. an expert index >= E */
} moe_status;

/* Layer shape and routing options.
 *   T            tokens (>= 0; moe_forward with T = 0 returns MOE_OK at once and
 *                touches no pointer)
 *   H            hidden size, a multiple of 128 (the down GEMM's weight tile
 *                is 128 output features), <= 16384 (the router keeps its
 *                tokens' rows of h in shared memory)
 *   I            expert intermediate size, a multiple of 64 (the gate/up
 *                GEMM's unit is 64 features, the down GEMM's K block 64
 *                elements; 128 for the block-scaled layers, whose scale tiles
 *                cover 128 elements of K), <= 16384
 *   E            experts, 1..1024
 *   top_k        experts per token, 1..min(E, 32) (one lane of the selecting
 *                warp per selected expert)
 *   renormalize  nonzero: the top_k weights are divided by their sum
 *   eps          RMSNorm epsilon (>= 0, finite)                              */
typedef struct {
  int32_t T, H, I, E, top_k;
  int32_t renormalize;
  float eps;
} moe_shape;

/* Bytes of device workspace moe_forward() needs for this shape.  Host only:
 * makes no CUDA call.  Returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED for
 * a bad shape. */
MOE_API moe_status moe_workspace_size(const moe_shape* shape, size_t* bytes);

/* The layer forward.
 *   x          [T, H]        bf16 token activations
 *   g_norm     [H]           bf16 RMSNorm gain
 *   w_router   [E, H]        fp32 router weight
 *   router_bias[E]           fp32 logit bias, or NULL for none
 *   w13        [E, 2I, H]    bf16; rows [0, I) of expert e are W_gate
 *                            (transposed, K-major), rows [I, 2I) are W_up
 *   w2         [E, H, I]     bf16; W_down of expert e (transposed, K-major)
 *   y          [T, H]        bf16 output (must not alias the inputs)
 *   workspace  device scratch of at least moe_workspace_size() bytes; its
 *              contents on entry do not matter; it holds the intermediate
 *              tensors (see moe_workspace_views) after the call.
 * Ownership: all buffers belong to the caller.  Errors: as above. */
MOE_API moe_status moe_forward(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm,
                       const float* w_router, const float* router_bias, const moe_bf16* w13,
                       const moe_bf16* w2, moe_bf16* y, void* workspace, size_t workspace_bytes,
                       moe_stream_t stream);

/* The steps of one moe_forward call, in order:
 *   1 RMSNorm + router logits, 2 top-k + softmax, 3 expert align, 4 gather,
 *   5 gate/up grouped GEMM + SwiGLU, 6 down grouped GEMM, 7 weighted combine.
 * For T <= MOE_FUSED_TOPK_MAX_T and E <= MOE_FUSED_TOPK_MAX_E, steps 2 and 3
 * run as one single-CTA kernel; otherwise step 2 is one multi-CTA kernel
 * (top-k with per-block expert counts) and step 3 two (scan, scatter).
 * So 6 launches per call (8 with the multi-CTA top-k and align);
 * moe_kernels_per_call_of gives the count for each entry point. */
#define MOE_NUM_KERNELS 7
#define MOE_FUSED_TOPK_MAX_T 256
#define MOE_FUSED_TOPK_MAX_E 256

/* Number of kernels one moe_forward call with this shape launches on the
 * current device (0 for T = 0).  Host-only apart from querying the device. */
MOE_API moe_status moe_kernels_per_call(const moe_shape* shape, int32_t* count);

/* The same for each entry point: call = MOE_CALL_FORWARD (moe_forward,
 * moe_forward_events, moe_forward_static_scratch), MOE_CALL_FORWARD_FUSED_FRONT
 * (moe_forward_fused_front), MOE_CALL_FORWARD_MX (moe_forward_mx),
 * MOE_CALL_FORWARD_FUSED_COMBINE (moe_forward_fused_combine),
 * MOE_CALL_FORWARD_MXFP4 (moe_forward_mxfp4), MOE_CALL_FORWARD_MXFP4A4
 * (moe_forward_mxfp4a4), MOE_CALL_FORWARD_NVFP4 (moe_forward_nvfp4) or
 * MOE_CALL_FORWARD_FUSED_MLP (moe_forward_fused_mlp; MOE_ERR_UNSUPPORTED for
 * shapes it refuses).  Another value of call: MOE_ERR_INVALID_ARG.  Host-only. */
#define MOE_CALL_FORWARD 0
#define MOE_CALL_FORWARD_FUSED_FRONT 1
#define MOE_CALL_FORWARD_MX 2
#define MOE_CALL_FORWARD_FUSED_COMBINE 3
#define MOE_CALL_FORWARD_MXFP4 4
#define MOE_CALL_FORWARD_MXFP4A4 5
#define MOE_CALL_FORWARD_NVFP4 6
#define MOE_CALL_FORWARD_FUSED_MLP 7
MOE_API moe_status moe_kernels_per_call_of(const moe_shape* shape, int32_t call, int32_t* count);

/* moe_forward, plus CUDA events recorded on `stream` around the kernels:
 * events[0] before kernel 1 and events[i] right after kernel i (i = 1..7),
 * so cudaEventElapsedTime(events[i-1], events[i]) is kernel i's time on the
 * stream (with top-k fused into the align kernel, events[2] follows events[1]
 * at once and the align interval includes the top-k; otherwise events[2] ends
 * the top-k/count kernel and events[3] the scan and scatter kernels; with the
 * single-launch front end, events[1] ends it and events[2..4] follow at once).  `events` holds n_events >= MOE_NUM_KERNELS + 1 cudaEvent_t
 * handles created by the caller (cudaEventCreate); the library records them
 * and does not create, wait on or destroy them.  Everything else is as for
 * moe_forward; with T = 0 no event is recorded. */
MOE_API moe_status moe_forward_events(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm,
                                      const float* w_router, const float* router_bias, const moe_bf16* w13,
                                      const moe_bf16* w2, moe_bf16* y, void* workspace, size_t workspace_bytes,
                                      moe_stream_t stream, void* const* events, int32_t n_events);

/* moe_forward with steps 1-4 (norm, router, top-k, align, gather) run as one
 * launch of one thread-block cluster: the decode dispatch as a single kernel
 * with a grid-wide barrier ("CuTeDSL chez Perplexity", "Synchronisation de la
 * grille"), here the cluster's hardware barrier (4 launches per call).  For
 * T <= MOE_FRONT_MAX_T and E <= MOE_FRONT_MAX_E on a device that runs a
 * cluster of at least 8 such CTAs; other shapes return MOE_ERR_UNSUPPORTED
 * before anything is enqueued.  Results are the same bits as moe_forward's;
 * the padding rows of the gathered input (moe_views.xg) are not written.
 * `events` is NULL, or as for moe_forward_events (the front end's time falls
 * in events[0]..events[1]).  moe_forward stays the faster choice on GB300:
 * there the expert GEMM cannot start its weight loads until the whole front
 * end has finished, and 16 SMs read the router weights more slowly than the
 * multi-launch router's grid. */
#define MOE_FRONT_MAX_T 64
#define MOE_FRONT_MAX_E 256
MOE_API moe_status moe_forward_fused_front(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm,
                                           const float* w_router, const float* router_bias, const moe_bf16* w13,
                                           const moe_bf16* w2, moe_bf16* y, void* workspace, size_t workspace_bytes,
                                           moe_stream_t stream, void* const* events, int32_t n_events);

/* moe_forward with step 7 (the top-k weighted combine) in the epilogue of
 * step 6, the down GEMM ("4 · La fusion de noyaux", §4.2 "GEMM + épilogue",
 * with one counter per piece of output as in §4.2 "GEMM + GEMM"): a unit of
 * the down GEMM that has stored its output rows of a 128-feature tile counts
 * one arrival per routed row in a per-(tile, token) counter of the workspace
 * (zeroed by the gather kernel), and the arrival that completes a token's k
 * rows sums them in routing-slot order j = 0..k-1 into y, with the separate
 * combine kernel's arithmetic: the same output bits as moe_forward, 5 launches
 * (7 with the multi-CTA top-k and align).  No thread ever waits on a counter.
 * `events` is NULL, or as for moe_forward_events (events[7] then follows
 * events[6] at once).  moe_forward stays the faster choice on GB300: the
 * epilogue's chain of store, fence, counter atomic and reads of the other
 * rows is as long as the kernel boundary it saves in decode, and in prefill
 * the epilogue waits on rows read back from DRAM and holds up the tensor
 * cores. */
MOE_API moe_status moe_forward_fused_combine(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm,
                                             const float* w_router, const float* router_bias, const moe_bf16* w13,
                                             const moe_bf16* w2, moe_bf16* y, void* workspace,
                                             size_t workspace_bytes, moe_stream_t stream, void* const* events,
                                             int32_t n_events);

/* moe_forward with both expert GEMMs in one persistent launch (the GEMM ->
 * GEMM fusion of "4 · La fusion de noyaux", §4.2 "GEMM + GEMM", grown into
 * the megakernel of §4.6): every CTA runs its stream-K share of the gate/up
 * GEMM, then its share of the down GEMM; a down-GEMM unit loads its
 * activation rows once every gate/up unit of its expert and token chunk has
 * counted the stores of its four epilogue warps in a per-chunk counter of the
 * workspace (zeroed by the align kernel; release add, acquire poll, proxy
 * fence before the TMA reads), while its weight tiles stream in ahead.  Same
 * K split as moe_forward, so the same output bits.  Decode tile plan only
 * (T * top_k <= 16 * E), else MOE_ERR_UNSUPPORTED before anything is
 * enqueued.  `events` as for moe_forward_events (events[6] then follows
 * events[5] at once).  moe_forward stays the faster choice on GB300: the
 * launch boundary saved (~4 us) is lost again because the fused kernel's
 * gate/up phase runs slower than the separate gate/up kernel. */
MOE_API moe_status moe_forward_fused_mlp(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm,
                                         const float* w_router, const float* router_bias, const moe_bf16* w13,
                                         const moe_bf16* w2, moe_bf16* y, void* workspace, size_t workspace_bytes,
                                         moe_stream_t stream, void* const* events, int32_t n_events);

/* Routing front end only (RMSNorm, router, top-k, align with `pad_rows`
 * rows of padding granularity), with the results copied out:
 *   topk_ids       [T, top_k] int32   selected experts, best first
 *   topk_w         [T, top_k] fp32    their weights
 *   expert_offsets [E + 1]    int32   start row of each expert's padded list;
 *                                     expert_offsets[E] = total rows P
 *   sorted_ids     [sorted_capacity] int32: rows [0, P) hold the flat index
 *                  t*top_k + j routed there (increasing within an expert),
 *                  padding rows hold T*top_k; entries in [P, T*top_k + E*(pad_rows-1))
 *                  are unspecified, entries beyond that are not written.
 * sorted_capacity must be >= T*top_k + E*(pad_rows - 1).  pad_rows: 1..256.
 * The workspace must be sized by moe_workspace_size() for the same shape. */
MOE_API moe_status moe_route_debug(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm,
                           const float* w_router, const float* router_bias, int32_t pad_rows,
                           int32_t* topk_ids, float* topk_w, int32_t* expert_offsets,
                           int32_t* sorted_ids, int64_t sorted_capacity, void* workspace,
                           size_t workspace_bytes, moe_stream_t stream);

/* Bytes of the fixed device scratch array used by moe_forward_static_scratch. */
#define MOE_STATIC_SCRATCH_BYTES (64ull << 20)

/* moe_forward without a caller-provided workspace and without allocating.
 * The pages have no counterpart of this call; it exists for callers that
 * cannot allocate device memory: hosts that give all device memory to their
 * own pool or run under a fixed budget, callers without a device allocator
 * (plain C, plug-ins), and latency-critical loops that avoid cudaMalloc /
 * cudaFree because those can block and synchronise the device.
 * The scratch is a file-scope __device__ array of MOE_STATIC_SCRATCH_BYTES
 * (64 MiB) inside the library; every GPU that loads the library holds it
 * until the process exits.  The caller still passes inputs and output, as
 * for moe_forward.
 *   - Shapes whose moe_workspace_size() exceeds MOE_STATIC_SCRATCH_BYTES are
 *     rejected with MOE_ERR_WORKSPACE before anything is enqueued (e.g. the
 *     decode layer H = I = 4096, E = 64, top_k = 8 fits for T <= 128: at
 *     T = 129 its tile plan changes and it needs 117 MB).
 *   - The first call on a device (with that device current) looks up the
 *     array's device address once (cudaGetSymbolAddress) and keeps it; make
 *     that first call before any stream capture.
 *   - Every call on a device shares the one array, which keeps the last
 *     call's contents; each call rewrites everything it reads, so nothing
 *     has to be cleared between calls.  Calls whose work overlaps on the GPU
 *     (other streams, other host threads) race on the array: serialise them.
 *   - The intermediate tensors are not exposed (no moe_workspace_views).
 *     Device-detected errors go to the error word at the start of the array;
 *     moe_static_scratch_device_status() reads it.
 *   - No cudaMalloc, cudaFree or allocating library routine is called. */
MOE_API moe_status moe_forward_static_scratch(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm,
                                              const float* w_router, const float* router_bias, const moe_bf16* w13,
                                              const moe_bf16* w2, moe_bf16* y, moe_stream_t stream);

/* The size of that array as compiled into the library (the value of
 * MOE_STATIC_SCRATCH_BYTES the library was built with), for bindings that
 * cannot read the macro.  Host-only; makes no CUDA call. */
MOE_API moe_status moe_static_scratch_bytes(size_t* bytes);

/* moe_device_status for moe_forward_static_scratch: waits for `stream`, then
 * reads the error word of the current device's static array (the one the
 * last moe_forward_static_scratch call on this device used; it is cleared by
 * the first kernel of every such call).  Returns MOE_OK, MOE_ERR_TIMEOUT or
 * MOE_ERR_DEVICE as moe_device_status does; `detail` (int32[4] or NULL)
 * receives the word.  Like the first moe_forward_static_scratch call, the
 * first call of either on a device looks up the array's address. */
MOE_API moe_status moe_static_scratch_device_status(moe_stream_t stream, int32_t* detail);

/* Device pointers to the intermediate tensors inside a workspace, valid for
 * the shape it was sized for (layout only; makes no CUDA call). */
typedef struct {
  void* error_word;   /* int32[4]: code, kernel id, detail, detail */
  void* h;            /* [T, H] bf16 RMSNorm output */
  void* logits;       /* [T, E] fp32 router logits (bias included) */
  void* topk_ids;     /* [T, top_k] int32 */
  void* topk_w;       /* [T, top_k] fp32 */
  void* counts;       /* [E] int32 tokens per expert */
  void* offsets;      /* [E + 1] int32 padded row offsets (16-row padding) */
  void* sorted_ids;   /* [P_max] int32 */
  void* slot_of;      /* [T * top_k] int32 row of each routed token */
  void* xg;           /* [P_max, H] bf16 gathered, padded expert inputs; written
                       * only where a gather kernel runs: moe_forward's decode
                       * tile plan (T * top_k <= 16 E) reads the rows of h in
                       * the gate/up GEMM instead (unless the combine is fused) */
  void* act;          /* [P_max, I] bf16 SwiGLU activations */
  void* out_rows;     /* [P_max, H] bf16 per-row expert outputs */
  int64_t P_max;      /* T*top_k + E*15: the most padded rows any routing can need */
} moe_views;

/* Device addresses of the block-scaled layers' extra intermediates (MXFP8,
 * MXFP4 and NVFP4; their token codes are in moe_views.xg, two per byte for the
 * FP4 layers).  Scales in the layouts described below. */
typedef struct {
  void* x_codes;    /* [P_max, H] E4M3 codes of the gathered token rows */
  void* x_scales;   /* their scales */
  void* act_codes;  /* [P_max, I] E4M3 codes of the SwiGLU activations */
  void* act_scales; /* their scales */
  int32_t x_chunk_rows;    /* token rows per scale chunk of x_scales (the gate/up GEMM's unit) */
  int32_t act_chunk_rows;  /* the same for act_scales (the down GEMM's unit) */
  void* x_gscale;          /* NVFP4 layer: [P_max] fp32 tensor scale of each gathered token row */
  void* act_gscale;        /* NVFP4 layer: [P_max] fp32 tensor scale of each activation row */
  int32_t nv_chunk_rows;   /* NVFP4 layer: token rows per scale chunk, both GEMMs (one CTA per unit) */
} moe_mx_views;

MOE_API moe_status moe_workspace_views_mx(const moe_shape* shape, void* workspace, size_t workspace_bytes,
                                          moe_views* views, moe_mx_views* mx_views);

MOE_API moe_status moe_workspace_views(const moe_shape* shape, void* workspace, size_t workspace_bytes,
                               moe_views* views);

/* Waits for `stream`, then reads the workspace's error word: MOE_OK, or the
 * device-side error of the last call that used this workspace
 * (MOE_ERR_TIMEOUT / MOE_ERR_DEVICE).  detail (may be NULL) receives the
 * four raw int32 words: the code, the id of the kernel that recorded it
 * (1 norm/router, 2 top-k, 3 align, 4 gather, 5 gate/up GEMM, 6 down GEMM,
 * 7 combine, 8 self-test), for the expert GEMMs a bit mask of the waits that
 * ran out (bit 1 producer: ring slot free; 2 MMA: accumulator free; 3 MMA:
 * ring slot loaded; 4 epilogue: accumulator complete; 5 epilogue: stream-K
 * partial sums; 6 epilogue: fused-combine rendezvous; 7 MMA: a stage's scales
 * written to TMEM; 8 scale warps: ring slot loaded), and the index of the CTA
 * that recorded the timeout. */
MOE_API moe_status moe_device_status(const void* workspace, size_t workspace_bytes, moe_stream_t stream,
                             int32_t* detail);

/* Static text for a status code. */
/* ---- FP8 expert weights (MXFP8) --------------------------------------
 * Block-scaled FP8 ("CuTeDSL chez Perplexity", "Prise en charge de Blackwell":
 * MXFP8, an absolute maximum over 32 elements): every 32 consecutive elements
 * along the reduction dimension share a power-of-two scale X = 2^E (one E8M0
 * byte, E + 127) with E = floor(log2(amax)) - 8 clamped to [-127, 127] (-127 for
 * an all-zero block); each element is stored as the E4M3 code of x / X, rounded
 * to nearest even and clamped to +-448.
 * Codes keep the matrix layout (one byte per element).  Scales are stored for
 * the block-scaled tensor-core MMA: per 128-row group and 128-element chunk of
 * the reduction dimension a 512-byte tile, byte r*16 + 4*j + b holding the
 * scale of row 32*j + r of the group and 32-element block b of the chunk.  For
 * W13 the rows of a group are the gate/up GEMM's tile rows: group e*(I/64) + t
 * holds features [64t, 64t+64) of expert e as, for g = 0..3, the 16 gate rows
 * 64t+16g .. +15 then the 16 matching up rows.  W2 groups are 128 consecutive
 * rows. */

/* Byte sizes of the MXFP8 copies of W13 and W2 for this shape. */
MOE_API moe_status moe_mx_weight_sizes(const moe_shape* shape, size_t* w13_codes, size_t* w13_scales,
                                       size_t* w2_codes, size_t* w2_scales);

/* Quantize the bf16 expert weights (layouts as for moe_forward) to MXFP8 on
 * the device (asynchronous on `stream`).  All pointers device, 16-byte aligned,
 * sized by moe_mx_weight_sizes. */
MOE_API moe_status moe_mx_quantize_weights(const moe_shape* shape, const moe_bf16* w13, const moe_bf16* w2,
                                           uint8_t* w13_codes, uint8_t* w13_scales, uint8_t* w2_codes,
                                           uint8_t* w2_scales, moe_stream_t stream);

/* Workspace bytes of moe_forward_mx (larger than moe_workspace_size's). */
MOE_API moe_status moe_workspace_size_mx(const moe_shape* shape, size_t* bytes);

/* The layer with MXFP8 expert weights: the same norm, router, top-k and
 * combine as moe_forward; each expert's input rows (the bf16 h) and its bf16
 * SwiGLU activations are quantized to MXFP8 the same way and the two expert
 * GEMMs run on the block-scaled tensor cores (tcgen05.mma kind::mxf8f6f4,
 * fp32 accumulation), in work units of 32 token rows (T * top_k / E <= 16)
 * or else 128, or 256 on CTA pairs where an expert's weight tiles come in
 * pairs (the tile plans of moe_forward).  Expert lists are padded to
 * 32 rows.  E <= 256 (else MOE_ERR_UNSUPPORTED).  events: NULL
 * or as for moe_forward_events (events[1] ends routing and align, events[4]
 * the gather + quantize, events[6] the activation quantize + down GEMM). */
MOE_API moe_status moe_forward_mx(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm,
                                  const float* w_router, const float* router_bias, const uint8_t* w13_codes,
                                  const uint8_t* w13_scales, const uint8_t* w2_codes, const uint8_t* w2_scales,
                                  moe_bf16* y, void* workspace, size_t workspace_bytes, moe_stream_t stream,
                                  void* const* events, int32_t n_events);

/* ---- FP4 expert weights (MXFP4) --------------------------------------
 * Block-scaled 4-bit weights (the same pages list Blackwell's block-scaled
 * FP4 formats beside MXFP8, "CuTeDSL chez Perplexity", "Prise en charge de
 * Blackwell"; the OCP Microscaling rule with E2M1 elements): every 32
 * consecutive elements along the reduction dimension share X = 2^E (one E8M0
 * byte, E + 127) with E = floor(log2(amax)) - 2 clamped to [-127, 127] (-127
 * for an all-zero block); each element is the E2M1 code of x / X (magnitudes
 * 0, 0.5, 1, 1.5, 2, 3, 4, 6; sign in bit 3) rounded to nearest with ties to
 * the even code and clamped to +-6.  Codes: the matrix layout with two codes
 * per byte, element 2i in the low nibble of byte i ([rows, K/2] bytes).
 * Scales: the MXFP8 layout above (the same tiles, the same W13 row order). */

/* Byte sizes of the MXFP4 copies of W13 and W2 for this shape (codes: half
 * the MXFP8 sizes; scales: the same). */
MOE_API moe_status moe_mxfp4_weight_sizes(const moe_shape* shape, size_t* w13_codes, size_t* w13_scales,
                                          size_t* w2_codes, size_t* w2_scales);

/* Quantize the bf16 expert weights (layouts as for moe_forward) to MXFP4 on
 * the device (asynchronous on `stream`).  All pointers device, sized by
 * moe_mxfp4_weight_sizes; codes 32-byte aligned (the tensor maps' rule for
 * packed 4-bit data), the rest 16-byte aligned; else MOE_ERR_INVALID_ARG. */
MOE_API moe_status moe_mxfp4_quantize_weights(const moe_shape* shape, const moe_bf16* w13, const moe_bf16* w2,
                                              uint8_t* w13_codes, uint8_t* w13_scales, uint8_t* w2_codes,
                                              uint8_t* w2_scales, moe_stream_t stream);

/* The layer with MXFP4 expert weights (W4A8): as moe_forward_mx (the same
 * routing, MXFP8 token rows and activations, tile plans, workspace
 * moe_workspace_size_mx and views moe_workspace_views_mx, events), with the
 * weights as E2M1 codes in the block-scaled MMA (tcgen05.mma
 * kind::mxf8f6f4, A = E2M1 weights, B = E4M3 tokens, fp32 accumulation).
 * Weight codes 32-byte aligned, else MOE_ERR_INVALID_ARG. */
MOE_API moe_status moe_forward_mxfp4(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm,
                                     const float* w_router, const float* router_bias, const uint8_t* w13_codes,
                                     const uint8_t* w13_scales, const uint8_t* w2_codes, const uint8_t* w2_scales,
                                     moe_bf16* y, void* workspace, size_t workspace_bytes, moe_stream_t stream,
                                     void* const* events, int32_t n_events);

/* The MXFP4 layer (W4A4): as moe_forward_mxfp4 (the same MXFP4 weights from
 * moe_mxfp4_quantize_weights, workspace, views and events), with each expert's
 * input rows and its SwiGLU activations quantized to MXFP4 by the same rule
 * as the weights, and both expert GEMMs on packed E2M1 operands (tcgen05.mma
 * kind::mxf4, two E8M0 scales per row per MMA of K = 64, fp32 accumulation).
 * H and I multiples of 128 like every block-scaled layer (else
 * MOE_ERR_UNSUPPORTED; a GEMM stage covers 256 elements of K, and an odd
 * multiple of 128 ends half way into the last one); weight codes 32-byte
 * aligned. */
MOE_API moe_status moe_forward_mxfp4a4(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm,
                                       const float* w_router, const float* router_bias, const uint8_t* w13_codes,
                                       const uint8_t* w13_scales, const uint8_t* w2_codes, const uint8_t* w2_scales,
                                       moe_bf16* y, void* workspace, size_t workspace_bytes, moe_stream_t stream,
                                       void* const* events, int32_t n_events);

/* ---- NVFP4 (E2M1 codes, E4M3 scales per 16, fp32 tensor scales) ---------
 * NVFP4 (the same pages name it beside MXFP8 / MXFP4, with an absolute
 * maximum over 16 elements; its published two-level form): every 16
 * consecutive elements along the reduction dimension share an E4M3 scale s
 * (sign 0), every tensor an fp32 scale g = amax_tensor / (448 * 6) (1 for an
 * all-zero tensor); s = E4M3(amax_16 / (6 g)) (nearest even, saturating to
 * 448) and each element the E2M1 code of x / (value(s) * g) (0 where that is
 * 0), each step one fp32 operation in this order.  The tensor of a weight is
 * one expert matrix (W13_e, W2_e); that of the token rows and activations one
 * row.  Codes: two per byte as for MXFP4.  Scales: 512-byte tiles per 128
 * rows and 64 elements of K, byte r*16 + 4*j + b = the scale of row 32*j + r
 * and 16-element block b of the 64 (W13 rows in the gate/up tile-row order as
 * for MXFP8). */

/* Byte sizes of the NVFP4 copies of W13 and W2 (their tensor scales: E floats
 * each, caller-sized). */
MOE_API moe_status moe_nvfp4_weight_sizes(const moe_shape* shape, size_t* w13_codes, size_t* w13_scales,
                                          size_t* w2_codes, size_t* w2_scales);

/* Quantize the bf16 expert weights to NVFP4 on the device (asynchronous on
 * `stream`): codes and block scales sized by moe_nvfp4_weight_sizes, tensor
 * scales w13_gscale[E], w2_gscale[E] (fp32; they hold the absolute maxima
 * until the last kernel of the call has run).  Codes 32-byte aligned, scales
 * 16-byte, tensor scales 4-byte aligned; else MOE_ERR_INVALID_ARG. */
MOE_API moe_status moe_nvfp4_quantize_weights(const moe_shape* shape, const moe_bf16* w13, const moe_bf16* w2,
                                              uint8_t* w13_codes, uint8_t* w13_scales, float* w13_gscale,
                                              uint8_t* w2_codes, uint8_t* w2_scales, float* w2_gscale,
                                              moe_stream_t stream);

/* The NVFP4 layer: as moe_forward_mxfp4a4 with NVFP4 weights, token rows and
 * activations (tcgen05.mma kind::mxf4nvf4, scale_vec::4X: four E4M3 scales per
 * row per MMA of K = 64; the fp32 tensor scales of the expert matrix and of the
 * token row multiply each accumulator in the epilogue), one CTA per work unit
 * in every tile plan.  H and I multiples of 128 (else MOE_ERR_UNSUPPORTED). */
MOE_API moe_status moe_forward_nvfp4(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm,
                                     const float* w_router, const float* router_bias, const uint8_t* w13_codes,
                                     const uint8_t* w13_scales, const float* w13_gscale, const uint8_t* w2_codes,
                                     const uint8_t* w2_scales, const float* w2_gscale, moe_bf16* y, void* workspace,
                                     size_t workspace_bytes, moe_stream_t stream, void* const* events,
                                     int32_t n_events);

/* QK-norm, in place: RMSNorm of every attention head of Q and of K
 * ("CuTeDSL chez Perplexity", "Norme QK"):
 *   out_j = bf16((w_j + weight_bias) * (x_j * rstd)),  rstd = 1/sqrt(mean_j x_j^2 + eps),
 * over the D elements of each head, with q_weight[D] applied to every head of Q
 * and k_weight[D] to every head of K.  Computed in fp32 in one fixed order
 * (see k_qk_norm.cu), so the result is within one bf16 ulp of the exact value.
 *   q [T, Hq, D] bf16, k [T, Hk, D] bf16: device, contiguous, 16-byte aligned,
 *   overwritten with the result; q_weight / k_weight [D] bf16.
 *   D: 64, 128 or 256.  Hq or Hk may be 0 (its pointers are then unused).
 * Errors: MOE_ERR_INVALID_ARG for a bad D, negative sizes, null or misaligned
 * pointers of a non-empty tensor, or a non-finite eps / weight_bias;
 * MOE_ERR_UNSUPPORTED for T * (Hq + Hk) >= 2^31 heads; T = 0 is a no-op.
 * Asynchronous on `stream`; no workspace. */
MOE_API moe_status moe_qk_norm(int64_t T, int32_t Hq, int32_t Hk, int32_t D, moe_bf16* q, moe_bf16* k,
                               const moe_bf16* q_weight, const moe_bf16* k_weight, float weight_bias, float eps,
                               moe_stream_t stream);

/* Self-test of the failure path of the library's bounded device waits (no
 * counterpart on the pages): enqueues one small kernel whose two waits -- on
 * an mbarrier phase that nothing completes and on a flag in the workspace's
 * error area that nothing sets -- give up after timeout_ns (1 .. 1e9) and
 * record MOE_ERR_TIMEOUT, with kernel id 8 in detail[1], in the workspace's
 * error word, then return normally.  moe_device_status() afterwards returns
 * MOE_ERR_TIMEOUT; the CUDA context stays usable, and the next moe_forward on
 * that workspace clears the word.  workspace: >= 64 bytes, 256-byte aligned;
 * its first 64 bytes are overwritten. */
MOE_API moe_status moe_selftest_wait_timeout(void* workspace, size_t workspace_bytes, int64_t timeout_ns,
                                             moe_stream_t stream);

MOE_API const char* moe_status_string(moe_status status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
