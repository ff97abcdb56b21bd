// moe_forward_impl.h -- the forward pass behind the ABI's forward entry points.
#pragma once

#include "../../include/moe.h"

namespace moe {

// Checks the arguments, then enqueues the kernels of one layer call on
// `stream`, with `workspace` (>= moe_workspace_size bytes) as scratch.  When
// `events` is non-null, events[0] is recorded before the first kernel and
// events[i] after the i-th kernel.  With single_launch_front, the norm,
// router, top-k, align and gather run as one cluster launch; shapes that do
// not fit it return MOE_ERR_UNSUPPORTED before anything is enqueued.  With
// fused_combine, the top-k weighted combine runs in the down GEMM's epilogue.
// With fused_mlp, both expert GEMMs run as one launch (small tile plan only,
// else MOE_ERR_UNSUPPORTED).
moe_status forward_impl(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm, const float* w_router,
                        const float* router_bias, const moe_bf16* w13, const moe_bf16* w2, moe_bf16* y,
                        void* workspace, size_t workspace_bytes, moe_stream_t stream, void* const* events,
                        bool single_launch_front = false, bool fused_combine = false, bool fused_mlp = false);

}  // namespace moe
