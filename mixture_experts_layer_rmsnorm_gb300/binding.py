"""Python binding of the C ABI in include/moe.h (argument marshalling only).

Every function here has the name of the C entry point it calls and forwards
plain integers / device pointers; all of the layer's work runs in the CUDA
kernels of libmoe_gb300.so.  There is no fallback: if the library cannot be
built or loaded, :func:`load` raises.

:class:`MoeLayer` is a convenience holder for torch tensors (weights and a
workspace on the GPU) that marshals their pointers into :func:`moe_forward`.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_TIMEOUT, \
    MOE_ERR_DEVICE = range(7)

_lock = threading.Lock()
_lib = None


class MoeShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32), ("E", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("renormalize", ctypes.c_int32), ("eps", ctypes.c_float)]


class MoeViews(ctypes.Structure):
    _fields_ = [("error_word", ctypes.c_void_p), ("h", ctypes.c_void_p), ("logits", ctypes.c_void_p),
                ("topk_ids", ctypes.c_void_p), ("topk_w", ctypes.c_void_p), ("counts", ctypes.c_void_p),
                ("offsets", ctypes.c_void_p), ("sorted_ids", ctypes.c_void_p), ("slot_of", ctypes.c_void_p),
                ("xg", ctypes.c_void_p), ("act", ctypes.c_void_p), ("out_rows", ctypes.c_void_p),
                ("P_max", ctypes.c_int64)]


class MoeMxViews(ctypes.Structure):
    _fields_ = [("x_codes", ctypes.c_void_p), ("x_scales", ctypes.c_void_p), ("act_codes", ctypes.c_void_p),
                ("act_scales", ctypes.c_void_p), ("x_chunk_rows", ctypes.c_int32), ("act_chunk_rows", ctypes.c_int32),
                ("x_gscale", ctypes.c_void_p), ("act_gscale", ctypes.c_void_p), ("nv_chunk_rows", ctypes.c_int32)]


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {moe_status_string(status)} (status {status})")
        self.status = status


def lib_path() -> str:
    return _build.LIB


def load(build: bool = True):
    """Load libmoe_gb300.so (compiling it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build else _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library {path} is missing; run __graft_entry__.build()")
            lib = ctypes.CDLL(path)
            p, sz, i32, i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int64
            sp = ctypes.POINTER(MoeShape)
            lib.moe_workspace_size.argtypes = [sp, ctypes.POINTER(sz)]
            lib.moe_forward.argtypes = [sp, p, p, p, p, p, p, p, p, sz, p]
            lib.moe_forward_events.argtypes = [sp, p, p, p, p, p, p, p, p, sz, p, p, i32]
            lib.moe_route_debug.argtypes = [sp, p, p, p, p, i32, p, p, p, p, i64, p, sz, p]
            lib.moe_forward_static_scratch.argtypes = [sp, p, p, p, p, p, p, p, p]
            lib.moe_static_scratch_bytes.argtypes = [ctypes.POINTER(sz)]
            lib.moe_static_scratch_device_status.argtypes = [p, ctypes.POINTER(ctypes.c_int32)]
            lib.moe_workspace_views.argtypes = [sp, p, sz, ctypes.POINTER(MoeViews)]
            lib.moe_device_status.argtypes = [p, sz, p, ctypes.POINTER(ctypes.c_int32)]
            lib.moe_kernels_per_call.argtypes = [sp, ctypes.POINTER(ctypes.c_int32)]
            lib.moe_kernels_per_call_of.argtypes = [sp, i32, ctypes.POINTER(ctypes.c_int32)]
            lib.moe_selftest_wait_timeout.argtypes = [p, sz, i64, p]
            lib.moe_qk_norm.argtypes = [i64, i32, i32, i32, p, p, p, p, ctypes.c_float, ctypes.c_float, p]
            psz = ctypes.POINTER(sz)
            lib.moe_mx_weight_sizes.argtypes = [sp, psz, psz, psz, psz]
            lib.moe_mx_quantize_weights.argtypes = [sp, p, p, p, p, p, p, p]
            lib.moe_workspace_size_mx.argtypes = [sp, psz]
            lib.moe_workspace_views_mx.argtypes = [sp, p, sz, ctypes.POINTER(MoeViews), ctypes.POINTER(MoeMxViews)]
            lib.moe_forward_mx.argtypes = [sp, p, p, p, p, p, p, p, p, p, p, sz, p, p, i32]
            lib.moe_mxfp4_weight_sizes.argtypes = [sp, psz, psz, psz, psz]
            lib.moe_mxfp4_quantize_weights.argtypes = [sp, p, p, p, p, p, p, p]
            lib.moe_forward_mxfp4.argtypes = [sp, p, p, p, p, p, p, p, p, p, p, sz, p, p, i32]
            lib.moe_forward_mxfp4a4.argtypes = [sp, p, p, p, p, p, p, p, p, p, p, sz, p, p, i32]
            lib.moe_nvfp4_weight_sizes.argtypes = [sp, psz, psz, psz, psz]
            lib.moe_nvfp4_quantize_weights.argtypes = [sp, p, p, p, p, p, p, p, p, p]
            lib.moe_forward_nvfp4.argtypes = [sp, p, p, p, p, p, p, p, p, p, p, p, p, sz, p, p, i32]
            lib.moe_forward_fused_front.argtypes = [sp, p, p, p, p, p, p, p, p, sz, p, p, i32]
            lib.moe_forward_fused_combine.argtypes = [sp, p, p, p, p, p, p, p, p, sz, p, p, i32]
            lib.moe_forward_fused_mlp.argtypes = [sp, p, p, p, p, p, p, p, p, sz, p, p, i32]
            lib.moe_status_string.argtypes = [ctypes.c_int]
            lib.moe_status_string.restype = ctypes.c_char_p
            for f in ("moe_workspace_size", "moe_forward", "moe_forward_events", "moe_route_debug",
                      "moe_workspace_views", "moe_device_status", "moe_forward_static_scratch",
                      "moe_static_scratch_bytes", "moe_static_scratch_device_status",
                      "moe_kernels_per_call", "moe_kernels_per_call_of", "moe_forward_fused_front",
                      "moe_selftest_wait_timeout",
                      "moe_qk_norm", "moe_mx_weight_sizes", "moe_mx_quantize_weights", "moe_workspace_size_mx",
                      "moe_workspace_views_mx", "moe_forward_mx", "moe_forward_fused_combine",
                      "moe_mxfp4_weight_sizes", "moe_mxfp4_quantize_weights", "moe_forward_mxfp4",
                      "moe_forward_mxfp4a4", "moe_nvfp4_weight_sizes", "moe_nvfp4_quantize_weights",
                      "moe_forward_nvfp4", "moe_forward_fused_mlp"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def shape(T, H, I, E, top_k, renormalize=True, eps=1e-6) -> MoeShape:
    return MoeShape(int(T), int(H), int(I), int(E), int(top_k), int(bool(renormalize)), float(eps))


def moe_status_string(status: int) -> str:
    return load().moe_status_string(int(status)).decode()


def moe_workspace_size(s: MoeShape) -> tuple[int, int]:
    n = ctypes.c_size_t(0)
    st = load().moe_workspace_size(ctypes.byref(s), ctypes.byref(n))
    return st, n.value


def moe_forward(s: MoeShape, x, g_norm, w_router, router_bias, w13, w2, y, workspace, workspace_bytes,
                stream) -> int:
    return load().moe_forward(ctypes.byref(s), x, g_norm, w_router, router_bias, w13, w2, y, workspace,
                              workspace_bytes, stream)


MOE_NUM_KERNELS = 7
MOE_FRONT_MAX_T = 64  # single-launch front end (norm .. gather) up to this many tokens ...
MOE_FRONT_MAX_E = 256  # ... and experts
MOE_FUSED_TOPK_MAX_T = 256  # top-k runs inside the align kernel up to this many tokens ...
MOE_FUSED_TOPK_MAX_E = 256  # ... and experts


def moe_kernels_per_call(s: MoeShape) -> tuple[int, int]:
    n = ctypes.c_int32(0)
    st = load().moe_kernels_per_call(ctypes.byref(s), ctypes.byref(n))
    return st, n.value


(MOE_CALL_FORWARD, MOE_CALL_FORWARD_FUSED_FRONT, MOE_CALL_FORWARD_MX, MOE_CALL_FORWARD_FUSED_COMBINE,
 MOE_CALL_FORWARD_MXFP4, MOE_CALL_FORWARD_MXFP4A4, MOE_CALL_FORWARD_NVFP4, MOE_CALL_FORWARD_FUSED_MLP) = \
    0, 1, 2, 3, 4, 5, 6, 7


def moe_kernels_per_call_of(s: MoeShape, call: int) -> tuple[int, int]:
    n = ctypes.c_int32(0)
    st = load().moe_kernels_per_call_of(ctypes.byref(s), int(call), ctypes.byref(n))
    return st, n.value


def kernels_per_call(T: int, H: int, I: int, E: int, top_k: int, call: int = MOE_CALL_FORWARD) -> int:
    """Kernel launches of one call of the entry point `call` (MOE_CALL_*)."""
    st, n = moe_kernels_per_call_of(shape(T, H, I, E, top_k), call)
    if st != MOE_OK:
        raise MoeError(st, "moe_kernels_per_call_of")
    return n


KERNEL_NAMES = ("norm_router", "topk_softmax", "align", "gather", "gemm_gate_up_swiglu", "gemm_down", "combine")


def moe_forward_events(s: MoeShape, x, g_norm, w_router, router_bias, w13, w2, y, workspace, workspace_bytes,
                       stream, events) -> int:
    """events: a sequence of MOE_NUM_KERNELS + 1 raw cudaEvent_t handles (ints)."""
    arr = (ctypes.c_void_p * len(events))(*events)
    return load().moe_forward_events(ctypes.byref(s), x, g_norm, w_router, router_bias, w13, w2, y, workspace,
                                     workspace_bytes, stream, arr, len(events))


def moe_forward_fused_front(s: MoeShape, x, g_norm, w_router, router_bias, w13, w2, y, workspace,
                            workspace_bytes, stream, events=None) -> int:
    """moe_forward with norm .. gather as one cluster launch (decode shapes only)."""
    if events is None:
        arr, n = None, 0
    else:
        arr, n = (ctypes.c_void_p * len(events))(*events), len(events)
    return load().moe_forward_fused_front(ctypes.byref(s), x, g_norm, w_router, router_bias, w13, w2, y, workspace,
                                          workspace_bytes, stream, arr, n)


def moe_forward_fused_combine(s: MoeShape, x, g_norm, w_router, router_bias, w13, w2, y, workspace,
                              workspace_bytes, stream, events=None) -> int:
    """moe_forward with the top-k weighted combine in the down GEMM's epilogue."""
    if events is None:
        arr, n = None, 0
    else:
        arr, n = (ctypes.c_void_p * len(events))(*events), len(events)
    return load().moe_forward_fused_combine(ctypes.byref(s), x, g_norm, w_router, router_bias, w13, w2, y,
                                            workspace, workspace_bytes, stream, arr, n)


def moe_forward_fused_mlp(s: MoeShape, x, g_norm, w_router, router_bias, w13, w2, y, workspace, workspace_bytes,
                          stream, events=None) -> int:
    """moe_forward with both expert GEMMs in one launch (decode tile plan only)."""
    if events is None:
        arr, n = None, 0
    else:
        arr, n = (ctypes.c_void_p * len(events))(*events), len(events)
    return load().moe_forward_fused_mlp(ctypes.byref(s), x, g_norm, w_router, router_bias, w13, w2, y, workspace,
                                        workspace_bytes, stream, arr, n)


def moe_static_scratch_bytes() -> tuple[int, int]:
    """Size of the library's fixed device scratch array, as compiled into it."""
    n = ctypes.c_size_t(0)
    st = load().moe_static_scratch_bytes(ctypes.byref(n))
    return st, n.value


def moe_static_scratch_device_status(stream) -> tuple[int, list]:
    """moe_device_status for moe_forward_static_scratch (the current device's array)."""
    d = (ctypes.c_int32 * 4)()
    st = load().moe_static_scratch_device_status(stream, d)
    return st, list(d)


def moe_forward_static_scratch(s: MoeShape, x, g_norm, w_router, router_bias, w13, w2, y, stream) -> int:
    """moe_forward with the library's fixed device scratch array instead of a
    caller workspace (for callers that cannot allocate device memory)."""
    return load().moe_forward_static_scratch(ctypes.byref(s), x, g_norm, w_router, router_bias, w13, w2, y, stream)


def moe_route_debug(s: MoeShape, x, g_norm, w_router, router_bias, pad_rows, topk_ids, topk_w, expert_offsets,
                    sorted_ids, sorted_capacity, workspace, workspace_bytes, stream) -> int:
    return load().moe_route_debug(ctypes.byref(s), x, g_norm, w_router, router_bias, pad_rows, topk_ids, topk_w,
                                  expert_offsets, sorted_ids, sorted_capacity, workspace, workspace_bytes, stream)


def moe_workspace_views(s: MoeShape, workspace, workspace_bytes) -> tuple[int, MoeViews]:
    v = MoeViews()
    st = load().moe_workspace_views(ctypes.byref(s), workspace, workspace_bytes, ctypes.byref(v))
    return st, v


def moe_device_status(workspace, workspace_bytes, stream) -> tuple[int, list]:
    d = (ctypes.c_int32 * 4)()
    st = load().moe_device_status(workspace, workspace_bytes, stream, d)
    return st, list(d)


def moe_qk_norm(T, Hq, Hk, D, q, k, q_weight, k_weight, weight_bias, eps, stream) -> int:
    return load().moe_qk_norm(int(T), int(Hq), int(Hk), int(D), q, k, q_weight, k_weight, float(weight_bias),
                              float(eps), stream)


def moe_selftest_wait_timeout(workspace, workspace_bytes, timeout_ns, stream) -> int:
    return load().moe_selftest_wait_timeout(workspace, workspace_bytes, int(timeout_ns), stream)


def moe_mx_weight_sizes(s: MoeShape) -> tuple[int, tuple[int, int, int, int]]:
    v = [ctypes.c_size_t(0) for _ in range(4)]
    st = load().moe_mx_weight_sizes(ctypes.byref(s), *[ctypes.byref(a) for a in v])
    return st, tuple(a.value for a in v)


def moe_mx_quantize_weights(s: MoeShape, w13, w2, w13_codes, w13_scales, w2_codes, w2_scales, stream) -> int:
    return load().moe_mx_quantize_weights(ctypes.byref(s), w13, w2, w13_codes, w13_scales, w2_codes, w2_scales,
                                          stream)


def moe_workspace_size_mx(s: MoeShape) -> tuple[int, int]:
    n = ctypes.c_size_t(0)
    st = load().moe_workspace_size_mx(ctypes.byref(s), ctypes.byref(n))
    return st, n.value


def moe_workspace_views_mx(s: MoeShape, workspace, workspace_bytes) -> tuple[int, MoeViews, MoeMxViews]:
    v, mv = MoeViews(), MoeMxViews()
    st = load().moe_workspace_views_mx(ctypes.byref(s), workspace, workspace_bytes, ctypes.byref(v), ctypes.byref(mv))
    return st, v, mv


def moe_forward_mx(s: MoeShape, x, g_norm, w_router, router_bias, w13_codes, w13_scales, w2_codes, w2_scales, y,
                   workspace, workspace_bytes, stream, events=None) -> int:
    if events is None:
        arr, n = None, 0
    else:
        arr, n = (ctypes.c_void_p * len(events))(*events), len(events)
    return load().moe_forward_mx(ctypes.byref(s), x, g_norm, w_router, router_bias, w13_codes, w13_scales, w2_codes,
                                 w2_scales, y, workspace, workspace_bytes, stream, arr, n)


def moe_mxfp4_weight_sizes(s: MoeShape) -> tuple[int, tuple[int, int, int, int]]:
    v = [ctypes.c_size_t(0) for _ in range(4)]
    st = load().moe_mxfp4_weight_sizes(ctypes.byref(s), *[ctypes.byref(a) for a in v])
    return st, tuple(a.value for a in v)


def moe_mxfp4_quantize_weights(s: MoeShape, w13, w2, w13_codes, w13_scales, w2_codes, w2_scales, stream) -> int:
    return load().moe_mxfp4_quantize_weights(ctypes.byref(s), w13, w2, w13_codes, w13_scales, w2_codes, w2_scales,
                                             stream)


def moe_forward_mxfp4(s: MoeShape, x, g_norm, w_router, router_bias, w13_codes, w13_scales, w2_codes, w2_scales, y,
                      workspace, workspace_bytes, stream, events=None) -> int:
    if events is None:
        arr, n = None, 0
    else:
        arr, n = (ctypes.c_void_p * len(events))(*events), len(events)
    return load().moe_forward_mxfp4(ctypes.byref(s), x, g_norm, w_router, router_bias, w13_codes, w13_scales,
                                    w2_codes, w2_scales, y, workspace, workspace_bytes, stream, arr, n)


def moe_forward_mxfp4a4(s: MoeShape, x, g_norm, w_router, router_bias, w13_codes, w13_scales, w2_codes, w2_scales,
                        y, workspace, workspace_bytes, stream, events=None) -> int:
    if events is None:
        arr, n = None, 0
    else:
        arr, n = (ctypes.c_void_p * len(events))(*events), len(events)
    return load().moe_forward_mxfp4a4(ctypes.byref(s), x, g_norm, w_router, router_bias, w13_codes, w13_scales,
                                      w2_codes, w2_scales, y, workspace, workspace_bytes, stream, arr, n)


def moe_nvfp4_weight_sizes(s: MoeShape) -> tuple[int, tuple[int, int, int, int]]:
    v = [ctypes.c_size_t(0) for _ in range(4)]
    st = load().moe_nvfp4_weight_sizes(ctypes.byref(s), *[ctypes.byref(a) for a in v])
    return st, tuple(a.value for a in v)


def moe_nvfp4_quantize_weights(s: MoeShape, w13, w2, w13_codes, w13_scales, w13_gscale, w2_codes, w2_scales,
                               w2_gscale, stream) -> int:
    return load().moe_nvfp4_quantize_weights(ctypes.byref(s), w13, w2, w13_codes, w13_scales, w13_gscale, w2_codes,
                                             w2_scales, w2_gscale, stream)


def moe_forward_nvfp4(s: MoeShape, x, g_norm, w_router, router_bias, w13_codes, w13_scales, w13_gscale, w2_codes,
                      w2_scales, w2_gscale, y, workspace, workspace_bytes, stream, events=None) -> int:
    if events is None:
        arr, n = None, 0
    else:
        arr, n = (ctypes.c_void_p * len(events))(*events), len(events)
    return load().moe_forward_nvfp4(ctypes.byref(s), x, g_norm, w_router, router_bias, w13_codes, w13_scales,
                                    w13_gscale, w2_codes, w2_scales, w2_gscale, y, workspace, workspace_bytes, stream,
                                    arr, n)


def _ptr(t):
    return None if t is None else t.data_ptr()


class MoeLayer:
    """One MoE layer's weights on the GPU plus a workspace sized for up to
    ``max_tokens`` tokens.  Inputs and outputs are torch tensors on the same
    device; bf16 tensors may be torch.bfloat16 or raw int16 bit patterns."""

    def __init__(self, g_norm, w_router, w13, w2, top_k, renormalize=True, eps=1e-6, router_bias=None,
                 max_tokens=1):
        import torch
        self.g_norm, self.w_router, self.w13, self.w2, self.bias = g_norm, w_router, w13, w2, router_bias
        self.E, two_i, self.H = w13.shape
        self.I = two_i // 2
        self.top_k, self.renormalize, self.eps = int(top_k), bool(renormalize), float(eps)
        self.device = w13.device
        self.max_tokens = 0
        self.workspace = None
        self.ensure_capacity(max_tokens)
        self._torch = torch

    def shape(self, T) -> MoeShape:
        return shape(T, self.H, self.I, self.E, self.top_k, self.renormalize, self.eps)

    def ensure_capacity(self, T):
        import torch
        if T <= self.max_tokens and self.workspace is not None:
            return
        st, n = moe_workspace_size(self.shape(max(T, 1)))
        if st != MOE_OK:
            raise MoeError(st, "moe_workspace_size")
        st, n_mx = moe_workspace_size_mx(self.shape(max(T, 1)))
        if st == MOE_OK:
            n = max(n, n_mx)  # room for the MXFP8 forward as well
        self.workspace = torch.empty(n, dtype=torch.uint8, device=self.device)
        self.max_tokens = max(T, 1)

    def workspace_bytes(self, T) -> int:
        st, n = moe_workspace_size(self.shape(T))
        if st != MOE_OK:
            raise MoeError(st, "moe_workspace_size")
        return n

    def forward(self, x, y=None, stream=None, events=None, fused_front=False, fused_combine=False, fused_mlp=False):
        """y = layer(x).  events: optional MOE_NUM_KERNELS + 1 cudaEvent_t handles
        recorded around the kernels (moe_forward_events).  fused_front: run the
        norm .. gather steps as one cluster launch (moe_forward_fused_front).
        fused_combine: the combine in the down GEMM's epilogue
        (moe_forward_fused_combine).  fused_mlp: both expert GEMMs in one
        launch (moe_forward_fused_mlp; decode tile plan only)."""
        import torch
        T = x.shape[0]
        self.ensure_capacity(T)
        if y is None:
            y = torch.empty((T, self.H), dtype=x.dtype, device=x.device)
        s = stream if stream is not None else torch.cuda.current_stream(x.device).cuda_stream
        args = (self.shape(T), _ptr(x), _ptr(self.g_norm), _ptr(self.w_router), _ptr(self.bias), _ptr(self.w13),
                _ptr(self.w2), _ptr(y), _ptr(self.workspace), self.workspace_bytes(T), s)
        if int(fused_front) + int(fused_combine) + int(fused_mlp) > 1:
            raise ValueError("fused_front, fused_combine and fused_mlp are separate entry points")
        if fused_mlp:
            st = moe_forward_fused_mlp(*args, events)
        elif fused_front:
            st = moe_forward_fused_front(*args, events)
        elif fused_combine:
            st = moe_forward_fused_combine(*args, events)
        elif events is None:
            st = moe_forward(*args)
        else:
            st = moe_forward_events(*args, events)
        if st != MOE_OK:
            raise MoeError(st, "moe_forward")
        return y

    def quantize_mx(self, stream=None):
        """Make the MXFP8 copies of W13 and W2 (moe_mx_quantize_weights) for forward_mx."""
        import torch
        st, (n13c, n13s, n2c, n2s) = moe_mx_weight_sizes(self.shape(1))
        if st != MOE_OK:
            raise MoeError(st, "moe_mx_weight_sizes")
        u8 = dict(dtype=torch.uint8, device=self.device)
        self.w13_codes, self.w13_scales = torch.empty(n13c, **u8), torch.empty(n13s, **u8)
        self.w2_codes, self.w2_scales = torch.empty(n2c, **u8), torch.empty(n2s, **u8)
        s = stream if stream is not None else torch.cuda.current_stream(self.device).cuda_stream
        st = moe_mx_quantize_weights(self.shape(1), _ptr(self.w13), _ptr(self.w2), _ptr(self.w13_codes),
                                     _ptr(self.w13_scales), _ptr(self.w2_codes), _ptr(self.w2_scales), s)
        if st != MOE_OK:
            raise MoeError(st, "moe_mx_quantize_weights")

    def quantize_mxfp4(self, stream=None):
        """Make the MXFP4 copies of W13 and W2 (moe_mxfp4_quantize_weights) for forward_mxfp4."""
        import torch
        st, (n13c, n13s, n2c, n2s) = moe_mxfp4_weight_sizes(self.shape(1))
        if st != MOE_OK:
            raise MoeError(st, "moe_mxfp4_weight_sizes")
        u8 = dict(dtype=torch.uint8, device=self.device)
        self.w13_codes4, self.w13_scales4 = torch.empty(n13c, **u8), torch.empty(n13s, **u8)
        self.w2_codes4, self.w2_scales4 = torch.empty(n2c, **u8), torch.empty(n2s, **u8)
        s = stream if stream is not None else torch.cuda.current_stream(self.device).cuda_stream
        st = moe_mxfp4_quantize_weights(self.shape(1), _ptr(self.w13), _ptr(self.w2), _ptr(self.w13_codes4),
                                        _ptr(self.w13_scales4), _ptr(self.w2_codes4), _ptr(self.w2_scales4), s)
        if st != MOE_OK:
            raise MoeError(st, "moe_mxfp4_quantize_weights")

    def forward_mxfp4(self, x, y=None, stream=None, events=None, fp4_tokens=False):
        """y = layer(x) with the MXFP4 expert weights (call quantize_mxfp4 first);
        fp4_tokens: the MXFP4 layer, with token rows and activations in MXFP4
        too (moe_forward_mxfp4a4), else MXFP8 tokens (moe_forward_mxfp4)."""
        import torch
        T = x.shape[0]
        self.ensure_capacity(T)
        if y is None:
            y = torch.empty((T, self.H), dtype=x.dtype, device=x.device)
        s = stream if stream is not None else torch.cuda.current_stream(x.device).cuda_stream
        fn, name = (moe_forward_mxfp4a4, "moe_forward_mxfp4a4") if fp4_tokens else (moe_forward_mxfp4,
                                                                                   "moe_forward_mxfp4")
        st = fn(self.shape(T), _ptr(x), _ptr(self.g_norm), _ptr(self.w_router), _ptr(self.bias),
                _ptr(self.w13_codes4), _ptr(self.w13_scales4), _ptr(self.w2_codes4), _ptr(self.w2_scales4), _ptr(y),
                _ptr(self.workspace), self.workspace_bytes_mx(T), s, events)
        if st != MOE_OK:
            raise MoeError(st, name)
        return y

    def quantize_nvfp4(self, stream=None):
        """Make the NVFP4 copies of W13 and W2 (moe_nvfp4_quantize_weights) for forward_nvfp4."""
        import torch
        st, (n13c, n13s, n2c, n2s) = moe_nvfp4_weight_sizes(self.shape(1))
        if st != MOE_OK:
            raise MoeError(st, "moe_nvfp4_weight_sizes")
        u8 = dict(dtype=torch.uint8, device=self.device)
        self.w13_codes_nv, self.w13_scales_nv = torch.empty(n13c, **u8), torch.empty(n13s, **u8)
        self.w2_codes_nv, self.w2_scales_nv = torch.empty(n2c, **u8), torch.empty(n2s, **u8)
        self.w13_gscale_nv = torch.empty(self.E, dtype=torch.float32, device=self.device)
        self.w2_gscale_nv = torch.empty(self.E, dtype=torch.float32, device=self.device)
        s = stream if stream is not None else torch.cuda.current_stream(self.device).cuda_stream
        st = moe_nvfp4_quantize_weights(self.shape(1), _ptr(self.w13), _ptr(self.w2), _ptr(self.w13_codes_nv),
                                        _ptr(self.w13_scales_nv), _ptr(self.w13_gscale_nv), _ptr(self.w2_codes_nv),
                                        _ptr(self.w2_scales_nv), _ptr(self.w2_gscale_nv), s)
        if st != MOE_OK:
            raise MoeError(st, "moe_nvfp4_quantize_weights")

    def forward_nvfp4(self, x, y=None, stream=None, events=None):
        """y = layer(x), the NVFP4 layer (call quantize_nvfp4 first)."""
        import torch
        T = x.shape[0]
        self.ensure_capacity(T)
        if y is None:
            y = torch.empty((T, self.H), dtype=x.dtype, device=x.device)
        s = stream if stream is not None else torch.cuda.current_stream(x.device).cuda_stream
        st = moe_forward_nvfp4(self.shape(T), _ptr(x), _ptr(self.g_norm), _ptr(self.w_router), _ptr(self.bias),
                               _ptr(self.w13_codes_nv), _ptr(self.w13_scales_nv), _ptr(self.w13_gscale_nv),
                               _ptr(self.w2_codes_nv), _ptr(self.w2_scales_nv), _ptr(self.w2_gscale_nv), _ptr(y),
                               _ptr(self.workspace), self.workspace_bytes_mx(T), s, events)
        if st != MOE_OK:
            raise MoeError(st, "moe_forward_nvfp4")
        return y

    def workspace_bytes_mx(self, T) -> int:
        st, n = moe_workspace_size_mx(self.shape(T))
        if st != MOE_OK:
            raise MoeError(st, "moe_workspace_size_mx")
        return n

    def forward_mx(self, x, y=None, stream=None, events=None):
        """y = layer(x) with the MXFP8 expert weights (call quantize_mx first)."""
        import torch
        T = x.shape[0]
        self.ensure_capacity(T)
        if y is None:
            y = torch.empty((T, self.H), dtype=x.dtype, device=x.device)
        s = stream if stream is not None else torch.cuda.current_stream(x.device).cuda_stream
        st = moe_forward_mx(self.shape(T), _ptr(x), _ptr(self.g_norm), _ptr(self.w_router), _ptr(self.bias),
                            _ptr(self.w13_codes), _ptr(self.w13_scales), _ptr(self.w2_codes), _ptr(self.w2_scales),
                            _ptr(y), _ptr(self.workspace), self.workspace_bytes_mx(T), s, events)
        if st != MOE_OK:
            raise MoeError(st, "moe_forward_mx")
        return y

    def views_mx(self, T):
        st, v, mv = moe_workspace_views_mx(self.shape(T), _ptr(self.workspace), self.workspace_bytes_mx(T))
        if st != MOE_OK:
            raise MoeError(st, "moe_workspace_views_mx")
        return v, mv

    def views(self, T):
        st, v = moe_workspace_views(self.shape(T), _ptr(self.workspace), self.workspace_bytes(T))
        if st != MOE_OK:
            raise MoeError(st, "moe_workspace_views")
        return v

    def view_tensor(self, T, name, dtype, shape_):
        """A torch view of one intermediate tensor inside the workspace."""
        import torch
        v = self.views(T)
        off = getattr(v, name) - self.workspace.data_ptr()
        n = 1
        for d in shape_:
            n *= d
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return self.workspace[off:off + nbytes].view(dtype).view(*shape_)

    def device_status(self, T, stream=None):
        import torch
        s = stream if stream is not None else torch.cuda.current_stream(self.device).cuda_stream
        return moe_device_status(_ptr(self.workspace), self.workspace_bytes(T), s)
