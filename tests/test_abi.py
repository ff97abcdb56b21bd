"""The C-ABI library loads on a host without a GPU, exports every entry point
include/moe.h declares, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

from mixture_experts_layer_rmsnorm_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_entry_points():
    txt = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", txt)))


def test_library_exports_every_declared_symbol():
    lib = binding.load()
    names = declared_entry_points()
    assert {"moe_forward", "moe_workspace_size", "moe_route_debug", "moe_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/moe.h but not exported"


def test_status_strings():
    for code in range(7):
        assert binding.moe_status_string(code)
    assert "unknown" in binding.moe_status_string(99)


def test_workspace_size_and_shape_checks():
    st, n = binding.moe_workspace_size(binding.shape(4096, 4096, 4096, 64, 8))
    assert st == binding.MOE_OK and n > 3 * 33728 * 4096 * 2
    bad = [
        (binding.shape(4, 100, 256, 8, 2), binding.MOE_ERR_UNSUPPORTED),   # H not a multiple of 128
        (binding.shape(4, 128, 200, 8, 2), binding.MOE_ERR_UNSUPPORTED),   # I not a multiple of 64
        (binding.shape(4, 128, 256, 8, 9), binding.MOE_ERR_INVALID_ARG),   # top_k > E
        (binding.shape(4, 128, 256, 2048, 2), binding.MOE_ERR_UNSUPPORTED),  # E > 1024
        (binding.shape(4, 128, 256, 64, 33), binding.MOE_ERR_UNSUPPORTED),  # top_k > 32
        (binding.shape(-1, 128, 256, 8, 2), binding.MOE_ERR_INVALID_ARG),
        (binding.shape(4, 128, 256, 8, 2, eps=-1.0), binding.MOE_ERR_INVALID_ARG),
        (binding.shape(4, 128, 256, 8, 2, eps=float("nan")), binding.MOE_ERR_INVALID_ARG),
    ]
    for s, want in bad:
        st, _ = binding.moe_workspace_size(s)
        assert st == want, (s.H, s.I, s.E, s.top_k, st)


def test_shape_rule_at_its_edges():
    """The supported shapes: H a multiple of 128 (the down GEMM's 128-feature
    weight tile) up to 16384 (the router's shared-memory rows of h); I a
    multiple of 64 (the gate/up GEMM's 64-feature unit, the down GEMM's
    64-element K block) up to 16384, and of 128 for the block-scaled layers
    (128-element scale tiles); 1 <= top_k <= min(E, 32) (one lane of the
    selecting warp per selected expert); E <= 1024."""
    ok, uns, inv = binding.MOE_OK, binding.MOE_ERR_UNSUPPORTED, binding.MOE_ERR_INVALID_ARG
    cases = [
        ((4, 128, 64, 8, 2), ok), ((4, 128, 192, 8, 2), ok), ((4, 128, 96, 8, 2), uns), ((4, 128, 32, 8, 2), uns),
        ((4, 16384, 256, 8, 2), ok), ((4, 16512, 256, 8, 2), uns), ((4, 128, 16384, 8, 2), ok),
        ((4, 128, 16448, 8, 2), uns), ((4, 128, 256, 1024, 2), ok), ((4, 128, 256, 1025, 2), uns),
        ((4, 128, 256, 64, 32), ok), ((4, 128, 256, 64, 33), uns), ((4, 128, 256, 8, 8), ok),
        ((4, 128, 256, 8, 9), inv), ((4, 128, 256, 8, 0), inv), ((4, 128, 256, 1, 1), ok),
    ]
    for (T, H, I, E, k), want in cases:
        st, _ = binding.moe_workspace_size(binding.shape(T, H, I, E, k))
        assert st == want, ((T, H, I, E, k), st, want)
    # block-scaled layers: I a multiple of 128
    for (T, H, I, E, k), want in [((4, 256, 192, 8, 2), uns), ((4, 256, 384, 8, 2), ok), ((4, 256, 128, 8, 2), ok)]:
        st, _ = binding.moe_workspace_size_mx(binding.shape(T, H, I, E, k))
        assert st == want, ((T, H, I, E, k), st, want)
        st, _ = binding.moe_mx_weight_sizes(binding.shape(T, H, I, E, k))
        assert st == want


def test_static_scratch_size_and_limit_without_a_gpu():
    st, cap = binding.moe_static_scratch_bytes()
    assert st == binding.MOE_OK and cap == 64 << 20
    _, need128 = binding.moe_workspace_size(binding.shape(128, 4096, 4096, 64, 8))
    _, need129 = binding.moe_workspace_size(binding.shape(129, 4096, 4096, 64, 8))
    assert need128 <= cap < need129
    A = 1 << 20  # never dereferenced: the size check comes first
    assert binding.moe_forward_static_scratch(binding.shape(129, 4096, 4096, 64, 8), A, A, A, None, A, A, A,
                                              None) == binding.MOE_ERR_WORKSPACE


def test_kernels_per_call_host_checks():
    st, n = binding.moe_kernels_per_call(binding.shape(0, 128, 256, 8, 2))
    assert st == binding.MOE_OK and n == 0
    st, _ = binding.moe_kernels_per_call(binding.shape(4, 100, 256, 8, 2))
    assert st == binding.MOE_ERR_UNSUPPORTED
    # norm/router, top-k + align, gather, the two GEMMs, combine; no gather on
    # the decode tile plan (the gate/up GEMM reads the rows of h itself: one
    # token through its tensor map, more through its row warps); large T: the
    # top-k and align take three kernels
    st, n = binding.moe_kernels_per_call(binding.shape(4, 128, 256, 8, 2))
    assert st == binding.MOE_OK and n == 5
    st, n = binding.moe_kernels_per_call(binding.shape(1, 128, 256, 8, 2))
    assert st == binding.MOE_OK and n == 5
    st, n = binding.moe_kernels_per_call(binding.shape(200, 128, 256, 8, 2))
    assert st == binding.MOE_OK and n == 6
    st, n = binding.moe_kernels_per_call(binding.shape(4096, 128, 256, 8, 2))
    assert st == binding.MOE_OK and n == 8
    s4 = binding.shape(4, 128, 256, 8, 2)
    assert binding.moe_kernels_per_call_of(s4, binding.MOE_CALL_FORWARD) == (binding.MOE_OK, 5)
    assert binding.moe_kernels_per_call_of(s4, binding.MOE_CALL_FORWARD_FUSED_FRONT) == (binding.MOE_OK, 4)
    assert binding.moe_kernels_per_call_of(s4, binding.MOE_CALL_FORWARD_MX) == (binding.MOE_OK, 7)
    assert binding.moe_kernels_per_call_of(s4, binding.MOE_CALL_FORWARD_MXFP4) == (binding.MOE_OK, 7)
    assert binding.moe_kernels_per_call_of(s4, binding.MOE_CALL_FORWARD_MXFP4A4) == (binding.MOE_OK, 7)
    assert binding.moe_kernels_per_call_of(s4, binding.MOE_CALL_FORWARD_NVFP4) == (binding.MOE_OK, 7)
    assert binding.moe_kernels_per_call_of(s4, 8)[0] == binding.MOE_ERR_INVALID_ARG
    assert binding.moe_kernels_per_call_of(s4, binding.MOE_CALL_FORWARD_FUSED_COMBINE) == (binding.MOE_OK, 5)
    assert binding.moe_kernels_per_call_of(s4, binding.MOE_CALL_FORWARD_FUSED_MLP) == (binding.MOE_OK, 5)
    s1 = binding.shape(1, 128, 256, 8, 2)
    assert binding.moe_kernels_per_call_of(s1, binding.MOE_CALL_FORWARD_FUSED_MLP) == (binding.MOE_OK, 4)
    s4096 = binding.shape(4096, 128, 256, 8, 2)
    assert binding.moe_kernels_per_call_of(s4096, binding.MOE_CALL_FORWARD_FUSED_COMBINE) == (binding.MOE_OK, 7)
    assert binding.moe_kernels_per_call_of(s4096, binding.MOE_CALL_FORWARD_FUSED_MLP)[0] == \
        binding.MOE_ERR_UNSUPPORTED
    # the fused MLP entry point refuses the prefill tile plan before touching a pointer
    _, need = binding.moe_workspace_size(s4096)
    A = 1 << 20
    assert binding.moe_forward_fused_mlp(s4096, A, A, A, None, A, A, A, A, need, None) == \
        binding.MOE_ERR_UNSUPPORTED
    assert binding.moe_kernels_per_call_of(s4, 8)[0] == binding.MOE_ERR_INVALID_ARG
    assert binding.moe_kernels_per_call_of(s4, -1)[0] == binding.MOE_ERR_INVALID_ARG


def test_selftest_wait_timeout_rejects_bad_arguments_without_a_gpu():
    A = 1 << 20
    assert binding.moe_selftest_wait_timeout(None, 64, 1000, None) == binding.MOE_ERR_INVALID_ARG
    assert binding.moe_selftest_wait_timeout(A, 32, 1000, None) == binding.MOE_ERR_INVALID_ARG
    assert binding.moe_selftest_wait_timeout(A + 16, 64, 1000, None) == binding.MOE_ERR_INVALID_ARG
    assert binding.moe_selftest_wait_timeout(A, 64, 0, None) == binding.MOE_ERR_INVALID_ARG
    assert binding.moe_selftest_wait_timeout(A, 64, 2_000_000_000, None) == binding.MOE_ERR_INVALID_ARG


def test_qk_norm_rejects_bad_arguments_without_a_gpu():
    A = 1 << 20
    ok = dict(T=4, Hq=2, Hk=1, D=128, q=A, k=A, qw=A, kw=A, wb=0.0, eps=1e-6)

    def call(**kw):
        a = dict(ok, **kw)
        return binding.moe_qk_norm(a["T"], a["Hq"], a["Hk"], a["D"], a["q"], a["k"], a["qw"], a["kw"], a["wb"],
                                   a["eps"], None)

    assert call(T=0) == binding.MOE_OK                       # nothing to do, nothing touched
    assert call(Hq=0, Hk=0) == binding.MOE_OK
    for bad in (dict(D=100), dict(D=32), dict(T=-1), dict(Hq=-1), dict(q=None), dict(kw=None), dict(q=A + 8),
                dict(eps=-1.0), dict(eps=float("nan")), dict(wb=float("inf"))):
        assert call(**bad) == binding.MOE_ERR_INVALID_ARG, bad


def test_forward_rejects_bad_arguments_without_a_gpu():
    # fake, aligned, never-dereferenced addresses: every case fails validation first
    s = binding.shape(4, 128, 256, 8, 2)
    _, need = binding.moe_workspace_size(s)
    A = 1 << 20
    args = dict(x=A, g=A, wr=A, b=None, w13=A, w2=A, y=A, ws=A, nbytes=need)

    def call(**kw):
        a = dict(args, **kw)
        return binding.moe_forward(s, a["x"], a["g"], a["wr"], a["b"], a["w13"], a["w2"], a["y"], a["ws"],
                                   a["nbytes"], None)

    assert call(nbytes=need - 1) == binding.MOE_ERR_WORKSPACE
    assert call(x=None) == binding.MOE_ERR_INVALID_ARG
    assert call(w13=None) == binding.MOE_ERR_INVALID_ARG
    assert call(y=None) == binding.MOE_ERR_INVALID_ARG
    assert call(x=A + 2) == binding.MOE_ERR_INVALID_ARG       # not 16-byte aligned
    assert call(ws=A + 16) == binding.MOE_ERR_INVALID_ARG     # workspace not 256-byte aligned
    assert binding.moe_forward(binding.shape(4, 100, 256, 8, 2), A, A, A, None, A, A, A, A, need, None) == \
        binding.MOE_ERR_UNSUPPORTED
    # T = 0 is a no-op that touches no pointer
    assert binding.moe_forward(binding.shape(0, 128, 256, 8, 2), None, None, None, None, None, None, None, None, 0,
                               None) == binding.MOE_OK


def test_mxfp4_sizes_and_argument_checks_without_a_gpu():
    s = binding.shape(4, 256, 384, 8, 2)
    st, (c13, s13, c2, s2) = binding.moe_mxfp4_weight_sizes(s)
    assert st == binding.MOE_OK
    assert (c13, c2) == (8 * 2 * 384 * 256 // 2, 8 * 256 * 384 // 2)  # two E2M1 codes per byte
    assert (s13, s2) == binding.moe_mx_weight_sizes(s)[1][1::2]      # the MXFP8 scale tiles
    _, need = binding.moe_workspace_size_mx(s)
    A = 1 << 20

    def fwd(w13c=A, w2c=A, w13s=A):
        return binding.moe_forward_mxfp4(s, A, A, A, None, w13c, w13s, w2c, A, A, A, need, None)

    assert fwd(w13c=A + 16) == binding.MOE_ERR_INVALID_ARG  # packed codes: 32-byte aligned
    s512 = binding.shape(4, 256, 512, 8, 2)
    _, need512 = binding.moe_workspace_size_mx(s512)
    assert binding.moe_forward_mxfp4a4(s512, A, A, A, None, A + 16, A, A, A, A, A, need512, None) == \
        binding.MOE_ERR_INVALID_ARG
    # the MXFP4 layer: H and I multiples of 128 (this shape has I = 384; I = 192 is refused)
    assert binding.moe_forward_mxfp4a4(s, A, A, A, None, A + 16, A, A, A, A, A, need, None) == \
        binding.MOE_ERR_INVALID_ARG
    s192 = binding.shape(4, 256, 192, 8, 2)
    assert binding.moe_forward_mxfp4a4(s192, A, A, A, None, A, A, A, A, A, A, 1 << 40, None) == \
        binding.MOE_ERR_UNSUPPORTED
    assert fwd(w2c=A + 16) == binding.MOE_ERR_INVALID_ARG
    assert fwd(w13s=None) == binding.MOE_ERR_INVALID_ARG
    assert binding.moe_forward_mxfp4(s, A, A, A, None, A, A, A, A, A, A, need - 1, None) == binding.MOE_ERR_WORKSPACE
    assert binding.moe_mxfp4_quantize_weights(s, A, A, A + 16, A, A, A, None) == binding.MOE_ERR_INVALID_ARG
    assert binding.moe_mxfp4_quantize_weights(s, A, A, A, A, A + 48, A, None) == binding.MOE_ERR_INVALID_ARG
    assert binding.moe_mxfp4_quantize_weights(binding.shape(4, 100, 384, 8, 2), A, A, A, A, A, A, None) == \
        binding.MOE_ERR_UNSUPPORTED


def test_nvfp4_sizes_and_argument_checks_without_a_gpu():
    s = binding.shape(4, 256, 512, 8, 2)
    st, (c13, s13, c2, s2) = binding.moe_nvfp4_weight_sizes(s)
    assert st == binding.MOE_OK
    assert (c13, c2) == (8 * 2 * 512 * 256 // 2, 8 * 256 * 512 // 2)
    assert (s13, s2) == (8 * 2 * 512 * 256 // 16, 8 * 256 * 512 // 16)  # one E4M3 byte per 16 elements
    _, need = binding.moe_workspace_size_mx(s)
    A = 1 << 20

    def fwd(**kw):
        a = dict(c13=A, g13=A, g2=A, nbytes=need, shape=s)
        a.update(kw)
        return binding.moe_forward_nvfp4(a["shape"], A, A, A, None, a["c13"], A, a["g13"], A, A, a["g2"], A, A,
                                         a["nbytes"], None)

    assert fwd(c13=A + 16) == binding.MOE_ERR_INVALID_ARG
    assert fwd(g13=None) == binding.MOE_ERR_INVALID_ARG
    assert fwd(g2=A + 2) == binding.MOE_ERR_INVALID_ARG
    assert fwd(nbytes=need - 1) == binding.MOE_ERR_WORKSPACE
    assert fwd(shape=binding.shape(4, 256, 192, 8, 2), nbytes=1 << 40) == binding.MOE_ERR_UNSUPPORTED
    q = binding.moe_nvfp4_quantize_weights
    assert q(s, A, A, A + 16, A, A, A, A, A, None) == binding.MOE_ERR_INVALID_ARG
    assert q(s, A, A, A, A, None, A, A, A, None) == binding.MOE_ERR_INVALID_ARG
    assert q(s, A, A, A, A, A, A, A, A + 1, None) == binding.MOE_ERR_INVALID_ARG


def test_route_debug_rejects_bad_arguments_without_a_gpu():
    s = binding.shape(4, 128, 256, 8, 2)
    _, need = binding.moe_workspace_size(s)
    A = 1 << 20
    cap = 4 * 2 + 8 * 15
    assert binding.moe_route_debug(s, A, A, A, None, 0, A, A, A, A, cap, A, need, None) == binding.MOE_ERR_INVALID_ARG
    assert binding.moe_route_debug(s, A, A, A, None, 257, A, A, A, A, 10**6, A, need, None) == \
        binding.MOE_ERR_INVALID_ARG
    assert binding.moe_route_debug(s, A, A, A, None, 16, A, A, A, A, cap - 1, A, need, None) == \
        binding.MOE_ERR_INVALID_ARG
    assert binding.moe_route_debug(s, A, A, A, None, 16, None, A, A, A, cap, A, need, None) == \
        binding.MOE_ERR_INVALID_ARG


def test_workspace_views_layout():
    T, H, I, E, k = 100, 256, 384, 16, 4
    s = binding.shape(T, H, I, E, k)
    _, need = binding.moe_workspace_size(s)
    base = 1 << 30
    st, v = binding.moe_workspace_views(s, base, need)
    assert st == binding.MOE_OK
    assert v.P_max == T * k + E * 15
    ptrs = [v.error_word, v.h, v.logits, v.topk_ids, v.topk_w, v.counts, v.offsets, v.sorted_ids, v.slot_of, v.xg,
            v.act, v.out_rows]
    assert ptrs == sorted(ptrs) and all(p % 256 == 0 for p in ptrs)
    assert v.out_rows + v.P_max * H * 2 <= base + need
    assert v.act + v.P_max * I * 2 <= v.out_rows
    st, _ = binding.moe_workspace_views(s, base, need - 1)
    assert st == binding.MOE_ERR_WORKSPACE
