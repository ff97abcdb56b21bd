"""GPU parity on small workloads the oracle computes completely.

Each case runs the whole layer through the C ABI and compares it with the CPU
oracle on the same seeded inputs: h, router logits, expert ids and the align
outputs bit for bit; the expert ids also against an fp64 selection (within the
fp32 router's summation error of a tie); routing weights within fp32 rounding;
every real row's SwiGLU activation and expert output element by element (one
bf16 step, at least 99% bit-equal); the layer output within the tolerance of
the fp64 oracle.
The shapes span several weight tiles, several token chunks per expert, ragged
tails, both launch plans (decode tiles and prefill tiles) and the degenerate
cases (T = 0, T = 1, E = 1, k = E, unnormalised weights, a router bias).
"""
import dataclasses

import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
from mixture_experts_layer_rmsnorm_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

CASES = [
    # name, T, H, I, E, k, renorm, zipf, seed
    ("tiny", 4, 128, 256, 8, 2, True, None, 0),
    ("T1", 1, 256, 256, 16, 4, True, None, 3),
    ("T2_wide_rows", 2, 5120, 256, 12, 3, True, None, 13),
    ("T3_bias", 3, 384, 256, 20, 5, True, 1.2, 14),
    ("ragged_decode", 37, 256, 384, 16, 4, True, None, 1),
    ("deep_k", 64, 1024, 512, 8, 2, True, None, 2),
    ("prefill_chunks", 1024, 256, 256, 4, 2, True, None, 4),
    ("prefill_ragged_norenorm", 300, 384, 128, 6, 3, False, None, 5),
    ("prefill_pairs_ragged", 700, 512, 384, 5, 2, True, None, 10),
    ("prefill_skewed", 512, 256, 256, 16, 4, True, 1.2, 11),
    ("skewed_bias", 96, 256, 256, 32, 6, True, 1.2, 7),
    ("multichunk_50_per_expert", 200, 256, 256, 8, 2, True, None, 9),
    ("single_expert", 20, 128, 128, 1, 1, True, None, 6),
    ("k_equals_E", 9, 128, 256, 4, 4, True, None, 8),
    # I a multiple of 64 but not of 128: an odd count of 64-feature gate/up
    # tiles and of 64-element K blocks in the down GEMM
    ("I192_decode", 40, 256, 192, 8, 2, True, None, 15),
    ("I320_prefill_odd_tiles", 512, 256, 320, 8, 2, True, None, 16),
    # the decode tile plan (T * k <= 16 E) under skewed routing: hot experts
    # with 45-64 rows take two or three 32-row chunks (the row warps' chunk
    # offsets and padded tails)
    ("decode_plan_hot_experts", 64, 256, 256, 16, 4, True, 1.2, 20),
    # 64 align blocks x 256 experts: more per-block counts than the scan
    # stages in shared memory (it reads them from global memory)
    ("align_counts_unstaged", 2048, 128, 128, 256, 2, True, None, 17),
]


@pytest.fixture(scope="module")
def o():
    return oracle.default()


def _layer_inputs(T, H, I, E, k, renorm, zipf, seed):
    cfg = inputs.LayerConfig(T=T, H=H, I=I, E=E, top_k=k, renormalize=renorm, seed=seed, zipf_bias=zipf)
    return inputs.make_layer_inputs(cfg)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_layer_parity(case, o):
    _, T, H, I, E, k, renorm, zipf, seed = case
    li = _layer_inputs(T, H, I, E, k, renorm, zipf, seed)
    dl = gu.DeviceLayer(li)
    g = dl.run(li.x)
    ids = gu.check_routing(o, li, li.x, g, label=case[0])
    # expert intermediates of every real row: SwiGLU activations and expert outputs, element by element
    real = np.nonzero(g["sorted"] < T * k)[0]
    gu.check_expert_rows(o, li, dl, T, g, ids, real, label=case[0])
    gu.check_output(o, li, li.x, g["y"])


FRONT_CASES = [c for c in CASES if c[1] <= binding.MOE_FRONT_MAX_T and c[4] <= binding.MOE_FRONT_MAX_E]


@pytest.mark.parametrize("case", FRONT_CASES, ids=[c[0] for c in FRONT_CASES])
def test_fused_front_parity(case, o):
    """The single-launch front end: the same routing bits as the oracle, and the
    same output bits as the multi-launch path."""
    _, T, H, I, E, k, renorm, zipf, seed = case
    li = _layer_inputs(T, H, I, E, k, renorm, zipf, seed)
    dl = gu.DeviceLayer(li)
    g = dl.run(li.x, fused_front=True)
    gu.check_routing(o, li, li.x, g)
    gu.check_output(o, li, li.x, g["y"])
    ref = dl.run(li.x)
    assert np.array_equal(g["y"], ref["y"]), "fused front end and multi-launch path disagree"
    assert np.array_equal(g["slot"], ref["slot"])


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fused_combine_parity(case, o):
    """The combine in the down GEMM's epilogue: the same output bits as the
    separate combine kernel (same rows, same order, same fp32 arithmetic), so
    within the oracle's tolerance too; and the same bits on a second call
    (arrival counters are zeroed per call)."""
    _, T, H, I, E, k, renorm, zipf, seed = case
    li = _layer_inputs(T, H, I, E, k, renorm, zipf, seed)
    dl = gu.DeviceLayer(li)
    ref = dl.run(li.x)
    xd = gu.dev_bf16(li.x)
    for _ in range(2):
        y = dl.layer.forward(xd, fused_combine=True)
        torch.cuda.synchronize()
        st, det = dl.layer.device_status(T)
        assert st == binding.MOE_OK, (st, det)
        assert np.array_equal(y.cpu().numpy().view(np.uint16), ref["y"]), "fused combine differs from the kernel"
    gu.check_output(o, li, li.x, ref["y"])


SMALL_PLAN_CASES = [c for c in CASES if c[1] * c[5] <= 16 * c[4]]  # T * top_k <= 16 * E: the decode tile plan


@pytest.mark.parametrize("case", SMALL_PLAN_CASES, ids=[c[0] for c in SMALL_PLAN_CASES])
def test_fused_mlp_parity(case, o):
    """Both expert GEMMs in one launch: the same K split as the separate GEMMs,
    so the same output bits as moe_forward on two calls in a row (completion
    counters are cleared per call), hence within the oracle's tolerance too."""
    _, T, H, I, E, k, renorm, zipf, seed = case
    li = _layer_inputs(T, H, I, E, k, renorm, zipf, seed)
    dl = gu.DeviceLayer(li)
    ref = dl.run(li.x)
    xd = gu.dev_bf16(li.x)
    for _ in range(2):
        y = dl.layer.forward(xd, fused_mlp=True)
        torch.cuda.synchronize()
        st, det = dl.layer.device_status(T)
        assert st == binding.MOE_OK, (st, det)
        assert np.array_equal(y.cpu().numpy().view(np.uint16), ref["y"]), "fused MLP differs from the split GEMMs"
    gu.check_output(o, li, li.x, ref["y"])


def test_fused_mlp_rejects_prefill_plan():
    li = _layer_inputs(200, 128, 128, 4, 2, True, None, 0)  # 100 rows per expert: the prefill tile plan
    dl = gu.DeviceLayer(li)
    with pytest.raises(binding.MoeError) as ei:
        dl.layer.forward(gu.dev_bf16(li.x), fused_mlp=True)
    assert ei.value.status == binding.MOE_ERR_UNSUPPORTED


def test_fused_front_rejects_large_batches():
    li = _layer_inputs(80, 128, 128, 4, 2, True, None, 0)
    dl = gu.DeviceLayer(li)
    with pytest.raises(binding.MoeError) as ei:
        dl.run(li.x, fused_front=True)
    assert ei.value.status == binding.MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("T", [5, 64, 300], ids=["fused_topk_T5", "fused_topk_T64", "multi_cta_T300"])
def test_tied_logits_pick_the_lower_expert(o, T):
    """Exactly equal logits are selected lowest expert index first, as the
    oracle's top-k does, in the single-CTA top-k + align and in the multi-CTA
    top-k.  Even tokens repeat token 0; with its normalised row u, experts 2, 5
    and 11 get the router row u (equal largest logits), experts 7, 9 and 13 a
    zero row (equal zero logits) and the others negative multiples of u, so
    those tokens select [2, 5, 11, 7, 9, 13] in that order."""
    E, k = 16, 6
    li = _layer_inputs(T, 256, 256, E, k, True, None, 21)
    x = li.x.copy()
    x[0::2] = x[0]
    h32, _, _ = o.route_f32(x[:1], li.g, li.cfg.eps, li.w_router, None)
    u = gu.widen(h32[0]).astype(np.float32) / 64.0
    wr = li.w_router.copy()
    for e in range(E):
        wr[e] = -(1.0 + e / 8.0) * u
    wr[[2, 5, 11]] = u
    wr[[7, 9, 13]] = 0.0
    li = dataclasses.replace(li, x=x, w_router=wr)
    dl = gu.DeviceLayer(li)
    g = dl.run(x)
    ids = gu.check_routing(o, li, x, g)
    assert (ids[0::2] == np.array([2, 5, 11, 7, 9, 13])).all()
    gu.check_output(o, li, x, g["y"])


@pytest.mark.parametrize("T", [3, 300], ids=["fused_topk", "multi_cta_topk"])
def test_non_finite_input_is_reported(o, T):
    """A token whose row holds an infinity has NaN logits, so no expert can be
    selected: the align reports MOE_ERR_DEVICE (the single-CTA form leaves an
    empty routing, the multi-CTA form routes the token to expert 0), nothing
    faults, and the next call on the same workspace is clean."""
    li = _layer_inputs(T, 256, 256, 8, 2, True, None, 22)
    bad = li.x.copy()
    bad[T // 2, 17] = 0x7F80  # +inf
    dl = gu.DeviceLayer(li)
    L = dl.layer
    L.forward(gu.dev_bf16(bad))
    torch.cuda.synchronize()
    st, det = L.device_status(T)
    assert st == binding.MOE_ERR_DEVICE, (st, det)
    g = dl.run(li.x)
    gu.check_routing(o, li, li.x, g)


def test_zero_tokens_is_a_noop():
    li = _layer_inputs(4, 128, 128, 4, 2, True, None, 0)
    dl = gu.DeviceLayer(li)
    L = dl.layer
    x = torch.empty((0, 128), dtype=torch.int16, device="cuda")
    y = torch.empty((0, 128), dtype=torch.int16, device="cuda")
    st = binding.moe_forward(L.shape(0), x.data_ptr(), L.g_norm.data_ptr(), L.w_router.data_ptr(), None,
                             L.w13.data_ptr(), L.w2.data_ptr(), y.data_ptr(), L.workspace.data_ptr(),
                             L.workspace.numel(), torch.cuda.current_stream().cuda_stream)
    assert st == binding.MOE_OK


def test_repeat_calls_are_identical(o):
    # same inputs, same bits: the permutation and the accumulation order are fixed
    li = _layer_inputs(50, 256, 256, 8, 2, True, None, 11)
    dl = gu.DeviceLayer(li)
    a = dl.run(li.x)
    b = dl.run(li.x)
    for key in ("y", "h", "logits", "ids", "w", "offsets", "sorted", "slot"):
        assert np.array_equal(a[key], b[key]), key


def test_route_debug_entry_point(o):
    li = _layer_inputs(33, 256, 256, 16, 4, True, None, 12)
    dl = gu.DeviceLayer(li)
    L = dl.layer
    T, E, k = 33, 16, 4
    for pad in (1, 16, 128):
        cap = T * k + E * (pad - 1)
        ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, k), dtype=torch.float32, device="cuda")
        offs = torch.empty(E + 1, dtype=torch.int32, device="cuda")
        srt = torch.full((cap,), -7, dtype=torch.int32, device="cuda")
        xd = gu.dev_bf16(li.x)
        st = binding.moe_route_debug(L.shape(T), xd.data_ptr(), L.g_norm.data_ptr(), L.w_router.data_ptr(), None,
                                     pad, ids.data_ptr(), w.data_ptr(), offs.data_ptr(), srt.data_ptr(), cap,
                                     L.workspace.data_ptr(), L.workspace.numel(),
                                     torch.cuda.current_stream().cuda_stream)
        assert st == binding.MOE_OK
        torch.cuda.synchronize()
        _, l32, _ = o.route_f32(li.x, li.g, li.cfg.eps, li.w_router, None)
        ids_ref = o.topk(l32, k)
        assert np.array_equal(ids.cpu().numpy(), ids_ref)
        counts, offsets, sorted_ids, _ = o.align(ids_ref, E, pad)
        assert np.array_equal(offs.cpu().numpy(), offsets)
        assert np.array_equal(srt.cpu().numpy()[:offsets[-1]], sorted_ids)
