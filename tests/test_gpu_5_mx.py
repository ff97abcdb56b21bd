"""GPU parity of the FP8 layer (MXFP8 expert weights, block-scaled tcgen05 MMA).

Every quantization decision is exact on both sides, so the E4M3 codes and E8M0
scales of the weights and of the gathered token rows are compared bit for bit
with the oracle's quantizer; the routing bit for bit as in the bf16 layer
(lists padded to 32 rows); the layer output against the oracle's FP8 layer
(the same recipe, fp64 arithmetic) within the layer tolerance.
"""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
from mixture_experts_layer_rmsnorm_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

CASES = [
    # name, T, H, I, E, k, renorm, zipf, seed
    ("mx_tiny", 4, 128, 256, 8, 2, True, None, 0),
    ("mx_T1", 1, 256, 256, 16, 4, True, None, 3),
    ("mx_ragged_decode", 37, 256, 384, 16, 4, True, None, 1),
    ("mx_mid_multichunk", 200, 256, 256, 8, 2, True, None, 9),
    ("mx_bias_norenorm", 3, 384, 256, 20, 5, False, 1.2, 14),
    ("mx_deep_k", 64, 1024, 512, 8, 2, True, None, 2),
    # prefill plan: 128-token units, several chunks per expert, ragged tails
    ("mx_prefill_chunks", 1024, 256, 256, 4, 2, True, None, 4),
    ("mx_prefill_ragged_norenorm", 300, 384, 128, 6, 3, False, None, 5),
    ("mx_prefill_skewed", 512, 256, 256, 16, 4, True, 1.2, 11),
]


@pytest.fixture(scope="module")
def o():
    return oracle.default()


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_mx_layer_parity(case, o):
    _, T, H, I, E, k, renorm, zipf, seed = case
    cfg = inputs.LayerConfig(T=T, H=H, I=I, E=E, top_k=k, renormalize=renorm, seed=seed, zipf_bias=zipf)
    li = inputs.make_layer_inputs(cfg)
    dl = gu.DeviceLayer(li)
    L = dl.layer
    L.quantize_mx()
    torch.cuda.synchronize()
    # weights: codes and scales bit for bit
    w13c, w13s = o.mx_quantize(li.w13)
    w2c, w2s = o.mx_quantize(li.w2)
    assert np.array_equal(L.w13_codes.cpu().numpy().reshape(E, 2 * I, H), w13c)
    assert np.array_equal(L.w2_codes.cpu().numpy().reshape(E, H, I), w2c)
    s13 = gu.ungroup_mx_scales(L.w13_scales.cpu().numpy(), E * 2 * I, H)[gu.w13_scale_rows(E, I)]
    assert np.array_equal(s13.reshape(E, 2 * I, H // 32), w13s)
    s2 = gu.ungroup_mx_scales(L.w2_scales.cpu().numpy(), E * H, I)
    assert np.array_equal(s2.reshape(E, H, I // 32), w2s)

    xd = gu.dev_bf16(li.x)
    y = L.forward_mx(xd)
    torch.cuda.synchronize()
    st, det = L.device_status(T)
    assert st == binding.MOE_OK, (st, det)
    v, mv = L.views_mx(T)
    ws0 = L.workspace.data_ptr()

    def view(addr, dtype, shape_):
        n = int(np.prod(shape_)) * torch.empty((), dtype=dtype).element_size()
        return L.workspace[addr - ws0: addr - ws0 + n].view(dtype).view(*shape_).cpu().numpy()

    g = {"h": view(v.h, torch.int16, (T, H)).view(np.uint16), "logits": view(v.logits, torch.float32, (T, E)),
         "ids": view(v.topk_ids, torch.int32, (T, k)), "w": view(v.topk_w, torch.float32, (T, k)),
         "counts": view(v.counts, torch.int32, (E,)), "offsets": view(v.offsets, torch.int32, (E + 1,))}
    P = int(g["offsets"][-1])
    g["sorted"] = view(v.sorted_ids, torch.int32, (v.P_max,))[:P]
    g["slot"] = view(v.slot_of, torch.int32, (T * k,))
    gu.check_routing(o, li, li.x, g, pad=32)
    # gathered token rows: codes and scales bit for bit on the real rows; the
    # scales are grouped by the GEMMs' token chunks (bn rows of an expert)
    # the gate/up GEMM's token rows per unit (its scale chunks): 32 / 64 by
    # decode plan, 128 or 256 in prefill; a chunk's scales take ceil(bn / 128) tiles
    bn = mv.x_chunk_rows
    small_mid = 32 if T * k <= 16 * E else 64 if T * k <= 64 * E else None
    assert bn == small_mid if small_mid else bn in (128, 256)
    G = -(-bn // 128)
    n_groups = 2 * (v.P_max // 32)
    xcodes = view(mv.x_codes, torch.uint8, (v.P_max, H))
    xs = gu.ungroup_mx_scales(view(mv.x_scales, torch.uint8, (n_groups * (H // 128) * 512,)), n_groups * 128, H)
    real = np.nonzero(g["sorted"] < T * k)[0]
    hc, hs = o.mx_quantize(g["h"][g["sorted"][real] // k])
    assert np.array_equal(xcodes[real], hc)
    offs = g["offsets"]
    chunk0 = np.concatenate([[0], np.cumsum(-(-np.diff(offs) // bn))])  # chunks before each expert
    e_of = np.searchsorted(offs, real, side="right") - 1
    within = real - offs[e_of]
    srow = (chunk0[e_of] + within // bn) * 128 * G + within % bn
    assert np.array_equal(xs[srow], hs)
    # the layer output against the oracle's FP8 layer
    r = o.moe_forward_mx(li.x, li.g, li.w_router, li.bias, w13c, w13s, w2c, w2s, k, renorm, cfg.eps)
    yg = gu.widen(y.cpu().numpy().view(np.uint16))
    err = yg - r["y64"]
    rel = np.linalg.norm(err) / np.linalg.norm(r["y64"])
    assert rel <= gu.REL_FRO_TOL, f"relative Frobenius error {rel:.3e}"
    assert np.abs(err).max() <= gu.MAX_ABS_TOL


def test_mx_rejects_more_than_256_experts():
    cfg = inputs.LayerConfig(T=4, H=128, I=128, E=300, top_k=2, seed=0)
    li = inputs.make_layer_inputs(cfg)
    dl = gu.DeviceLayer(li)
    dl.layer.quantize_mx()
    with pytest.raises(binding.MoeError) as ei:
        dl.layer.forward_mx(gu.dev_bf16(li.x))
    assert ei.value.status == binding.MOE_ERR_UNSUPPORTED
