"""GPU parity of the block-scaled layers: MXFP8 expert weights (E4M3 codes) and
MXFP4 expert weights (E2M1 codes, two per byte), both with MXFP8 token rows and
activations, on the block-scaled tcgen05 MMA.

Every quantization decision is exact on both sides, so the weight codes and
E8M0 scales and those of the gathered token rows are compared bit for bit with
the oracle's quantizers; the routing bit for bit as in the bf16 layer (lists
padded to 32 rows); the layer output against the oracle's layer of the same
format (the same recipe, fp64 arithmetic) within the layer tolerance.
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
    ("mx_multichunk_50_per_expert", 200, 256, 256, 8, 2, True, None, 9),
    ("mx_bias_norenorm", 3, 384, 256, 20, 5, False, 1.2, 14),
    ("mx_deep_k", 64, 1024, 512, 8, 2, True, None, 2),
    # prefill plan: 128-token units, several chunks per expert, ragged tails
    ("mx_prefill_chunks", 1024, 256, 256, 4, 2, True, None, 4),
    ("mx_prefill_ragged_norenorm", 300, 384, 128, 6, 3, False, None, 5),
    ("mx_prefill_skewed", 512, 256, 256, 16, 4, True, 1.2, 11),
    # H and I multiples of 256: no partial last stage in the packed-FP4 layers
    ("a4_ragged_decode", 37, 256, 512, 16, 4, True, None, 21),
    ("a4_bias_norenorm", 3, 512, 256, 20, 5, False, 1.2, 22),
    ("a4_prefill_ragged_norenorm", 300, 512, 256, 6, 3, False, None, 23),
]
FORMATS = ["mxfp8", "mxfp4", "mxfp4a4", "nvfp4"]


@pytest.fixture(scope="module")
def o():
    return oracle.default()


def unpack_e2m1(packed, shape_):
    """Two E2M1 codes per byte, element 2i in the low nibble of byte i -> one code per byte."""
    b = packed.reshape(-1)
    out = np.empty(b.size * 2, np.uint8)
    out[0::2] = b & 0xF
    out[1::2] = b >> 4
    return out.reshape(shape_)


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_mx_layer_parity(case, fmt, o):
    _, T, H, I, E, k, renorm, zipf, seed = case
    nv = fmt == "nvfp4"
    a4 = fmt == "mxfp4a4" or nv  # packed E2M1 token codes
    cfg = inputs.LayerConfig(T=T, H=H, I=I, E=E, top_k=k, renormalize=renorm, seed=seed, zipf_bias=zipf)
    li = inputs.make_layer_inputs(cfg)
    dl = gu.DeviceLayer(li)
    L = dl.layer
    fp4 = fmt != "mxfp8"
    if nv:
        L.quantize_nvfp4()
        codes13, scales13, codes2, scales2 = L.w13_codes_nv, L.w13_scales_nv, L.w2_codes_nv, L.w2_scales_nv
        quantize, unpack = None, unpack_e2m1
    elif fp4:
        L.quantize_mxfp4()
        codes13, scales13, codes2, scales2 = L.w13_codes4, L.w13_scales4, L.w2_codes4, L.w2_scales4
        quantize, unpack = o.mx4_quantize, unpack_e2m1
    else:
        L.quantize_mx()
        codes13, scales13, codes2, scales2 = L.w13_codes, L.w13_scales, L.w2_codes, L.w2_scales
        quantize, unpack = o.mx_quantize, lambda c, shp: c.reshape(shp)
    torch.cuda.synchronize()
    # weights: codes and scales (and NVFP4's tensor scales) bit for bit; an
    # NVFP4 scale tile covers 64 elements of K with 16-element blocks, i.e. the
    # MXFP8 tile of a matrix twice as wide
    if nv:
        w13c, w13s, w13g = o.nv4_quantize_experts(li.w13)
        w2c, w2s, w2g = o.nv4_quantize_experts(li.w2)
        assert np.array_equal(L.w13_gscale_nv.cpu().numpy(), w13g)
        assert np.array_equal(L.w2_gscale_nv.cpu().numpy(), w2g)
    else:
        w13c, w13s = quantize(li.w13)
        w2c, w2s = quantize(li.w2)
    wide, bs = (2, 16) if nv else (1, 32)
    assert np.array_equal(unpack(codes13.cpu().numpy(), (E, 2 * I, H)), w13c)
    assert np.array_equal(unpack(codes2.cpu().numpy(), (E, H, I)), w2c)
    s13 = gu.ungroup_mx_scales(scales13.cpu().numpy(), E * 2 * I, wide * H)[gu.w13_scale_rows(E, I)]
    assert np.array_equal(s13.reshape(E, 2 * I, H // bs), w13s)
    s2 = gu.ungroup_mx_scales(scales2.cpu().numpy(), E * H, wide * I)
    assert np.array_equal(s2.reshape(E, H, I // bs), w2s)

    xd = gu.dev_bf16(li.x)
    y = L.forward_nvfp4(xd) if nv else L.forward_mxfp4(xd, fp4_tokens=a4) if fp4 else L.forward_mx(xd)
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
    # the gate/up GEMM's token rows per unit (its scale chunks): 32 in the
    # decode plan, 128 or 256 in prefill; a chunk's scales take ceil(bn / 128) tiles
    bn = mv.nv_chunk_rows if nv else mv.x_chunk_rows
    assert bn == 32 if T * k <= 16 * E else bn in ((128,) if nv else (128, 256))
    G = -(-bn // 128)
    n_groups = (1 if nv else 2) * (v.P_max // 32)
    if a4:  # E2M1 token codes, two per byte
        xcodes = unpack_e2m1(view(mv.x_codes, torch.uint8, (v.P_max, H // 2)), (v.P_max, H))
    else:
        xcodes = view(mv.x_codes, torch.uint8, (v.P_max, H))
    xs = gu.ungroup_mx_scales(view(mv.x_scales, torch.uint8, (n_groups * (wide * H // 128) * 512,)), n_groups * 128,
                              wide * H)
    real = np.nonzero(g["sorted"] < T * k)[0]
    if nv:
        hc, hs, hg = o.nv4_quantize(g["h"][g["sorted"][real] // k], per_row=True)
        assert np.array_equal(view(mv.x_gscale, torch.float32, (v.P_max,))[real], hg)
    else:
        hc, hs = (o.mx4_quantize if a4 else o.mx_quantize)(g["h"][g["sorted"][real] // k])
    assert np.array_equal(xcodes[real], hc)
    offs = g["offsets"]
    chunk0 = np.concatenate([[0], np.cumsum(-(-np.diff(offs) // bn))])  # chunks before each expert
    e_of = np.searchsorted(offs, real, side="right") - 1
    within = real - offs[e_of]
    srow = (chunk0[e_of] + within // bn) * 128 * G + within % bn
    assert np.array_equal(xs[srow], hs)
    # the layer output against the oracle's layer of the same weight format
    if nv:
        r = o.moe_forward_nv4(li.x, li.g, li.w_router, li.bias, w13c, w13s, w13g, w2c, w2s, w2g, k, renorm, cfg.eps)
    else:
        fwd = o.moe_forward_mx4a4 if a4 else o.moe_forward_mx4 if fp4 else o.moe_forward_mx
        r = fwd(li.x, li.g, li.w_router, li.bias, w13c, w13s, w2c, w2s, k, renorm, cfg.eps)
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


def test_mxfp4_codes_every_value_class(o):
    """E2M1 quantizer on rows built to hit every code, every tie between
    neighbouring magnitudes, saturation, signed zeros, tiny and huge blocks."""
    rng = np.random.default_rng(41)
    mags = np.array([0.0, 0.25, 0.5, 0.75, 1.0, 1.25, 1.5, 1.75, 2.0, 2.5, 3.0, 3.5, 4.0, 5.0, 6.0, 7.0])
    rows = []
    for p in (-130, -100, -8, 0, 5, 100):
        for _ in range(8):
            v = rng.choice(mags, 32) * rng.choice([-1.0, 1.0], 32)
            v[0] = 4.0 * rng.choice([1.0, 1.5])  # block maximum fixes the scale at 2^p
            rows.append(v * 2.0 ** p)
    x = torch.tensor(np.array(rows).reshape(8, -1), dtype=torch.float64).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    R, K = xb.shape  # 8 x 192 -> pad K to a multiple of 128
    xpad = np.zeros((128, 256), np.uint16)
    xpad[:R, :K] = xb
    codes = torch.empty(128 * 128, dtype=torch.uint8, device="cuda")
    scales = torch.empty(512 * 2, dtype=torch.uint8, device="cuda")
    # W2 of a one-expert layer with H = 128 rows and I = 256: its quantizer runs on plain rows
    s = binding.shape(1, 128, 256, 1, 1)
    w13 = torch.zeros((1, 512, 128), dtype=torch.int16, device="cuda")
    w2 = torch.from_numpy(xpad.view(np.int16)).cuda()
    c13 = torch.empty(512 * 128 // 2, dtype=torch.uint8, device="cuda")
    s13 = torch.empty(4 * 512, dtype=torch.uint8, device="cuda")
    st = binding.moe_mxfp4_quantize_weights(s, w13.data_ptr(), w2.data_ptr(), c13.data_ptr(), s13.data_ptr(),
                                            codes.data_ptr(), scales.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == binding.MOE_OK
    torch.cuda.synchronize()
    oc, os_ = o.mx4_quantize(xpad)
    assert np.array_equal(unpack_e2m1(codes.cpu().numpy(), (128, 256)), oc)
    assert np.array_equal(gu.ungroup_mx_scales(scales.cpu().numpy(), 128, 256), os_)


def test_mxfp4_rejects_unaligned_codes():
    cfg = inputs.LayerConfig(T=4, H=128, I=128, E=4, top_k=2, seed=0)
    li = inputs.make_layer_inputs(cfg)
    dl = gu.DeviceLayer(li)
    L = dl.layer
    L.quantize_mxfp4()
    L.w13_codes4 = L.w13_codes4[16:]  # 16-byte aligned, not 32
    with pytest.raises(binding.MoeError) as ei:
        L.forward_mxfp4(gu.dev_bf16(li.x))
    assert ei.value.status == binding.MOE_ERR_INVALID_ARG


def test_block_scaled_layers_reject_i_not_multiple_of_128():
    """The bf16 layer takes I = 192 (a multiple of 64); the block-scaled layers,
    whose scale tiles cover 128 elements of K, refuse it before anything runs."""
    cfg = inputs.LayerConfig(T=4, H=256, I=192, E=4, top_k=2, seed=0)
    li = inputs.make_layer_inputs(cfg)
    dl = gu.DeviceLayer(li)
    L = dl.layer
    for quantize in (L.quantize_mx, L.quantize_mxfp4, L.quantize_nvfp4):
        with pytest.raises(binding.MoeError) as ei:
            quantize()
        assert ei.value.status == binding.MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("span", [(-4, 4), (-120, 120), (-30, -20)])
def test_nvfp4_weight_quantizer_extreme_ranges(o, span):
    """NVFP4 weights whose rows span 2^lo .. 2^hi: one tensor scale for the
    matrix sends the small rows' block scales to 0 (codes 0) or into E4M3's
    subnormals; codes, block scales and the tensor scale bit for bit with the
    oracle's fp32 decisions."""
    lo, hi = span
    rng = np.random.default_rng(hi - lo)
    E, H, I = 2, 256, 256
    w13 = rng.standard_normal((E, 2 * I, H)) * np.exp2(rng.uniform(lo, hi, (E, 2 * I, 1)))
    w2 = rng.standard_normal((E, H, I)) * np.exp2(rng.uniform(lo, hi, (E, H, 1)))
    w13[0, 3, :16] = 0.0  # an all-zero block
    w13[1, 5, :] *= -1.0
    w13[1, 7, 16:32] = [6, 3, 1.5, -0.5, 0, -0.0, 4, 2, 1, 0.75, 0.25, 5, -6, 7, 2.5, 3.5]  # ties and signs
    b13 = torch.tensor(w13).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    b2 = torch.tensor(w2).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    s_ = binding.shape(1, H, I, E, 1)
    st, (n13c, n13s, n2c, n2s) = binding.moe_nvfp4_weight_sizes(s_)
    dev = lambda a: torch.from_numpy(a.view(np.int16)).cuda()
    u8 = lambda n: torch.empty(n, dtype=torch.uint8, device="cuda")
    c13, sc13, c2, sc2 = u8(n13c), u8(n13s), u8(n2c), u8(n2s)
    g13 = torch.empty(E, dtype=torch.float32, device="cuda")
    g2 = torch.empty(E, dtype=torch.float32, device="cuda")
    d13, d2 = dev(b13), dev(b2)  # held until the asynchronous quantize has run
    st = binding.moe_nvfp4_quantize_weights(s_, d13.data_ptr(), d2.data_ptr(), c13.data_ptr(),
                                            sc13.data_ptr(), g13.data_ptr(), c2.data_ptr(), sc2.data_ptr(),
                                            g2.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == binding.MOE_OK
    torch.cuda.synchronize()
    oc13, os13, og13 = o.nv4_quantize_experts(b13)
    oc2, os2, og2 = o.nv4_quantize_experts(b2)
    assert np.array_equal(g13.cpu().numpy(), og13) and np.array_equal(g2.cpu().numpy(), og2)
    assert np.array_equal(unpack_e2m1(c13.cpu().numpy(), (E, 2 * I, H)), oc13)
    assert np.array_equal(unpack_e2m1(c2.cpu().numpy(), (E, H, I)), oc2)
    s13 = gu.ungroup_mx_scales(sc13.cpu().numpy(), E * 2 * I, 2 * H)[gu.w13_scale_rows(E, I)]
    assert np.array_equal(s13.reshape(E, 2 * I, H // 16), os13)
    assert np.array_equal(gu.ungroup_mx_scales(sc2.cpu().numpy(), E * H, 2 * I).reshape(E, H, I // 16), os2)
    if hi - lo > 100:
        assert (os13 == 0).sum() > 0, "some blocks' scales should underflow to 0 under one tensor scale"
