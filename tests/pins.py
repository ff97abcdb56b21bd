"""Pins of the CPU oracle to things other than itself.

Each ``pin_*`` takes an :class:`oracle.Oracle` and raises AssertionError when
the oracle disagrees with a closed form, a library routine, a brute-force
computation or an invariant that the pages and the mathematics fix.  They are
run against the real oracle (``test_oracle_pins.py``) and against copies of
the oracle with a planted mistake (``test_oracle_mutations.py``), which must
each fail at least one pin.
"""
from __future__ import annotations

import math

import numpy as np
import scipy.special
import torch
import torch.nn.functional as F

from mixture_experts_layer_rmsnorm_gb300 import inputs


def bits(vals) -> np.ndarray:
    """bf16 bits of values that are exactly representable in bf16."""
    f = np.asarray(vals, dtype=np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exactly representable in bf16"
    return (u >> 16).astype(np.uint16)


def widen(b) -> np.ndarray:
    return inputs.bf16_bits_to_f32(np.asarray(b, dtype=np.uint16)).astype(np.float64)


def torch_bf16_bits(v32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def rand_layer(T, H, I, E, seed, bias=False):
    cfg = inputs.LayerConfig(T=T, H=H, I=I, E=E, top_k=1, seed=seed, zipf_bias=1.2 if bias else None)
    li = inputs.make_layer_inputs(cfg)
    return li


# ---------------------------------------------------------------- conversions

def pin_bf16_conversions(o):
    # single rounding from fp64, ties to even (hand-derived values)
    assert o.f64_to_bf16(1.0) == 0x3F80
    assert o.f64_to_bf16(-2.0) == 0xC000
    assert o.f64_to_bf16(1 + 2 ** -8) == 0x3F80            # tie -> even
    assert o.f64_to_bf16(1 + 3 * 2 ** -8) == 0x3F82        # tie -> even (up)
    assert o.f64_to_bf16(1 + 2 ** -8 + 2 ** -30) == 0x3F81  # above the tie: one rounding, not two
    assert o.f64_to_bf16(1 + 2 ** -8 - 2 ** -30) == 0x3F80
    # fp32 -> bf16 against torch's conversion (a library routine)
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(4096) * np.exp(rng.uniform(-20, 20, 4096))).astype(np.float32)
    ours = np.array([o.f32_to_bf16(float(a)) for a in v], dtype=np.uint16)
    assert np.array_equal(ours, torch_bf16_bits(v))


# ------------------------------------------------------------------- RMSNorm

def pin_rmsnorm_constant_row(o):
    # x = c * 1  =>  mean(x^2) = c^2 exactly, so h_j = c g_j / sqrt(c^2 + eps)
    H, eps = 256, 1e-6
    for c in (0.5, -3.0, 0.0078125):
        x = bits(np.full((1, H), c))
        g = inputs.normal_bf16(3, 2, (H,), 1.0, 0.1)
        _, he = o.rmsnorm_f64(x, g, eps)
        want = c * widen(g) / math.sqrt(c * c + eps)
        assert np.allclose(he[0], want, rtol=1e-14, atol=0)


def pin_rmsnorm_single_rounding(o):
    # x = 1, g = 1, eps chosen so that h = 1/sqrt(1+eps) sits 2^-30 below the
    # bf16 tie 1 - 2^-9: one rounding gives 1 - 2^-8 (0x3F7F); rounding to fp32
    # first would land on the tie and give 1.0 (0x3F80).
    v = 1.0 - 2.0 ** -9 - 2.0 ** -30
    eps = 1.0 / (v * v) - 1.0
    h, he = o.rmsnorm_f64(bits(np.ones((1, 128))), bits(np.ones(128)), eps)
    assert abs(he[0, 0] - v) < 1e-13
    assert np.all(h == 0x3F7F)


def pin_rmsnorm_torch(o):
    # against torch.nn.functional.rms_norm in fp64 (a library routine)
    T, H, eps = 5, 384, 1e-6
    x = inputs.normal_bf16(4, 1, (T, H))
    g = inputs.normal_bf16(4, 2, (H,), 1.0, 0.1)
    h, he = o.rmsnorm_f64(x, g, eps)
    ref = F.rms_norm(torch.from_numpy(widen(x)), (H,), weight=torch.from_numpy(widen(g)), eps=eps).numpy()
    assert np.allclose(he, ref, rtol=1e-13, atol=1e-300)
    # the stored h is the bf16 rounding of the exact value: within half an ulp
    hv = widen(h)
    ulp = np.exp2(np.floor(np.log2(np.abs(ref))) - 7)
    assert np.all(np.abs(hv - ref) <= 0.5 * ulp * (1 + 1e-9))


def pin_rmsnorm_unit_gain(o):
    # g = 1 => mean_j h_j^2 = ms / (ms + eps) exactly (in exact arithmetic)
    H, eps = 512, 1e-2
    x = inputs.normal_bf16(5, 1, (3, H))
    g = bits(np.ones(H))
    _, he = o.rmsnorm_f64(x, g, eps)
    ms = (widen(x) ** 2).mean(axis=1)
    assert np.allclose((he ** 2).mean(axis=1), ms / (ms + eps), rtol=1e-13)


# ------------------------------------------------------------------- QK-norm

def pin_qknorm_power_of_two_heads(o):
    # x = c (a power of two), eps = 0: mean(x^2) = c^2 and rstd = 1/|c| exactly, so
    # x * rstd = sign(c) and out_j = sign(c) * (w_j + weight_bias) -- exact bf16
    # values for these gains, known by hand
    D = 64
    w = np.resize(np.array([0.5, -0.25, 2.0, 0.0, -1.5, 0.75, 3.0, -2.0], np.float32), D)
    for c in (0.25, -4.0):
        x = bits(np.full((3, D), c))
        out = o.qk_norm_f64(x, bits(w), 0.0, 0.0)
        assert np.array_equal(out, np.broadcast_to(bits(np.sign(c) * w), (3, D)))
        out = o.qk_norm_f64(x, bits(w), 1.0, 0.0)  # the bias is added to the gain
        assert np.array_equal(out, np.broadcast_to(bits(np.sign(c) * (w + 1.0)), (3, D)))


def pin_qknorm_torch(o):
    # against torch.nn.functional.rms_norm in fp64 with weight w + weight_bias
    # (a library routine), rounded once to bf16 by integer arithmetic
    for D, wb, eps in ((64, 1.0, 1e-2), (128, 0.0, 1e-6), (256, 0.5, 1e-3)):
        x = inputs.normal_bf16(21, 1, (7, 3, D))
        w = inputs.normal_bf16(21, 2, (D,), 0.0, 0.3)
        out = o.qk_norm_f64(x, w, wb, eps)
        ref = F.rms_norm(torch.from_numpy(widen(x)), (D,), weight=torch.from_numpy(widen(w) + wb), eps=eps).numpy()
        want = torch_bf16_bits_from_f64(ref)
        # equal but where fp64 rounding of the two orders straddles a bf16 rounding boundary
        diff = np.abs(out.astype(np.int32) - want.astype(np.int32))
        assert diff.max() <= 1 and np.mean(diff == 0) > 0.999


def pin_qknorm_per_head(o):
    # each head is normalised on its own: scaling one head of a token leaves the
    # others unchanged, and a head scaled by a power of two gives the same output
    D = 128
    x = inputs.normal_bf16(22, 1, (2, 4, D))
    w = inputs.normal_bf16(22, 2, (D,), 1.0, 0.1)
    base = o.qk_norm_f64(x, w, 0.0, 0.0)
    x2 = widen(x).copy()
    x2[:, 1] *= 64.0
    out2 = o.qk_norm_f64(bits(x2.astype(np.float32)), w, 0.0, 0.0)
    assert np.array_equal(out2, base)
    # unit gain: mean(out^2) = ms / (ms + eps) up to the bf16 rounding of out
    eps = 0.05
    out = widen(o.qk_norm_f64(x, bits(np.ones(D, np.float32)), 0.0, eps))
    ms = (widen(x) ** 2).mean(axis=-1)
    assert np.allclose((out ** 2).mean(axis=-1), ms / (ms + eps), rtol=1e-2)


# ---------------------------------------------------------------------- MXFP8

def _torch_e4m3_bits(v32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v32, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def pin_e4m3_decode_torch(o):
    # every finite code against torch's float8_e4m3fn (a library routine)
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([o.e4m3_decode(int(c)) for c in codes])
    assert np.array_equal(ours, ref)


def pin_e4m3_encode(o):
    # hand-derived codes: 1.0, the largest finite value, saturation, the smallest
    # subnormal, and ties to an even mantissa
    assert o.e4m3_encode(1.0) == 0x38 and o.e4m3_encode(-1.0) == 0xB8
    assert o.e4m3_encode(448.0) == 0x7E and o.e4m3_encode(500.0) == 0x7E and o.e4m3_encode(-1e6) == 0xFE
    assert o.e4m3_encode(2.0 ** -9) == 0x01 and o.e4m3_encode(2.0 ** -10) == 0x00  # tie -> 0 (even)
    assert o.e4m3_encode(3 * 2.0 ** -10) == 0x02                                   # tie -> 2 (even)
    assert o.e4m3_encode(1.0625) == 0x38 and o.e4m3_encode(1.1875) == 0x3A
    # in range: torch's round-to-nearest-even cast, on random values of all
    # magnitudes and on every midpoint between neighbouring codes
    rng = np.random.default_rng(7)
    v = (rng.standard_normal(20000) * np.exp2(rng.uniform(-12, 8, 20000))).astype(np.float32)
    v = v[np.abs(v) <= 448]
    vals = np.array(sorted({o.e4m3_decode(c) for c in range(0x7F)}))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    for arr in (v, mids, -mids):
        ours = np.array([o.e4m3_encode(float(a)) for a in arr], np.uint8)
        assert np.array_equal(ours, _torch_e4m3_bits(arr))


def pin_mx_block_scale(o):
    # block absolute maximum amax = r * 2^p: scale exponent p - 8, the maximum's
    # code 256 * r (r = 1 -> 0x78, r = 1.75 -> 448 = 0x7E, r = 1.90625 -> 488, saturated)
    for p, r, code in ((0, 1.0, 0x78), (-6, 1.75, 0x7E), (3, 1.90625, 0x7E), (-20, 1.5, 0x7C)):
        x = np.zeros((1, 64), np.float32)
        x[0, 5] = r * 2.0 ** p
        x[0, 40] = -r * 2.0 ** p
        x[0, 7] = 2.0 ** (p - 5)
        codes, scales = o.mx_quantize(bits(x))
        assert scales.tolist() == [[p - 8 + 127, p - 8 + 127]]
        assert codes[0, 5] == code and codes[0, 40] == code | 0x80
        assert o.e4m3_decode(int(codes[0, 7])) == 2.0 ** 3  # 2^(p-5) / 2^(p-8)
    codes, scales = o.mx_quantize(np.zeros((2, 32), np.uint16))
    assert np.all(codes == 0) and np.all(scales == 0)


def pin_mx_roundtrip_error(o):
    # dequantize(quantize(x)): at most half an E4M3 step per element, except the
    # values above 448 X (block maxima with a mantissa above 1.75), clamped to 448 X
    x = inputs.normal_bf16(23, 1, (16, 256), 0.0, 0.02)
    codes, scales = o.mx_quantize(x)
    d = o.mx_dequantize(codes, scales)
    xv = widen(x)
    X = np.exp2(np.repeat(scales.astype(np.float64) - 127, 32, axis=1))
    r = np.abs(xv) / X
    assert np.all(r < 512)  # the block maximum lies in [256, 512) X
    sat = r > 448
    assert np.array_equal(d[sat], np.sign(xv[sat]) * 448 * X[sat])
    step = np.maximum(np.exp2(np.floor(np.log2(np.maximum(r, 2.0 ** -6))) - 3), 2.0 ** -9) * X
    assert np.all(np.abs(d - xv)[~sat] <= step[~sat] / 2 * (1 + 1e-12))


def _torch_mx_dequant(v64: np.ndarray) -> np.ndarray:
    """Independent MXFP8 round trip of fp64 rows (values exact in bf16): block
    exponents from frexp, codes from torch's fp8 cast of the clamped scaled values."""
    v = v64.reshape(-1, 32)
    amax = np.abs(v).max(axis=1)
    _, e = np.frexp(amax)                   # amax = m * 2^e, m in [0.5, 1)
    ex = np.where(amax > 0, e - 1 - 8, -127)
    ex = np.clip(ex, -127, 127)
    scaled = np.clip(v / np.exp2(ex)[:, None], -448, 448).astype(np.float32)
    q = torch.from_numpy(scaled).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    return (q * np.exp2(ex)[:, None]).reshape(v64.shape)


def pin_mx_layer_torch(o):
    # the FP8 layer against a torch restatement: the same routing, MXFP8 round
    # trips of h, the weights and the bf16 activation, fp64 products and sums
    T, H, I, E, k = 3, 64, 96, 4, 2
    li = rand_layer(T, H, I, E, seed=24)
    w13c, w13s = o.mx_quantize(li.w13)
    w2c, w2s = o.mx_quantize(li.w2)
    res = o.moe_forward_mx(li.x, li.g, li.w_router, None, w13c, w13s, w2c, w2s, k, True, 1e-6)
    ref = o.moe_forward(li.x, li.g, li.w_router, None, li.w13, li.w2, k, True, 1e-6)
    assert np.array_equal(res["ids"], ref["ids"]) and np.allclose(res["w"], ref["w"], rtol=0, atol=0)
    W13 = _torch_mx_dequant(widen(li.w13))
    W2 = _torch_mx_dequant(widen(li.w2))
    y = np.zeros((T, H))
    for t in range(T):
        hq = _torch_mx_dequant(widen(ref["h16"][t]))
        for j in range(k):
            e = int(res["ids"][t, j])
            gate = W13[e, :I] @ hq
            up = W13[e, I:] @ hq
            a = widen(torch_bf16_bits_from_f64(gate / (1 + np.exp(-gate)) * up))
            y[t] += res["w"][t, j] * (W2[e] @ _torch_mx_dequant(a))
    assert np.allclose(res["y64"], y, rtol=1e-12, atol=1e-15)
    # and close to the bf16 layer: the MXFP8 error of a 64-long dot product
    rel = np.linalg.norm(res["y64"] - ref["y64"]) / np.linalg.norm(ref["y64"])
    assert 1e-4 < rel < 0.1


# ---------------------------------------------------------------------- MXFP4

E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # the OCP E2M1 table (codes 0..7)


def _rne_e2m1(a: np.ndarray) -> np.ndarray:
    """E2M1 rounding restated per binade with numpy's round-half-even rint:
    steps of 0.5 below 2, 1 below 4, 2 below 8; the value 8 saturates to 6."""
    a = np.abs(a)
    q = np.where(a < 2, np.rint(a * 2) / 2, np.where(a < 4, np.rint(a), 2 * np.rint(a / 2)))
    return np.minimum(q, 6.0)


def pin_e2m1_decode(o):
    for c in range(16):
        v = E2M1_MAGNITUDES[c & 7]
        assert o.e2m1_decode(c) == (-v if c & 8 else v)


def pin_e2m1_encode(o):
    # hand-derived: ties go to the even mantissa bit (0.25 -> 0, 0.75 -> 1,
    # 1.25 -> 1, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4), above 6 saturates
    for v, c in ((0.25, 0), (0.26, 1), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6), (5.5, 7),
                 (7.0, 7), (1e9, 7), (-0.3, 9), (-6.0, 15), (-1e9, 15)):
        assert o.e2m1_encode(v) == c, (v, c)
    # random values of all magnitudes and every midpoint between neighbours
    rng = np.random.default_rng(8)
    v = rng.standard_normal(20000) * np.exp2(rng.uniform(-4, 4, 20000))
    mids = (np.array(E2M1_MAGNITUDES[:-1]) + np.array(E2M1_MAGNITUDES[1:])) / 2
    for arr in (v, mids, -mids):
        got = np.array([o.e2m1_decode(o.e2m1_encode(float(a))) for a in arr])
        assert np.array_equal(np.abs(got), _rne_e2m1(arr)) and np.all((got == 0) | (np.sign(got) == np.sign(arr)))


def pin_mx4_block_scale(o):
    # block absolute maximum amax = r * 2^p: scale exponent p - 2, the maximum's
    # value 4 r (r = 1 -> 4 = code 6, r = 1.5 -> 6 = code 7, r = 1.75 -> 7,
    # saturated to 6); an element 2^(p-3) becomes 0.5 (code 1)
    for p, r, code in ((0, 1.0, 6), (-6, 1.5, 7), (3, 1.75, 7), (-20, 1.25, 6)):
        x = np.zeros((1, 64), np.float32)
        x[0, 5] = r * 2.0 ** p
        x[0, 40] = -r * 2.0 ** p
        x[0, 7] = 2.0 ** (p - 3)
        codes, scales = o.mx4_quantize(bits(x))
        assert scales.tolist() == [[p - 2 + 127, p - 2 + 127]]
        assert codes[0, 5] == code and codes[0, 40] == code | 8 and codes[0, 7] == 1
    codes, scales = o.mx4_quantize(np.zeros((2, 32), np.uint16))
    assert np.all(codes == 0) and np.all(scales == 0)


def pin_mx4_roundtrip_error(o):
    # dequantize(quantize(x)): at most half an E2M1 step of the value's binade
    # (0.25 X below 2 X, 0.5 X below 4 X, 1 X above), except the values above
    # 6 X (block maxima with a mantissa above 1.5), clamped to 6 X
    x = inputs.normal_bf16(25, 1, (16, 256), 0.0, 0.02)
    codes, scales = o.mx4_quantize(x)
    d = o.mx4_dequantize(codes, scales)
    xv = widen(x)
    X = np.exp2(np.repeat(scales.astype(np.float64) - 127, 32, axis=1))
    r = np.abs(xv) / X
    assert np.all(r < 8) and np.all(r.reshape(-1, 32).max(axis=1) >= 4)  # block maxima in [4, 8) X
    sat = r > 6
    assert np.array_equal(d[sat], np.sign(xv[sat]) * 6 * X[sat])
    half = np.where(r < 2, 0.25, np.where(r < 4, 0.5, 1.0)) * X
    assert np.all(np.abs(d - xv)[~sat] <= half[~sat] * (1 + 1e-12))


def _np_mx4_dequant(v64: np.ndarray) -> np.ndarray:
    """Independent MXFP4 round trip of fp64 rows (values exact in bf16): block
    exponents from frexp, values from the per-binade rint restatement."""
    v = v64.reshape(-1, 32)
    amax = np.abs(v).max(axis=1)
    _, e = np.frexp(amax)                   # amax = m * 2^e, m in [0.5, 1)
    ex = np.clip(np.where(amax > 0, e - 1 - 2, -127), -127, 127)
    s = v / np.exp2(ex)[:, None]
    q = np.sign(s) * _rne_e2m1(s)
    return (q * np.exp2(ex)[:, None]).reshape(v64.shape)


def pin_mx4_layer_restated(o):
    # the FP4-weight layer against a restatement: the same routing, MXFP4 round
    # trips of the weights (numpy), MXFP8 round trips of h and of the bf16
    # activation (torch's fp8 cast), fp64 products and sums
    T, H, I, E, k = 3, 64, 96, 4, 2
    li = rand_layer(T, H, I, E, seed=26)
    w13c, w13s = o.mx4_quantize(li.w13)
    w2c, w2s = o.mx4_quantize(li.w2)
    res = o.moe_forward_mx4(li.x, li.g, li.w_router, None, w13c, w13s, w2c, w2s, k, True, 1e-6)
    ref = o.moe_forward(li.x, li.g, li.w_router, None, li.w13, li.w2, k, True, 1e-6)
    assert np.array_equal(res["ids"], ref["ids"])
    W13 = _np_mx4_dequant(widen(li.w13))
    W2 = _np_mx4_dequant(widen(li.w2))
    y = np.zeros((T, H))
    for t in range(T):
        hq = _torch_mx_dequant(widen(ref["h16"][t]))
        for j in range(k):
            e = int(res["ids"][t, j])
            gate = W13[e, :I] @ hq
            up = W13[e, I:] @ hq
            a = widen(torch_bf16_bits_from_f64(gate / (1 + np.exp(-gate)) * up))
            y[t] += res["w"][t, j] * (W2[e] @ _torch_mx_dequant(a))
    assert np.allclose(res["y64"], y, rtol=1e-12, atol=1e-15)
    # further from the bf16 layer than the FP8-weight layer, but close
    rel = np.linalg.norm(res["y64"] - ref["y64"]) / np.linalg.norm(ref["y64"])
    assert 1e-3 < rel < 0.5


def pin_mx4a4_layer_restated(o):
    # the MXFP4 layer (FP4 weights, FP4 tokens and activations) against a
    # restatement: numpy MXFP4 round trips of the weights, of h and of the bf16
    # activation, fp64 products and sums
    T, H, I, E, k = 3, 64, 96, 4, 2
    li = rand_layer(T, H, I, E, seed=27)
    w13c, w13s = o.mx4_quantize(li.w13)
    w2c, w2s = o.mx4_quantize(li.w2)
    res = o.moe_forward_mx4a4(li.x, li.g, li.w_router, None, w13c, w13s, w2c, w2s, k, True, 1e-6)
    ref = o.moe_forward(li.x, li.g, li.w_router, None, li.w13, li.w2, k, True, 1e-6)
    assert np.array_equal(res["ids"], ref["ids"])
    W13 = _np_mx4_dequant(widen(li.w13))
    W2 = _np_mx4_dequant(widen(li.w2))
    y = np.zeros((T, H))
    for t in range(T):
        hq = _np_mx4_dequant(widen(ref["h16"][t]))
        for j in range(k):
            e = int(res["ids"][t, j])
            gate = W13[e, :I] @ hq
            up = W13[e, I:] @ hq
            a = widen(torch_bf16_bits_from_f64(gate / (1 + np.exp(-gate)) * up))
            y[t] += res["w"][t, j] * (W2[e] @ _np_mx4_dequant(a))
    assert np.allclose(res["y64"], y, rtol=1e-12, atol=1e-15)
    # the FP4 tokens move the result further from the W4A8 layer's
    w4a8 = o.moe_forward_mx4(li.x, li.g, li.w_router, None, w13c, w13s, w2c, w2s, k, True, 1e-6)
    assert np.linalg.norm(res["y64"] - w4a8["y64"]) > 1e-3 * np.linalg.norm(w4a8["y64"])


# --------------------------------------------------------------------- NVFP4


def pin_nv4_hand_cases(o):
    # tensor maximum 2688 = 448 * 6 -> tensor scale 1; per 16-element block:
    # amax 6 -> scale 1.0 (E4M3 0x38), codes of 6, 3, -1.5, 0.5, 0 = 7, 5, 11, 1, 0;
    # amax 2688 -> scale 448 (0x7E), 2688 -> code 7; amax 0.75 -> scale 0.125 (0x20),
    # 0.75 -> 7, 0.25 -> 4; amax 5 -> 5/6 rounds to 0.8125 (0x35) and 5 / 0.8125
    # saturates to 6 (code 7); an all-zero block -> scale 0, codes 0
    x = np.zeros((1, 80), np.float64)
    x[0, :5] = [6, 3, -1.5, 0.5, 0]
    x[0, 16] = 2688
    x[0, 32:34] = [0.75, 0.25]
    x[0, 48] = 5
    for per_row in (True, False):
        c, sc, g = o.nv4_quantize(torch_bf16_bits_from_f64(x), per_row=per_row)
        assert g.tolist() == [1.0]
        assert sc.tolist() == [[0x38, 0x7E, 0x20, 0x35, 0]]
        assert c[0, :5].tolist() == [7, 5, 11, 1, 0] and c[0, 16] == 7 and c[0, 32:34].tolist() == [7, 4]
        assert c[0, 48] == 7 and not c[0, 64:].any()
    # a tensor of zeros: tensor scale 1, every scale and code 0
    c, sc, g = o.nv4_quantize(np.zeros((2, 32), np.uint16), per_row=False)
    assert g.tolist() == [1.0] and not sc.any() and not c.any()


def _np_nv4(x16: np.ndarray, per_row: bool):
    """NVFP4 restated with numpy float32 arithmetic, torch's E4M3 cast for the
    block scales and the per-binade rint for E2M1: (codes, scales, g)."""
    import torch
    x = widen(x16).astype(np.float32)
    R, K = x.shape
    amax_r = np.abs(x).max(axis=1) if per_row else np.full(R, np.abs(x).max(), np.float32)
    g = np.where(amax_r > 0, amax_r / np.float32(2688), np.float32(1)).astype(np.float32)
    blk = np.abs(x).reshape(R, K // 16, 16).max(axis=2)
    u = (blk / (np.float32(6) * g)[:, None]).astype(np.float32)
    s8 = torch.from_numpy(np.minimum(u, np.float32(448))).to(torch.float8_e4m3fn)
    sc = s8.view(torch.uint8).numpy()
    X = (s8.to(torch.float32).numpy() * g[:, None]).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):  # X = 0 blocks take code 0 below
        q = (x.reshape(R, K // 16, 16) / X[:, :, None]).astype(np.float32)
    mag = _rne_e2m1(q.astype(np.float64))
    code = np.searchsorted(np.array(E2M1_MAGNITUDES), mag)
    code = code | np.where(np.signbit(q), 8, 0)
    code = np.where(X[:, :, None] > 0, code, 0).reshape(R, K).astype(np.uint8)
    return code, sc, (g if per_row else g[:1])


def pin_nv4_restated(o):
    rng = np.random.default_rng(31)
    for per_row in (True, False):
        x = rng.standard_normal((24, 256)) * np.exp2(rng.uniform(-12, 8, (24, 1)))
        x[3, 16:32] = 0.0                      # an all-zero block
        x[5, :] = x[5, :] * 1e-3               # a row far below the tensor maximum
        x16 = torch_bf16_bits_from_f64(x)
        c, sc, g = o.nv4_quantize(x16, per_row=per_row)
        c2, sc2, g2 = _np_nv4(x16, per_row)
        assert np.array_equal(g, g2) and np.array_equal(sc, sc2) and np.array_equal(c, c2)


def pin_nv4_roundtrip_error(o):
    # |x - q X| is at most half an E2M1 step of x/X's binade (0.25 X, 0.5 X, X),
    # except above 6 X, where it saturates to 6 X
    x16 = inputs.normal_bf16(33, 1, (16, 256), 0.0, 0.02)
    c, sc, g = o.nv4_quantize(x16, per_row=True)
    d = o.nv4_dequantize(c, sc, g, per_row=True)
    x = widen(x16)
    X = np.repeat(np.array([[o.e4m3_decode(int(b)) for b in row] for row in sc]), 16, axis=1) * \
        g.astype(np.float64)[:, None]
    r = np.abs(x) / X
    sat = r > 6
    assert np.allclose(d[sat], np.sign(x[sat]) * 6 * X[sat], rtol=1e-12)
    half = np.where(r < 2, 0.25, np.where(r < 4, 0.5, 1.0)) * X
    assert np.all(np.abs(d - x)[~sat] <= half[~sat] * (1 + 1e-6))
    assert np.linalg.norm(d - x) < 0.1 * np.linalg.norm(x)


def pin_nv4_layer_restated(o):
    # the NVFP4 layer against a restatement whose round trips use _np_nv4
    T, H, I, E, k = 3, 64, 96, 4, 2
    li = rand_layer(T, H, I, E, seed=28)
    w13c, w13s, w13g = o.nv4_quantize_experts(li.w13)
    w2c, w2s, w2g = o.nv4_quantize_experts(li.w2)
    res = o.moe_forward_nv4(li.x, li.g, li.w_router, None, w13c, w13s, w13g, w2c, w2s, w2g, k, True, 1e-6)
    ref = o.moe_forward(li.x, li.g, li.w_router, None, li.w13, li.w2, k, True, 1e-6)
    assert np.array_equal(res["ids"], ref["ids"])

    def deq(x16, per_row):
        c, sc, g = _np_nv4(np.atleast_2d(x16), per_row)
        vals = np.array(E2M1_MAGNITUDES)[c & 7] * np.where(c & 8, -1.0, 1.0)
        import torch
        sv = torch.from_numpy(sc.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        gg = g.astype(np.float64)[:, None] if per_row else np.float64(g[0])
        return vals * np.repeat(sv, 16, axis=1) * gg

    W13 = np.stack([deq(li.w13[e], False) for e in range(E)])
    W2 = np.stack([deq(li.w2[e], False) for e in range(E)])
    y = np.zeros((T, H))
    for t in range(T):
        hq = deq(ref["h16"][t], True)[0]
        for j in range(k):
            e = int(res["ids"][t, j])
            gate = W13[e, :I] @ hq
            up = W13[e, I:] @ hq
            a = torch_bf16_bits_from_f64(gate / (1 + np.exp(-gate)) * up)
            y[t] += res["w"][t, j] * (W2[e] @ deq(a, True)[0])
    assert np.allclose(res["y64"], y, rtol=1e-12, atol=1e-15)
    rel = np.linalg.norm(res["y64"] - ref["y64"]) / np.linalg.norm(ref["y64"])
    assert 1e-3 < rel < 0.5


# -------------------------------------------------------------------- router

def pin_router_f64_numpy(o):
    T, H, E = 4, 256, 16
    h = inputs.normal_bf16(6, 1, (T, H))
    wr = inputs.normal_f32(6, 3, (E, H), 0.0, 0.02)
    b = inputs.normal_f32(6, 9, (E,), 0.0, 1.0)
    l = o.router_logits_f64(h, wr, b)
    ref = widen(h) @ wr.astype(np.float64).T + b.astype(np.float64)
    scale = np.abs(widen(h)) @ np.abs(wr.astype(np.float64)).T + np.abs(b)
    assert np.all(np.abs(l - ref) <= 1e-13 * scale)


def pin_route_f32_exact_integers(o):
    # eps = 0 and x_j = +-2  =>  rstd = 1/2 exactly and h_j = +-g_j exactly; with
    # small-integer g, Wr and bias every fp32 partial sum is exact, so the
    # logits must equal the integer dot products whatever the order.
    rng = np.random.default_rng(7)
    T, H, E = 3, 512, 12
    sgn = rng.choice([-1.0, 1.0], size=(T, H))
    x = bits(2.0 * sgn)
    gi = rng.integers(1, 9, size=H) * rng.choice([-1, 1], size=H)
    g = bits(gi.astype(np.float32))
    wri = rng.integers(-8, 9, size=(E, H))
    bi = rng.integers(-50, 51, size=E)
    h32, l32, rstd = o.route_f32(x, g, 0.0, wri.astype(np.float32), bi.astype(np.float32))
    assert np.all(rstd == np.float32(0.5))
    hint = (sgn * gi).astype(np.int64)
    assert np.array_equal(h32, bits(hint.astype(np.float32)))
    want = hint @ wri.T.astype(np.int64) + bi
    assert np.array_equal(l32.astype(np.int64), want)


def pin_route_f32_order(o):
    # Values chosen so that each plausible other order gives a different fp32 result.
    H = 512
    x = bits(np.full((1, H), 2.0))
    g = bits(np.ones(H))  # eps = 0  =>  h = 1 exactly
    big = 2.0 ** 24
    wr = np.zeros((4, H), np.float32)
    wr[0, 0] = big; wr[0, 8:16] = 1.0        # chunk 1 is its own lane: 2^24 + 8 (sequential: 2^24)
    wr[1, 0] = big; wr[1, 256:264] = 1.0     # chunk 32 follows chunk 0 in lane 0: 2^24
    wr[2, 0] = big; wr[2, 1:8] = 1.0         # inside one chunk, sequential: 2^24
    wr[3, 0] = big; wr[3, 8:16] = 0.125      # lane 1 = 1; lane 16 = -2^24, lane 17 = 1: butterfly gives 2
    wr[3, 128] = -big; wr[3, 136:144] = 0.125
    _, l32, _ = o.route_f32(x, g, 0.0, wr)
    assert l32[0, 0] == np.float32(big + 8)
    assert l32[0, 1] == np.float32(big)
    assert l32[0, 2] == np.float32(big)
    assert l32[0, 3] == np.float32(2.0)
    # each step is one fused multiply-add: -(1+2^-7+2^-17) + (1+2^-7)(1+2^-17) = 2^-24
    # exactly; a rounded product would tie to even and give 0
    gv = np.zeros(H, np.float32); gv[0] = 1.0; gv[1] = 1.0 + 2.0 ** -7
    wf = np.zeros((1, H), np.float32); wf[0, 0] = -(1.0 + 2.0 ** -7 + 2.0 ** -17); wf[0, 1] = 1.0 + 2.0 ** -17
    _, lf, _ = o.route_f32(x, bits(gv), 0.0, wf)
    assert lf[0, 0] == np.float32(2.0 ** -24)
    # sum of squares in the same order: x_0 = 2^12, x_8..15 = 1  =>  ss = 2^24 + 8
    H2 = 256
    xv = np.zeros(H2, np.float32); xv[0] = 4096.0; xv[8:16] = 1.0
    _, _, rstd = o.route_f32(bits(xv[None, :]), bits(np.ones(H2)), 0.0, np.zeros((1, H2), np.float32))
    ss = np.float32(big + 8)
    want = np.float32(1.0) / np.sqrt(ss / np.float32(H2))
    assert rstd[0] == want


def pin_route_f32_bounds(o):
    # fp32 canonical logits vs fp64 logits of the same h: within the fp32 error bound
    T, H, E = 6, 1024, 32
    x = inputs.normal_bf16(8, 1, (T, H))
    g = inputs.normal_bf16(8, 2, (H,), 1.0, 0.1)
    wr = inputs.normal_f32(8, 3, (E, H), 0.0, 0.02)
    b = inputs.normal_f32(8, 9, (E,), 0.0, 1.0)
    h32, l32, rstd = o.route_f32(x, g, 1e-6, wr, b)
    l64 = o.router_logits_f64(h32, wr, b)
    hw = np.abs(widen(h32)) @ np.abs(wr.astype(np.float64)).T
    bound = (H / 32 + 8) * 2.0 ** -24 * hw + 2.0 ** -24 * (np.abs(l64) + np.abs(b))
    assert np.all(np.abs(l32 - l64) <= bound)
    # the fp32 norm output is within one bf16 ulp of the fp64 one, and almost always equal
    h64, he = o.rmsnorm_f64(x, g, 1e-6)
    d = np.abs(widen(h32) - widen(h64))
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(he), 1e-30))) - 7)
    assert np.all(d <= ulp * 1.0000001)
    assert np.mean(d > 0) < 0.01


# ---------------------------------------------------------------- selection

def pin_topk_numpy(o):
    rng = np.random.default_rng(9)
    for dtype in (np.float32, np.float64):
        for (T, E, k) in ((7, 64, 8), (5, 8, 8), (3, 256, 6), (4, 5, 1)):
            l = rng.standard_normal((T, E)).astype(dtype)
            ids = o.topk(l, k)
            ref = np.argsort(-l, axis=1, kind="stable")[:, :k]
            assert np.array_equal(ids, ref)
            # many exact ties: the stable sort puts the lower index first
            lt = rng.integers(0, 4, size=(T, E)).astype(dtype)
            assert np.array_equal(o.topk(lt, k), np.argsort(-lt, axis=1, kind="stable")[:, :k])


def pin_topk_duplicate_router_rows(o):
    # two identical router rows give bit-identical logits; a large bias on both
    # makes them the top two: expert 3 must come first, then 5
    T, H, E = 6, 256, 8
    x = inputs.normal_bf16(10, 1, (T, H))
    g = inputs.normal_bf16(10, 2, (H,), 1.0, 0.1)
    wr = inputs.normal_f32(10, 3, (E, H), 0.0, 0.02)
    wr[5] = wr[3]
    b = np.zeros(E, np.float32); b[3] = b[5] = 100.0
    _, l32, _ = o.route_f32(x, g, 1e-6, wr, b)
    assert np.array_equal(l32[:, 3], l32[:, 5])
    ids = o.topk(l32, 3)
    assert np.all(ids[:, 0] == 3) and np.all(ids[:, 1] == 5)


def pin_weights(o):
    rng = np.random.default_rng(11)
    T, E, k = 9, 16, 4
    l = rng.standard_normal((T, E)) * 3
    ids = np.argsort(-l, axis=1, kind="stable")[:, :k].astype(np.int32)
    w = o.route_weights_f64(l, ids, True)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-15)
    ref = scipy.special.softmax(np.take_along_axis(l, ids, axis=1), axis=1)
    assert np.allclose(w, ref, rtol=1e-14, atol=0)
    w2 = o.route_weights_f64(l, ids, False)
    ref2 = np.take_along_axis(scipy.special.softmax(l, axis=1), ids, axis=1)
    assert np.allclose(w2, ref2, rtol=1e-14, atol=0)
    assert np.all(w2.sum(axis=1) <= 1.0 + 1e-15)
    # k = E with renormalisation is the full softmax
    idsE = np.argsort(-l, axis=1, kind="stable").astype(np.int32)
    wE = o.route_weights_f64(l, idsE, True)
    assert np.allclose(wE, np.take_along_axis(scipy.special.softmax(l, axis=1), idsE, axis=1), rtol=1e-14)


# --------------------------------------------------------------------- align

def brute_align(ids_flat, E, pad):
    N = len(ids_flat)
    rows, offsets = [], [0]
    for e in range(E):
        lst = [i for i in range(N) if ids_flat[i] == e]
        while len(lst) % pad:
            lst.append(N)
        rows += lst
        offsets.append(len(rows))
    return np.array(rows, np.int32), np.array(offsets, np.int32)


def pin_align_bruteforce(o):
    rng = np.random.default_rng(12)
    cases = [(0, 4, 2, 16), (1, 8, 2, 16), (4, 8, 2, 16), (13, 64, 8, 16), (16, 7, 3, 1), (30, 5, 5, 128),
             (64, 128, 6, 16)]
    for (T, E, k, pad) in cases:
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32) if T else \
            np.zeros((0, k), np.int32)
        flat = ids.reshape(-1)
        counts, offsets, sorted_ids, slot_of = o.align(flat, E, pad)
        rows, offs = brute_align(list(flat), E, pad)
        assert np.array_equal(offsets, offs)
        assert np.array_equal(sorted_ids, rows)
        assert np.array_equal(counts, np.bincount(flat, minlength=E))
        N = flat.size
        # invariants: every entry exactly once; slot_of inverts sorted_ids; segments padded
        real = sorted_ids[sorted_ids < N]
        assert np.array_equal(np.sort(real), np.arange(N))
        if N:
            assert np.array_equal(sorted_ids[slot_of], np.arange(N))
        assert np.all(np.diff(offsets) % pad == 0)


# --------------------------------------------------------------- expert MLP

def _torch_swiglu(h64, w13_e, w2_e, round_act=False):
    I = w13_e.shape[0] // 2
    W = torch.from_numpy(widen(w13_e))
    Wd = torch.from_numpy(widen(w2_e))
    hh = torch.from_numpy(np.asarray(h64, dtype=np.float64))
    a = F.silu(hh @ W[:I].T) * (hh @ W[I:].T)
    return a.numpy(), (a @ Wd.T).numpy()


def pin_expert_torch(o):
    H, I = 256, 384
    li = rand_layer(2, H, I, 1, seed=13)
    h64 = widen(li.x[0])  # any bf16 row will do as the expert's input
    a, out = o.expert_f64(h64, li.w13[0], li.w2[0], round_act=False)
    a_ref, o_ref = _torch_swiglu(h64, li.w13[0], li.w2[0])
    assert np.allclose(a, a_ref, rtol=1e-12, atol=1e-15)
    assert np.allclose(out, o_ref, rtol=1e-11, atol=1e-14)
    # with the activation stored as bf16, a is the rounding of the exact value
    a_r, _ = o.expert_f64(li.x[0], li.w13[0], li.w2[0], round_act=True)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(a_ref), 1e-30))) - 7)
    assert np.all(np.abs(a_r - a_ref) <= 0.5 * ulp * (1 + 1e-9))
    assert np.array_equal(a_r, widen(torch_bf16_bits_from_f64(a_r)))  # stored as bf16 values


# ------------------------------------------------------------- whole layer

def _dense_reference(li, k, renorm, eps):
    """Brute force: y = sum over ALL experts of G_e * SwiGLU_e(h), with G_e the
    routing weight of e if e is among the token's k selected experts, else 0."""
    x64 = widen(li.x)
    g64 = widen(li.g)
    T, H = li.x.shape
    # norm: library routine (torch rms_norm, fp64)
    he = F.rms_norm(torch.from_numpy(x64), (H,), weight=torch.from_numpy(g64), eps=eps).numpy()
    # logits: numpy fp64 matmul of the bf16-rounded h
    h_round = widen(torch_bf16_bits_from_f64(he))
    l64 = h_round @ li.w_router.astype(np.float64).T
    if li.bias is not None:
        l64 = l64 + li.bias.astype(np.float64)
    return he, h_round, l64


def torch_bf16_bits_from_f64(v: np.ndarray) -> np.ndarray:
    """bf16 rounding of fp64 values through exact integer arithmetic on the
    significand (ties to even), independent of any fp32 intermediate."""
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(np.abs(v))
    q = np.round(np.ldexp(m, 8))  # numpy rounds half to even
    r = np.sign(v) * np.ldexp(q, e - 8)
    return (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def pin_layer_dense_bruteforce(o):
    for (T, H, I, E, k, renorm, bias, seed) in ((4, 128, 256, 8, 2, True, False, 0),
                                                (6, 256, 128, 5, 3, False, True, 14),
                                                (3, 128, 128, 4, 4, True, False, 15)):
        li = rand_layer(T, H, I, E, seed=seed, bias=bias)
        eps = 1e-6
        res = o.moe_forward(li.x, li.g, li.w_router, li.bias, li.w13, li.w2, k, renorm, eps, round_inter=False)
        he, h_round, l64 = _dense_reference(li, k, renorm, eps)
        # the selection is taken on the fp32 logits (the kernel's precision); a stable
        # sort of them (library routine) gives the experts and their order
        ids = np.argsort(-res["l32"], axis=1, kind="stable")[:, :k]
        assert np.array_equal(res["ids"], ids)
        p = scipy.special.softmax(l64, axis=1)
        G = np.zeros((T, E))
        for t in range(T):
            sel = p[t, ids[t]]
            if renorm:
                sel = sel / sel.sum()
            G[t, ids[t]] = sel
        y = np.zeros((T, H))
        for e in range(E):  # dense: every expert, gate zero where not selected
            _, oe = _torch_swiglu(he, li.w13[e], li.w2[e])
            y += G[:, e:e + 1] * oe
        assert np.allclose(res["y64"], y, rtol=1e-11, atol=1e-13)
        assert np.allclose(res["w"], np.take_along_axis(G, ids, axis=1), rtol=1e-13, atol=0)
        assert np.array_equal(res["y16"], torch_bf16_bits_from_f64(res["y64"]))
        assert np.array_equal(res["h16"], torch_bf16_bits_from_f64(he))


def pin_layer_single_expert(o):
    # E = 1, k = 1, renormalised: the layer is a dense SwiGLU MLP on RMSNorm(x)
    T, H, I = 5, 256, 256
    li = rand_layer(T, H, I, 1, seed=16)
    eps = 1e-6
    res = o.moe_forward(li.x, li.g, li.w_router, None, li.w13, li.w2, 1, True, eps, round_inter=False)
    he = F.rms_norm(torch.from_numpy(widen(li.x)), (H,), weight=torch.from_numpy(widen(li.g)), eps=eps).numpy()
    _, y = _torch_swiglu(he, li.w13[0], li.w2[0])
    assert np.all(res["ids"] == 0) and np.allclose(res["w"], 1.0, atol=1e-15)
    assert np.allclose(res["y64"], y, rtol=1e-11, atol=1e-13)


def pin_layer_rounded_mode(o):
    # storage-type mode: within the bf16 error of h and of the activation
    T, H, I, E, k = 4, 128, 256, 8, 2
    li = rand_layer(T, H, I, E, seed=0)
    r1 = o.moe_forward(li.x, li.g, li.w_router, None, li.w13, li.w2, k, True, 1e-6, round_inter=True)
    r0 = o.moe_forward(li.x, li.g, li.w_router, None, li.w13, li.w2, k, True, 1e-6, round_inter=False)
    assert np.array_equal(r1["ids"], r0["ids"])
    rel = np.linalg.norm(r1["y64"] - r0["y64"]) / np.linalg.norm(r0["y64"])
    assert 0 < rel < 2e-2


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
