"""Planted mistakes in copies of the CPU oracle must each fail at least one pin.

Each mutation is a plausible slip (a dropped term, a wrong sign or index, a
transposed operand, a wrong order) applied as a text edit to a copy of
moe_oracle.c, compiled into a temporary library on the CPU.  The real oracle
is never modified.
"""
import os

import pytest

import oracle
import pins

MUTATIONS = {
    "eps_dropped": ("sqrt(ss / (double)H + eps)", "sqrt(ss / (double)H)"),
    "mean_not_divided": ("sqrt(ss / (double)H + eps)", "sqrt(ss + eps)"),
    "gain_dropped": ("double v = bf16_to_f64(x[j]) * rstd * bf16_to_f64(g[j]);",
                     "double v = bf16_to_f64(x[j]) * rstd;"),
    "gate_up_swapped": ("const uint16_t* wg = W13e + i * H;\n    const uint16_t* wu = W13e + (I + i) * H;",
                        "const uint16_t* wg = W13e + (I + i) * H;\n    const uint16_t* wu = W13e + i * H;"),
    "silu_sign": ("gate / (1.0 + exp(-gate))", "gate / (1.0 + exp(gate))"),
    "w2_transposed": ("acc += a[i] * bf16_to_f64(wd[i]);", "acc += a[i] * bf16_to_f64(W2e[i * H + n]);"),
    "bias_dropped": ("logits[e] = acc + (bias ? (double)bias[e] : 0.0);", "logits[e] = acc;"),
    "tie_to_higher_f32": ("if (!taken[e] && (best < 0 || l[e] > l[best])) best = e;\n      taken[best] = 1;\n"
                          "      ids[t * k + j] = (int32_t)best;\n    }\n  }\n  free(taken);\n}\n\nvoid oracle_topk_f64",
                          "if (!taken[e] && (best < 0 || l[e] >= l[best])) best = e;\n      taken[best] = 1;\n"
                          "      ids[t * k + j] = (int32_t)best;\n    }\n  }\n  free(taken);\n}\n\nvoid oracle_topk_f64"),
    "renorm_ignored": ("    if (renorm)\n      for (int j = 0; j < k; ++j) w[t * k + j] /= s;", ""),
    "softmax_not_shifted_sum": ("for (int64_t e = 0; e < E; ++e) z += exp(l[e] - m);",
                                "for (int64_t e = 0; e < E; ++e) z += exp(l[e]);"),
    "combine_unweighted": ("acc += w[s * k + j] * c.o[(s * k + j) * H + n];", "acc += c.o[(s * k + j) * H + n];"),
    "butterfly_reversed": ("for (int off = 16; off >= 1; off >>= 1) {", "for (int off = 1; off <= 16; off <<= 1) {"),
    "chunks_blocked": ("for (int64_t c = L; c * 8 < H; c += 32)",
                       "for (int64_t c = L * ((H / 8 + 31) / 32); c < (L + 1) * ((H / 8 + 31) / 32) && c * 8 < H; c += 1)"),
    "no_fma_in_router": ("acc = fmaf(a[j], b[j], acc);", "acc = acc + a[j] * b[j];"),
    "align_unstable": ("  for (int64_t i = 0; i < N; ++i) {\n    int32_t e = ids[i];",
                       "  for (int64_t i = N - 1; i >= 0; --i) {\n    int32_t e = ids[i];"),
    "align_unpadded": ("int64_t padded = (counts[e] + pad - 1) / pad * pad;", "int64_t padded = counts[e];"),
    "h_not_rounded_to_bf16": ("if (h) h[j] = f64_to_bf16(v);", "if (h) h[j] = f32_to_bf16((float)v);"),
    "act_round_dropped": ("a[i] = round_act ? bf16_to_f64(f64_to_bf16(v)) : v;", "a[i] = v;"),
    "mx_emax_7": ("return mx_block_exponent_of(amax, 8); }", "return mx_block_exponent_of(amax, 7); }"),
    "e4m3_round_half_up": ("double q = nearbyint(a / ldexp(1.0, ex - 3));", "double q = floor(a / ldexp(1.0, ex - 3) + 0.5);"),
    "e4m3_no_saturation": ("      e = 15;\n      m = 6;", "      e = 15;\n      m = 7;"),
    "e4m3_subnormal_scale": ("double v = e == 0 ? ldexp((double)m, -9)", "double v = e == 0 ? ldexp((double)m, -10)"),
    "mx_act_not_quantized": ("  mx_token_roundtrip(afmt, I, a16, a);",
                             "  for (int64_t i = 0; i < I; ++i) a[i] = bf16_to_f64(a16[i]);"),
    "mx_token_not_quantized": ("  mx_token_roundtrip(afmt, H, h16, hq);",
                               "  for (int64_t j = 0; j < H; ++j) hq[j] = bf16_to_f64(h16[j]);"),
    "mx4_emax_1": ("int ex = mx_block_exponent_of(amax, 2);", "int ex = mx_block_exponent_of(amax, 1);"),
    "e2m1_tie_to_odd": ("if (d < bd || (d == bd && (c & 1) == 0)) {", "if (d < bd || (d == bd && (c & 1) == 1)) {"),
    "e2m1_binade_off": ("double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);",
                        "double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e);"),
    "mx4_weights_as_e4m3": ("  else if (wfmt)\n    oracle_mx4_dequantize(rows, K, codes, scales, out);",
                            "  else if (0)\n    oracle_mx4_dequantize(rows, K, codes, scales, out);"),
    "e2m1_sign_dropped": ("  return (uint8_t)((sgn << 3) | best);", "  return (uint8_t)best;"),
    "mx4a4_tokens_as_mxfp8": ("  } else if (afmt) {\n    oracle_mx4_quantize(1, K, x16, c, sc);",
                              "  } else if (0) {\n    oracle_mx4_quantize(1, K, x16, c, sc);"),
    "nv4_global_scale_ignored": ("static float nv4_global_of(float amax) { return amax > 0.0f ? amax / 2688.0f : 1.0f; }",
                                 "static float nv4_global_of(float amax) { return amax > 0.0f ? 1.0f : 1.0f; }"),
    "nv4_block_scale_not_six": ("    const float six_g = 6.0f * g;", "    const float six_g = 4.0f * g;"),
    "nv4_scale_skips_global": ("      const float X = (float)oracle_e4m3_decode(sc) * g;",
                               "      const float X = (float)oracle_e4m3_decode(sc);"),
    "nv4_token_tensor_scale": ("    oracle_nv4_quantize(1, K, x16, 1, c, sc, &g);\n    oracle_nv4_dequantize(1, K, c, sc, &g, 1, out);",
                               "    oracle_nv4_quantize(1, K, x16, 1, c, sc, &g);\n    g = 1.0f;\n    oracle_nv4_dequantize(1, K, c, sc, &g, 1, out);"),
    "qk_bias_dropped": ("(bf16_to_f64(w[j]) + weight_bias)", "(bf16_to_f64(w[j]))"),
    "qk_bias_multiplied": ("(bf16_to_f64(w[j]) + weight_bias)", "(bf16_to_f64(w[j]) * weight_bias)"),
    "qk_eps_dropped": ("sqrt(ss / (double)D + eps)", "sqrt(ss / (double)D)"),
    "qk_sum_not_mean": ("sqrt(ss / (double)D + eps)", "sqrt(ss + eps)"),
    "qk_x_unsquared": ("      ss += xv * xv;\n    }\n    double rstd = 1.0 / sqrt(ss / (double)D",
                       "      ss += fabs(xv);\n    }\n    double rstd = 1.0 / sqrt(ss / (double)D"),
}


def _build_variant(tmp_path, name, old, new):
    src = open(oracle._SRC).read()
    assert old in src, f"mutation {name}: pattern not found"
    mutated = src.replace(old, new, 1)
    cpath = os.path.join(tmp_path, f"oracle_{name}.c")
    with open(cpath, "w") as f:
        f.write(mutated)
    return oracle.Oracle(oracle.build_lib(force=True, src=cpath, out=os.path.join(tmp_path, f"lib_{name}.so")))


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    o = _build_variant(str(tmp_path), name, old, new)
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"planted mistake {name!r} passed every pin"
