"""Stored values: the pages' printed figures (byte/FLOP accounting) and the
oracle's own regression values on the tiny workload."""
import json
import os

import numpy as np

from mixture_experts_layer_rmsnorm_gb300 import accounting, inputs

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_pages_elementwise_fusion_bytes():
    d = _load("pages_figures.json")["elementwise_fusion"]
    m = 1000
    un = accounting.elementwise_bytes(d["n_ops"], m, d["elem_bytes"], fused=False)
    fu = accounting.elementwise_bytes(d["n_ops"], m, d["elem_bytes"], fused=True)
    assert un == d["unfused_bytes_per_element"] * m
    assert fu == d["fused_bytes_per_element"] * m
    assert un // fu == d["factor"]


def test_pages_gemm_epilogue_bytes():
    d = _load("pages_figures.json")["gemm_epilogue_saving"]
    c = accounting.matrix_bytes(d["M"], d["N"])
    # 4096^2 * 2 B = 33.55e6 B, printed as "33,5 Mo" (truncated to one decimal)
    assert 0 <= c / 1e6 - d["C_megabytes"] < 0.1
    assert 0 <= 2 * c / 1e6 - d["saved_megabytes"] < 0.2


def test_pages_gemm_flops():
    d = _load("pages_figures.json")["gemm_flops"]
    f = accounting.gemm_flops(d["M"], d["N"], d["K"])
    assert abs(f - d["flop"]) / d["flop"] < d["rel_tol"]


def test_pages_vector_width():
    d = _load("pages_figures.json")["vector_width"]
    assert d["bits"] // (8 * accounting.BF16) == d["bf16_per_thread"]
    assert d["bits"] // (8 * accounting.FP32) == d["fp32_per_thread"]


def test_layer_flops_formula():
    # 6*T*k*H*I for the two expert GEMMs, 2*T*E*H for the router
    T, H, I, E, k = 4096, 4096, 4096, 64, 8
    f = accounting.layer_flops(T, H, I, E, k)
    assert f["gemm1"] + f["gemm2"] == 6 * T * k * H * I
    assert f["router"] == 2 * T * E * H


def test_oracle_tiny_regression(oracle_default):
    d = _load("tiny_oracle.json")
    c = d["config"]
    cfg = inputs.LayerConfig(T=c["T"], H=c["H"], I=c["I"], E=c["E"], top_k=c["top_k"],
                             renormalize=c["renormalize"], eps=c["eps"], seed=c["seed"])
    li = inputs.make_layer_inputs(cfg)
    r = oracle_default.moe_forward(li.x, li.g, li.w_router, li.bias, li.w13, li.w2, cfg.top_k,
                                   cfg.renormalize, cfg.eps)
    assert r["ids"].tolist() == d["topk_ids"]
    assert np.allclose(r["w"], np.array(d["topk_w"]), rtol=1e-14, atol=0)
    assert np.array_equal(r["y16"], np.array(d["y_bf16_bits"], dtype=np.uint16))
    assert np.array_equal(r["h16"][:, :8], np.array(d["h_bf16_bits_first8"], dtype=np.uint16))
    assert np.array_equal(r["l32"], np.array(d["logits_f32_first8"], dtype=np.float32))
