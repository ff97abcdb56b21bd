"""Byte and FLOP accounting of the fused MoE layer (host-side arithmetic only).

Traffic model: an operation that reads and writes a tensor of m elements of
s bytes moves 2*m*s bytes; fusing n such elementwise passes into one moves
2*m*s instead of n*2*m*s ("4 · La fusion de noyaux", §4.1, fusion arithmetic).
A GEMM of M x N x K costs 2*M*N*K floating-point operations (the same page's
quiz on two 4096^3 GEMMs: 1.37e11 FLOP each), and a bf16 matrix of M x N
elements occupies 2*M*N bytes (§4.2 "GEMM + épilogue": 33.5 MB for 4096^2).

Per-call figures of the layer (T tokens, H hidden, I expert intermediate, E
experts, k = top_k, n_touched = distinct experts that received a token):
  weight bytes      n_touched * (2I*H + H*I) * 2     (W13 and W2 of touched experts)
  router bytes      E*H*4 + H*2                      (fp32 router, bf16 norm gain)
  token bytes       T*H*2 in + T*H*2 out
  FLOP              2*(T*k)*(2I)*H + 2*(T*k)*H*I + 2*T*E*H   (= 6*T*k*H*I + router)
"""
from __future__ import annotations

import numpy as np

BF16 = 2
FP32 = 4


def elementwise_bytes(n_ops: int, m: int, s: int, fused: bool) -> int:
    """Bytes moved by n elementwise passes over m elements of s bytes."""
    return 2 * m * s if fused else n_ops * 2 * m * s


def gemm_flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K


def matrix_bytes(M: int, N: int, elem: int = BF16) -> int:
    return M * N * elem


def n_touched(topk_ids: np.ndarray, E: int) -> int:
    return int(np.unique(np.asarray(topk_ids).reshape(-1)).size) if np.asarray(topk_ids).size else 0


def mx_bytes(n_elems: int) -> int:
    """MXFP8 bytes of n elements: one E4M3 code each plus one E8M0 scale per 32."""
    return n_elems + n_elems // 32


def mx4_bytes(n_elems: int) -> int:
    """MXFP4 bytes of n elements: E2M1 codes two per byte plus one E8M0 scale per 32."""
    return n_elems // 2 + n_elems // 32


def nv4_bytes(n_elems: int) -> int:
    """NVFP4 bytes of n elements: E2M1 codes two per byte plus one E4M3 scale per 16
    (the fp32 tensor scales, one per matrix or row, are left out)."""
    return n_elems // 2 + n_elems // 16


def weight_bytes(n_elems: int, mx) -> int:
    """Bytes of n weight elements: bf16 (mx false), MXFP8 (mx true), MXFP4
    (mx == "mxfp4", FP4 weights with MXFP8 tokens, or "mxfp4a4", the MXFP4 layer)
    or NVFP4 (mx == "nvfp4")."""
    if mx == "nvfp4":
        return nv4_bytes(n_elems)
    if mx in ("mxfp4", "mxfp4a4"):
        return mx4_bytes(n_elems)
    return mx_bytes(n_elems) if mx else n_elems * BF16


def token_bytes(n_elems: int, mx) -> int:
    """Bytes of n quantized token elements: MXFP4 in the MXFP4 layer, NVFP4 in
    the NVFP4 layer, else MXFP8."""
    if mx == "nvfp4":
        return nv4_bytes(n_elems)
    return mx4_bytes(n_elems) if mx == "mxfp4a4" else mx_bytes(n_elems)


def expert_weight_bytes(H: int, I: int, mx=False) -> dict:
    """Bytes of one expert's weights: gate/up (W13) and down (W2); mx: MXFP8
    copies (true) or MXFP4 copies ("mxfp4")."""
    if mx:
        return {"w13": weight_bytes(2 * I * H, mx), "w2": weight_bytes(H * I, mx)}
    return {"w13": 2 * I * H * BF16, "w2": H * I * BF16}


def layer_bytes(T: int, H: int, I: int, E: int, k: int, touched: int, mx=False) -> dict:
    ew = expert_weight_bytes(H, I, mx)
    d = {
        "weights_w13": touched * ew["w13"],
        "weights_w2": touched * ew["w2"],
        "router": E * H * FP32 + H * BF16,
        "tokens": 2 * T * H * BF16,
    }
    d["weights"] = d["weights_w13"] + d["weights_w2"]
    d["total"] = d["weights"] + d["router"] + d["tokens"]
    return d


def layer_flops(T: int, H: int, I: int, E: int, k: int) -> dict:
    g1 = gemm_flops(T * k, 2 * I, H)
    g2 = gemm_flops(T * k, H, I)
    r = gemm_flops(T, E, H)
    return {"gemm1": g1, "gemm2": g2, "router": r, "total": g1 + g2 + r}


def gemm1_kernel_bytes(T: int, H: int, I: int, k: int, touched: int, mx=False) -> int:
    """Algorithmic bytes of the gate/up expert GEMM: touched W13, the T*k
    gathered token rows read once, the T*k activation rows (bf16) written once.
    mx: MXFP8 (true) or MXFP4 ("mxfp4") weights with MXFP8 token rows, or
    the MXFP4 layer ("mxfp4a4")."""
    if mx:
        return weight_bytes(touched * 2 * I * H, mx) + token_bytes(T * k * H, mx) + T * k * I * BF16
    return touched * 2 * I * H * BF16 + T * k * H * BF16 + T * k * I * BF16


def gemm2_kernel_bytes(T: int, H: int, I: int, k: int, touched: int, mx=False) -> int:
    if mx:
        return weight_bytes(touched * H * I, mx) + token_bytes(T * k * I, mx) + T * k * H * BF16
    return touched * H * I * BF16 + T * k * I * BF16 + T * k * H * BF16
