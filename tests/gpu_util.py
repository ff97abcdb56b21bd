"""Helpers of the GPU parity tests: run the CUDA path through the C ABI on
seeded inputs, read back its intermediates, compare with the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

from mixture_experts_layer_rmsnorm_gb300 import binding, inputs

# spec tolerance of the layer output against the fp64 oracle
REL_FRO_TOL = 5e-3
MAX_ABS_TOL = 3e-2
PAD = 16


def dev_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to("cuda")


def dev_f32(a: np.ndarray | None):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda")


def widen(bits: np.ndarray) -> np.ndarray:
    return inputs.bf16_bits_to_f32(np.asarray(bits, dtype=np.uint16)).astype(np.float64)


class DeviceLayer:
    """A layer's weights on the GPU (from host arrays of the input generator)."""

    def __init__(self, li: inputs.LayerInputs, max_tokens: int | None = None):
        c = li.cfg
        self.li = li
        self.layer = binding.MoeLayer(dev_bf16(li.g), dev_f32(li.w_router), dev_bf16(li.w13), dev_bf16(li.w2),
                                      c.top_k, c.renormalize, c.eps, router_bias=dev_f32(li.bias),
                                      max_tokens=max_tokens or c.T)

    def run(self, x: np.ndarray, fused_front: bool = False) -> dict:
        c = self.li.cfg
        T, H, I, E, k = x.shape[0], c.H, c.I, c.E, c.top_k
        xd = dev_bf16(x)
        y = self.layer.forward(xd, fused_front=fused_front)
        torch.cuda.synchronize()
        st, det = self.layer.device_status(T)
        assert st == binding.MOE_OK, f"device status {st} {det}"
        L = self.layer
        v = L.views(T)
        out = {"y": y.cpu().numpy().view(np.uint16)}
        if T == 0:
            return out
        out["h"] = L.view_tensor(T, "h", torch.int16, (T, H)).cpu().numpy().view(np.uint16)
        out["logits"] = L.view_tensor(T, "logits", torch.float32, (T, E)).cpu().numpy()
        out["ids"] = L.view_tensor(T, "topk_ids", torch.int32, (T, k)).cpu().numpy()
        out["w"] = L.view_tensor(T, "topk_w", torch.float32, (T, k)).cpu().numpy()
        out["counts"] = L.view_tensor(T, "counts", torch.int32, (E,)).cpu().numpy()
        out["offsets"] = L.view_tensor(T, "offsets", torch.int32, (E + 1,)).cpu().numpy()
        P = int(out["offsets"][-1])
        out["sorted"] = L.view_tensor(T, "sorted_ids", torch.int32, (v.P_max,)).cpu().numpy()[:P]
        out["slot"] = L.view_tensor(T, "slot_of", torch.int32, (T * k,)).cpu().numpy()
        out["P_max"] = v.P_max
        self._P = P
        return out

    def act_rows(self, T, rows):
        c = self.li.cfg
        v = self.layer.views(T)
        a = self.layer.view_tensor(T, "act", torch.int16, (v.P_max, c.I))
        o = self.layer.view_tensor(T, "out_rows", torch.int16, (v.P_max, c.H))
        idx = torch.as_tensor(np.asarray(rows, dtype=np.int64), device="cuda")
        return a[idx].cpu().numpy().view(np.uint16), o[idx].cpu().numpy().view(np.uint16)


def check_routing(o, li: inputs.LayerInputs, x: np.ndarray, g: dict, pad: int = PAD):
    """Bit-exact checks of h, logits, expert ids and the align outputs; the
    routing weights within fp32 rounding of the oracle's fp64 softmax."""
    c = li.cfg
    h32, l32, _ = o.route_f32(x, li.g, c.eps, li.w_router, li.bias)
    assert np.array_equal(g["h"], h32), "RMSNorm output differs from the oracle's fp32 path"
    assert np.array_equal(g["logits"].view(np.uint32), l32.view(np.uint32)), "router logits differ"
    ids = o.topk(l32, c.top_k)
    assert np.array_equal(g["ids"], ids), "selected experts differ"
    l64 = o.router_logits_f64(h32, li.w_router, li.bias)
    w_ref = o.route_weights_f64(l64, ids, c.renormalize)
    assert np.allclose(g["w"], w_ref, rtol=2e-5, atol=1e-7), f"weights: max err {np.abs(g['w'] - w_ref).max()}"
    counts, offsets, sorted_ids, slot_of = o.align(ids, c.E, pad)
    assert np.array_equal(g["counts"], counts)
    assert np.array_equal(g["offsets"], offsets)
    assert np.array_equal(g["sorted"], sorted_ids)
    assert np.array_equal(g["slot"], slot_of)
    return ids


def check_output(o, li: inputs.LayerInputs, x: np.ndarray, y_bits: np.ndarray, sample=None, nthreads=None):
    c = li.cfg
    r = o.moe_forward(x, li.g, li.w_router, li.bias, li.w13, li.w2, c.top_k, c.renormalize, c.eps,
                      sample=sample, nthreads=nthreads)
    rows = r["sample"]
    yg = widen(y_bits[rows])
    y64 = r["y64"]
    err = yg - y64
    rel = np.linalg.norm(err) / max(np.linalg.norm(y64), 1e-30)
    mx = np.abs(err).max() if err.size else 0.0
    assert rel <= REL_FRO_TOL, f"relative Frobenius error {rel:.3e} > {REL_FRO_TOL}"
    assert mx <= MAX_ABS_TOL, f"max abs error {mx:.3e} > {MAX_ABS_TOL}"
    return rel, mx


def ungroup_mx_scales(buf: np.ndarray, rows: int, K: int) -> np.ndarray:
    """Scales in the block-scaled MMA's tile layout (512 bytes per 128-row group
    and 128-element chunk: byte r*16 + 4*j + b = row 32*j + r, block b) ->
    [rows, K/32] in scale-row order."""
    ng, kc = rows // 128, K // 128
    t = np.asarray(buf, np.uint8)[: ng * kc * 512].reshape(ng, kc, 32, 4, 4)  # [g][c][r][j][b]
    return t.transpose(0, 3, 2, 1, 4).reshape(ng * 128, kc * 4)


def w13_scale_rows(E: int, I: int) -> np.ndarray:
    """Scale row of each W13 row (e*2I + i): the gate/up GEMM's tile-row order."""
    i = np.arange(2 * I)
    up, f = i // I, i % I
    m = 32 * ((f % 64) // 16) + 16 * up + f % 16
    R = [(e * (I // 64) + f // 64) * 128 + m for e in range(E)]
    return np.concatenate(R)
