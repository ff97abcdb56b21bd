"""Helpers of the GPU parity tests: run the CUDA path through the C ABI on
seeded inputs, read back its intermediates, compare with the CPU oracle."""
from __future__ import annotations

import concurrent.futures as cf
import json
import os

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


# the fp64 logit gap below which the fp32 router may order two experts
# differently from exact arithmetic (its summation error is ~1e-6 at H = 4096)
SELECTION_GAP_TOL = 1e-5


def _report(record: dict):
    """Append a JSON line to the file named by MOE_TEST_REPORT (if set)."""
    path = os.environ.get("MOE_TEST_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(record) + "\n")


def boundary_gaps(l64: np.ndarray, k: int) -> np.ndarray:
    """Per token, the fp64 gap between the k-th and (k+1)-th largest logit
    (inf when k = E)."""
    if k >= l64.shape[1]:
        return np.full(l64.shape[0], np.inf)
    srt = -np.sort(-l64, axis=1)
    return srt[:, k - 1] - srt[:, k]


def check_selection_f64(o, li: inputs.LayerInputs, x: np.ndarray, h_gpu: np.ndarray, ids_gpu: np.ndarray,
                        label: str = ""):
    """The GPU's expert choice against an exact-arithmetic selection, independent
    of the fp32 summation order the kernel and the oracle's fp32 path share.

    (a) fp64 logits of the GPU's h (bit-equal to the oracle's fp32-path h),
        selected by the oracle's fp64 top-k (largest first, ties to the lower
        index): wherever the GPU's j-th expert differs from the fp64 j-th, the
        two experts' fp64 logits must lie within SELECTION_GAP_TOL.
    (b) the same from the fp64 RMSNorm's h (rounded once to bf16): the two h
        differ by at most one bf16 step at a few elements, which moves logit e
        by at most d_e = sum_j |Wr[e,j]| |dh_j| (computed exactly); a swap of
        experts a and b must then lie within SELECTION_GAP_TOL + d_a + d_b.
    Returns the smallest fp64 boundary gap (k-th minus (k+1)-th logit) over the
    tokens, which shows how close the batch came to a tie."""
    c = li.cfg
    k = c.top_k
    rows = np.arange(x.shape[0])[:, None]
    l64 = o.router_logits_f64(h_gpu, li.w_router, li.bias)
    ids64 = o.topk(l64, k)
    diff = ids_gpu != ids64
    gap = np.abs(l64[rows, ids_gpu] - l64[rows, ids64])
    assert (gap[diff] <= SELECTION_GAP_TOL).all(), \
        f"GPU selection differs from the fp64 top-k at fp64 gaps up to {gap[diff].max():.3e}"
    h64, _ = o.rmsnorm_f64(x, li.g, c.eps)
    l64b = o.router_logits_f64(h64, li.w_router, li.bias)
    ids64b = o.topk(l64b, k)
    dh = np.abs(widen(h64) - widen(h_gpu))
    dl = dh @ np.abs(li.w_router.astype(np.float64)).T  # [T, E]: bound on each logit's move
    diffb = ids_gpu != ids64b
    gapb = np.abs(l64b[rows, ids_gpu] - l64b[rows, ids64b])
    tolb = SELECTION_GAP_TOL + dl[rows, ids_gpu] + dl[rows, ids64b]
    assert (gapb[diffb] <= tolb[diffb]).all(), "GPU selection differs from the fp64-norm top-k beyond the h bound"
    gaps = boundary_gaps(l64, k)
    min_gap = float(gaps.min()) if gaps.size else float("inf")
    _report({"check": "selection_f64", "label": label, "T": int(x.shape[0]), "E": int(c.E), "k": int(k),
             "min_boundary_gap": min_gap, "swaps_vs_f64": int(diff.sum()), "swaps_vs_f64_norm": int(diffb.sum()),
             "h_elems_differing_from_f64_norm": int((dh > 0).sum())})
    return min_gap


def check_routing(o, li: inputs.LayerInputs, x: np.ndarray, g: dict, pad: int = PAD, label: str = ""):
    """Bit-exact checks of h, logits, expert ids and the align outputs against
    the oracle's fp32 path; the expert ids against an fp64 selection (gap rule
    of check_selection_f64); the routing weights within fp32 rounding of the
    oracle's fp64 softmax."""
    c = li.cfg
    h32, l32, _ = o.route_f32(x, li.g, c.eps, li.w_router, li.bias)
    assert np.array_equal(g["h"], h32), "RMSNorm output differs from the oracle's fp32 path"
    assert np.array_equal(g["logits"].view(np.uint32), l32.view(np.uint32)), "router logits differ"
    ids = o.topk(l32, c.top_k)
    assert np.array_equal(g["ids"], ids), "selected experts differ"
    check_selection_f64(o, li, x, g["h"], g["ids"], label)
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


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (8 significant bits; subnormal spacing below 2^-126)."""
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def round_bf16(v: np.ndarray) -> np.ndarray:
    """fp64 values rounded once to bf16 (nearest, ties to even), as fp64; normal range only."""
    m, e = np.frexp(np.asarray(v, np.float64))
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


def check_expert_rows(o, li: inputs.LayerInputs, dl: "DeviceLayer", T: int, g: dict, ids: np.ndarray, rows,
                      threads: int | None = None, label: str = ""):
    """The GPU's SwiGLU activation and expert-output rows against the oracle's
    expert on the same bf16 h, element by element.

    act: the oracle rounds its fp64 activation to bf16 once, the GPU its fp32
    one; every element must be within one bf16 step of the larger of the two
    plus 1e-5 of the row's largest value (fp32 accumulation noise near zero),
    and at least 99% bit-equal.
    out: the GPU rounds its fp32 sum of act x W2 to bf16; the reference is the
    oracle's fp64 output rounded once to bf16.  Every element within one bf16
    step plus 1e-5 of the row maximum plus the exact effect of the GPU's act
    differences (sum_i |W2[n,i]| |d act_i|).  At least 99% of the elements
    bit-equal to that reference, or, where the GPU's act differs from the
    oracle's, to the down projection of the GPU's own act in exact (fp64)
    arithmetic rounded once to bf16: at K = 4096 the act differences alone
    move a few percent of the outputs across a bf16 rounding boundary."""
    k = li.cfg.top_k
    rows = np.asarray(rows, np.int64)
    if rows.size == 0:
        return
    act, out = dl.act_rows(T, rows)
    items = []
    for r_i, p in enumerate(rows):
        t, j = divmod(int(g["sorted"][p]), k)
        items.append((r_i, int(p), t, int(ids[t, j])))

    def ref(it):
        _, _, t, e = it
        return o.expert_f64(g["h"][t], li.w13[e], li.w2[e], round_act=True)

    with cf.ThreadPoolExecutor(max_workers=threads or max(1, min(16, os.cpu_count() or 1))) as ex:
        refs = list(ex.map(ref, items))
    eq_a = eq_o = n_a = n_o = 0
    by_e: dict[int, list] = {}
    for it, rf in zip(items, refs):
        by_e.setdefault(it[3], []).append((it, rf))
    for e, lst in by_e.items():
        for (r_i, p, t, _), (a_ref, o_ref) in lst:
            a_g = widen(act[r_i])
            da = np.abs(a_g - a_ref)
            tol_a = bf16_ulp(np.maximum(np.abs(a_ref), np.abs(a_g))) + 1e-5 * np.abs(a_ref).max()
            assert (da <= tol_a).all(), f"{label} act row {p} (token {t}, expert {e}): max excess {(da - tol_a).max():.3e}"
            o16 = round_bf16(o_ref)
            o_g = widen(out[r_i])
            do = np.abs(o_g - o16)
            nz = np.nonzero(da)[0]  # the act elements that differ (few): their exact effect on every output
            prop = np.abs(widen(li.w2[e][:, nz])) @ da[nz] if nz.size else 0.0
            tol_o = bf16_ulp(np.maximum(np.abs(o16), np.abs(o_g))) + 1e-5 * np.abs(o_ref).max() + prop
            assert (do <= tol_o).all(), f"{label} out row {p} (token {t}, expert {e}): max excess {(do - tol_o).max():.3e}"
            eq = do == 0
            miss = np.nonzero(~eq)[0]
            if miss.size and nz.size:
                own = round_bf16(widen(li.w2[e][miss]) @ a_g)  # exact down projection of the GPU's act
                eq[miss] = o_g[miss] == own
            eq_a += int((da == 0).sum()); n_a += da.size
            eq_o += int(eq.sum()); n_o += do.size
    assert eq_a >= 0.99 * n_a, f"{label} act: only {eq_a / n_a:.4f} of elements bit-equal"
    assert eq_o >= 0.99 * n_o, f"{label} out: only {eq_o / n_o:.4f} of elements bit-equal"
    _report({"check": "expert_rows", "label": label, "T": int(T), "rows": int(rows.size),
             "act_bit_equal": eq_a / n_a, "out_bit_equal": eq_o / n_o})


def rows_per_expert(offsets: np.ndarray, sorted_ids: np.ndarray, n_routed: int, positions=(0, -1)) -> np.ndarray:
    """Real rows of every expert's list at the given positions within the list
    (negative: from the end), e.g. its first and last routed rows."""
    out = []
    for e in range(offsets.size - 1):
        seg = np.arange(offsets[e], offsets[e + 1])
        seg = seg[sorted_ids[seg] < n_routed]
        if seg.size == 0:
            continue
        for q in positions:
            if -seg.size <= q < seg.size:
                out.append(seg[q])
    return np.unique(np.asarray(out, np.int64))
