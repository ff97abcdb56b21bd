"""GPU parity of the block-scaled layers at the decode and prefill workloads'
full sizes (H = I = 4096, E = 64, top_k = 8; T = 8 and T = 4096) and at the
fine-grained workload's T = 1024 (H = 7168, I = 2048, E = 256, top_k = 8: 32
rows per expert, one-CTA 128-token units), in the launch configuration the
benchmark times: the MXFP8 layer, MXFP4 weights with MXFP8 tokens, the MXFP4
layer and the NVFP4 layer.

The outputs of sampled tokens (every token at T = 8, 32 spread over the larger
batches) are compared with the oracle's layer of the same format within the
layer tolerance.  The oracle quantizes only the weights of
the experts its own routing selects for the sampled tokens (in parallel; the
other experts' codes stay zero and a correct routing never reads them).
"""
import concurrent.futures as cf
import gc

import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
from mixture_experts_layer_rmsnorm_gb300 import inputs

pytestmark = pytest.mark.gpu

FORMATS = ["mxfp8", "mxfp4", "mxfp4a4", "nvfp4"]


@pytest.fixture(scope="module")
def o():
    return oracle.default()


@pytest.fixture(scope="module")
def layer():
    cfg = inputs.WORKLOADS["prefill_T4096"]  # decode and prefill share the layer's weights
    li = inputs.make_layer_inputs(inputs.LayerConfig(T=1, H=cfg.H, I=cfg.I, E=cfg.E, top_k=cfg.top_k, seed=cfg.seed))
    dl = gu.DeviceLayer(li, max_tokens=4096)
    _quantize_all(dl)
    yield dl
    del dl
    gc.collect()
    torch.cuda.empty_cache()


class OracleWeights:
    """The oracle's quantized copies of a layer's expert weights, filled in per
    expert on demand (zero elsewhere)."""

    def __init__(self, o, li, fmt):
        self.o, self.li, self.fmt = o, li, fmt
        E, two_i, H = li.w13.shape
        I = two_i // 2
        bs = 16 if fmt == "nvfp4" else 32
        self.w13c = np.zeros((E, two_i, H), np.uint8)
        self.w13s = np.zeros((E, two_i, H // bs), np.uint8)
        self.w2c = np.zeros((E, H, I), np.uint8)
        self.w2s = np.zeros((E, H, I // bs), np.uint8)
        self.w13g = np.ones(E, np.float32)
        self.w2g = np.ones(E, np.float32)
        self.done = set()

    def _one(self, e):
        o, li = self.o, self.li
        if self.fmt == "nvfp4":
            self.w13c[e], self.w13s[e], g13 = o.nv4_quantize(li.w13[e], per_row=False)
            self.w2c[e], self.w2s[e], g2 = o.nv4_quantize(li.w2[e], per_row=False)
            self.w13g[e], self.w2g[e] = g13[0], g2[0]
        else:
            q = o.mx_quantize if self.fmt == "mxfp8" else o.mx4_quantize
            self.w13c[e], self.w13s[e] = q(li.w13[e])
            self.w2c[e], self.w2s[e] = q(li.w2[e])

    def ensure(self, experts):
        todo = sorted(set(int(e) for e in experts) - self.done)
        with cf.ThreadPoolExecutor(max_workers=max(1, min(16, len(todo)))) as ex:
            list(ex.map(self._one, todo))
        self.done.update(todo)

    def forward(self, x, sample):
        o, c = self.o, self.li.cfg
        args = (x, self.li.g, self.li.w_router, self.li.bias)
        if self.fmt == "nvfp4":
            return o.moe_forward_nv4(*args, self.w13c, self.w13s, self.w13g, self.w2c, self.w2s, self.w2g, c.top_k,
                                     c.renormalize, c.eps, sample=sample)
        fwd = {"mxfp8": o.moe_forward_mx, "mxfp4": o.moe_forward_mx4, "mxfp4a4": o.moe_forward_mx4a4}[self.fmt]
        return fwd(*args, self.w13c, self.w13s, self.w2c, self.w2s, c.top_k, c.renormalize, c.eps, sample=sample)


_cache = {}


def _quantize_all(dl):
    dl.layer.quantize_mx()
    dl.layer.quantize_mxfp4()
    dl.layer.quantize_nvfp4()
    torch.cuda.synchronize()


@pytest.fixture(scope="module")
def finegrained_layer():
    cfg = inputs.WORKLOADS["finegrained_T1024"]
    li = inputs.make_layer_inputs(inputs.LayerConfig(T=1, H=cfg.H, I=cfg.I, E=cfg.E, top_k=cfg.top_k, seed=cfg.seed))
    dl = gu.DeviceLayer(li, max_tokens=1024)
    _quantize_all(dl)
    yield dl
    del dl
    gc.collect()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("T", [8, 4096])
@pytest.mark.parametrize("fmt", FORMATS)
def test_block_scaled_full(layer, o, fmt, T):
    if fmt not in _cache:
        _cache[fmt] = OracleWeights(o, layer.li, fmt)
    _check(layer, o, fmt, T, _cache[fmt])


@pytest.mark.parametrize("fmt", FORMATS)
def test_block_scaled_finegrained(finegrained_layer, o, fmt):
    # the oracle's weight copies of this layer (11 GB per format) are not kept,
    # nor those of the decode/prefill layer from here on
    _cache.clear()
    _check(finegrained_layer, o, fmt, 1024, OracleWeights(o, finegrained_layer.li, fmt))
    gc.collect()


def _check(layer, o, fmt, T, ow):
    li = layer.li
    cfg = inputs.LayerConfig(T=T, H=li.cfg.H, I=li.cfg.I, E=li.cfg.E, top_k=li.cfg.top_k, seed=li.cfg.seed)
    x = inputs.make_tokens(cfg)
    L = layer.layer
    xd = gu.dev_bf16(x)
    if fmt == "mxfp8":
        y = L.forward_mx(xd)
    elif fmt == "nvfp4":
        y = L.forward_nvfp4(xd)
    else:
        y = L.forward_mxfp4(xd, fp4_tokens=fmt == "mxfp4a4")
    torch.cuda.synchronize()
    st, det = L.device_status(T)
    assert st == 0, (st, det)
    yb = y.cpu().numpy().view(np.uint16)
    # every token of a decode batch; 32 tokens spread over a prefill-size batch
    sample = np.unique(np.linspace(0, T - 1, min(T, 32)).astype(np.int64))
    # the experts the oracle's own routing gives the sampled tokens
    _, logits, _ = o.route_f32(x[sample], li.g, li.cfg.eps, li.w_router, li.bias)
    experts = np.unique(o.topk(logits, li.cfg.top_k))
    ow.ensure(experts)
    r = ow.forward(x, sample)
    assert set(np.unique(r["ids"]).tolist()) <= ow.done
    err = gu.widen(yb[sample]) - r["y64"]
    rel = np.linalg.norm(err) / np.linalg.norm(r["y64"])
    assert rel <= gu.REL_FRO_TOL, f"relative Frobenius error {rel:.3e}"
    assert np.abs(err).max() <= gu.MAX_ABS_TOL
