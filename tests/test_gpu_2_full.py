"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times.

Routing (h, logits, expert ids, align) is checked bit for bit for every token;
the layer output on a sample of tokens the oracle computes one by one.
Workloads: decode (H = I = 4096, E = 64, top_k = 8; T = 1, 8, 32, 64),
prefill (same shapes, T = 4096), fine-grained (H = 7168, I = 2048, E = 256,
top_k = 8; T = 16, 128, 1024) and skewed routing (H = 4096, I = 1408,
E = 128, top_k = 6, T = 512, Zipf(1.2) router bias, seed 7).
"""
import gc

import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
from mixture_experts_layer_rmsnorm_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def o():
    return oracle.default()


def _free():
    gc.collect()
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def decode_layer():
    cfg = inputs.WORKLOADS["prefill_T4096"]  # decode and prefill share the layer's weights
    li = inputs.make_layer_inputs(inputs.LayerConfig(T=1, H=cfg.H, I=cfg.I, E=cfg.E, top_k=cfg.top_k, seed=cfg.seed))
    dl = gu.DeviceLayer(li, max_tokens=4096)
    yield dl
    del dl
    _free()


def _sample(T, n):
    return np.unique(np.linspace(0, T - 1, min(T, n)).astype(np.int64))


@pytest.mark.parametrize("T", [1, 8, 32, 64, 4096])
def test_decode_prefill_full(decode_layer, o, T):
    li = decode_layer.li
    cfg = inputs.LayerConfig(T=T, H=li.cfg.H, I=li.cfg.I, E=li.cfg.E, top_k=li.cfg.top_k, seed=li.cfg.seed)
    x = inputs.make_tokens(cfg)
    g = decode_layer.run(x)
    li_T = inputs.LayerInputs(cfg=cfg, x=x, g=li.g, w_router=li.w_router, bias=None, w13=li.w13, w2=li.w2)
    gu.check_routing(o, li_T, x, g)
    gu.check_output(o, li_T, x, g["y"], sample=_sample(T, 8 if T <= 64 else 6))


@pytest.fixture(scope="module")
def finegrained_layer():
    cfg = inputs.WORKLOADS["finegrained_T1024"]
    li = inputs.make_layer_inputs(inputs.LayerConfig(T=1, H=cfg.H, I=cfg.I, E=cfg.E, top_k=cfg.top_k, seed=cfg.seed))
    dl = gu.DeviceLayer(li, max_tokens=1024)
    yield dl
    del dl
    _free()


@pytest.mark.parametrize("T", [16, 128, 1024])
def test_finegrained_full(finegrained_layer, o, T):
    li = finegrained_layer.li
    cfg = inputs.LayerConfig(T=T, H=li.cfg.H, I=li.cfg.I, E=li.cfg.E, top_k=li.cfg.top_k, seed=li.cfg.seed)
    x = inputs.make_tokens(cfg)
    g = finegrained_layer.run(x)
    li_T = inputs.LayerInputs(cfg=cfg, x=x, g=li.g, w_router=li.w_router, bias=None, w13=li.w13, w2=li.w2)
    gu.check_routing(o, li_T, x, g)
    gu.check_output(o, li_T, x, g["y"], sample=_sample(T, 4))


def test_skewed_full(o):
    cfg = inputs.WORKLOADS["skewed_T512"]
    li = inputs.make_layer_inputs(cfg)
    dl = gu.DeviceLayer(li)
    g = dl.run(li.x)
    ids = gu.check_routing(o, li, li.x, g)
    counts = np.bincount(ids.reshape(-1), minlength=cfg.E)
    assert counts.max() > 8 * counts.mean() and (counts == 0).sum() > 0, "routing should be skewed"
    # sample tokens of the hottest expert and a spread of others
    hot = int(np.argmax(counts))
    hot_tokens = np.nonzero((ids == hot).any(axis=1))[0][:3]
    sample = np.unique(np.concatenate([hot_tokens, _sample(cfg.T, 5)]))
    gu.check_output(o, li, li.x, g["y"], sample=sample)
    del dl
    _free()
