"""The layer forward inside a CUDA graph.

A serving loop captures a decode step once and replays it.  Every entry point
is asynchronous on the given stream, allocates nothing and makes no host
synchronisation, so it can be captured with stream capture (here through
torch.cuda.graph).  The tensor maps and scalars are taken when the call is
made, at capture time; the data are read from the caller's buffers at replay.

For each entry point and shape this test:
  - captures one call, replays it, and checks that the output is bit for bit
    the output of the same call made directly (same kernels, same inputs);
  - writes a second batch into the same input buffer, replays again, and
    checks the result against a direct call on that batch (the graph reads
    the buffer's current contents);
  - checks the device error word afterwards.
"""
import numpy as np
import pytest
import torch

import gpu_util as gu
from mixture_experts_layer_rmsnorm_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

SHAPES = [
    # name, T, H, I, E, k
    ("one_token", 1, 1024, 512, 16, 4),
    ("decode", 24, 1024, 512, 16, 4),
    ("prefill_pairs", 700, 512, 384, 8, 2),
]


def _layer(T, H, I, E, k, seed=31):
    cfg = inputs.LayerConfig(T=T, H=H, I=I, E=E, top_k=k, seed=seed)
    li = inputs.make_layer_inputs(cfg)
    return cfg, gu.DeviceLayer(li, max_tokens=T)


def _check_graph(call, x, x_next, T, H, layer):
    y_direct = torch.empty((T, H), dtype=torch.int16, device="cuda")
    y_graph = torch.full((T, H), -1, dtype=torch.int16, device="cuda")
    call(x, y_direct)  # also sets every launch's one-time configuration
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(x, y_graph)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y_graph, y_direct), int((y_graph != y_direct).sum())
    # a new batch in the captured input buffer
    x.copy_(x_next)
    call(x, y_direct)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y_graph, y_direct), int((y_graph != y_direct).sum())
    st, det = layer.device_status(T)
    assert st == binding.MOE_OK, det


@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
def test_forward_in_graph(shape):
    _, T, H, I, E, k = shape
    cfg, dl = _layer(T, H, I, E, k)
    x = gu.dev_bf16(inputs.make_tokens(cfg, batch_index=1))
    x_next = gu.dev_bf16(inputs.make_tokens(cfg, batch_index=2))
    _check_graph(lambda a, b: dl.layer.forward(a, b), x, x_next, T, H, dl.layer)


@pytest.mark.parametrize("variant", ["fused_front", "fused_combine", "fused_mlp"])
def test_variants_in_graph(variant):
    cfg, dl = _layer(24, 1024, 512, 16, 4)
    x = gu.dev_bf16(inputs.make_tokens(cfg, batch_index=1))
    x_next = gu.dev_bf16(inputs.make_tokens(cfg, batch_index=2))
    _check_graph(lambda a, b: dl.layer.forward(a, b, **{variant: True}), x, x_next, 24, 1024, dl.layer)


@pytest.mark.parametrize("fmt", ["mx", "mxfp4", "mxfp4a4", "nvfp4"])
def test_block_scaled_in_graph(fmt):
    cfg, dl = _layer(24, 1024, 512, 16, 4)
    L = dl.layer
    if fmt == "mx":
        L.quantize_mx()
        call = lambda a, b: L.forward_mx(a, b)  # noqa: E731
    elif fmt == "nvfp4":
        L.quantize_nvfp4()
        call = lambda a, b: L.forward_nvfp4(a, b)  # noqa: E731
    else:
        L.quantize_mxfp4()
        call = lambda a, b: L.forward_mxfp4(a, b, fp4_tokens=(fmt == "mxfp4a4"))  # noqa: E731
    x = gu.dev_bf16(inputs.make_tokens(cfg, batch_index=1))
    x_next = gu.dev_bf16(inputs.make_tokens(cfg, batch_index=2))
    _check_graph(call, x, x_next, 24, 1024, L)
