"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times.

Routing (h, logits, expert ids, align) is checked bit for bit for every token,
and the expert ids against an fp64 selection; the layer output on every token
of the decode batches (T <= 128) and on samples of the larger batches that the
oracle computes one by one; the SwiGLU activation and expert output rows of
several rows of every touched expert, element by element.
Workloads: decode (H = I = 4096, E = 64, top_k = 8; T = 1, 8, 32, 64),
prefill (same shapes, T = 4096), fine-grained (H = 7168, I = 2048, E = 256,
top_k = 8; T = 16, 128, 1024) and skewed routing (H = 4096, I = 1408,
E = 128, top_k = 6, T = 512, Zipf(1.2) router bias, seed 7).

The prefill sample (at least 256 tokens) is chosen from the routing so that,
in every expert's list, every 256-row token chunk of the prefill tile plan,
both halves of each chunk (the two CTAs of a pair each take one half), each
expert's last partial chunk and every row position 0..255 within a chunk
are reached by at least one sampled token.
"""
import gc

import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
from mixture_experts_layer_rmsnorm_gb300 import inputs

pytestmark = pytest.mark.gpu

PREFILL_CHUNK = 256  # token rows per unit of the prefill tile plan (a CTA pair: two halves)


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


def _spread(T, n):
    return np.unique(np.linspace(0, T - 1, min(T, n)).astype(np.int64))


def chunk_cover_sample(g: dict, T: int, k: int, n_min: int, chunk: int = PREFILL_CHUNK) -> np.ndarray:
    """Tokens whose routed rows reach every (expert, chunk, half) cell, every
    row position within a chunk and every expert's last chunk (greedy cover),
    topped up with evenly spread tokens to at least n_min."""
    offsets, srt = g["offsets"], g["sorted"]
    N = T * k
    feats_of_token = [set() for _ in range(T)]
    for e in range(offsets.size - 1):
        n_e = int(offsets[e + 1] - offsets[e])
        last_chunk = (n_e - 1) // chunk if n_e else -1
        for r in range(n_e):
            sid = int(srt[offsets[e] + r])
            if sid >= N:
                continue
            c, pos = divmod(r, chunk)
            rows_c = min(chunk, n_e - c * chunk)
            half = (rows_c + 31) // 32 * 32 // 2
            t = sid // k
            feats_of_token[t].add(("cell", e, c, pos >= half))
            feats_of_token[t].add(("pos", pos))
            if c == last_chunk:
                feats_of_token[t].add(("last", e))
    need = set().union(*feats_of_token)
    chosen = []
    while need:
        t = max(range(T), key=lambda i: len(feats_of_token[i] & need))
        gain = feats_of_token[t] & need
        if not gain:
            break
        chosen.append(t)
        need -= gain
    assert not need
    sample = np.unique(np.concatenate([np.asarray(chosen, np.int64), _spread(T, n_min)]))
    extra = [t for t in range(T) if t not in set(sample.tolist())]
    if sample.size < n_min:
        sample = np.unique(np.concatenate([sample, np.asarray(extra[: n_min - sample.size], np.int64)]))
    return sample


def _check_full(o, dl, li_T, x, g, T, sample, label, row_positions):
    ids = gu.check_routing(o, li_T, x, g, label=label)
    gu.check_output(o, li_T, x, g["y"], sample=sample)
    k = li_T.cfg.top_k
    rows = gu.rows_per_expert(g["offsets"], g["sorted"], T * k, row_positions)
    gu.check_expert_rows(o, li_T, dl, T, g, ids, rows, label=label)


@pytest.mark.parametrize("T", [1, 8, 32, 64, 4096])
def test_decode_prefill_full(decode_layer, o, T):
    li = decode_layer.li
    cfg = inputs.LayerConfig(T=T, H=li.cfg.H, I=li.cfg.I, E=li.cfg.E, top_k=li.cfg.top_k, seed=li.cfg.seed)
    x = inputs.make_tokens(cfg)
    g = decode_layer.run(x)
    li_T = inputs.LayerInputs(cfg=cfg, x=x, g=li.g, w_router=li.w_router, bias=None, w13=li.w13, w2=li.w2)
    if T <= 64:
        sample, positions = None, (0, -1)
    else:
        sample = chunk_cover_sample(g, T, cfg.top_k, 256)
        assert sample.size >= 256
        # both halves' first and last rows of the first chunk, the second chunk's start, the list's last row
        positions = (0, 127, 128, 255, 256, -1)
    _check_full(o, decode_layer, li_T, x, g, T, sample, f"decode_prefill_T{T}", positions)


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
    sample = None if T <= 128 else chunk_cover_sample(g, T, cfg.top_k, 64)
    # T = 1024: 32 rows per expert, one chunk each; first, middle and last rows
    _check_full(o, finegrained_layer, li_T, x, g, T, sample, f"finegrained_T{T}", (0, 15, -1))


def test_skewed_full(o):
    cfg = inputs.WORKLOADS["skewed_T512"]
    li = inputs.make_layer_inputs(cfg)
    dl = gu.DeviceLayer(li)
    g = dl.run(li.x)
    ids = g["ids"]
    counts = np.bincount(ids.reshape(-1), minlength=cfg.E)
    assert counts.max() > 8 * counts.mean() and (counts == 0).sum() > 0, "routing should be skewed"
    # every token of the hottest expert's first rows, and a cover of the hot experts' chunks
    hot = int(np.argmax(counts))
    hot_tokens = np.nonzero((ids == hot).any(axis=1))[0][:16]
    sample = np.unique(np.concatenate([hot_tokens, chunk_cover_sample(g, cfg.T, cfg.top_k, 64)]))
    assert sample.size >= 64
    _check_full(o, dl, li, li.x, g, cfg.T, sample, "skewed_T512", (0, 127, 128, 255, 256, -1))
    del dl
    _free()
