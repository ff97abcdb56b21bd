"""Seeded synthetic inputs for the fused MoE layer workloads.

This module is the one place both sides of a parity check get their inputs
from: the CUDA path's callers (bench, GPU tests) and the CPU oracle's callers.
It holds none of the MoE method's arithmetic: it only draws numbers from the
counter-based generator defined in ``moe_gen.c`` (splitmix64 -> Box-Muller ->
round to fp32 / bf16) and lays them out in the tensor shapes of the layer.

Tensor streams (one generator stream per tensor, all from the same seed):
  1 x[T,H] bf16        N(0, 1)
  2 g_norm[H] bf16     1 + N(0, 0.1)
  3 W_router[E,H] f32  N(0, 0.02)
  4 W13[E,2I,H] bf16   N(0, 0.02)   rows [0,I) gate, rows [I,2I) up
  5 W2[E,H,I] bf16     N(0, 0.02)
  6 router-bias expert permutation (skewed-routing workload only)
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_gen.c")
_LIB = os.path.join(_HERE, "libmoegen.so")
_lock = threading.Lock()
_lib = None

STREAM_X, STREAM_G, STREAM_WR, STREAM_W13, STREAM_W2, STREAM_BIAS_PERM = 1, 2, 3, 4, 5, 6


def build_lib(force: bool = False) -> str:
    """Compile the generator with the host C compiler (no CUDA involved)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build_lib())
            u64, p = ctypes.c_uint64, ctypes.c_void_p
            lib.moe_gen_normal_bf16.argtypes = [u64, u64, u64, ctypes.c_double, ctypes.c_double, p, ctypes.c_int]
            lib.moe_gen_normal_f32.argtypes = [u64, u64, u64, ctypes.c_double, ctypes.c_double, p, ctypes.c_int]
            lib.moe_gen_u64.argtypes = [u64, u64, u64, p, ctypes.c_int]
            _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal_bf16(seed: int, stream: int, shape, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """Raw bf16 bits (uint16) of N(mean, std) draws, element i from counter i."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.uint16)
    if n:
        _load().moe_gen_normal_bf16(seed, stream, n, mean, std, out.ctypes.data, _threads())
    return out.reshape(shape)


def normal_f32(seed: int, stream: int, shape, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.float32)
    if n:
        _load().moe_gen_normal_f32(seed, stream, n, mean, std, out.ctypes.data, _threads())
    return out.reshape(shape)


def raw_u64(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    if n:
        _load().moe_gen_u64(seed, stream, n, out.ctypes.data, 1)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen raw bf16 bits to float32 (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def zipf_router_bias(seed: int, E: int, s: float = 1.2) -> np.ndarray:
    """Per-expert router bias for the skewed-routing workload.

    The experts are put in a seeded random order (Fisher-Yates driven by
    stream 6); the expert of rank r (1-based) gets bias ln(p_r) with
    p_r = r^-s / sum_q q^-s, a Zipf(s) law over ranks.
    """
    r = raw_u64(seed, STREAM_BIAS_PERM, E)
    perm = list(range(E))
    for i in range(E - 1, 0, -1):
        j = int(r[i] % np.uint64(i + 1))
        perm[i], perm[j] = perm[j], perm[i]
    z = sum(q ** (-s) for q in range(1, E + 1))
    bias = np.empty(E, dtype=np.float64)
    for rank in range(1, E + 1):
        bias[perm[rank - 1]] = math.log((rank ** (-s)) / z)
    return bias.astype(np.float32)


@dataclass
class LayerConfig:
    """One MoE layer workload: shapes, routing options and seed."""
    T: int
    H: int
    I: int
    E: int
    top_k: int
    renormalize: bool = True
    eps: float = 1e-6
    seed: int = 0
    zipf_bias: float | None = None  # Zipf exponent of the router bias, or None
    name: str = ""

    def key(self) -> str:
        return self.name or f"T{self.T}_H{self.H}_I{self.I}_E{self.E}_k{self.top_k}"


@dataclass
class LayerInputs:
    cfg: LayerConfig
    x: np.ndarray         # [T,H] uint16 (bf16 bits)
    g: np.ndarray         # [H] uint16
    w_router: np.ndarray  # [E,H] float32
    bias: np.ndarray | None  # [E] float32
    w13: np.ndarray       # [E,2I,H] uint16
    w2: np.ndarray        # [E,H,I] uint16
    extra: dict = field(default_factory=dict)


def make_weights(cfg: LayerConfig):
    """Layer parameters (router, expert weights, norm gain, optional bias)."""
    s = cfg.seed
    g = normal_bf16(s, STREAM_G, (cfg.H,), 1.0, 0.1)
    wr = normal_f32(s, STREAM_WR, (cfg.E, cfg.H), 0.0, 0.02)
    w13 = normal_bf16(s, STREAM_W13, (cfg.E, 2 * cfg.I, cfg.H), 0.0, 0.02)
    w2 = normal_bf16(s, STREAM_W2, (cfg.E, cfg.H, cfg.I), 0.0, 0.02)
    bias = zipf_router_bias(s, cfg.E, cfg.zipf_bias) if cfg.zipf_bias is not None else None
    return g, wr, bias, w13, w2


def make_tokens(cfg: LayerConfig, batch_index: int = 0) -> np.ndarray:
    """Token activations x[T,H]; batch_index selects an independent batch."""
    stream = STREAM_X if batch_index == 0 else (STREAM_X + 1000 * batch_index)
    return normal_bf16(cfg.seed, stream, (cfg.T, cfg.H), 0.0, 1.0)


def make_layer_inputs(cfg: LayerConfig) -> LayerInputs:
    g, wr, bias, w13, w2 = make_weights(cfg)
    return LayerInputs(cfg=cfg, x=make_tokens(cfg), g=g, w_router=wr, bias=bias, w13=w13, w2=w2)


# The workloads of the layer (shapes, distributions, seeds) by name.
WORKLOADS = {
    "tiny": LayerConfig(T=4, H=128, I=256, E=8, top_k=2, seed=0, name="tiny"),
    "decode_T1": LayerConfig(T=1, H=4096, I=4096, E=64, top_k=8, seed=0, name="decode_T1"),
    "decode_T8": LayerConfig(T=8, H=4096, I=4096, E=64, top_k=8, seed=0, name="decode_T8"),
    "decode_T32": LayerConfig(T=32, H=4096, I=4096, E=64, top_k=8, seed=0, name="decode_T32"),
    "decode_T64": LayerConfig(T=64, H=4096, I=4096, E=64, top_k=8, seed=0, name="decode_T64"),
    "prefill_T4096": LayerConfig(T=4096, H=4096, I=4096, E=64, top_k=8, seed=0, name="prefill_T4096"),
    "finegrained_T16": LayerConfig(T=16, H=7168, I=2048, E=256, top_k=8, seed=0, name="finegrained_T16"),
    "finegrained_T128": LayerConfig(T=128, H=7168, I=2048, E=256, top_k=8, seed=0, name="finegrained_T128"),
    "finegrained_T1024": LayerConfig(T=1024, H=7168, I=2048, E=256, top_k=8, seed=0, name="finegrained_T1024"),
    "skewed_T512": LayerConfig(T=512, H=4096, I=1408, E=128, top_k=6, seed=7, zipf_bias=1.2, name="skewed_T512"),
}
