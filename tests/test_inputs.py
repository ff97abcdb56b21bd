"""The seeded input generator against a pure-Python restatement of its
published definition (splitmix64 finaliser, Box-Muller, round to nearest)."""
import math

import numpy as np
import torch

from mixture_experts_layer_rmsnorm_gb300 import inputs

M64 = (1 << 64) - 1


def _mix64(z):
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def _normal(seed, stream, i):
    base = _mix64(seed ^ ((stream * 0xD1B54A32D192ED03) & M64))
    def u(c):
        r = _mix64((base + (c + 1) * 0x9E3779B97F4A7C15) & M64)
        return ((r >> 11) + 1) * 2.0 ** -53
    p = i // 2
    rad = math.sqrt(-2.0 * math.log(u(2 * p)))
    th = 2.0 * math.pi * u(2 * p + 1)
    return rad * math.sin(th) if i & 1 else rad * math.cos(th)


def test_generator_matches_definition():
    n = 257
    got = inputs.normal_f32(5, 3, (n,), 0.25, 2.0)
    want = np.array([0.25 + 2.0 * _normal(5, 3, i) for i in range(n)], dtype=np.float32)
    assert np.array_equal(got, want)
    gb = inputs.normal_bf16(5, 3, (n,), 0.25, 2.0)
    wb = torch.from_numpy(want).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(gb, wb)


def test_generator_thread_independent_and_streams_differ():
    a = inputs.normal_bf16(0, 4, (100003,))
    lib = inputs._load()
    b = np.empty(100003, np.uint16)
    lib.moe_gen_normal_bf16(0, 4, 100003, 0.0, 1.0, b.ctypes.data, 1)
    assert np.array_equal(a, b)
    c = inputs.normal_bf16(0, 5, (100003,))
    assert not np.array_equal(a, c)


def test_distributions():
    x = inputs.bf16_bits_to_f32(inputs.normal_bf16(0, 1, (1 << 20,)))
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1) < 5e-3
    w = inputs.normal_f32(0, 3, (1 << 20,), 0.0, 0.02)
    assert abs(w.std() - 0.02) < 1e-4


def test_zipf_bias():
    b = inputs.zipf_router_bias(7, 128, 1.2)
    p = np.exp(b.astype(np.float64))
    assert abs(p.sum() - 1) < 1e-5
    s = np.sort(p)[::-1]
    r = np.arange(1, 129)
    assert np.allclose(s, r ** -1.2 / (r ** -1.2).sum(), rtol=1e-5)
    assert len(set(np.argsort(-b)[:5])) == 5
