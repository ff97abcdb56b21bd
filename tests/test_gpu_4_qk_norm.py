"""GPU parity of the QK-norm kernel against the fp64 oracle.

Inputs from the seeded generator: q, k ~ N(0, 1) bf16 (some heads scaled by
powers of two, so head norms differ widely), gains N(1, 0.1) with weight bias 0
(Qwen-style) or N(0, 0.1) with weight bias 1.  The kernel computes in fp32 in
one fixed order; against the fp64 oracle every output is within one bf16 ulp and
almost all are bit-identical.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_rmsnorm_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

CASES = [
    # name, T, Hq, Hk, D, weight_bias, eps, seed
    ("decode_qwen", 1, 32, 4, 128, 0.0, 1e-6, 0),
    ("ragged_d64", 37, 8, 2, 64, 0.0, 1e-6, 1),
    ("d256_bias", 5, 4, 1, 256, 1.0, 1e-5, 2),
    ("q_only", 9, 6, 0, 128, 0.0, 1e-6, 3),
    ("k_only", 3, 0, 5, 64, 1.0, 1e-6, 4),
    ("prefill_qwen", 4096, 32, 4, 128, 0.0, 1e-6, 5),
]


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def _ulps(a, b):
    """Distance in bf16 ulps of finite values of the same sign region (bit-pattern order)."""
    def key(u):
        u = u.astype(np.int32)
        return np.where(u & 0x8000, -(u & 0x7FFF), u & 0x7FFF)
    return np.abs(key(a) - key(b))


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_qk_norm_parity(case):
    _, T, Hq, Hk, D, wb, eps, seed = case
    q = inputs.normal_bf16(seed, 31, (T, Hq, D))
    k = inputs.normal_bf16(seed, 32, (T, Hk, D))
    # spread the head norms over several binades
    scale = np.exp2(np.arange(Hq + Hk) % 7 - 3).astype(np.float32)
    q = (inputs.bf16_bits_to_f32(q) * scale[None, :Hq, None]).astype(np.float32).view(np.uint32) >> 16
    k = (inputs.bf16_bits_to_f32(k) * scale[None, Hq:, None]).astype(np.float32).view(np.uint32) >> 16
    q = q.astype(np.uint16)
    k = k.astype(np.uint16)
    mean = 0.0 if wb else 1.0
    qw = inputs.normal_bf16(seed, 33, (D,), mean, 0.1)
    kw = inputs.normal_bf16(seed, 34, (D,), mean, 0.1)
    o = oracle.default()
    q_ref = o.qk_norm_f64(q, qw, wb, eps)
    k_ref = o.qk_norm_f64(k, kw, wb, eps)
    qd, kd, qwd, kwd = _dev(q), _dev(k), _dev(qw), _dev(kw)
    st = binding.moe_qk_norm(T, Hq, Hk, D, qd.data_ptr() if Hq else None, kd.data_ptr() if Hk else None,
                             qwd.data_ptr() if Hq else None, kwd.data_ptr() if Hk else None, wb, eps,
                             torch.cuda.current_stream().cuda_stream)
    assert st == binding.MOE_OK
    q_out = qd.cpu().numpy().view(np.uint16)
    k_out = kd.cpu().numpy().view(np.uint16)
    for got, ref in ((q_out, q_ref), (k_out, k_ref)):
        if ref.size == 0:
            continue
        d = _ulps(got, ref)
        assert d.max() <= 1, f"max {d.max()} ulps"
        assert np.mean(d == 0) > 0.99, f"only {np.mean(d == 0):.4f} bit-identical"


def test_qk_norm_zero_tokens_is_a_noop():
    assert binding.moe_qk_norm(0, 32, 4, 128, None, None, None, None, 0.0, 1e-6,
                               torch.cuda.current_stream().cuda_stream) == binding.MOE_OK
