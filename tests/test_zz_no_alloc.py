"""moe_forward_static_scratch: the layer forward for callers that cannot
allocate device memory (their host owns all device memory, runs under a fixed
budget, or must keep cudaMalloc/cudaFree out of a latency-critical loop).

The entry point takes no workspace: its scratch is a fixed __device__ array
inside the library.  This test calls it through the C ABI twice in a row, on
two different batches, and checks each output against the existing
moe_forward entry point (with a caller workspace) on the same inputs, within
the tolerance the parity tests use.  It also checks that a shape needing more
scratch than the array holds is refused.  It runs last (file name) so that a
run stopping at the first failure has already run every other test, and it
needs nothing from earlier tests.
"""
import numpy as np
import pytest
import torch

import gpu_util as gu
from mixture_experts_layer_rmsnorm_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def _rel_and_max(a_bits, b_bits):
    a, b = gu.widen(a_bits), gu.widen(b_bits)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30), float(np.abs(a - b).max())


def test_static_scratch_matches_moe_forward_on_two_calls():
    cfg = inputs.LayerConfig(T=48, H=1024, I=512, E=16, top_k=4, seed=21)
    li = inputs.make_layer_inputs(cfg)
    dl = gu.DeviceLayer(li, max_tokens=64)
    L = dl.layer
    stream = torch.cuda.current_stream().cuda_stream
    for T, batch in ((48, 1), (37, 2)):  # two calls in a row, different batches and sizes
        c = inputs.LayerConfig(T=T, H=cfg.H, I=cfg.I, E=cfg.E, top_k=cfg.top_k, seed=cfg.seed)
        x = gu.dev_bf16(inputs.make_tokens(c, batch_index=batch))
        y_ref = L.forward(x)
        y = torch.full((T, cfg.H), -1, dtype=torch.int16, device="cuda")
        st = binding.moe_forward_static_scratch(L.shape(T), x.data_ptr(), L.g_norm.data_ptr(), L.w_router.data_ptr(),
                                                None, L.w13.data_ptr(), L.w2.data_ptr(), y.data_ptr(), stream)
        assert st == binding.MOE_OK, binding.moe_status_string(st)
        torch.cuda.synchronize()
        rel, mx = _rel_and_max(y.cpu().numpy().view(np.uint16), y_ref.cpu().numpy().view(np.uint16))
        assert rel <= gu.REL_FRO_TOL and mx <= gu.MAX_ABS_TOL, (T, rel, mx)


def test_static_scratch_refuses_shapes_beyond_the_array():
    s = binding.shape(4096, 4096, 4096, 64, 8)
    _, need = binding.moe_workspace_size(s)
    assert need > binding.MOE_STATIC_SCRATCH_BYTES
    A = 1 << 20  # never dereferenced: the size check comes first
    st = binding.moe_forward_static_scratch(s, A, A, A, None, A, A, A, None)
    assert st == binding.MOE_ERR_WORKSPACE
