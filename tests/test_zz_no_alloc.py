"""moe_forward_static_scratch: the layer forward for callers that cannot
allocate device memory (their host owns all device memory, runs under a fixed
budget, or must keep cudaMalloc/cudaFree out of a latency-critical loop).

The entry point takes no workspace: its scratch is a fixed __device__ array
inside the library.  This test calls it through the C ABI twice in a row, on
two different batches (the second smaller, so regions the first call wrote
and the second does not rewrite would show up), and checks after each call:
  - the device error word of the static array (moe_static_scratch_device_status)
    reports MOE_OK;
  - the output is bit-for-bit the output of the existing moe_forward entry
    point (caller workspace) on the same inputs: both run the same kernels in
    the same order, so any difference would be a stale or misplaced scratch
    region;
  - the output is within the tolerance the parity tests use against the oracle.
It also checks that the array's size is read from the library, and that a
shape needing more scratch than the array holds is refused before anything
is enqueued.  It runs last (file name) so that a run stopping at the first
failure has already run every other test, and it needs nothing from earlier
tests.
"""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
from mixture_experts_layer_rmsnorm_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def test_static_scratch_matches_moe_forward_on_two_calls():
    cfg = inputs.LayerConfig(T=48, H=1024, I=512, E=16, top_k=4, seed=21)
    li = inputs.make_layer_inputs(cfg)
    dl = gu.DeviceLayer(li, max_tokens=64)
    L = dl.layer
    stream = torch.cuda.current_stream().cuda_stream
    o = oracle.default()
    for T, batch in ((48, 1), (37, 2)):  # two calls in a row, different batches and sizes
        c = inputs.LayerConfig(T=T, H=cfg.H, I=cfg.I, E=cfg.E, top_k=cfg.top_k, seed=cfg.seed)
        x_host = inputs.make_tokens(c, batch_index=batch)
        x = gu.dev_bf16(x_host)
        y_ref = L.forward(x)
        torch.cuda.synchronize()
        st, det = L.device_status(T)
        assert st == binding.MOE_OK, det
        y = torch.full((T, cfg.H), -1, dtype=torch.int16, device="cuda")
        st = binding.moe_forward_static_scratch(L.shape(T), x.data_ptr(), L.g_norm.data_ptr(), L.w_router.data_ptr(),
                                                None, L.w13.data_ptr(), L.w2.data_ptr(), y.data_ptr(), stream)
        assert st == binding.MOE_OK, binding.moe_status_string(st)
        st, det = binding.moe_static_scratch_device_status(stream)
        assert st == binding.MOE_OK, (T, binding.moe_status_string(st), det)
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref), (T, int((y != y_ref).sum()))
        li_T = inputs.LayerInputs(cfg=c, x=x_host, g=li.g, w_router=li.w_router, bias=None, w13=li.w13, w2=li.w2)
        gu.check_output(o, li_T, x_host, y.cpu().numpy().view(np.uint16))


def test_static_scratch_refuses_shapes_beyond_the_array():
    st, cap = binding.moe_static_scratch_bytes()
    assert st == binding.MOE_OK and cap == 64 << 20
    # the decode layer (H = I = 4096, E = 64, top_k = 8) fits for T <= 128;
    # at T = 129 its tile plan changes and its scratch no longer fits
    _, need128 = binding.moe_workspace_size(binding.shape(128, 4096, 4096, 64, 8))
    _, need129 = binding.moe_workspace_size(binding.shape(129, 4096, 4096, 64, 8))
    assert need128 <= cap < need129
    A = 1 << 20  # never dereferenced: the size check comes first
    st = binding.moe_forward_static_scratch(binding.shape(129, 4096, 4096, 64, 8), A, A, A, None, A, A, A, None)
    assert st == binding.MOE_ERR_WORKSPACE
