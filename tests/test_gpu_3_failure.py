"""Failure detection on the GPU without a fault: a bounded device wait that runs
out is reported to the host through the workspace error word, and the CUDA
context stays usable.

The self-test kernel waits on an mbarrier phase that nothing completes and on a
flag that nothing sets, with a 2 ms limit; both waits give up, record
MOE_ERR_TIMEOUT with the kernel's id, and the kernel returns.  Afterwards a
normal layer call on the same workspace clears the word and matches the oracle.
"""
import time

import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
from mixture_experts_layer_rmsnorm_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

KERNEL_ID_SELFTEST = 8


def test_wait_that_runs_out_is_reported_and_context_survives():
    cfg = inputs.LayerConfig(T=4, H=128, I=256, E=8, top_k=2, renormalize=True, seed=0)
    li = inputs.make_layer_inputs(cfg)
    dl = gu.DeviceLayer(li)
    L = dl.layer
    L.ensure_capacity(cfg.T)
    ws, nbytes = L.workspace.data_ptr(), L.workspace_bytes(cfg.T)
    stream = torch.cuda.current_stream().cuda_stream

    t0 = time.perf_counter()
    assert binding.moe_selftest_wait_timeout(ws, nbytes, 2_000_000, stream) == binding.MOE_OK
    st, detail = binding.moe_device_status(ws, nbytes, stream)
    elapsed = time.perf_counter() - t0
    assert st == binding.MOE_ERR_TIMEOUT, (st, detail)
    assert detail[0] == binding.MOE_ERR_TIMEOUT and detail[1] == KERNEL_ID_SELFTEST
    assert elapsed < 5.0  # the waits gave up on time; nothing hung

    # the context still works, and the next call clears the error word
    g = dl.run(li.x)
    gu.check_routing(oracle.default(), li, li.x, g)
    gu.check_output(oracle.default(), li, li.x, g["y"])
    st, detail = binding.moe_device_status(ws, nbytes, stream)
    assert st == binding.MOE_OK and detail[0] == 0
