"""Concurrent host threads.  In a fresh process (so that every launcher's
once-per-device configuration runs for the first time while two threads race
to it), two threads drive their own layer, workspace and stream through the
bf16, fused-front-end, MXFP8 and MXFP4 entry points at once; each thread's
outputs must equal, bit for bit, the same calls made from one thread.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, threading
sys.path.insert(0, ROOT); sys.path.insert(0, ROOT + "/tests")
import numpy as np, torch
import gpu_util as gu
from mixture_experts_layer_rmsnorm_gb300 import inputs

def make(seed, T):
    cfg = inputs.LayerConfig(T=T, H=256, I=512, E=16, top_k=4, seed=seed)
    li = inputs.make_layer_inputs(cfg)
    dl = gu.DeviceLayer(li, max_tokens=T)
    return dl, li

def run(dl, li, stream, out):
    L = dl.layer
    with torch.cuda.stream(stream):
        L.quantize_mx(stream=stream.cuda_stream)
        L.quantize_mxfp4(stream=stream.cuda_stream)
        x = gu.dev_bf16(li.x)
        res = []
        for _ in range(5):
            res.append(L.forward(x, stream=stream.cuda_stream).clone())
            res.append(L.forward(x, stream=stream.cuda_stream, fused_front=True).clone())
            res.append(L.forward_mx(x, stream=stream.cuda_stream).clone())
            res.append(L.forward_mxfp4(x, stream=stream.cuda_stream, fp4_tokens=True).clone())
        stream.synchronize()
    out.extend(r.cpu().numpy() for r in res)

layers = [make(11, 24), make(12, 40)]
streams = [torch.cuda.Stream(), torch.cuda.Stream()]
outs = [[], []]
threads = [threading.Thread(target=run, args=(layers[i][0], layers[i][1], streams[i], outs[i])) for i in range(2)]
for t in threads: t.start()
for t in threads: t.join()
for i in range(2):
    ref = []
    run(layers[i][0], layers[i][1], torch.cuda.Stream(), ref)
    assert len(outs[i]) == len(ref) == 20, (len(outs[i]), len(ref))
    for a, b in zip(outs[i], ref):
        assert np.array_equal(a, b)
    for j in range(4, 20):  # repeated calls are identical too
        assert np.array_equal(outs[i][j], outs[i][j % 4])
print("threads ok")
"""


def test_two_host_threads_fresh_process():
    code = "ROOT = %r\n" % ROOT + CHILD
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0 and "threads ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
