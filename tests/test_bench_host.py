"""Host-side logic of bench.py: roofline arithmetic, clock parsing, the
replica (N > 1) timing reduction over gloo ranks, and the accounting of the
workloads.  No GPU needed."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench
from mixture_experts_layer_rmsnorm_gb300 import accounting


def test_roofline_arithmetic():
    r = bench.roofline("hbm", 6.44e9, 1e-3, 6782.8, None)
    assert r["unit"] == "GB/s" and abs(r["achieved"] - 6440.0) < 1e-6
    assert abs(r["frac"] - 6440.0 / 6782.8) < 1e-4
    t = bench.roofline("tensor", 3.3e12, 2e-3, 1877.6, None)
    assert t["unit"] == "TFLOP/s" and abs(t["achieved"] - 1650.0) < 1e-6


def test_clock_parsing():
    rows = ["0, 1965, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 1455, 2070, 1380.1, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 1500, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    c = bench.parse_clock_samples(rows)
    assert c["sm_mhz"] == 1500 and c["sm_max_mhz"] == 2070 and c["reasons"] == ["sw_power_cap"]
    assert bench.parse_clock_samples([])["sm_mhz"] is None


def test_workload_accounting_matches_layer_shapes():
    # decode T=64 touches every expert: weight bytes = 64 experts x (2*4096*4096 + 4096*4096) x 2 B
    lb = accounting.layer_bytes(64, 4096, 4096, 64, 8, 64)
    assert lb["weights"] == 64 * 3 * 4096 * 4096 * 2
    assert abs(lb["weights"] / 1e9 - 6.44) < 0.01
    f = accounting.layer_flops(4096, 4096, 4096, 64, 8)
    assert abs((f["gemm1"] + f["gemm2"]) / 1e12 - 3.30) < 0.01


def test_kernel_source_sha_is_stable():
    a = bench.kernel_source_sha("gemm_gate_up_swiglu")
    assert a == bench.kernel_source_sha("gemm_gate_up_swiglu") and len(a) == 16


def test_kernel_source_hash_ignores_comments_only():
    code = "int f(int x) {\n  return x + 1;  // one\n}\n"
    assert bench._code_only(code) == bench._code_only("/* doc */\n" + code.replace("// one", "// two\n\n"))
    assert bench._code_only(code) != bench._code_only(code.replace("x + 1", "x + 2"))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, loc = bench.dist_env()
    bench.barrier(w)
    m = bench.reduce_max(10.0 + rank, w)
    q.put((r, loc, m))
    dist.destroy_process_group()


def test_replica_timing_reduction_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 0, 11.0), (1, 1, 11.0)]
