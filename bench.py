#!/usr/bin/env python3
"""Benchmark of the fused MoE layer forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One JSON line on stdout (rank 0).  Workloads (synthetic, seeded, the shapes
and distributions of the layer's configurations):
  decode       (default) H = I = 4096, E = 64, top_k = 8; one step = one layer
               call at each of T = 1, 8, 32, 64 tokens (the thin-M sweep)
  prefill      same layer, T = 4096
  finegrained  H = 7168, I = 2048, E = 256, top_k = 8; T = 16, 128, 1024
  skewed       H = 4096, I = 1408, E = 128, top_k = 6, T = 512, Zipf(1.2) router bias
  tiny         T = 4, H = 128, I = 256, E = 8, top_k = 2
The L2 cache is flushed (a 256 MB write) before every layer call; the flush
is outside the timed intervals, which are CUDA events on the launch stream
around each call (and around each of its kernels).

--impl reference times the CPU oracle (the reference of this build) on the
host cores on a bounded sample of the same workload.

N > 1 (torchrun): every rank runs an independent replica of the workload on
its own GPU; the only cross-rank traffic is the host-side barrier and the max
of the timings.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused-MoE layer µs & tokens/s; % HBM roofline (decode), % bf16 TC peak (prefill)"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

WORKLOADS = {
    "decode": dict(H=4096, I=4096, E=64, k=8, Ts=[1, 8, 32, 64], seed=0, zipf=None,
                   label="decode sweep T in {1,8,32,64}, H=I=4096, E=64, top_k=8, bf16"),
    "prefill": dict(H=4096, I=4096, E=64, k=8, Ts=[4096], seed=0, zipf=None,
                    label="prefill T=4096, H=I=4096, E=64, top_k=8, bf16"),
    "finegrained": dict(H=7168, I=2048, E=256, k=8, Ts=[16, 128, 1024], seed=0, zipf=None,
                        label="fine-grained T in {16,128,1024}, H=7168, I=2048, E=256, top_k=8, bf16"),
    "skewed": dict(H=4096, I=1408, E=128, k=6, Ts=[512], seed=7, zipf=1.2,
                   label="skewed routing T=512, H=4096, I=1408, E=128, top_k=6, Zipf(1.2) bias, bf16"),
    "tiny": dict(H=128, I=256, E=8, k=2, Ts=[4], seed=0, zipf=None,
                 label="tiny T=4, H=128, I=256, E=8, top_k=2, bf16"),
    # small cases of the same per-unit shapes, for ncu captures (inputs > L2, < 2 GB on the device)
    "decode_ncu": dict(H=4096, I=4096, E=16, k=8, Ts=[64], seed=0, zipf=None,
                       label="ncu case: T=64, H=I=4096, E=16, top_k=8 (32 tokens/expert)"),
    "decode_rows_ncu": dict(H=4096, I=4096, E=8, k=8, Ts=[16], seed=0, zipf=None,
                            label="ncu case: T=16, H=I=4096, E=8, top_k=8 (decode tile plan, 16 rows per expert: "
                                  "the gate/up GEMM with row warps)"),
    "router_ncu": dict(H=4096, I=256, E=64, k=8, Ts=[1, 64], seed=0, zipf=None,
                       label="ncu case: router of the decode layer (H=4096, E=64) with small experts (I=256)"),
    "router_prefill_ncu": dict(H=4096, I=256, E=64, k=8, Ts=[4096], seed=0, zipf=None,
                               label="ncu case: router of the prefill layer (T=4096, H=4096, E=64) with small "
                                     "experts (I=256)"),
    "t1_ncu": dict(H=4096, I=4096, E=8, k=8, Ts=[1], seed=0, zipf=None,
                   label="ncu case: T=1, H=I=4096, E=8, top_k=8 (all 8 experts touched, as decode T=1)"),
    "prefill_ncu": dict(H=4096, I=4096, E=8, k=8, Ts=[512], seed=0, zipf=None,
                        label="ncu case: T=512, H=I=4096, E=8, top_k=8 (prefill tiles, 512 tokens/expert)"),
}
# QK-norm ("CuTeDSL chez Perplexity", "Norme QK"): attention heads of a Qwen3-style layer
QK_WORKLOADS = {
    "qk_norm": dict(Hq=32, Hk=4, D=128, Ts=[1, 64, 4096], wb=0.0, eps=1e-6, seed=0,
                    label="QK-norm sweep T in {1,64,4096}, 32 Q heads + 4 K heads, head_dim 128, bf16"),
}
KERNEL_SOURCES = {  # files whose content the ncu traffic figure of a kernel depends on
    "gemm_gate_up_swiglu": ["k_expert_gemm.cu", "tc_ptx.cuh", "moe_kernels.cuh", "moe_api.cu"],
    "gemm_down": ["k_expert_gemm.cu", "tc_ptx.cuh", "moe_kernels.cuh", "moe_api.cu"],
}


# ----------------------------------------------------------------- host logic

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS if k in d}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def _code_only(text: str) -> str:
    """C/CUDA source without comments, whitespace runs collapsed: what the
    compiled kernel depends on (a comment edit keeps the counters valid)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return re.sub(r"\s+", " ", text).strip()


def kernel_source_sha(name: str) -> str:
    h = hashlib.sha256()
    for fn in KERNEL_SOURCES.get(name, []):
        with open(os.path.join(ROOT, "mixture_experts_layer_rmsnorm_gb300", "csrc", fn), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic_per_launch(name: str, workload: str):
    """DRAM bytes per launch of `name` from the committed ncu summary, if it was
    taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload, {}).get(name)
    if not e or e.get("source_sha") != kernel_source_sha(name):
        return None
    return e.get("dram_bytes_per_launch")


def roofline(bound, algorithmic, seconds, peak, traffic):
    """achieved = algorithmic bytes (or FLOPs) per launch / average launch time."""
    if bound == "hbm":
        achieved = algorithmic / seconds / 1e9
        unit = "GB/s"
    else:
        achieved = algorithmic / seconds / 1e12
        unit = "TFLOP/s"
    return {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": traffic}


def parse_clock_samples(lines):
    """nvidia-smi CSV rows (noheader, nounits) -> clocks summary for the JSON line."""
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for ln in lines:
        parts = [p.strip() for p in ln.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1]))
            mx.append(float(parts[2]))
        except ValueError:
            continue
        for n, v in zip(names, parts[5:9]):
            if v.lower().startswith("active"):
                reasons.add(n)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
            "samples": len(sm)}


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        return parse_clock_samples(self.lines)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int) -> float:
    """Max of a host scalar over ranks (gloo); identity on one rank."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------- workloads

def make_host_inputs(wl):
    from mixture_experts_layer_rmsnorm_gb300 import inputs
    cfg0 = inputs.LayerConfig(T=wl["Ts"][0], H=wl["H"], I=wl["I"], E=wl["E"], top_k=wl["k"], seed=wl["seed"],
                              zipf_bias=wl["zipf"])
    g, wr, bias, w13, w2 = inputs.make_weights(cfg0)
    xs = {}
    for T in wl["Ts"]:
        cfg = inputs.LayerConfig(T=T, H=wl["H"], I=wl["I"], E=wl["E"], top_k=wl["k"], seed=wl["seed"],
                                 zipf_bias=wl["zipf"])
        xs[T] = inputs.make_tokens(cfg)
    return dict(g=g, wr=wr, bias=bias, w13=w13, w2=w2, xs=xs)


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                low = ln.lower()
                if low.startswith("model name") or low.startswith("cpu part") or low.startswith("hardware"):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def cpu_oracle_rate(wl, host, per_batch_cap, reps=1, min_seconds=0.0, max_reps=50, nthreads=None):
    """Tokens/s of the CPU oracle (as it stands; all host cores unless nthreads)
    on a bounded sample: from each of the workload's batches, up to
    per_batch_cap tokens spread over the batch; repeated `reps` times, or more
    until min_seconds of CPU work have been timed (at most max_reps)."""
    import numpy as np
    import oracle
    total_tok, total_s, r = 0, 0.0, 0
    while r < reps or (total_s < min_seconds and r < max_reps):
        for T in wl["Ts"]:
            sample = np.unique(np.linspace(0, T - 1, min(T, per_batch_cap)).astype(np.int64))
            t0 = time.perf_counter()
            oracle.moe_forward(host["xs"][T], host["g"], host["wr"], host["bias"], host["w13"], host["w2"], wl["k"],
                               True, 1e-6, sample=sample, nthreads=nthreads)
            total_s += time.perf_counter() - t0
            total_tok += sample.size
        r += 1
    return total_tok / total_s, total_tok, total_s, nthreads or oracle.threads(), r


# ----------------------------------------------------------------- QK-norm

def qk_host_inputs(wl):
    import numpy as np
    from mixture_experts_layer_rmsnorm_gb300 import inputs
    D, Hq, Hk, seed = wl["D"], wl["Hq"], wl["Hk"], wl["seed"]
    qs = {T: inputs.normal_bf16(seed + 1000 * T, 31, (T, Hq, D)) for T in wl["Ts"]}
    ks = {T: inputs.normal_bf16(seed + 1000 * T, 32, (T, Hk, D)) for T in wl["Ts"]}
    qw = inputs.normal_bf16(seed, 33, (D,), 1.0, 0.1)
    kw = inputs.normal_bf16(seed, 34, (D,), 1.0, 0.1)
    return dict(qs=qs, ks=ks, qw=qw, kw=kw, np=np)


def qk_cpu_rate(wl, host, min_seconds, max_tokens=256):
    """Tokens/s of the CPU oracle's QK-norm on up to max_tokens tokens of each batch."""
    import oracle
    o = oracle.default()
    ntok, secs, reps = 0, 0.0, 0
    while secs < min_seconds and reps < 1000:
        for T in wl["Ts"]:
            n = min(T, max_tokens)
            t0 = time.perf_counter()
            o.qk_norm_f64(host["qs"][T][:n], host["qw"], wl["wb"], wl["eps"])
            o.qk_norm_f64(host["ks"][T][:n], host["kw"], wl["wb"], wl["eps"])
            secs += time.perf_counter() - t0
            ntok += n
        reps += 1
    return ntok / secs, ntok, secs, reps


def run_qk_norm(args, wl, world, rank, local):
    import torch
    from mixture_experts_layer_rmsnorm_gb300 import binding

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    host = qk_host_inputs(wl)
    np = host["np"]
    Ts, Hq, Hk, D = wl["Ts"], wl["Hq"], wl["Hk"], wl["D"]

    def d16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)

    qd = {T: d16(host["qs"][T]) for T in Ts}
    kd = {T: d16(host["ks"][T]) for T in Ts}
    qwd, kwd = d16(host["qw"]), d16(host["kw"])
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(64 << 20, dtype=torch.float32, device=dev)

    def call(T, q, k):
        st = binding.moe_qk_norm(T, Hq, Hk, D, q.data_ptr(), k.data_ptr(), qwd.data_ptr(), kwd.data_ptr(),
                                 wl["wb"], wl["eps"], stream.cuda_stream)
        if st != binding.MOE_OK:
            raise binding.MoeError(st, "moe_qk_norm")

    # batches of 32 MB or more: R copies (R x bytes > 256 MB, twice L2) run back to
    # back between one pair of events, so every call reads and writes HBM; smaller
    # ones: one call after an L2 flush (their time is launch and memory latency)
    reps = {}
    for T in Ts:
        nbytes = 2 * T * (Hq + Hk) * D * 2
        reps[T] = 1 if nbytes < (32 << 20) else -(-(256 << 20) // nbytes) + 1
    qcopies = {T: [qd[T]] + [qd[T].clone() for _ in range(reps[T] - 1)] for T in Ts}
    kcopies = {T: [kd[T]] + [kd[T].clone() for _ in range(reps[T] - 1)] for T in Ts}

    for _ in range(args.warmup):
        for T in Ts:
            for r in range(reps[T]):
                call(T, qcopies[T][r], kcopies[T][r])
    ev = {T: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)] for T in Ts}
    sampler = ClockSampler(local)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    for s_ in range(args.steps):
        for T in Ts:
            flush.fill_(s_ & 0xFF)
            flush_rd.sum()
            a, b = ev[T][s_]
            a.record(stream)
            for r in range(reps[T]):  # in place: each call normalises the previous call's output
                call(T, qcopies[T][r], kcopies[T][r])
            b.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    per_T, total_ms, total_bytes = {}, 0.0, 0
    for T in Ts:
        ms = [a.elapsed_time(b) / reps[T] for a, b in ev[T]]
        med = statistics.median(ms)
        nbytes = 2 * T * (Hq + Hk) * D * 2 + 2 * D * 2
        total_ms += sum(ms)
        total_bytes += nbytes * len(ms)
        per_T[str(T)] = {"us_median": round(med * 1e3, 2), "tokens_per_s": round(T / (med * 1e-3), 1),
                         "bytes": nbytes, "GBps": round(nbytes / (med * 1e-3) / 1e9, 1),
                         "timing": ("one call after an L2 flush" if reps[T] == 1 else
                                    f"{reps[T]} calls on distinct buffers back to back, per-call mean")}
    ms_step = reduce_max(total_ms / args.steps, world)
    value = world * sum(Ts) / (ms_step * 1e-3)
    peaks, peak_kind = load_peaks()
    achieved = total_bytes / (total_ms * 1e-3) / 1e9
    big = str(max(Ts))
    roof = {"bound": "hbm", "achieved": round(achieved, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": None,
            "peak_source": f"hbm_gbs ({peak_kind}, copy bandwidth)", "kernel": "qk_norm_kernel<128>",
            "algorithmic_per_launch": total_bytes / (args.steps * len(Ts)),
            "avg_launch_us": round(total_ms / (args.steps * len(Ts)) * 1e3, 2),
            "largest_T": {"T": int(big), "GBps": per_T[big]["GBps"],
                          "frac": round(per_T[big]["GBps"] / peaks["hbm_gbs"], 4)}}
    # end to end: pinned host q, k -> device, the call, the result back, every step
    hq = {T: torch.from_numpy(host["qs"][T].view(np.int16)).pin_memory() for T in Ts}
    hk = {T: torch.from_numpy(host["ks"][T].view(np.int16)).pin_memory() for T in Ts}
    oq = {T: torch.empty_like(hq[T]).pin_memory() for T in Ts}
    ok_ = {T: torch.empty_like(hk[T]).pin_memory() for T in Ts}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        for T in Ts:
            qd[T].copy_(hq[T], non_blocking=True)
            kd[T].copy_(hk[T], non_blocking=True)
            call(T, qd[T], kd[T])
            oq[T].copy_(qd[T], non_blocking=True)
            ok_[T].copy_(kd[T], non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1) / args.steps, world)
    io = sum(2 * T * (Hq + Hk) * D for T in Ts)
    out = {"metric": "QK-norm us & tokens/s; % HBM roofline", "value": round(value, 1), "unit": "tokens/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic (seeded generator)",
           "config": {"workload": wl["label"], "Hq": Hq, "Hk": Hk, "head_dim": D, "weight_bias": wl["wb"],
                      "eps": wl["eps"], "l2": "flushed before every call (256 MB write + 256 MB read), outside the "
                                               "timed CUDA-event intervals",
                      "parallelism": f"replicas x{world}", "per_T": per_T},
           "roofline": roof,
           "e2e": {"value": round(world * sum(Ts) / (e2e_ms * 1e-3), 1), "unit": "tokens/s",
                   "h2d_bytes_per_step": io, "d2h_bytes_per_step": io, "ms_per_step": round(e2e_ms, 4)},
           "gpu_launches": args.steps * sum(reps.values()), "clocks": clocks}
    return out, host


# ----------------------------------------------------------------- our arm

def run_ours(args, wl, world, rank, local):
    import numpy as np
    import torch
    from mixture_experts_layer_rmsnorm_gb300 import accounting, binding

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    t_setup = time.time()
    host = make_host_inputs(wl)

    def d16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)

    layer = binding.MoeLayer(d16(host["g"]), torch.from_numpy(host["wr"]).to(dev), d16(host["w13"]),
                             d16(host["w2"]), wl["k"], True, 1e-6,
                             router_bias=None if host["bias"] is None else torch.from_numpy(host["bias"]).to(dev),
                             max_tokens=max(wl["Ts"]))
    Ts = wl["Ts"]
    H = wl["H"]
    xs = {T: d16(host["xs"][T]) for T in Ts}
    ys = {T: torch.empty((T, H), dtype=torch.int16, device=dev) for T in Ts}
    # L2 flush: write 256 MB (2x L2), then read another 256 MB so that the
    # write's dirty lines are written back here rather than inside the timed call
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(64 << 20, dtype=torch.float32, device=dev)

    def flush_l2(v):
        flush.fill_(v & 0xFF)
        flush_rd.sum()

    stream = torch.cuda.current_stream(dev)
    nk = binding.MOE_NUM_KERNELS

    def new_events():
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)]
        for e in evs:
            e.record(stream)  # creates the CUDA event behind the torch object
        return evs

    call_ev = {T: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)] for T in Ts}
    kern_ev = {T: [new_events() for _ in range(args.steps)] for T in Ts}
    setup_s = time.time() - t_setup

    ff, fc, fm = args.fused_front, args.fused_combine, args.fused_mlp
    mx = ("nvfp4" if args.nvfp4 else "mxfp4a4" if args.mxfp4a4 else "mxfp4" if args.mxfp4
          else args.mx)  # formats for the byte counts
    if args.nvfp4:
        layer.quantize_nvfp4()
    elif args.mxfp4 or args.mxfp4a4:
        layer.quantize_mxfp4()
    elif mx:
        layer.quantize_mx()

    def fwd(x, y, events=None):
        if args.nvfp4:
            return layer.forward_nvfp4(x, y, events=events)
        if args.mxfp4 or args.mxfp4a4:
            return layer.forward_mxfp4(x, y, events=events, fp4_tokens=args.mxfp4a4)
        if mx:
            return layer.forward_mx(x, y, events=events)
        return layer.forward(x, y, events=events, fused_front=ff, fused_combine=fc, fused_mlp=fm)

    def kpc(T):  # our kernels per layer call
        call = (binding.MOE_CALL_FORWARD_NVFP4 if args.nvfp4 else
                binding.MOE_CALL_FORWARD_MXFP4A4 if args.mxfp4a4 else
                binding.MOE_CALL_FORWARD_MXFP4 if args.mxfp4 else binding.MOE_CALL_FORWARD_MX if mx else
                binding.MOE_CALL_FORWARD_FUSED_FRONT if ff else
                binding.MOE_CALL_FORWARD_FUSED_COMBINE if fc else
                binding.MOE_CALL_FORWARD_FUSED_MLP if fm else binding.MOE_CALL_FORWARD)
        return binding.kernels_per_call(T, H, wl["I"], wl["E"], wl["k"], call)

    graphs = {}  # batch size -> CUDA graph of one layer call (the timed calls replay it)

    def one_step(step_idx=None, per_kernel=False, eager_ev=None):
        for T in Ts:
            flush_l2(step_idx or 0)
            if step_idx is None:
                fwd(xs[T], ys[T])
            elif per_kernel:
                fwd(xs[T], ys[T], events=[e.cuda_event for e in kern_ev[T][step_idx]])
            else:
                a, b = (eager_ev or call_ev)[T][step_idx]
                a.record(stream)
                if T in graphs and eager_ev is None:
                    graphs[T].replay()
                else:
                    fwd(xs[T], ys[T])
                b.record(stream)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    for T in Ts:
        st, det = layer.device_status(T)
        if st != binding.MOE_OK:
            raise binding.MoeError(st, f"device status after warm-up (T={T}, detail {det})")

    # routing facts (touched experts) of each batch, from the last warm-up call
    touched = {}
    for T in Ts:
        fwd(xs[T], ys[T])
        ids = layer.view_tensor(T, "topk_ids", torch.int32, (T, wl["k"])).cpu().numpy()
        touched[T] = accounting.n_touched(ids, wl["E"])
    torch.cuda.synchronize()
    # A serving loop captures the decode step once and replays it: each
    # batch's layer call, captured into a CUDA graph (same kernels, launch
    # attributes and arguments; the inputs are read from xs[T] at replay)
    if not args.eager:
        for T in Ts:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fwd(xs[T], ys[T])
            graphs[T] = g
        for T in Ts:
            graphs[T].replay()
        torch.cuda.synchronize()
        for T in Ts:
            st, det = layer.device_status(T)
            if st != binding.MOE_OK:
                raise binding.MoeError(st, f"device status after a graph replay (T={T}, detail {det})")

    gpu_index = local
    cvd = os.environ.get("CUDA_VISIBLE_DEVICES")
    if cvd:
        try:
            gpu_index = int(cvd.split(",")[local])
        except (ValueError, IndexError):
            gpu_index = local
    sampler = ClockSampler(gpu_index)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    t_wall0 = time.perf_counter()
    for s in range(args.steps):
        one_step(s)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    barrier(world)
    # second pass, same work: CUDA events recorded by the library around each kernel
    for s in range(args.steps):
        one_step(s, per_kernel=True)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    # the plain calls made directly (no graph), for comparison
    eager_ev = {T: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    for _ in range(args.steps)] for T in Ts}
    for s in range(args.steps):
        one_step(s, eager_ev=eager_ev)
    torch.cuda.synchronize()
    # extra, not the headline: the same calls with the L2 left warm (no flush),
    # each batch called `reps` times back to back
    warm = {}
    for T in Ts:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        fwd(xs[T], ys[T])
        a.record(stream)
        for _ in range(args.steps):
            fwd(xs[T], ys[T])
        b.record(stream)
        torch.cuda.synchronize()
        warm[T] = a.elapsed_time(b) / args.steps

    # per-call device times (plain calls) and per-kernel times (second pass)
    per_T = {}
    kern_ms = {n: 0.0 for n in binding.KERNEL_NAMES}
    total_ms = 0.0
    eager_ms = 0.0
    for T in Ts:
        calls = [a.elapsed_time(b) for a, b in call_ev[T]]
        kt = {n: [] for n in binding.KERNEL_NAMES}
        for evs in kern_ev[T]:
            for i, n in enumerate(binding.KERNEL_NAMES):
                dt = evs[i].elapsed_time(evs[i + 1])
                kern_ms[n] += dt
                kt[n].append(dt)
        total_ms += sum(calls)
        lb = accounting.layer_bytes(T, H, wl["I"], wl["E"], wl["k"], touched[T], mx)
        us = statistics.median(calls) * 1e3
        calls_eager = [a.elapsed_time(b) for a, b in eager_ev[T]]
        eager_ms += sum(calls_eager)
        per_T[str(T)] = {"us_median": round(us, 2), "us_mean": round(sum(calls) / len(calls) * 1e3, 2),
                         "us_median_eager": round(statistics.median(calls_eager) * 1e3, 2),
                         "tokens_per_s": round(T / (us * 1e-6), 1), "experts_touched": touched[T],
                         "weight_GB": round(lb["weights"] / 1e9, 4),
                         "weight_GBps": round(lb["weights"] / (us * 1e-6) / 1e9, 1),
                         "hbm_frac_of_8TBps": round(lb["weights"] / (us * 1e-6) / 1e9 / NOMINAL_HBM_GBS, 4),
                         "kernels_per_call": kpc(T),
                         "us_unflushed_mean": round(warm[T] * 1e3, 2),
                         "kernel_us_median": {n: round(statistics.median(v) * 1e3, 2) for n, v in kt.items()}}
    ms_per_step = total_ms / args.steps
    tokens_per_step = sum(Ts)
    ms_max = reduce_max(ms_per_step, world)
    value = world * tokens_per_step / (ms_max * 1e-3)
    eager_ms_max = reduce_max(eager_ms / args.steps, world)

    # dominant kernel and its roofline
    peaks, peak_kind = load_peaks()
    dom = max(kern_ms, key=kern_ms.get)
    launches = args.steps * len(Ts)
    avg_s = kern_ms[dom] / launches * 1e-3
    prefill_like = all(T * wl["k"] > 64 * wl["E"] for T in Ts)
    if dom in ("gemm_gate_up_swiglu", "gemm_down") and prefill_like:
        fl = accounting.layer_flops
        per = [fl(T, H, wl["I"], wl["E"], wl["k"])["gemm1" if dom == "gemm_gate_up_swiglu" else "gemm2"]
               for T in Ts]
        if mx in ("mxfp4a4", "nvfp4"):  # kind::mxf4 / mxf4nvf4: the measured bf16 peak x the nominal dense
            # ratio 13.5 / 2.25
            roof = roofline("tensor", sum(per) / len(per), avg_s, 6.0 * peaks["bf16_tflops"], None)
            roof["peak_source"] = f"6 x bf16_tflops ({peak_kind}; nominal dense fp4 / bf16 ratio)"
        elif mx:  # block-scaled FP8 / FP4xFP8 MMAs (kind::mxf8f6f4, the FP8 rate): the measured bf16 peak x
            # the nominal dense ratio 4.5 / 2.25
            roof = roofline("tensor", sum(per) / len(per), avg_s, 2.0 * peaks["bf16_tflops"], None)
            roof["peak_source"] = f"2 x bf16_tflops ({peak_kind}; nominal dense fp8 / bf16 ratio)"
        else:
            roof = roofline("tensor", sum(per) / len(per), avg_s, peaks["bf16_tflops"],
                            ncu_traffic_per_launch(dom, args.workload))
            roof["peak_source"] = f"bf16_tflops ({peak_kind})"
    else:
        if dom == "gemm_gate_up_swiglu" and fm:  # both GEMMs in one launch
            per = [accounting.gemm1_kernel_bytes(T, H, wl["I"], wl["k"], touched[T], mx) +
                   accounting.gemm2_kernel_bytes(T, H, wl["I"], wl["k"], touched[T], mx) for T in Ts]
        elif dom == "gemm_gate_up_swiglu":
            per = [accounting.gemm1_kernel_bytes(T, H, wl["I"], wl["k"], touched[T], mx) for T in Ts]
        elif dom == "gemm_down":
            per = [accounting.gemm2_kernel_bytes(T, H, wl["I"], wl["k"], touched[T], mx) for T in Ts]
        else:
            per = [accounting.layer_bytes(T, H, wl["I"], wl["E"], wl["k"], touched[T], mx)["total"] for T in Ts]
        traffic = None if mx else ncu_traffic_per_launch(dom, args.workload)
        roof = roofline("hbm", sum(per) / len(per), avg_s, peaks["hbm_gbs"], traffic)
        roof["peak_source"] = f"hbm_gbs ({peak_kind}, copy bandwidth)"
    roof["kernel"] = "expert_mlp_fused (gate/up and down GEMMs in one launch)" if (fm and dom == "gemm_gate_up_swiglu") \
        else dom
    roof["algorithmic_per_launch"] = sum(per) / len(per)
    roof["avg_launch_us"] = round(avg_s * 1e6, 2)

    # end to end through the public API with host buffers: H2D of x, forward, D2H of y
    pinned_x = {T: torch.from_numpy(host["xs"][T].view(np.int16)).pin_memory() for T in Ts}
    pinned_y = {T: torch.empty((T, H), dtype=torch.int16).pin_memory() for T in Ts}
    e2e_ms = 0.0
    for s in range(args.steps):
        for T in Ts:
            flush_l2(s)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            xs[T].copy_(pinned_x[T], non_blocking=True)
            fwd(xs[T], ys[T])
            pinned_y[T].copy_(ys[T], non_blocking=True)
            b.record(stream)
            b.synchronize()
            e2e_ms += a.elapsed_time(b)
    e2e_ms_step = reduce_max(e2e_ms / args.steps, world)
    e2e = {"value": round(world * tokens_per_step / (e2e_ms_step * 1e-3), 1), "unit": "tokens/s",
           "h2d_bytes_per_step": sum(T * H * 2 for T in Ts), "d2h_bytes_per_step": sum(T * H * 2 for T in Ts),
           "ms_per_step": round(e2e_ms_step, 4)}

    prefill = None
    if args.workload == "decode" and not args.no_prefill and not ff and not fm:
        prefill = prefill_section(args, wl, layer, fwd, flush_l2, stream, gpu_index, world, d16, mx)

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_max, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": ("nvfp4 (e2m1 + e4m3 per 16 + fp32 per tensor) x nvfp4, fp32 accumulation" if args.nvfp4 else
                  "mxfp4 (e2m1 + e8m0 per 32) x mxfp4, fp32 accumulation" if args.mxfp4a4 else
                  "mxfp4 (e2m1 + e8m0 per 32) x mxfp8, fp32 accumulation" if args.mxfp4 else
                  "mxfp8 (e4m3 + e8m0 per 32) x mxfp8, fp32 accumulation" if mx else "bf16"),
        "data": "synthetic (seeded generator; random-init weights)",
        "config": {"workload": wl["label"], "tokens_per_step": tokens_per_step,
                   "layer_calls_per_step": len(Ts),
                   "expert_weights": ("NVFP4 weights and tokens (moe_forward_nvfp4; bytes counted as codes + "
                                      "block scales)" if args.nvfp4 else
                                      "MXFP4 weights and tokens (moe_forward_mxfp4a4; bytes counted as codes + "
                                      "scales)" if args.mxfp4a4 else
                                      "MXFP4 (moe_forward_mxfp4; weight bytes counted as codes + scales)"
                                      if args.mxfp4 else
                                      "MXFP8 (moe_forward_mx; weight bytes counted as codes + scales)" if mx
                                      else "bf16"),
                   "front_end": ("moe_forward_fused_front: norm .. gather in one cluster launch" if ff
                                 else "moe_forward: multi-launch front end"),
                   "combine": ("moe_forward_fused_combine: in the down GEMM's epilogue" if fc
                               else "separate kernel"),
                   "expert_gemms": ("moe_forward_fused_mlp: both in one launch" if fm else "two launches"),
                   "l2": "flushed before every layer call (256 MB write, then a 256 MB read of another buffer so "
                         "no dirty lines remain); flush outside the timed CUDA-event intervals",
                   "timing": (("CUDA events on the launch stream around the replay of a CUDA graph holding one "
                               "layer call per batch size (captured once with stream capture: the same kernels, "
                               "launch attributes and arguments as the plain call, inputs read from the device "
                               "buffer at replay); " if graphs else
                               "CUDA events on the launch stream around each plain layer call; ") +
                              "per_T.us_median_eager and `eager` time the plain calls made directly; kernel times "
                              "from a pass of the same calls through the events entry point (with 4 kernels per "
                              "call, 'norm_router' is the single-launch front end: norm, router, top-k, align and "
                              "gather)"),
                   "eager": {"value": round(world * tokens_per_step / (eager_ms_max * 1e-3), 1),
                             "ms_per_step": round(eager_ms_max, 4)},
                   "parallelism": f"replicas x{world} (no cross-GPU data path)", "per_T": per_T,
                   "kernel_ms_per_step": {n: round(v / args.steps, 4) for n, v in kern_ms.items()},
                   "wall_s_timed_region": round(t_wall, 3), "setup_s": round(setup_s, 1)},
        "roofline": roof,
        "e2e": e2e,
        # kernels of the timed pass (top-k runs inside the align kernel for small T and E); the per-kernel pass
        # launches as many again
        "gpu_launches": sum(args.steps * kpc(T) for T in Ts),
        "clocks": clocks,
    }
    if prefill is not None:
        out["prefill"] = prefill
    return out, host


PREFILL_T = 4096
PREFILL_MIN_TIMED_S = 2.5  # long enough for >= 10 clock samples at 200 ms


def prefill_section(args, wl, layer, fwd, flush_l2, stream, gpu_index, world, d16, mx):
    """The prefill configuration (T = 4096 on the decode layer's weights: the
    same H, I, E, top_k and seed) through the same entry point: flushed calls
    timed with CUDA events on the launch stream, repeated until the timed
    region lasts at least PREFILL_MIN_TIMED_S (clock samples during it), then
    a per-kernel pass of `steps` calls; the gate/up GEMM's tensor roofline."""
    import numpy as np
    import torch
    from mixture_experts_layer_rmsnorm_gb300 import accounting, binding, inputs

    T, H, I, E, k = PREFILL_T, wl["H"], wl["I"], wl["E"], wl["k"]
    cfg = inputs.LayerConfig(T=T, H=H, I=I, E=E, top_k=k, seed=wl["seed"], zipf_bias=wl["zipf"])
    x = d16(inputs.make_tokens(cfg))
    y = torch.empty((T, H), dtype=torch.int16, device=x.device)
    for _ in range(args.warmup):
        flush_l2(0)
        fwd(x, y)
    torch.cuda.synchronize()
    st, det = layer.device_status(T)
    if st != binding.MOE_OK:
        raise binding.MoeError(st, f"device status after prefill warm-up (detail {det})")
    ids = layer.view_tensor(T, "topk_ids", torch.int32, (T, k)).cpu().numpy()
    touched = accounting.n_touched(ids, E)
    # one flushed call's time sets how many calls fill the timed region
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    flush_l2(1)
    a.record(stream)
    fwd(x, y)
    b.record(stream)
    torch.cuda.synchronize()
    est_s = a.elapsed_time(b) * 1e-3 + 2e-4  # + the flush
    n_calls = max(args.steps, int(PREFILL_MIN_TIMED_S / est_s) + 1)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_calls)]
    sampler = ClockSampler(gpu_index)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    for i in range(n_calls):
        flush_l2(i)
        evs[i][0].record(stream)
        fwd(x, y)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    calls = [e0.elapsed_time(e1) for e0, e1 in evs]
    nk = binding.MOE_NUM_KERNELS
    kern = {n: [] for n in binding.KERNEL_NAMES}
    for i in range(args.steps):
        ke = [torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)]
        for e in ke:
            e.record(stream)
        flush_l2(i)
        fwd(x, y, events=[e.cuda_event for e in ke])
        torch.cuda.synchronize()
        for j, n in enumerate(binding.KERNEL_NAMES):
            kern[n].append(ke[j].elapsed_time(ke[j + 1]))
    torch.cuda.synchronize()
    med_ms = statistics.median(calls)
    ms_max = reduce_max(med_ms, world)
    peaks, peak_kind = load_peaks()
    fl = accounting.layer_flops(T, H, I, E, k)
    ratio = 6.0 if mx in ("mxfp4a4", "nvfp4") else 2.0 if mx else 1.0  # MMA kind / bf16 nominal dense rate
    peak_b, peak_s = ratio * peaks["bf16_tflops"], ratio * peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    g1_ms = statistics.median(kern["gemm_gate_up_swiglu"])
    roof = roofline("tensor", fl["gemm1"], g1_ms * 1e-3, peak_b,
                    None if mx else ncu_traffic_per_launch("gemm_gate_up_swiglu", "prefill"))
    roof.update({"kernel": "gemm_gate_up_swiglu", "algorithmic_per_launch": fl["gemm1"],
                 "avg_launch_us": round(g1_ms * 1e3, 2),
                 "peak_source": (f"{ratio:g} x " if ratio != 1.0 else "") + f"bf16_tflops ({peak_kind}, burst)",
                 "peak_sustained": peak_s, "frac_of_sustained": round(fl["gemm1"] / (g1_ms * 1e-3) / 1e12 / peak_s, 4)})
    layer_tf = fl["total"] / (med_ms * 1e-3) / 1e12
    return {"workload": f"prefill T={T}, H={H}, I={I}, E={E}, top_k={k} (the decode layer's weights)",
            "T": T, "experts_touched": touched, "calls_timed": n_calls,
            "us_median": round(med_ms * 1e3, 2), "us_mean": round(sum(calls) / len(calls) * 1e3, 2),
            "us_min": round(min(calls) * 1e3, 2), "tokens_per_s": round(world * T / (ms_max * 1e-3), 1),
            # the first `steps` calls, before a sustained load meets the power cap
            "us_median_first_calls": round(statistics.median(calls[: args.steps]) * 1e3, 2),
            "layer_tflops": round(layer_tf, 2), "layer_frac_of_peak": round(layer_tf / peak_b, 4),
            "layer_frac_of_sustained": round(layer_tf / peak_s, 4),
            "flops": {n: int(v) for n, v in fl.items()},
            "kernel_us_median": {n: round(statistics.median(v) * 1e3, 2) for n, v in kern.items()},
            "roofline": roof, "clocks": clocks,
            "timing": "flushed calls (256 MB write + 256 MB read before each), CUDA events on the launch stream, "
                      "back to back for >= 2.5 s (us_median over all of them, sustained; us_median_first_calls over "
                      "the first `steps`); kernel times from a second pass through moe_forward_events"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="decode", choices=sorted(WORKLOADS) + sorted(QK_WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-tokens-per-batch", type=int, default=32,
                    help="CPU oracle sample: at most this many tokens of each batch per step")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="minimum timed CPU-oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true",
                    help="time the plain layer calls made directly, not their replay from a CUDA graph")
    ap.add_argument("--no-prefill", action="store_true",
                    help="decode workload: skip the prefill (T=4096) object of the JSON line")
    ap.add_argument("--nvfp4", action="store_true",
                    help="time moe_forward_nvfp4: the NVFP4 layer (NVFP4 weights, token rows and activations)")
    ap.add_argument("--mxfp4a4", action="store_true",
                    help="time moe_forward_mxfp4a4: the MXFP4 layer (MXFP4 weights, token rows and activations)")
    ap.add_argument("--mxfp4", action="store_true",
                    help="time moe_forward_mxfp4: MXFP4 expert weights, MXFP8 token rows and activations")
    ap.add_argument("--mx", action="store_true",
                    help="time moe_forward_mx: MXFP8 expert weights and activations (decode shapes)")
    ap.add_argument("--fused-front", action="store_true",
                    help="time moe_forward_fused_front (norm .. gather in one cluster launch; T <= 64)")
    ap.add_argument("--fused-combine", action="store_true",
                    help="time moe_forward_fused_combine (the combine in the down GEMM's epilogue)")
    ap.add_argument("--fused-mlp", action="store_true",
                    help="time moe_forward_fused_mlp (both expert GEMMs in one launch; decode tile plan)")
    args = ap.parse_args()
    if sum([args.mx, args.mxfp4, args.mxfp4a4, args.nvfp4, args.fused_front, args.fused_combine, args.fused_mlp]) > 1:
        ap.error("--mx, --mxfp4, --mxfp4a4, --nvfp4, --fused-front, --fused-combine and --fused-mlp are separate entry "
                 "points; pick one")
    if args.warmup < 3:
        print("bench: at least 3 warm-up steps are required; using 3", file=sys.stderr)
        args.warmup = 3
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    if args.workload in QK_WORKLOADS:
        wl = QK_WORKLOADS[args.workload]
        if args.impl == "reference":
            if rank == 0:
                host = qk_host_inputs(wl)
                rate, ntok, secs, reps = qk_cpu_rate(wl, host, min_seconds=min(args.cpu_seconds, 5.0))
                print(json.dumps({"impl": "reference", "metric": "QK-norm us & tokens/s; % HBM roofline",
                                  "value": round(rate, 1), "unit": "tokens/s", "n_gpus": world, "steps": reps,
                                  "warmup": 0, "higher_is_better": True, "dtype": "f64", "data": "synthetic",
                                  "config": {"workload": wl["label"], "reference": "CPU oracle (fp64 C)"},
                                  "cpu_baseline": {"value": round(rate, 1), "unit": "tokens/s", "cores": 1,
                                                   "kind": "oracle", "sample": f"{ntok} tokens, {secs:.1f} s"},
                                  "e2e": {"value": round(rate, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                          "d2h_bytes_per_step": 0}}), flush=True)
        else:
            out, host = run_qk_norm(args, wl, world, rank, local)
            if rank == 0 and world == 1 and not args.no_cpu_baseline:
                rate, ntok, secs, reps = qk_cpu_rate(wl, host, min_seconds=min(args.cpu_seconds, 5.0))
                out["cpu_baseline"] = {"value": round(rate, 1), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                       "sample": f"{ntok} tokens (up to 256 of each batch, {reps} passes), "
                                                 f"{secs:.1f} s"}
            if rank == 0:
                print(json.dumps(out), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    wl = WORKLOADS[args.workload]

    if args.impl == "reference":
        if rank == 0:
            host = make_host_inputs(wl)
            cap = args.ref_tokens_per_batch
            cpu_oracle_rate(wl, host, cap, reps=args.warmup)  # warm-up steps, untimed
            rate, ntok, secs, cores, _ = cpu_oracle_rate(wl, host, cap, reps=args.steps)
            out = {"impl": "reference", "metric": METRIC, "value": round(rate, 3), "unit": "tokens/s", "n_gpus": world,
                   "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 1),
                   "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                   "data": "synthetic (seeded generator; random-init weights)",
                   "config": {"workload": wl["label"], "reference": "CPU oracle (fp64 C, all host cores)",
                              "step": f"up to {cap} tokens of each batch T={wl['Ts']}"},
                   "cpu_baseline": {"value": round(rate, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                    "sample": f"{ntok} tokens over {args.steps} steps (up to {cap} per batch of "
                                              f"T={wl['Ts']}), {secs:.1f} s"},
                   "e2e": {"value": round(rate, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}}
            print(json.dumps(out), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    out, host = run_ours(args, wl, world, rank, local)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cap = args.ref_tokens_per_batch
        rate, ntok, secs, cores, reps = cpu_oracle_rate(wl, host, cap, reps=1, min_seconds=args.cpu_seconds)
        # one thread, a smaller sample (a token each from every batch)
        r1, n1, s1, _, p1 = cpu_oracle_rate(wl, host, 1, reps=1, min_seconds=min(3.0, args.cpu_seconds), max_reps=3,
                                            nthreads=1)
        out["cpu_baseline"] = {"value": round(rate, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                               "cpu": cpu_model(),
                               "sample": f"{ntok} tokens: {reps} passes over up to {cap} tokens of each batch "
                                         f"T={wl['Ts']} ({secs:.1f} s)",
                               "single_thread": {"value": round(r1, 3), "unit": "tokens/s",
                                                 "sample": f"{n1} tokens in {p1} passes ({s1:.1f} s)"}}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
