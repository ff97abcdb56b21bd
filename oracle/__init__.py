"""CPU oracle of the fused MoE layer forward -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg import this package.  It wraps ``moe_oracle.c`` (plain fp64 C,
compiled with the host compiler) through ctypes and shares no code with the
CUDA path.  The definitions it follows are cited in ``moe_oracle.c``.

Every function here is pinned by ``tests/test_oracle_pins.py`` to something
other than the oracle itself (closed forms, library routines, brute force,
invariants); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_default = None


def build_lib(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle with gcc.  -ffp-contract=off keeps every fp32
    multiply and add separately rounded unless the source asks for fmaf."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
                               "-fno-fast-math", "-o", tmp, src, "-lm"])
        os.replace(tmp, out)
    return out


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def threads() -> int:
    return max(1, os.cpu_count() or 1)


class Oracle:
    """ctypes view of one compiled copy of moe_oracle.c."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        i64, p, i, d, f = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_float
        lib.oracle_rmsnorm_f64.argtypes = [i64, i64, p, p, d, p, p]
        lib.oracle_router_logits_f64.argtypes = [i64, i64, i64, p, p, p, p]
        lib.oracle_route_f32.argtypes = [i64, i64, i64, p, p, f, p, p, p, p, p, i]
        lib.oracle_topk_f32.argtypes = [i64, i64, i, p, p]
        lib.oracle_topk_f64.argtypes = [i64, i64, i, p, p]
        lib.oracle_route_weights_f64.argtypes = [i64, i64, i, p, p, i, p]
        lib.oracle_align.argtypes = [i64, i64, p, i64, p, p, p, i64, p]
        lib.oracle_align.restype = i64
        lib.oracle_expert_f64.argtypes = [i64, i64, p, p, p, p, i, p, p]
        lib.oracle_moe_forward.argtypes = [i64, i64, i64, i64, i, i, d, p, p, p, p, p, p, i64, p, i, i,
                                           p, p, p, p, p, p, p]
        lib.oracle_moe_forward.restype = i
        lib.oracle_qk_norm_f64.argtypes = [i64, i64, p, p, d, d, p]
        lib.oracle_e4m3_encode.argtypes = [d]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = d
        lib.oracle_mx_quantize.argtypes = [i64, i64, p, p, p]
        lib.oracle_mx_dequantize.argtypes = [i64, i64, p, p, p]
        lib.oracle_expert_mx_f64.argtypes = [i64, i64, p, p, p, p, p, p, p]
        lib.oracle_moe_forward_mx.argtypes = [i64, i64, i64, i64, i, i, d, p, p, p, p, p, p, p, p, i64, p, i,
                                              p, p, p, p]
        lib.oracle_moe_forward_mx.restype = i
        lib.oracle_e2m1_encode.argtypes = [d]
        lib.oracle_e2m1_encode.restype = ctypes.c_uint8
        lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e2m1_decode.restype = d
        lib.oracle_mx4_quantize.argtypes = [i64, i64, p, p, p]
        lib.oracle_mx4_dequantize.argtypes = [i64, i64, p, p, p]
        lib.oracle_expert_mx4_f64.argtypes = [i64, i64, p, p, p, p, p, p, p]
        lib.oracle_moe_forward_mx4.argtypes = [i64, i64, i64, i64, i, i, d, p, p, p, p, p, p, p, p, i64, p, i,
                                               p, p, p, p]
        lib.oracle_moe_forward_mx4.restype = i
        lib.oracle_moe_forward_mx4a4.argtypes = [i64, i64, i64, i64, i, i, d, p, p, p, p, p, p, p, p, i64, p, i,
                                                 p, p, p, p]
        lib.oracle_moe_forward_mx4a4.restype = i
        lib.oracle_nv4_quantize.argtypes = [i64, i64, p, i, p, p, p]
        lib.oracle_nv4_dequantize.argtypes = [i64, i64, p, p, p, i, p]
        lib.oracle_moe_forward_nv4.argtypes = [i64, i64, i64, i64, i, i, d, p, p, p, p, p, p, p, p, p, p, i64, p,
                                               i, p, p, p, p]
        lib.oracle_moe_forward_nv4.restype = i
        lib.oracle_f64_to_bf16.argtypes = [d]
        lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
        lib.oracle_f32_to_bf16.argtypes = [f]
        lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
        self.lib = lib
        self.path = lib_path

    def f64_to_bf16(self, v: float) -> int:
        return int(self.lib.oracle_f64_to_bf16(float(v)))

    def f32_to_bf16(self, v: float) -> int:
        return int(self.lib.oracle_f32_to_bf16(float(v)))

    def rmsnorm_f64(self, x, g, eps):
        """h (bf16 bits, [T,H]) and the unrounded fp64 values."""
        x = _c(x, np.uint16); g = _c(g, np.uint16)
        T, H = x.shape
        h = np.empty((T, H), np.uint16); he = np.empty((T, H), np.float64)
        self.lib.oracle_rmsnorm_f64(T, H, _p(x), _p(g), float(eps), _p(h), _p(he))
        return h, he

    def qk_norm_f64(self, x, w, weight_bias, eps):
        """QK-norm of head vectors x[..., D] (bf16 bits) with gain w[D] + weight_bias."""
        x = _c(x, np.uint16); w = _c(w, np.uint16)
        D = x.shape[-1]
        out = np.empty(x.shape, np.uint16)
        self.lib.oracle_qk_norm_f64(x.size // D, D, _p(x), _p(w), float(weight_bias), float(eps), _p(out))
        return out

    def e4m3_encode(self, v: float) -> int:
        return int(self.lib.oracle_e4m3_encode(float(v)))

    def e4m3_decode(self, c: int) -> float:
        return float(self.lib.oracle_e4m3_decode(int(c)))

    def mx_quantize(self, x):
        """MXFP8 of bf16 rows x[..., K]: (codes [..., K] uint8, scales [..., K/32] uint8)."""
        x = _c(x, np.uint16)
        K = x.shape[-1]
        rows = x.size // K
        codes = np.empty(x.shape, np.uint8)
        scales = np.empty(x.shape[:-1] + (K // 32,), np.uint8)
        self.lib.oracle_mx_quantize(rows, K, _p(x), _p(codes), _p(scales))
        return codes, scales

    def mx_dequantize(self, codes, scales):
        codes = _c(codes, np.uint8); scales = _c(scales, np.uint8)
        K = codes.shape[-1]
        out = np.empty(codes.shape, np.float64)
        self.lib.oracle_mx_dequantize(codes.size // K, K, _p(codes), _p(scales), _p(out))
        return out

    def e2m1_encode(self, v: float) -> int:
        return int(self.lib.oracle_e2m1_encode(float(v)))

    def e2m1_decode(self, c: int) -> float:
        return float(self.lib.oracle_e2m1_decode(int(c)))

    def mx4_quantize(self, x):
        """MXFP4 of bf16 rows x[..., K]: (E2M1 codes [..., K] uint8 one per byte, scales [..., K/32] uint8)."""
        x = _c(x, np.uint16)
        K = x.shape[-1]
        rows = x.size // K
        codes = np.empty(x.shape, np.uint8)
        scales = np.empty(x.shape[:-1] + (K // 32,), np.uint8)
        self.lib.oracle_mx4_quantize(rows, K, _p(x), _p(codes), _p(scales))
        return codes, scales

    def mx4_dequantize(self, codes, scales):
        codes = _c(codes, np.uint8); scales = _c(scales, np.uint8)
        K = codes.shape[-1]
        out = np.empty(codes.shape, np.float64)
        self.lib.oracle_mx4_dequantize(codes.size // K, K, _p(codes), _p(scales), _p(out))
        return out

    def nv4_quantize(self, x, per_row):
        """NVFP4 of bf16 rows x[..., K]: (E2M1 codes [..., K] one per byte, E4M3
        block scales [..., K/16], fp32 tensor scales: [rows] per row, else [1])."""
        x = _c(x, np.uint16)
        K = x.shape[-1]
        rows = x.size // K
        codes = np.empty(x.shape, np.uint8)
        scales = np.empty(x.shape[:-1] + (K // 16,), np.uint8)
        g = np.empty(rows if per_row else 1, np.float32)
        self.lib.oracle_nv4_quantize(rows, K, _p(x), int(bool(per_row)), _p(codes), _p(scales), _p(g))
        return codes, scales, g

    def nv4_quantize_experts(self, w):
        """NVFP4 of expert weights w[E, rows, K] with one tensor scale per expert matrix:
        (codes [E, rows, K], scales [E, rows, K/16], g [E])."""
        w = _c(w, np.uint16)
        cs = [self.nv4_quantize(w[e], per_row=False) for e in range(w.shape[0])]
        return (np.stack([c[0] for c in cs]), np.stack([c[1] for c in cs]),
                np.concatenate([c[2] for c in cs]).astype(np.float32))

    def nv4_dequantize(self, codes, scales, g, per_row):
        codes = _c(codes, np.uint8); scales = _c(scales, np.uint8); g = _c(g, np.float32)
        K = codes.shape[-1]
        out = np.empty(codes.shape, np.float64)
        self.lib.oracle_nv4_dequantize(codes.size // K, K, _p(codes), _p(scales), _p(g), int(bool(per_row)), _p(out))
        return out

    def moe_forward_nv4(self, x, g, w_router, bias, w13c, w13s, w13g, w2c, w2s, w2g, top_k, renorm, eps,
                        sample=None, nthreads=None):
        """The NVFP4 layer (NVFP4 weights with a tensor scale per expert matrix,
        NVFP4 tokens and activations with one per row): ids, w, y64, y16, sample."""
        x = _c(x, np.uint16); g = _c(g, np.uint16); wr = _c(w_router, np.float32)
        w13c = _c(w13c, np.uint8); w13s = _c(w13s, np.uint8); w2c = _c(w2c, np.uint8); w2s = _c(w2s, np.uint8)
        w13g = _c(w13g, np.float32); w2g = _c(w2g, np.float32)
        T, H = x.shape; E = wr.shape[0]; I = w13c.shape[1] // 2
        b = None if bias is None else _c(bias, np.float32)
        smp = np.arange(T, dtype=np.int64) if sample is None else _c(sample, np.int64)
        S = smp.size; k = int(top_k)
        out = dict(ids=np.empty((S, k), np.int32), w=np.empty((S, k), np.float64),
                   y64=np.empty((S, H), np.float64), y16=np.empty((S, H), np.uint16), sample=smp)
        rc = self.lib.oracle_moe_forward_nv4(T, H, I, E, k, int(bool(renorm)), float(eps), _p(x), _p(g), _p(wr),
                                             _p(b), _p(w13c), _p(w13s), _p(w13g), _p(w2c), _p(w2s), _p(w2g), S,
                                             _p(smp), int(nthreads or threads()), _p(out["ids"]), _p(out["w"]),
                                             _p(out["y64"]), _p(out["y16"]))
        if rc != 0:
            raise ValueError("oracle_moe_forward_nv4: bad input")
        return out

    def expert_mx4_f64(self, h, w13c, w13s, w2c, w2s):
        """One token (bf16 h) through one expert with MXFP4 weights: (activation [I], output [H]) f64."""
        h = _c(h, np.uint16)
        w13c = _c(w13c, np.uint8); w13s = _c(w13s, np.uint8); w2c = _c(w2c, np.uint8); w2s = _c(w2s, np.uint8)
        H = h.shape[-1]; I = w13c.shape[0] // 2
        a = np.empty(I, np.float64); o = np.empty(H, np.float64)
        self.lib.oracle_expert_mx4_f64(H, I, _p(h), _p(w13c), _p(w13s), _p(w2c), _p(w2s), _p(a), _p(o))
        return a, o

    def moe_forward_mx4(self, x, g, w_router, bias, w13c, w13s, w2c, w2s, top_k, renorm, eps, sample=None,
                        nthreads=None):
        """The FP4-weight layer (MXFP4 weights, MXFP8 tokens and activations); as moe_forward_mx."""
        return self.moe_forward_mx(x, g, w_router, bias, w13c, w13s, w2c, w2s, top_k, renorm, eps, sample,
                                   nthreads, _fn=self.lib.oracle_moe_forward_mx4)

    def moe_forward_mx4a4(self, x, g, w_router, bias, w13c, w13s, w2c, w2s, top_k, renorm, eps, sample=None,
                          nthreads=None):
        """The MXFP4 layer (MXFP4 weights, MXFP4 tokens and activations); as moe_forward_mx."""
        return self.moe_forward_mx(x, g, w_router, bias, w13c, w13s, w2c, w2s, top_k, renorm, eps, sample,
                                   nthreads, _fn=self.lib.oracle_moe_forward_mx4a4)

    def expert_mx_f64(self, h, w13c, w13s, w2c, w2s):
        """One token (bf16 h) through one FP8 expert: (activation [I] f64 after MXFP8, output [H] f64)."""
        h = _c(h, np.uint16)
        w13c = _c(w13c, np.uint8); w13s = _c(w13s, np.uint8); w2c = _c(w2c, np.uint8); w2s = _c(w2s, np.uint8)
        H = h.shape[-1]; I = w13c.shape[0] // 2
        a = np.empty(I, np.float64); o = np.empty(H, np.float64)
        self.lib.oracle_expert_mx_f64(H, I, _p(h), _p(w13c), _p(w13s), _p(w2c), _p(w2s), _p(a), _p(o))
        return a, o

    def moe_forward_mx(self, x, g, w_router, bias, w13c, w13s, w2c, w2s, top_k, renorm, eps, sample=None,
                       nthreads=None, _fn=None):
        """The FP8 layer (MXFP8 weights and activations) for the sampled tokens:
        ids [S,k], w [S,k], y64 [S,H], y16 [S,H] bf16 bits, sample [S]."""
        x = _c(x, np.uint16); g = _c(g, np.uint16); wr = _c(w_router, np.float32)
        w13c = _c(w13c, np.uint8); w13s = _c(w13s, np.uint8); w2c = _c(w2c, np.uint8); w2s = _c(w2s, np.uint8)
        T, H = x.shape; E = wr.shape[0]; I = w13c.shape[1] // 2
        b = None if bias is None else _c(bias, np.float32)
        smp = np.arange(T, dtype=np.int64) if sample is None else _c(sample, np.int64)
        S = smp.size; k = int(top_k)
        out = dict(ids=np.empty((S, k), np.int32), w=np.empty((S, k), np.float64),
                   y64=np.empty((S, H), np.float64), y16=np.empty((S, H), np.uint16), sample=smp)
        fn = _fn or self.lib.oracle_moe_forward_mx
        rc = fn(T, H, I, E, k, int(bool(renorm)), float(eps), _p(x), _p(g), _p(wr), _p(b), _p(w13c), _p(w13s),
                _p(w2c), _p(w2s), S, _p(smp), nthreads or threads(), _p(out["ids"]), _p(out["w"]), _p(out["y64"]),
                _p(out["y16"]))
        if rc != 0:
            raise ValueError("oracle_moe_forward_mx: bad arguments")
        return out

    def router_logits_f64(self, h, w_router, bias=None):
        h = _c(h, np.uint16); wr = _c(w_router, np.float32)
        T, H = h.shape; E = wr.shape[0]
        b = None if bias is None else _c(bias, np.float32)
        out = np.empty((T, E), np.float64)
        self.lib.oracle_router_logits_f64(T, H, E, _p(h), _p(wr), _p(b), _p(out))
        return out

    def route_f32(self, x, g, eps, w_router, bias=None, nthreads=None):
        """Kernel-precision front end: (h bf16 bits [T,H], logits fp32 [T,E], rstd fp32 [T])."""
        x = _c(x, np.uint16); g = _c(g, np.uint16); wr = _c(w_router, np.float32)
        T, H = x.shape; E = wr.shape[0]
        b = None if bias is None else _c(bias, np.float32)
        h = np.empty((T, H), np.uint16); l = np.empty((T, E), np.float32); r = np.empty(T, np.float32)
        self.lib.oracle_route_f32(T, H, E, _p(x), _p(g), float(eps), _p(wr), _p(b), _p(h), _p(l), _p(r),
                                  nthreads or threads())
        return h, l, r

    def topk(self, logits, k):
        logits = np.ascontiguousarray(logits)
        T, E = logits.shape
        ids = np.empty((T, k), np.int32)
        if logits.dtype == np.float32:
            self.lib.oracle_topk_f32(T, E, k, _p(logits), _p(ids))
        else:
            logits = _c(logits, np.float64)
            self.lib.oracle_topk_f64(T, E, k, _p(logits), _p(ids))
        return ids

    def route_weights_f64(self, logits64, ids, renorm):
        l = _c(logits64, np.float64); ids = _c(ids, np.int32)
        T, E = l.shape; k = ids.shape[1]
        w = np.empty((T, k), np.float64)
        self.lib.oracle_route_weights_f64(T, E, k, _p(l), _p(ids), int(bool(renorm)), _p(w))
        return w

    def align(self, ids, E, pad):
        """(counts[E], offsets[E+1], sorted_ids[P], slot_of[N]) for flat routing ids."""
        ids = _c(np.asarray(ids).reshape(-1), np.int32)
        N = ids.size
        cap = N + E * (pad - 1)
        counts = np.empty(E, np.int32); offsets = np.empty(E + 1, np.int32)
        sorted_ids = np.empty(max(cap, 1), np.int32); slot_of = np.empty(max(N, 1), np.int32)
        total = self.lib.oracle_align(N, E, _p(ids), pad, _p(counts), _p(offsets), _p(sorted_ids), cap,
                                      _p(slot_of))
        assert total >= 0
        return counts, offsets, sorted_ids[:total].copy(), slot_of[:N].copy()

    def expert_f64(self, h, w13_e, w2_e, round_act=True):
        """One token through one expert: (a[I] fp64, o[H] fp64).  h: bf16 bits or float64 [H]."""
        w13_e = _c(w13_e, np.uint16); w2_e = _c(w2_e, np.uint16)
        H = w13_e.shape[1]; I = w13_e.shape[0] // 2
        a = np.empty(I, np.float64); o = np.empty(H, np.float64)
        h = np.ascontiguousarray(h)
        if h.dtype == np.uint16:
            self.lib.oracle_expert_f64(H, I, _p(h), None, _p(w13_e), _p(w2_e), int(round_act), _p(a), _p(o))
        else:
            h = _c(h, np.float64)
            self.lib.oracle_expert_f64(H, I, None, _p(h), _p(w13_e), _p(w2_e), int(round_act), _p(a), _p(o))
        return a, o

    def moe_forward(self, x, g, w_router, bias, w13, w2, top_k, renorm, eps, sample=None, round_inter=True,
                    nthreads=None):
        """Layer forward for the sampled tokens (all tokens if sample is None).

        Returns a dict: ids [S,k] int32, w [S,k] f64, y64 [S,H] f64, y16 [S,H] bf16 bits,
        h16 [S,H] bf16 bits, l32 [S,E] f32, l64 [S,E] f64, sample [S] int64.
        """
        x = _c(x, np.uint16); g = _c(g, np.uint16); wr = _c(w_router, np.float32)
        w13 = _c(w13, np.uint16); w2 = _c(w2, np.uint16)
        T, H = x.shape; E = wr.shape[0]; I = w13.shape[1] // 2
        b = None if bias is None else _c(bias, np.float32)
        smp = np.arange(T, dtype=np.int64) if sample is None else _c(sample, np.int64)
        S = smp.size; k = int(top_k)
        out = dict(ids=np.empty((S, k), np.int32), w=np.empty((S, k), np.float64),
                   y64=np.empty((S, H), np.float64), y16=np.empty((S, H), np.uint16),
                   h16=np.empty((S, H), np.uint16), l32=np.empty((S, E), np.float32),
                   l64=np.empty((S, E), np.float64), sample=smp)
        rc = self.lib.oracle_moe_forward(T, H, I, E, k, int(bool(renorm)), float(eps), _p(x), _p(g), _p(wr), _p(b),
                                         _p(w13), _p(w2), S, _p(smp), int(bool(round_inter)), nthreads or threads(),
                                         _p(out["ids"]), _p(out["w"]), _p(out["y64"]), _p(out["y16"]),
                                         _p(out["h16"]), _p(out["l32"]), _p(out["l64"]))
        if rc != 0:
            raise ValueError("oracle_moe_forward: bad arguments")
        return out


def default() -> Oracle:
    """The oracle built from moe_oracle.c (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build_lib())
    return _default


def __getattr__(name):
    # module-level shorthands: oracle.moe_forward(...), oracle.align(...), ...
    if name in ("f64_to_bf16", "f32_to_bf16", "rmsnorm_f64", "router_logits_f64", "route_f32", "topk",
                "route_weights_f64", "align", "expert_f64", "moe_forward", "qk_norm_f64", "mx_quantize",
                "mx_dequantize", "moe_forward_mx"):
        return getattr(default(), name)
    raise AttributeError(name)
