"""Fused MoE layer forward (RMSNorm -> router/top-k -> align -> gate/up GEMM + SwiGLU
-> down GEMM -> combine) for one GB300, behind a C ABI.

The compiled library is loaded lazily by :mod:`mixture_experts_layer_rmsnorm_gb300.binding`
so that the seeded input generator (:mod:`.inputs`) can be imported on hosts without
a GPU.
"""
