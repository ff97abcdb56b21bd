"""Writes tests/golden/tiny_oracle.json: the CPU oracle's outputs on the tiny
workload (T=4, H=128, I=256, E=8, top_k=2, renormalised, eps=1e-6, seed 0).

It calls only the oracle (and the seeded input generator).  Re-run it only
when a change to the oracle's arithmetic is justified by the pages; the
regression test then checks that every later build of the oracle, on either
host architecture, reproduces these values.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from mixture_experts_layer_rmsnorm_gb300 import inputs  # noqa: E402


def main():
    cfg = inputs.WORKLOADS["tiny"]
    li = inputs.make_layer_inputs(cfg)
    r = oracle.moe_forward(li.x, li.g, li.w_router, li.bias, li.w13, li.w2, cfg.top_k, cfg.renormalize, cfg.eps)
    out = {
        "_about": "CPU oracle outputs on the tiny workload; written by tests/golden/make_golden.py",
        "config": {"T": cfg.T, "H": cfg.H, "I": cfg.I, "E": cfg.E, "top_k": cfg.top_k,
                   "renormalize": cfg.renormalize, "eps": cfg.eps, "seed": cfg.seed},
        "topk_ids": r["ids"].tolist(),
        "topk_w": [[float(v) for v in row] for row in r["w"]],
        "y_bf16_bits": [[int(v) for v in row] for row in r["y16"]],
        "h_bf16_bits_first8": [[int(v) for v in row[:8]] for row in r["h16"]],
        "logits_f32_first8": [[float(v) for v in row] for row in r["l32"]],
    }
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
