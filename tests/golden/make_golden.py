"""Writes the stored values under tests/golden/ that the oracle produces.

Calls only oracle/ (and synth/ for the seeded inputs); nothing here comes from
the CUDA path.  Run:  python tests/golden/make_golden.py

skew_bias_scale.json: the scale c of the Zipf-shaped router bias
  bias_e = -s * c * ln(r_e),  s = 1.2,  r a seeded permutation of 1..E,
for the skewed-routing workload (Qwen3-MoE shape).  c starts at 1 and is
multiplied by 1.5 until the oracle's routing has at least 8 experts with no
token and one expert holding more than 10% of the T*k assignments (the
hotspot and empty-expert regime the Awesome-ML-SYS-Tutorial MoE/EP guide
describes for EP: "Hotspot Expert" load imbalance, never-activated experts).
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth  # noqa: E402


def calibrate_skew(cfg):
    inp = synth.make_inputs(cfg, bias_scale=1.0, weights=False)
    c = 1.0
    while True:
        bias = synth.zipf_bias(cfg.seed, cfg.E, c)
        r = oracle.route(inp.x, inp.w_router, bias, cfg.k)
        counts = np.bincount(r["ids"].reshape(-1), minlength=cfg.E)
        empty = int((counts == 0).sum())
        top = float(counts.max()) / cfg.R
        if empty >= 8 and top > 0.10:
            return dict(c=c, empty_experts=empty, top_expert_share=top,
                        min_kgap=float(r["kgap"].min()))
        c *= 1.5


def main():
    out = {}
    for name, cfg in synth.CONFIGS.items():
        if cfg.skew:
            out[name] = calibrate_skew(cfg)
            print(name, out[name])
    with open(os.path.join(HERE, "skew_bias_scale.json"), "w") as f:
        json.dump(out, f, indent=1, sort_keys=True)
        f.write("\n")


if __name__ == "__main__":
    main()
