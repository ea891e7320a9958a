"""Derives rho for the M = 10 verify-block input recipe
x_t = sqrt(rho) u + sqrt(1 - rho) z_t (u shared by the step's tokens, z_t per
token), so that on average half of each token's top-8 experts overlap the
previous token's top-8 (4.0 of 8). Routing is computed by the CPU oracle only,
on layer copy 0 of the Ling-shape layer, over steps 0..63; rho is bisected on
a grid of 2^-10. Writes overlap_rho.json beside this file.

Run:  python tests/golden/derive_overlap_rho.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from moe_decode_gb300 import synth  # noqa: E402

STEPS, M, TARGET = 64, 10, 4.0


def stats(Wg, rho):
    ov, uniq = [], []
    for s in range(STEPS):
        x = synth.to_u16(synth.x_overlap(synth.LING, s, M, rho))
        idx, _, _ = oracle.route(x, Wg, 8)
        for t in range(1, M):
            ov.append(len(set(idx[t]) & set(idx[t - 1])))
        uniq.append(len(set(idx.ravel())))
    return float(np.mean(ov)), float(np.mean(uniq))


def main():
    Wg = synth.to_u16(synth.router_weight(synth.LING, 0))
    lo, hi = 0, 1024
    while hi - lo > 1:
        mid = (lo + hi) // 2
        o, _ = stats(Wg, mid / 1024)
        if o < TARGET:
            lo = mid
        else:
            hi = mid
    cands = [(abs(stats(Wg, r / 1024)[0] - TARGET), r) for r in (lo, hi)]
    r = min(cands)[1]
    o, u = stats(Wg, r / 1024)
    out = {"rho": r / 1024, "mean_consecutive_overlap": o, "mean_distinct_experts": u,
           "target_overlap": TARGET, "steps": STEPS, "M": M, "layer_copy": 0,
           "router": "CPU oracle (oracle.route), fp32"}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "overlap_rho.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print(json.dumps(out))


if __name__ == "__main__":
    main()
