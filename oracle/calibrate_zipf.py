"""Calibrate the Zipf router-bias magnitude of the long skewed-prefill workload.

Each of the four skewed layers adds b_e = beta * r_e^-1.1 to expert e's
selection score (r = a seeded rank permutation, rank 1 hottest). beta is found
by bisection on [0, 4] (40 steps) so that, on the workload's own 4096 tokens
routed by the oracle, the hottest expert's token count is 20x the mean count.
The bias enters the selection score only ("YoungAi - DeepSeek V4.1 Flash on one
DGX Spark", section 3: "selection score += delta-b").

Run:  python -m oracle.calibrate_zipf   (writes synth/zipf_beta.json)
Routing here is the oracle's own; nothing else is executed.
"""
import json
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

TARGET = 20.0


def load_ratio(shape, L, profile, beta):
    r = oracle.select(shape, L, (beta * profile).astype(np.float32))
    counts = np.bincount(r["idx"].ravel(), minlength=shape.n_experts)
    return counts.max() / counts.mean(), counts


def main():
    wl = synth.WORKLOADS["prefill_t4096_zipf4"]
    shape = wl.shape
    x = synth.make_tokens(wl.name)
    out = {"target_max_over_mean": TARGET, "zipf_s": synth.ZIPF_S, "tokens": int(x.shape[0]), "beta": {},
           "achieved": {}}
    for seed in wl.layer_seeds:
        t0 = time.time()
        router = synth.normal_f32(shape.n_experts * shape.hidden, seed, synth.S_ROUTER, 0.02)
        L = oracle.logits(shape, router.reshape(shape.n_experts, shape.hidden), x)
        profile = synth.zipf_profile(shape.n_experts, seed)
        lo, hi = 0.0, 4.0
        for _ in range(40):
            mid = 0.5 * (lo + hi)
            ratio, _ = load_ratio(shape, L, profile, mid)
            if ratio < TARGET:
                lo = mid
            else:
                hi = mid
        beta = float(np.float32(0.5 * (lo + hi)))
        ratio, counts = load_ratio(shape, L, profile, beta)
        out["beta"][str(seed)] = beta
        out["achieved"][str(seed)] = {"max_over_mean": float(ratio), "max": int(counts.max()),
                                      "min": int(counts.min()), "mean": float(counts.mean())}
        print(f"layer seed {seed:#x}: beta={beta:.6f} max/mean={ratio:.3f} ({time.time() - t0:.1f}s)")
    with open(synth.ZIPF_BETA_FILE, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
