"""Calibrate the draft-logit noise of the 32-layer speculation-round workload.

The round workload (batch 32, context 16384, 32 layers, gamma 3, vocab
128256) asks for draft and target logits drawn so that the mean acceptance
alpha = E[sum_x min(p(x), q(x))] is about 0.9 (the acceptance at which MagicDec
notes, quick-read summary, say self-speculation with a compressed KV easily
operates).  Draft logits are target + sigma_n * N(0, 1); this script bisects
sigma_n with the float64 oracle's softmax over the seeded logits and writes
tests/golden/round_sigma.json.  Only ``oracle/`` computes anything here.

    python tests/golden/calibrate_round_sigma.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

from long_context_speculative_split_gb300 import workloads as wl  # noqa: E402
from oracle.sampling import softmax  # noqa: E402

TARGET_ALPHA = 0.9


def mean_alpha(sigma_n, cfg):
    t, d = wl.logits(cfg, "cpu", seed=0, sigma_n=sigma_n)
    p = softmax(t[:, : cfg["gamma"]])
    q = softmax(d)
    return float(np.minimum(p, q).sum(axis=-1).mean())


def main():
    cfg = wl.WORKLOADS["round_b32_ctx16k_32layers"]
    lo, hi = 0.0, 3.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if mean_alpha(mid, cfg) > TARGET_ALPHA:
            lo = mid
        else:
            hi = mid
    sigma = 0.5 * (lo + hi)
    out = {"workload": cfg["name"], "target_alpha": TARGET_ALPHA, "sigma_n": sigma,
           "alpha_at_sigma_n": mean_alpha(sigma, cfg),
           "omega_expected": (1 - TARGET_ALPHA ** (cfg["gamma"] + 1)) / (1 - TARGET_ALPHA),
           "written_by": "tests/golden/calibrate_round_sigma.py (oracle softmax only)"}
    with open(os.path.join(HERE, "round_sigma.json"), "w") as f:
        json.dump(out, f, indent=1)
    print(out)


if __name__ == "__main__":
    main()
