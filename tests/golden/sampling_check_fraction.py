"""Fraction of sequences whose speculation round the GPU parity test can compare exactly.

"Wann beschleunigt spekulatives Decoding das LLM-Serving?", "Eine
Verifizierungsrunde verstehen": a round accepts candidates left to right and
ends with one correction or bonus draw.  The GPU decisions are compared with
the float64 oracle's exactly, except for a sequence where the oracle reports a
tested acceptance with |u*q - p| < 1e-6, or a final draw whose target lies
within 1e-6 of a bucket edge (relative to the total).  Which sequences those
are is fixed by the inputs and the oracle alone, so the fraction of fully
compared sequences is known before any kernel runs.  This script computes it
with ``oracle/`` only (the draft tokens are the oracle's own draws) and writes
tests/golden/sampling_check_fraction.json; the GPU test asserts that the
fraction it achieves is this one, within a few points (the GPU's draft tokens
differ from the oracle's only inside the band).

    python tests/golden/sampling_check_fraction.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

from long_context_speculative_split_gb300 import workloads as wl  # noqa: E402
from oracle.sampling import draft_draw, rejection_sample  # noqa: E402

BAND = 1e-6

# (case id, workload, overrides, seed): the cases of tests/test_gpu_sampling.py
CASES = [
    ("tiny_b2", "tiny_b2", {}, 0),
    ("b32_ctx8k", "b32_ctx8k", {}, 0),
    ("b128_ctx32k", "b128_ctx32k", {}, 0),
    ("ragged_b256_ctx4k_64k", "ragged_b256_ctx4k_64k", {}, 0),
    ("odd_vocab_b300", "b32_ctx8k", dict(B=300, V=4099, gamma=5, sigma=2.0, sigma_n=1.0), 4),
    ("masked_vocab_b64", "b32_ctx8k", dict(B=64, V=32000, mask_frac=0.6), 6),
    ("gamma1_b40", "b32_ctx8k", dict(B=40, V=5000, gamma=1), 7),
    ("gamma16_b24", "b32_ctx8k", dict(B=24, V=5000, gamma=16), 8),
    ("qwen_vocab_b48", "b32_ctx8k", dict(B=48, V=152064), 9),
    ("odd_vocab_five_chunks_b100", "b32_ctx8k", dict(B=100, V=65539), 10),
    ("odd_vocab_ten_chunks_b50", "b32_ctx8k", dict(B=50, V=147459), 11),
]


def fully_checked_fraction(cfg, seed):
    t, d = wl.logits(cfg, "cpu", seed=seed)
    u = wl.uniforms(cfg, "cpu", seed=seed)
    tok, _ = draft_draw(d, u)
    ref = rejection_sample(t, d, tok, u)
    gamma = cfg["gamma"]
    with np.errstate(invalid="ignore"):
        amb = ref["accept_margin"] < BAND
    first = np.where(amb.any(axis=1), amb.argmax(axis=1), gamma + 1)
    full = (first > gamma) & ~(ref["draw_margin"] < BAND)
    return float(full.mean()), int(full.sum()), int(full.size)


def main():
    out = {"band": BAND, "cases": {},
           "written_by": "tests/golden/sampling_check_fraction.py (oracle draft_draw and rejection_sample only)"}
    for cid, name, over, seed in CASES:
        cfg = dict(wl.WORKLOADS[name], **over)
        frac, n, tot = fully_checked_fraction(cfg, seed)
        out["cases"][cid] = {"fraction": frac, "fully_checked": n, "sequences": tot, "seed": seed}
        print(cid, frac, n, tot, flush=True)
    with open(os.path.join(HERE, "sampling_check_fraction.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
