"""Shared helpers of the GPU parity tests: tolerances and comparisons against the oracle.

Tolerances (attention): max-abs error <= 2e-2 and relative L2 error <= 1e-3
against the float64 oracle, bf16 inputs upcast exactly.  SnapKV: index sets
equal except positions whose oracle score lies within 1e-5 (relative) of the
K-th kept score.  Sampling: decisions equal except where |u*q - p| < 1e-6 or
the inverse-CDF target lies within 1e-6 (relative) of a bucket edge.
"""
import numpy as np
import pytest
import torch

ATT_MAX_ABS = 2e-2
ATT_REL_L2 = 1e-3
LSE_ABS = 1e-3
SNAP_REL = 1e-5
SAMPLE_BAND = 1e-6


def gpu_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from long_context_speculative_split_gb300 import build
    build.build()
    return torch.device("cuda:0")


def to64(t):
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.double().numpy()


def assert_attention_close(got, ref, what="out"):
    g = to64(got) if isinstance(got, torch.Tensor) else np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), "%s has non-finite values" % what
    err = np.abs(g - r)
    rel = np.linalg.norm((g - r).ravel()) / max(np.linalg.norm(r.ravel()), 1e-300)
    assert err.max() <= ATT_MAX_ABS, "%s max-abs %.3e" % (what, err.max())
    assert rel <= ATT_REL_L2, "%s rel-L2 %.3e" % (what, rel)
    return err.max(), rel


def assert_lse_close(got, ref):
    g = to64(got)
    assert np.all(np.isfinite(g))
    assert np.abs(g - np.asarray(ref)).max() <= LSE_ABS


def assert_index_sets_match(gpu_idx, ref_idx, pooled_ref, kth):
    """gpu_idx / ref_idx: 1-D ascending kept positions of one (sequence, KV head)."""
    g = [int(x) for x in gpu_idx]
    assert g == sorted(g) and len(set(g)) == len(g), "GPU indices not strictly ascending"
    assert len(g) == len(ref_idx)
    diff = set(g) ^ set(int(x) for x in ref_idx)
    for j in diff:
        assert np.isfinite(kth), "sets differ but every prefix row is kept by rule"
        assert abs(pooled_ref[j] - kth) <= SNAP_REL * abs(kth), \
            "position %d (score %.9g) differs outside the band around %.9g" % (j, pooled_ref[j], kth)
    return len(diff)
