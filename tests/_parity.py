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


# ---------------------------------------------------------------- canaries
# Out-of-bounds writes by a kernel would only be caught by a compared value they happen to
# corrupt; instead every output of the parity tests can sit between two guard regions of one
# allocation, filled with a poison bit pattern (a NaN for float types, the same bits for
# integers), and padded rows that a call must leave alone can be poisoned too.  After the
# call the poison must be intact, bit for bit.
_BITS = {torch.float32: torch.int32, torch.int32: torch.int32, torch.bfloat16: torch.int16,
         torch.int16: torch.int16}
_POISON = {torch.int32: 0x7FBADBAD, torch.int16: 0x7FBA}   # NaN payloads as f32 / bf16


def poison_value(dtype):
    return _POISON[_BITS[dtype]]


def poison_(t):
    """Fill t (any tensor of a guarded dtype) with the poison pattern; returns t."""
    t.view(_BITS[t.dtype]).fill_(poison_value(t.dtype))
    return t


def is_poison(t):
    """Elementwise: does t still hold the poison pattern?"""
    return t.view(_BITS[t.dtype]) == poison_value(t.dtype)


class Guarded:
    """An output tensor `t` between two 4 KB poisoned guard regions of one allocation (the
    offset keeps t 256-byte aligned).  `init` fills t (default: poison, so elements a call
    must write and does not stay visibly unwritten)."""
    GUARD_BYTES = 4096

    def __init__(self, shape, dtype, device, init=None):
        esz = torch.empty((), dtype=dtype).element_size()
        self.g = self.GUARD_BYTES // esz
        n = int(np.prod(shape)) if len(shape) else 1
        self.buf = poison_(torch.empty(2 * self.g + n, dtype=dtype, device=device))
        self.t = self.buf[self.g:self.g + n].view(*shape)
        if init is not None:
            self.t.copy_(init)

    def check(self, what="output"):
        head, tail = self.buf[:self.g], self.buf[self.buf.numel() - self.g:]
        assert bool(is_poison(head).all()), "%s: the guard region before it was written" % what
        assert bool(is_poison(tail).all()), "%s: the guard region after it was written" % what


def check_guards(**guards):
    for name, g in guards.items():
        g.check(name)
