"""mgd_spec_sample_noalloc, the entry point for callers that cannot allocate
device memory (a host framework that owns every byte through its own pool, or a
serving loop whose memory is planned once at start-up and may not call
cudaMalloc per token).  It keeps its scratch in a library-owned device array
instead of a caller workspace; these tests check, through the C ABI, that two
calls in a row give exactly the tokens of the workspace entry point, and that
requests larger than the fixed array are refused with a clear error.

This file is collected last on purpose: it must pass in a fresh process and
after every other test."""
import pytest
import torch

from _parity import gpu_or_skip
from long_context_speculative_split_gb300 import mgd, ops
from long_context_speculative_split_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    dev = gpu_or_skip()
    c = dict(wl.WORKLOADS["b32_ctx8k"], B=64)
    B, g, V = c["B"], c["gamma"], c["V"]
    for seed in (31, 32):  # two calls in a row; the second reuses the array the first left behind
        t, d = wl.logits(c, dev, seed=seed)
        u = wl.uniforms(c, dev, seed=seed)
        tok_ref = ops.draft_draw(d, u)
        out_ref, nacc_ref = ops.rejection_sample(t, d, tok_ref, u)

        tok = torch.full((B, g), -5, dtype=torch.int32, device=dev)
        mgd.mgd_spec_sample_noalloc(None, d, tok, u, B, g, V, mgd.MGD_DRAW_DRAFT, -1, None, None)
        out = torch.full((B, g + 1), -5, dtype=torch.int32, device=dev)
        nacc = torch.full((B,), -5, dtype=torch.int32, device=dev)
        mgd.mgd_spec_sample_noalloc(t, d, tok, u, B, g, V, mgd.MGD_VERIFY, -1, out, nacc)
        torch.cuda.synchronize()
        # same kernels, same inputs: integer results must be identical
        assert torch.equal(tok, tok_ref)
        assert torch.equal(nacc, nacc_ref)
        assert torch.equal(out, out_ref)
        # the verify that reuses the draws' statistics, after draws into the same scratch
        ws = ops.workspace(mgd.mgd_spec_workspace_size(B, g, V), dev)
        ops.draft_draw(d, u, draft_tokens=tok_ref, ws=ws)
        out_ref, nacc_ref = ops.rejection_sample(t, d, tok_ref, u, ws=ws, reuse_draft_stats=True)
        mgd.mgd_spec_sample_noalloc(None, d, tok, u, B, g, V, mgd.MGD_DRAW_DRAFT, -1, None, None)
        mgd.mgd_spec_sample_noalloc(t, d, tok, u, B, g, V, mgd.MGD_VERIFY_DRAWN, -1, out, nacc)
        torch.cuda.synchronize()
        assert mgd.mgd_workspace_errors(ws) == 0
        assert torch.equal(tok, tok_ref)
        assert torch.equal(nacc, nacc_ref)
        assert torch.equal(out, out_ref)


def test_noalloc_refuses_requests_beyond_its_array():
    gpu_or_skip()
    B, g, V = 4096, 4, 128256
    assert mgd.mgd_spec_workspace_size(B, g, V) > mgd.MGD_NOALLOC_SCRATCH_BYTES
    # every pointer is NULL: the size check refuses the call first; were it ever to stop doing
    # so, the null-pointer check of the sampling call would refuse it before any launch, and
    # the status below would fail the test instead of a kernel touching memory
    with pytest.raises(mgd.MgdError) as e:
        mgd.mgd_spec_sample_noalloc(None, None, None, None, B, g, V, mgd.MGD_VERIFY, -1, None, None)
    assert e.value.status == mgd.MGD_ERR_UNSUPPORTED
    assert "scratch" in str(e.value)
