"""Concurrent calls on two CUDA streams with distinct workspaces (the header's thread-safety
contract): the results equal those of the same calls made one after the other.

Integer outputs (selected indices, drawn tokens, accept counts) must be identical; attention
outputs may differ only by float reassociation inside a CTA (the epilogue adds the four warps'
partial outputs in arrival order), far below the oracle tolerances."""
import pytest
import torch

from _parity import gpu_or_skip
from long_context_speculative_split_gb300 import mgd, ops
from long_context_speculative_split_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _inputs(dev, seed):
    c = dict(wl.WORKLOADS["b32_ctx8k"], B=8, lens=4096, V=32000)
    kv_len = wl.lengths(c, seed)
    k, v = wl.kv_cache(c, dev, seed, kv_len=kv_len, cap=4096)
    q = wl.queries(c, dev, seed)
    qw = wl.window_queries(c, dev, seed)
    t, d = wl.logits(c, dev, seed)
    u = wl.uniforms(c, dev, seed)
    return c, kv_len.to(dev), k, v, q, qw, t, d, u


def _run(c, kv_len, k, v, q, qw, t, d, u, stream):
    dev = k.device
    B, g = c["B"], c["gamma"]
    ws_v = ops.workspace(mgd.mgd_verify_workspace_size(B, g + 1, c["Hq"], c["Hkv"], c["D"], 4096), dev)
    ws_s = ops.workspace(mgd.mgd_snapkv_workspace_size(B, c["Hq"], c["Hkv"], c["D"], 4096, c["W"]), dev)
    ws_p = ops.workspace(mgd.mgd_spec_workspace_size(B, g, c["V"]), dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        out, lse = ops.verify_attn(q, k, v, kv_len, ws=ws_v, stream=stream)
        sel = ops.snapkv_select(qw, k, v, kv_len, c["W"], c["pool"], c["K"], ws=ws_s, stream=stream)
        tok = torch.full((B, g), -1, dtype=torch.int32, device=dev)
        ops.draft_draw(d, u, draft_tokens=tok, ws=ws_p, stream=stream)
        toks, nacc = ops.rejection_sample(t, d, tok, u, ws=ws_p, stream=stream)
    return dict(out=out, lse=lse, sel=sel["sel_idx"], dlen=sel["draft_len"], tok=tok, toks=toks, nacc=nacc,
                ws=(ws_v, ws_s, ws_p))


def test_two_streams_match_serial_runs():
    dev = gpu_or_skip()
    a_in, b_in = _inputs(dev, 1), _inputs(dev, 2)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    # serial reference: one after the other on one stream
    ra = _run(*a_in, stream=s1)
    torch.cuda.synchronize()
    rb = _run(*b_in, stream=s1)
    torch.cuda.synchronize()
    # concurrent: the two calls sequences issued on two streams before any synchronisation
    ca = _run(*a_in, stream=s1)
    cb = _run(*b_in, stream=s2)
    torch.cuda.synchronize()
    for ref, got in ((ra, ca), (rb, cb)):
        for ws in got["ws"]:
            assert mgd.mgd_workspace_errors(ws) == 0
        assert torch.equal(ref["sel"], got["sel"]) and torch.equal(ref["dlen"], got["dlen"])
        assert torch.equal(ref["tok"], got["tok"])
        assert torch.equal(ref["toks"], got["toks"]) and torch.equal(ref["nacc"], got["nacc"])
        torch.testing.assert_close(got["out"], ref["out"], rtol=1e-5, atol=1e-6)
        torch.testing.assert_close(got["lse"], ref["lse"], rtol=1e-6, atol=1e-6)
