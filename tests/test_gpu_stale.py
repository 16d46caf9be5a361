"""Stale-workspace detection by the sampling and commit calls.

Every call leaves its workspace header ready for the next call instead of
clearing it first; a header that was not left ready (a stale claim count, a
stale check-in count or block-id sum) is detected at the call's last check-in
and raises MGD_DEVERR_STALE_WS.  The same buffer zero-filled again gives the
results of a fresh workspace with no error bits.  (The attention and SnapKV
calls are covered in test_gpu_attention.py.)"""
import pytest
import torch

from _parity import gpu_or_skip
from long_context_speculative_split_gb300 import mgd, ops

pytestmark = pytest.mark.gpu

# int32 words of the 256-byte header: err[0], err[1], next_unit, next_unit2, seq, claimed, then the
# 64-bit check-in word (low word: block-id sum; high word: id-sum bits 32..39 and the count << 8)
STALE_FIELDS = ((5, 2), (7, 1 << 8), (6, 9))


def _logits(B, gamma, V, dev, seed):
    g = torch.Generator().manual_seed(seed)
    t = (3.0 * torch.randn((B, gamma + 1, V), generator=g)).to(dev)
    d = (t[:, :gamma].cpu() + 0.5 * torch.randn((B, gamma, V), generator=g)).to(dev)
    u = torch.rand((B, gamma + 1, 3), generator=g).to(dev)
    return t, d, u


@pytest.mark.parametrize("B,V", [(32, 128256), (300, 1000)], ids=["b32_v128k", "b300_v1000"])
def test_sampling_stale_workspace_is_detected(B, V):
    dev = gpu_or_skip()
    gamma = 3
    t, d, u = _logits(B, gamma, V, dev, seed=B)
    need = mgd.mgd_spec_workspace_size(B, gamma, V)
    fresh = ops.workspace(need, dev)
    tok0 = ops.draft_draw(d, u, ws=fresh)
    out0, n0 = ops.rejection_sample(t, d, tok0, u, ws=fresh)
    torch.cuda.synchronize()
    assert mgd.mgd_workspace_errors(fresh) == 0
    ws = ops.workspace(need, dev)
    hdr = ws[:256].view(torch.int32)
    for field, value in STALE_FIELDS:
        ws.zero_()
        hdr[field] = value
        ops.draft_draw(d, u, ws=ws, row=0)
        assert mgd.mgd_workspace_errors(ws) & mgd.MGD_DEVERR_STALE_WS, ("draw", field, value)
        ws.zero_()
        hdr[field] = value
        ops.rejection_sample(t, d, tok0, u, ws=ws)
        assert mgd.mgd_workspace_errors(ws) & mgd.MGD_DEVERR_STALE_WS, ("reject", field, value)
    ws.zero_()
    tok = ops.draft_draw(d, u, ws=ws)
    out, n = ops.rejection_sample(t, d, tok, u, ws=ws)
    torch.cuda.synchronize()
    assert mgd.mgd_workspace_errors(ws) == 0
    assert torch.equal(tok, tok0) and torch.equal(out, out0) and torch.equal(n, n0)


def test_commit_stale_workspace_is_detected():
    dev = gpu_or_skip()
    B, Hkv, cap, dcap, D, gamma = 20, 8, 200, 64, 128, 3
    g = torch.Generator().manual_seed(5)
    k = torch.randn((B, Hkv, cap, D), generator=g).to(torch.bfloat16).to(dev)
    v = torch.randn((B, Hkv, cap, D), generator=g).to(torch.bfloat16).to(dev)
    kd0 = torch.randn((B, Hkv, dcap, D), generator=g).to(torch.bfloat16).to(dev)
    vd0 = torch.randn((B, Hkv, dcap, D), generator=g).to(torch.bfloat16).to(dev)
    kv_len0 = torch.randint(gamma + 1, cap + 1, (B,), generator=g, dtype=torch.int32).to(dev)
    dl0 = torch.randint(0, dcap - gamma - 1, (B,), generator=g, dtype=torch.int32).to(dev)
    nacc = torch.randint(0, gamma + 1, (B,), generator=g, dtype=torch.int32).to(dev)

    def run(ws):
        kl, dl, kd, vd = kv_len0.clone(), dl0.clone(), kd0.clone(), vd0.clone()
        ops.commit_round(nacc, gamma, kl, k, v, kd, vd, dl, ws=ws)
        torch.cuda.synchronize()
        return kl, dl, kd, vd

    need = mgd.mgd_commit_workspace_size(B)
    fresh = run(ops.workspace(need, dev))
    ws = ops.workspace(need, dev)
    hdr = ws[:256].view(torch.int32)
    for field, value in STALE_FIELDS:
        ws.zero_()
        hdr[field] = value
        run(ws)
        assert mgd.mgd_workspace_errors(ws) & mgd.MGD_DEVERR_STALE_WS, (field, value)
    ws.zero_()
    got = run(ws)
    assert mgd.mgd_workspace_errors(ws) == 0
    for a, b in zip(got, fresh):
        assert torch.equal(a, b)
