"""GPU parity of the commit / rollback step (mgd_commit_round) against the oracle:
byte copies and integer updates, so every result must be bit-exact; sequences
with out-of-range values must be left untouched and flagged."""
import numpy as np
import pytest
import torch

from _parity import Guarded, check_guards, gpu_or_skip
from long_context_speculative_split_gb300 import mgd, ops
from oracle.commit import commit_round as ref_commit

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("gamma", [1, 3, 4])
def test_commit_matches_oracle(dtype, gamma):
    dev = gpu_or_skip()
    B, Hkv, cap, dcap, D = 37, 8, 300, 70, 128
    g = torch.Generator().manual_seed(gamma * 10 + (dtype == torch.float32))
    k = torch.randn((B, Hkv, cap, D), generator=g).to(dtype)
    v = torch.randn((B, Hkv, cap, D), generator=g).to(dtype)
    kd = torch.randn((B, Hkv, dcap, D), generator=g).to(dtype)
    vd = torch.randn((B, Hkv, dcap, D), generator=g).to(dtype)
    kv_len = torch.randint(gamma + 1, cap + 1, (B,), generator=g, dtype=torch.int32)
    draft_len = torch.randint(0, dcap - gamma, (B,), generator=g, dtype=torch.int32)
    nacc = torch.randint(0, gamma + 1, (B,), generator=g, dtype=torch.int32)
    # out-of-range cases: too many accepted, too short, draft overflow
    nacc[3] = gamma + 1
    kv_len[5] = gamma
    draft_len[7] = dcap - 1
    nacc[7] = gamma
    ref_len, ref_kd, ref_vd, ref_dl, bad = ref_commit(kv_len, nacc, gamma, k.view(torch.int16) if dtype == torch.bfloat16 else k,
                                                      v.view(torch.int16) if dtype == torch.bfloat16 else v,
                                                      kd.view(torch.int16) if dtype == torch.bfloat16 else kd,
                                                      vd.view(torch.int16) if dtype == torch.bfloat16 else vd, draft_len)
    assert bad[3] and bad[5] and bad[7]
    # the updated arrays between poisoned guard regions
    g = dict(kv_len=Guarded((B,), torch.int32, dev, init=kv_len), draft_len=Guarded((B,), torch.int32, dev, init=draft_len),
             k_draft=Guarded(tuple(kd.shape), dtype, dev, init=kd), v_draft=Guarded(tuple(vd.shape), dtype, dev, init=vd))
    kl_d, dl_d, kd_d, vd_d = g["kv_len"].t, g["draft_len"].t, g["k_draft"].t, g["v_draft"].t
    ws = ops.workspace(mgd.mgd_commit_workspace_size(B), dev)
    ops.commit_round(nacc.to(dev), gamma, kl_d, k.to(dev), v.to(dev), kd_d, vd_d, dl_d, ws=ws)
    assert mgd.mgd_workspace_errors(ws) & mgd.MGD_DEVERR_COMMIT
    check_guards(**g)
    np.testing.assert_array_equal(kl_d.cpu().numpy(), ref_len)
    np.testing.assert_array_equal(dl_d.cpu().numpy(), ref_dl)
    view = (lambda t: t.cpu().view(torch.int16).numpy()) if dtype == torch.bfloat16 else (lambda t: t.cpu().numpy())
    np.testing.assert_array_equal(view(kd_d), ref_kd)
    np.testing.assert_array_equal(view(vd_d), ref_vd)


def test_commit_after_a_sampled_round():
    """Feed the sampler's num_accepted straight into the commit step."""
    dev = gpu_or_skip()
    from long_context_speculative_split_gb300 import workloads as wl
    c = dict(wl.WORKLOADS["b32_ctx8k"], B=16, V=2048)
    t, d = wl.logits(c, dev)
    u = wl.uniforms(c, dev)
    tok = ops.draft_draw(d, u)
    out, nacc = ops.rejection_sample(t, d, tok, u)
    B, Hkv, cap, D, gamma = 16, 8, 64, 128, c["gamma"]
    k = torch.randn((B, Hkv, cap, D), device=dev).bfloat16()
    v = torch.randn((B, Hkv, cap, D), device=dev).bfloat16()
    kd = torch.zeros((B, Hkv, 32, D), device=dev).bfloat16()
    vd = torch.zeros_like(kd)
    kv_len = torch.full((B,), cap, dtype=torch.int32, device=dev)
    dl = torch.full((B,), 10, dtype=torch.int32, device=dev)
    ops.commit_round(nacc, gamma, kv_len, k, v, kd, vd, dl)
    emitted = (out >= 0).sum(dim=1).int()
    assert torch.equal(dl - 10, emitted)
    assert torch.equal(cap - kv_len, gamma + 1 - emitted)
