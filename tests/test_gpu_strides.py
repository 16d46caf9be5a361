"""Caches held in a larger pool: K/V are views [:, :, :kv_cap] of [B, Hkv, pool_cap, D] tensors, so the
head and batch strides passed through the C ABI are not the dense ones.  Every call that takes KV strides
must give the oracle's answer on those views (the tensor maps and pointer arithmetic use the strides)."""
import math

import numpy as np
import pytest
import torch

from _parity import assert_attention_close, assert_index_sets_match, assert_lse_close, gpu_or_skip
from long_context_speculative_split_gb300 import ops
from long_context_speculative_split_gb300 import workloads as wl
from oracle.attention import attention, draft_attention
from oracle.commit import commit_round as ref_commit
from oracle.snapkv import snapkv_select as ref_snapkv
from oracle.streaming import streaming_select as ref_streaming

pytestmark = pytest.mark.gpu

B, Hq, Hkv, D = 3, 32, 8, 128
CAP, POOL = 1500, 1600          # logical capacity, pool rows per (sequence, KV head)
LENS = [1500, 777, 65]


def _pool(dev, seed):
    cfg = dict(B=B, Hq=Hq, Hkv=Hkv, D=D, dtype="bf16", lens=LENS, W=32, hh=0.01, gamma=3)
    kv_len = torch.tensor(LENS, dtype=torch.int32)
    kp, vp = wl.kv_cache(cfg, dev, seed, kv_len=kv_len, cap=POOL)
    k, v = kp[:, :, :CAP], vp[:, :, :CAP]
    assert not k.is_contiguous() and k.stride(1) == POOL * D
    return cfg, kv_len, k, v


def test_verify_and_draft_on_pool_views():
    dev = gpu_or_skip()
    cfg, kv_len, k, v = _pool(dev, 11)
    q = wl.queries(cfg, dev, 11)
    out, lse = ops.verify_attn(q, k, v, kv_len.to(dev))
    ref, ref_lse = attention(q, k, v, kv_len, 1.0 / math.sqrt(D))
    assert_attention_close(out, ref)
    assert_lse_close(lse, ref_lse)
    # a draft cache that is itself a view of a larger pool
    dlen = torch.tensor([300, 1, 299], dtype=torch.int32)
    kd, vd = k[:, :, :300], v[:, :, :300]
    qd = wl.draft_queries(cfg, dev, 11)
    dout, dl = ops.draft_attn(qd, kd, vd, dlen.to(dev))
    rd, rdl = draft_attention(qd, kd, vd, dlen, 1.0 / math.sqrt(D))
    assert_attention_close(dout, rd[:, 0])
    assert_lse_close(dl, rdl[:, 0])


@pytest.mark.parametrize("W,pool,K", [(32, 7, 256), (8, 1, 100)], ids=["tc05_window128rows", "small_window32rows"])
def test_snapkv_on_pool_views(W, pool, K):
    dev = gpu_or_skip()
    cfg, kv_len, k, v = _pool(dev, 12)
    cfg = dict(cfg, W=W)
    qw = wl.window_queries(cfg, dev, 12)
    res = ops.snapkv_select(qw, k, v, kv_len.to(dev), W, pool, K, want_scores=True)
    torch.cuda.synchronize()
    ref = ref_snapkv(qw, k, v, kv_len, W, pool, K, 1.0 / math.sqrt(D))
    for b in range(B):
        Keff = min(K, LENS[b])
        assert int(res["draft_len"][b]) == Keff
        for h in range(Hkv):
            got = res["sel_idx"][b, h].cpu().numpy()
            assert_index_sets_match(got[:Keff], ref["sel_idx"][b, h, :Keff], ref["pooled"][b, h], ref["kth"][b, h])
            idx = torch.from_numpy(got[:Keff].astype(np.int64)).to(dev)
            assert torch.equal(res["k_draft"][b, h, :Keff], k[b, h, idx])
            assert torch.equal(res["v_draft"][b, h, :Keff], v[b, h, idx])


def test_streaming_and_commit_on_pool_views():
    dev = gpu_or_skip()
    cfg, kv_len, k, v = _pool(dev, 13)
    res = ops.streaming_select(k, v, kv_len.to(dev), 4, 128)
    torch.cuda.synchronize()
    ref = ref_streaming(k.view(torch.int16), v.view(torch.int16), kv_len, 4, 128)
    np.testing.assert_array_equal(res["sel_idx"].cpu().numpy(), ref["sel_idx"])
    np.testing.assert_array_equal(res["draft_len"].cpu().numpy(), ref["draft_len"])
    np.testing.assert_array_equal(res["k_draft"].cpu().view(torch.int16).numpy(), ref["k_draft"])
    np.testing.assert_array_equal(res["v_draft"].cpu().view(torch.int16).numpy(), ref["v_draft"])
    # commit into a draft cache that is a view of a larger pool
    gamma = 3
    dpool_k = torch.zeros((B, Hkv, 200, D), dtype=torch.bfloat16, device=dev)
    dpool_v = torch.zeros_like(dpool_k)
    kd, vd = dpool_k[:, :, :150], dpool_v[:, :, :150]
    dl = torch.tensor([10, 0, 149], dtype=torch.int32)
    nacc = torch.tensor([3, 0, 1], dtype=torch.int32)
    ref_len, ref_kd, ref_vd, ref_dl, bad = ref_commit(kv_len, nacc, gamma, k.cpu().view(torch.int16),
                                                      v.cpu().view(torch.int16), kd.cpu().view(torch.int16),
                                                      vd.cpu().view(torch.int16), dl)
    kl_d, dl_d = kv_len.to(dev), dl.to(dev)
    ops.commit_round(nacc.to(dev), gamma, kl_d, k, v, kd, vd, dl_d)
    np.testing.assert_array_equal(kl_d.cpu().numpy(), ref_len)
    np.testing.assert_array_equal(dl_d.cpu().numpy(), ref_dl)
    np.testing.assert_array_equal(kd.cpu().view(torch.int16).numpy(), ref_kd)
    np.testing.assert_array_equal(vd.cpu().view(torch.int16).numpy(), ref_vd)
    assert bool(bad[2]) and not bad[0] and not bad[1]  # 149 + 2 rows > 150: left unchanged and flagged
