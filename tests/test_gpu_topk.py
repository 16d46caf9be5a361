"""GPU parity of one dynamic top-K draft step (mgd_topk_draft_attn) against the float64 oracle.

The kept rows must match the oracle's except at positions whose oracle score lies
within 1e-5 (relative) of the lowest kept score; the gathered rows must equal the
source rows bit for bit; the attention output must match the oracle's attention over
the rows the GPU kept (attention tolerances), and the oracle's own output where the
two kept sets agree."""
import math

import numpy as np
import pytest
import torch

from _parity import assert_attention_close, assert_index_sets_match, assert_lse_close, gpu_or_skip
from long_context_speculative_split_gb300 import ops
from long_context_speculative_split_gb300 import workloads as wl
from oracle.attention import draft_attention
from oracle.topk import topk_attention

pytestmark = pytest.mark.gpu


def _check(res, q, k, v, kv_len, K, scale, pairs=None):
    """Compare (b, h) pairs (all by default); q [B,Hq,D] and k, v on the device."""
    B, Hq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    pairs = pairs or [(b, h) for b in range(B) for h in range(Hkv)]
    L = kv_len.cpu().numpy()
    ndiff = 0
    for b, h in pairs:
        n = int(L[b])
        qs = q[b:b + 1, h * G:(h + 1) * G]
        ref = topk_attention(qs, k[b:b + 1, h:h + 1, :n], v[b:b + 1, h:h + 1, :n], L[b:b + 1], K, scale)
        Keff = min(K, n)
        assert int(res["draft_len"][b]) == Keff
        got = res["sel_idx"][b, h].cpu().numpy()
        assert np.all(got[Keff:] == -1)
        ref_idx = ref["sel_idx"][0, 0, :Keff]
        sc = ref["score"][0, 0]
        kth = np.min(sc[ref_idx[:-1]]) if 0 < Keff - 1 < n - 1 else np.nan
        d = assert_index_sets_match(got[:Keff], ref_idx, sc, kth)
        ndiff += d
        idx = torch.from_numpy(got[:Keff].astype(np.int64)).to(k.device)
        assert torch.equal(res["k_draft"][b, h, :Keff], k[b, h, idx])
        assert torch.equal(res["v_draft"][b, h, :Keff], v[b, h, idx])
        # attention over the rows the GPU kept
        o, lse = draft_attention(qs[:, None], k[b:b + 1, h:h + 1, idx], v[b:b + 1, h:h + 1, idx],
                                 np.array([Keff]), scale)
        assert_attention_close(res["out"][b:b + 1, h * G:(h + 1) * G], o[:, 0], "out[b=%d,h=%d]" % (b, h))
        assert_lse_close(res["lse"][b:b + 1, h * G:(h + 1) * G], lse[:, 0])
        if d == 0:
            assert_attention_close(res["out"][b:b + 1, h * G:(h + 1) * G], ref["out"])
    return ndiff


CASES = [
    # B, Hq, Hkv, D, lens, cap, K
    (3, 32, 8, 128, [700, 300, 1], 700, 64),     # ragged, a one-row context
    (2, 32, 8, 128, [100, 40], 128, 128),        # K >= L: plain decode attention
    (2, 8, 2, 64, [2000, 1999], 2048, 1),        # only the query's own row
    (1, 64, 8, 128, [4097], 4100, 513),          # G = 8, a ragged last tile
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "L%s_K%d_G%d_D%d" % ("-".join(map(str, c[4])), c[6],
                                                                           c[1] // c[2], c[3]))
def test_bf16_cases_match_oracle(case):
    dev = gpu_or_skip()
    B, Hq, Hkv, D, lens, cap, K = case
    cfg = dict(B=B, Hq=Hq, Hkv=Hkv, D=D, dtype="bf16", lens=lens, W=1, hh=0.01, gamma=1)
    kv_len = torch.tensor(lens, dtype=torch.int32)
    k, v = wl.kv_cache(cfg, dev, seed=5, kv_len=kv_len, cap=cap)
    q = wl.window_queries(cfg, dev, seed=5)[:, 0].contiguous()
    res = ops.topk_draft_attn(q, k, v, kv_len.to(dev), K)
    torch.cuda.synchronize()
    _check(res, q, k, v, kv_len, K, 1.0 / math.sqrt(D))


def test_tiny_config_float32():
    dev = gpu_or_skip()
    c = wl.WORKLOADS["tiny_b2"]
    kv_len = wl.lengths(c)
    k, v = wl.kv_cache(c, dev, kv_len=kv_len)
    q = wl.draft_queries(c, dev)[:, 0].contiguous()
    res = ops.topk_draft_attn(q, k, v, kv_len.to(dev), c["K"])
    torch.cuda.synchronize()
    _check(res, q, k, v, kv_len, c["K"], 1.0 / math.sqrt(c["D"]))


def test_full_size_sampled():
    """Batch 32 x context 8192, K = 512, in the launch configuration the benchmark uses."""
    dev = gpu_or_skip()
    c = wl.WORKLOADS["b32_ctx8k"]
    kv_len = wl.lengths(c)
    k, v = wl.kv_cache(c, dev, kv_len=kv_len)
    q = wl.draft_queries(c, dev)[:, 0].contiguous()
    res = ops.topk_draft_attn(q, k, v, kv_len.to(dev), c["K"])
    torch.cuda.synchronize()
    assert bool(torch.isfinite(res["out"]).all())
    rng = np.random.default_rng(2)
    pairs = [(0, 0), (c["B"] - 1, c["Hkv"] - 1), (int(rng.integers(c["B"])), int(rng.integers(c["Hkv"])))]
    _check(res, q, k, v, kv_len, c["K"], 1.0 / math.sqrt(c["D"]), pairs)
    del k, v
    torch.cuda.empty_cache()
