"""GPU parity of SnapKV draft-cache selection against the float64 oracle.

Index sets must match except at positions whose oracle score lies within 1e-5
(relative) of the K-th kept score; the gathered rows must equal the source
rows bit for bit; draft_len must equal min(K, L)."""
import math

import numpy as np
import pytest
import torch

from _parity import (Guarded, assert_attention_close, assert_index_sets_match, assert_lse_close, check_guards,
                     gpu_or_skip, is_poison)
from long_context_speculative_split_gb300 import ops
from long_context_speculative_split_gb300 import workloads as wl
from oracle.attention import draft_attention as ref_draft
from oracle.snapkv import max_pool, select_indices, snapkv_select as ref_select, window_scores

pytestmark = pytest.mark.gpu


def _check_pair(res, k, v, b, h, L, W, P, K, ref_scores_row, D):
    pooled = np.zeros(ref_scores_row.shape)
    n = L - W
    pooled[:n] = max_pool(ref_scores_row, n, P)
    ref_idx = select_indices(pooled, L, W, K)
    n_top = len(ref_idx) - W
    kth = np.min(pooled[ref_idx[:n_top]]) if 0 < n_top < n else np.nan
    Keff = min(K, L)
    got = res["sel_idx"][b, h].cpu().numpy()
    assert int(res["draft_len"][b]) == Keff
    assert np.all(got[Keff:] == -1)
    ndiff = assert_index_sets_match(got[:Keff], ref_idx, pooled, kth)
    idx = torch.from_numpy(got[:Keff].astype(np.int64)).to(k.device)
    assert torch.equal(res["k_draft"][b, h, :Keff], k[b, h, idx])
    assert torch.equal(res["v_draft"][b, h, :Keff], v[b, h, idx])
    if res["scores"] is not None and n > 0:
        gs = res["scores"][b, h, :n].double().cpu().numpy()
        np.testing.assert_allclose(gs, pooled[:n], rtol=1e-4, atol=1e-9)
    return ndiff, ref_idx


def test_tiny_config_float32_full():
    dev = gpu_or_skip()
    c = wl.WORKLOADS["tiny_b2"]
    kv_len = wl.lengths(c)
    k, v = wl.kv_cache(c, dev, kv_len=kv_len)
    qw = wl.window_queries(c, dev)
    res = ops.snapkv_select(qw, k, v, kv_len.to(dev), c["W"], c["pool"], c["K"], want_scores=True)
    torch.cuda.synchronize()
    ref = ref_select(qw, k, v, kv_len, c["W"], c["pool"], c["K"], 1.0 / math.sqrt(c["D"]))
    for b in range(c["B"]):
        _check_pair(res, k, v, b, 0, int(kv_len[b]), c["W"], c["pool"], c["K"], ref["scores"][b, 0], c["D"])


CASES = [
    # B, Hq, Hkv, D, lens, cap, W, P, K
    (2, 32, 8, 128, [700, 300], 700, 32, 7, 128),
    (2, 8, 2, 64, [100, 40], 128, 16, 5, 200),       # K >= L: every row kept
    (1, 8, 2, 128, [32], 64, 32, 3, 64),             # L == W: only the window
    (2, 64, 8, 128, [1000, 999], 1000, 32, 7, 256),  # 256 window rows -> two row groups
    (3, 32, 8, 128, [5000, 4000, 2500], 5000, 32, 7, 512),
    (1, 32, 8, 128, [777], 800, 8, 1, 100),          # no pooling, short window
    # lengths at tile (128) and scoring-slice (1536) edges: a slice holding only window keys,
    # a window that straddles a slice edge, a prefix of one key
    (4, 32, 8, 128, [1537, 1568, 3112, 33], 3200, 32, 7, 256),
    (2, 64, 8, 128, [3000, 1600], 3000, 16, 5, 300),  # G = 8 x W = 16 window rows on the tensor-core scorer
    (2, 32, 8, 64, [1500, 900], 1500, 32, 7, 256),    # 128 window rows at head_dim 64 (the mma.sync scorer)
    # windows of <= 8 rows: key sums taken from the logits pass 1 keeps
    (2, 32, 8, 128, [2000, 700], 2000, 2, 3, 128),
    (2, 8, 2, 64, [900, 400], 900, 2, 1, 64),
    # capacities long enough that the scorer's slices grow past 1536 keys (at most 64 per sequence)
    (1, 8, 2, 128, [200000], 200000, 32, 7, 1024),
    (2, 8, 2, 128, [150001, 70000], 160000, 32, 7, 512),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "L%s_W%d_P%d_K%d_G%d" % ("-".join(map(str, c[4])), c[6], c[7],
                                                                                c[8], c[1] // c[2]))
def test_bf16_cases_match_oracle(case):
    dev = gpu_or_skip()
    B, Hq, Hkv, D, lens, cap, W, P, K = case
    cfg = dict(B=B, Hq=Hq, Hkv=Hkv, D=D, dtype="bf16", lens=lens, W=W, hh=0.01, gamma=1)
    kv_len = torch.tensor(lens, dtype=torch.int32)
    k, v = wl.kv_cache(cfg, dev, seed=3, kv_len=kv_len, cap=cap)
    qw = wl.window_queries(cfg, dev, seed=3)
    # every output between poisoned guard regions; the draft cache has 64 spare rows per
    # (sequence, KV head) that the call must leave as they are (poisoned here)
    dcap = K + 64
    g = dict(sel_idx=Guarded((B, Hkv, dcap), torch.int32, dev), k_draft=Guarded((B, Hkv, dcap, D), k.dtype, dev),
             v_draft=Guarded((B, Hkv, dcap, D), k.dtype, dev), draft_len=Guarded((B,), torch.int32, dev),
             scores=Guarded((B, Hkv, cap), torch.float32, dev, init=torch.zeros(())))
    res = ops.snapkv_select(qw, k, v, kv_len.to(dev), W, P, K, draft_cap=dcap, want_scores=True,
                            out={n: x.t for n, x in g.items()})
    torch.cuda.synchronize()
    check_guards(**g)
    for b in range(B):
        keff = min(K, lens[b])
        assert bool(is_poison(res["k_draft"][b, :, keff:]).all()) and bool(is_poison(res["v_draft"][b, :, keff:]).all())
    s = window_scores(qw, k, kv_len, W, 1.0 / math.sqrt(D))
    for b in range(B):
        for h in range(Hkv):
            _check_pair(res, k, v, b, h, lens[b], W, P, K, s[b, h], D)


@pytest.mark.parametrize("name,seed", [("b32_ctx8k", 2), ("b128_ctx32k", 3), ("ragged_b256_ctx4k_64k", 4)],
                         ids=["b32_ctx8k", "b128_ctx32k", "ragged_b256_ctx4k_64k"])
def test_full_size_sampled(name, seed):
    """Full-size workloads (including ragged lengths 4k-64k at batch 256) with sampled pairs:
    the first, the last, the longest sequence's and one random (sequence, KV head).  Then the
    draft step over the selected caches: draft attention over each sampled pair's compacted
    cache is compared with the oracle's draft attention over the oracle's own selection,
    gathered from the input cache (where the two index sets differ inside the tie band the
    outputs legitimately differ and only the selection check above applies)."""
    dev = gpu_or_skip()
    c = wl.WORKLOADS[name]
    kv_len = wl.lengths(c)
    k, v = wl.kv_cache(c, dev, kv_len=kv_len, cap=wl.capacity(c))
    qw = wl.window_queries(c, dev)
    res = ops.snapkv_select(qw, k, v, kv_len.to(dev), c["W"], c["pool"], c["K"], want_scores=True)
    qd = wl.draft_queries(c, dev)
    dout, dlse = ops.draft_attn(qd, res["k_draft"], res["v_draft"], res["draft_len"])
    torch.cuda.synchronize()
    assert bool(torch.isfinite(dout).all()) and bool(torch.isfinite(dlse).all())
    G, D = c["Hq"] // c["Hkv"], c["D"]
    scale = 1.0 / math.sqrt(D)
    rng = np.random.default_rng(seed)
    pairs = [(0, 0), (c["B"] - 1, c["Hkv"] - 1), (int(np.argmax(kv_len.numpy())), 3),
             (int(rng.integers(c["B"])), int(rng.integers(c["Hkv"])))]
    drafts_compared = 0
    for b, h in pairs:
        L = int(kv_len[b])
        hs = slice(h * G, (h + 1) * G)
        s = window_scores(qw[b:b + 1, :, hs], k[b:b + 1, h:h + 1, :L], kv_len[b:b + 1], c["W"], scale)
        ndiff, ref_idx = _check_pair(res, k, v, b, h, L, c["W"], c["pool"], c["K"], s[0, 0], c["D"])
        if ndiff:
            continue
        sel = torch.from_numpy(np.asarray(ref_idx, dtype=np.int64))
        kd = k[b, h, :L].cpu()[sel][None, None]
        vd = v[b, h, :L].cpu()[sel][None, None]
        ref, ref_lse = ref_draft(qd[b:b + 1, :, hs], kd, vd, torch.tensor([len(ref_idx)]), scale)
        assert_attention_close(dout[b:b + 1, hs], ref[:, 0], "draft[b=%d,h=%d]" % (b, h))
        assert_lse_close(dlse[b:b + 1, hs], ref_lse[:, 0])
        drafts_compared += 1
    assert drafts_compared >= len(pairs) - 1
    del k, v
    torch.cuda.empty_cache()


@pytest.mark.parametrize("W,pool,D", [(32, 7, 128), (2, 3, 128), (16, 5, 64)],
                         ids=["tc05_window128rows", "logit_sums_8rows", "mma_sync_D64"])
def test_per_sequence_budgets(W, pool, D):
    """MagicDec notes, section 4.3: every sequence keeps K_eff = min(K_b, L_b) rows of its own budget K_b;
    a budget outside [W, draft_cap] skips that sequence (flagged) and leaves the others intact."""
    dev = gpu_or_skip()
    lens = [3000, 2000, 500, 40, 1500]
    B, Hq, Hkv, cap, dcap = len(lens), 32, 8, 3000, 1024
    budgets = [512, W + 32, 1000, 100, W - 1]   # the third and fourth cover their sequence; the last is invalid
    cfg = dict(B=B, Hq=Hq, Hkv=Hkv, D=D, dtype="bf16", lens=lens, W=W, hh=0.01, gamma=1)
    kv_len = torch.tensor(lens, dtype=torch.int32)
    k, v = wl.kv_cache(cfg, dev, seed=8, kv_len=kv_len, cap=cap)
    qw = wl.window_queries(cfg, dev, seed=8)
    kb = torch.tensor(budgets, dtype=torch.int32, device=dev)
    from long_context_speculative_split_gb300 import mgd
    ws = ops.workspace(mgd.mgd_snapkv_workspace_size(B, Hq, Hkv, D, cap, W), dev)
    res = ops.snapkv_select(qw, k, v, kv_len.to(dev), W, pool, kb, draft_cap=dcap, ws=ws, want_scores=True)
    torch.cuda.synchronize()
    assert mgd.mgd_workspace_errors(ws) == 0x2                      # MGD_DEVERR_SNAP_LEN from the last budget
    assert int(res["draft_len"][B - 1]) == 0 and bool((res["sel_idx"][B - 1] == -1).all())
    s = window_scores(qw[:B - 1], k[:B - 1], kv_len[:B - 1], W, 1.0 / math.sqrt(D))
    for b in range(B - 1):
        for h in range(Hkv):
            _check_pair(res, k, v, b, h, lens[b], W, pool, budgets[b], s[b, h], D)
