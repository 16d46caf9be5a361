"""Oracle: dynamic top-K attention drafting, one draft step (float64, CPU).

TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__.py``.  Pins live in
``tests/test_oracle_topk.py``.

MagicDec notes, section 4.4: top-K attention reaches a very high acceptance
rate with a much smaller KV budget than static selection, but is impractical
as a draft because of its selection cost; dynamic selectors search the KV
cache again for every query.  The pages give no algorithm.  The reading used
here is the SnapKV selection with the draft query itself as the observation
window (one row, no pooling), then attention over the kept rows, written out
directly from that definition for one (sequence, KV head):

  1. the draft query of head g sits at position L - 1 (its own K/V row is the
     last cache row); p_g[j] = softmax_j(scale * <q_g, k_j>) over j < L;
  2. score[j] = sum over the G heads of the KV head of p_g[j], for the earlier
     positions j < L - 1;
  3. K_eff = min(K, L) rows are kept: the newest row L - 1 and the K_eff - 1
     earlier positions with the largest score (ties towards the lower
     position), in ascending order;
  4. out_g = sum over kept j of softmax over the kept rows of
     (scale * <q_g, k_j>) times v_j;  lse_g = log of that softmax's normaliser.
"""
import numpy as np

from .attention import _f64, _ints


def topk_keep(score, L, K):
    """Step 3: kept positions (ascending) for scores of positions 0 .. L-2."""
    K_eff = min(K, L)
    n_pre = L - 1
    ranked = sorted(range(n_pre), key=lambda j: (-score[j], j))   # largest first, ties -> lower j
    kept = sorted(ranked[: K_eff - 1]) + [L - 1]
    return np.asarray(kept, dtype=np.int64)


def topk_attention(q, k, v, kv_len, K, scale):
    """q [B, Hq, D], k, v [B, Hkv, L_cap, D] -> dict(out [B, Hq, D], lse [B, Hq], sel_idx [B, Hkv, K] (-1 padded),
    draft_len [B], score [B, Hkv, L_cap] (entries < kv_len - 1 meaningful))."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    kv_len = _ints(kv_len)
    B, Hq, D = q.shape
    Hkv, L_cap = k.shape[1], k.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D))
    lse = np.zeros((B, Hq))
    sel = np.full((B, Hkv, K), -1, dtype=np.int64)
    score = np.zeros((B, Hkv, L_cap))
    dlen = np.zeros(B, dtype=np.int64)
    for b in range(B):
        L = int(kv_len[b])
        for hk in range(Hkv):
            logits = np.stack([(k[b, hk, :L] @ q[b, hk * G + g]) * scale for g in range(G)])   # [G, L]
            p = np.exp(logits - logits.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            score[b, hk, : L - 1] = p[:, : L - 1].sum(axis=0)
            kept = topk_keep(score[b, hk], L, K)
            sel[b, hk, : len(kept)] = kept
            dlen[b] = len(kept)
            for g in range(G):
                s = logits[g, kept]
                m = s.max()
                e = np.exp(s - m)
                out[b, hk * G + g] = (e[:, None] * v[b, hk, kept]).sum(axis=0) / e.sum()
                lse[b, hk * G + g] = m + np.log(e.sum())
    return dict(out=out, lse=lse, sel_idx=sel, draft_len=dlen, score=score)
