"""Oracle: SnapKV-style static draft-KV selection (float64, CPU).

TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__.py``.  Pins live in
``tests/test_oracle_snapkv.py``.

Where this comes from
---------------------
MagicDec notes, section 4.4, names SnapKV as a *static* selector: the sparse
KV used for drafting is collected once and no search runs per generated token;
appendix A.1 says that this compressed KV is produced at prefill and reused by
every draft step, and the quick-read summary gives its size as the draft KV
budget K.  The pages never spell out SnapKV's own arithmetic, so the steps
below are the plainest reading of "observation-window scores, max-pool along
the sequence, per-(sequence, KV-head) top-K, gather into a compacted cache":

  1. window scores: the last W positions of each context are the observation
     window; their queries q_win[b, w, h] (position L_b - W + w) attend
     causally over keys 0 .. L_b - W + w with scale * <q, k>; the softmax
     probabilities are summed over the W window queries and over the G query
     heads that share a KV head, for every prefix key j < L_b - W;
  2. max-pool: pooled[j] = max of the scores at positions t with
     |t - j| <= P // 2 and 0 <= t < L_b - W (stride 1, same length, positions
     outside the prefix are ignored); P is odd;
  3. selection: K_eff = min(K, L_b) rows are kept; the budget includes the W
     window rows, so the top K_eff - W prefix positions by pooled score
     (ties broken towards the lower position) are kept together with every
     window position L_b - W .. L_b - 1; indices are stored in ascending
     order;
  4. gather: the kept K and V rows are copied, in that order, into the
     compacted draft cache; draft_len[b] = K_eff.
"""
import numpy as np

from .attention import _f64, _ints


def window_scores(q_win, k, kv_len, W, scale):
    """Step 1.  q_win [B, W, Hq, D], k [B, Hkv, L_cap, D] -> s [B, Hkv, L_cap] float64.

    Only entries j < kv_len[b] - W are meaningful; the rest are left at zero.
    """
    q_win, k = _f64(q_win), _f64(k)
    kv_len = _ints(kv_len)
    B, Wq, Hq, D = q_win.shape
    assert Wq == W
    Hkv, L_cap = k.shape[1], k.shape[2]
    G = Hq // Hkv
    s = np.zeros((B, Hkv, L_cap), dtype=np.float64)
    for b in range(B):
        L = int(kv_len[b])
        n_pre = L - W
        assert n_pre >= 0
        for hk in range(Hkv):
            for g in range(G):
                h = hk * G + g
                for w in range(W):
                    pos = L - W + w                      # position of this window query
                    logits = (k[b, hk, : pos + 1, :] @ q_win[b, w, h, :]) * scale
                    e = np.exp(logits - np.max(logits))
                    p = e / np.sum(e)
                    s[b, hk, :n_pre] += p[:n_pre]
    return s


def max_pool(row, n, P):
    """Step 2 on one score row: pooled[j] = max(row[t]) over |t - j| <= P//2, 0 <= t < n."""
    assert P % 2 == 1, "pool kernel must be odd"
    r = P // 2
    out = np.zeros(n, dtype=np.float64)
    for j in range(n):
        out[j] = np.max(row[max(0, j - r): min(n, j + r + 1)])
    return out


def select_indices(pooled, L, W, K):
    """Step 3 on one (sequence, KV head): returns the ascending kept positions (length min(K, L))."""
    K_eff = min(K, L)
    n_pre = L - W
    n_top = K_eff - W
    assert 0 <= n_top <= n_pre
    # rank prefix positions by (score descending, position ascending)
    order = np.lexsort((np.arange(n_pre), -pooled[:n_pre]))
    keep = np.sort(order[:n_top])
    return np.concatenate([keep, np.arange(n_pre, L)]).astype(np.int64)


def snapkv_select(q_win, k, v, kv_len, W, P, K, scale):
    """Steps 1-4.  Returns a dict with

    sel_idx [B, Hkv, K] int64 (-1 beyond draft_len), k_draft / v_draft [B, Hkv, K, D]
    float64 (rows beyond draft_len zero), draft_len [B], and for tolerance checks
    scores [B, Hkv, L_cap], pooled [B, Hkv, L_cap] and kth [B, Hkv] (the pooled
    score of the lowest-ranked kept prefix position; nan when no prefix row is kept
    by rank because K_eff - W is 0 or covers the whole prefix).
    """
    k64, v64 = _f64(k), _f64(v)
    kv_len = _ints(kv_len)
    B, Hkv, L_cap, D = k64.shape
    s = window_scores(q_win, k64, kv_len, W, scale)
    pooled = np.zeros_like(s)
    sel = -np.ones((B, Hkv, K), dtype=np.int64)
    kd = np.zeros((B, Hkv, K, D), dtype=np.float64)
    vd = np.zeros((B, Hkv, K, D), dtype=np.float64)
    draft_len = np.zeros(B, dtype=np.int64)
    kth = np.full((B, Hkv), np.nan)
    for b in range(B):
        L = int(kv_len[b])
        n_pre = L - W
        for hk in range(Hkv):
            pooled[b, hk, :n_pre] = max_pool(s[b, hk], n_pre, P)
            idx = select_indices(pooled[b, hk], L, W, K)
            n = len(idx)
            sel[b, hk, :n] = idx
            kd[b, hk, :n] = k64[b, hk, idx]
            vd[b, hk, :n] = v64[b, hk, idx]
            n_top = n - W
            if 0 < n_top < n_pre:
                kth[b, hk] = np.min(pooled[b, hk, idx[:n_top]])
        draft_len[b] = min(K, L)
    return dict(sel_idx=sel, k_draft=kd, v_draft=vd, draft_len=draft_len,
                scores=s, pooled=pooled, kth=kth)
