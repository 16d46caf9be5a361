"""Oracle: exact softmax attention for the verify and draft passes (float64, CPU).

TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__.py``.  Parity pins live in
``tests/test_oracle_attention.py``.

What is computed
----------------
MagicDec notes, section 3.2: verification of gamma draft tokens and ordinary
decoding read the same KV cache, so the verify pass is decode attention with
T = gamma + 1 query rows per sequence (the +1 row yields the target
distribution for the bonus token of the verification round described in "Wann
beschleunigt spekulatives Decoding das LLM-Serving?", "Eine Verifizierungsrunde
verstehen").  The draft pass (quick-read summary: the target model itself
drafts over a compressed KV of budget K) is the same operation with T = 1 over
the compacted cache.

Readings taken where the pages are silent (the pages give no formula for the
attention itself):
  * layouts: q [B, T, Hq, D]; k, v [B, Hkv, L_cap, D]; kv_len [B].
  * grouped-query attention: query head h reads KV head h // G, G = Hq / Hkv.
  * kv_len[b] counts every cached row *including* the T rows being verified;
    row t sits at position kv_len[b] - T + t and sees keys 0 .. kv_len[b]-T+t
    (causal among the appended rows).  With T = 1 every cached row is seen.
  * scores are scale * <q, k>; no positional encoding is applied here (the
    synthetic inputs stand for already-rotated q and k).

For every (b, t, h) this is the plain two-pass softmax: m = max_j s_j,
Z = sum_j exp(s_j - m), O = sum_j exp(s_j - m) v_j / Z, lse = m + log Z.
There is no split over keys and no running rescaling: this is the exact
result that a split-KV flash-decoding kernel reaches faster.
"""
import numpy as np


def _f64(x):
    """Exact upcast of any float tensor/array (float32, bfloat16 via torch) to float64."""
    if hasattr(x, "detach"):  # a torch tensor: bf16 -> f32 -> f64 is exact
        x = x.detach().cpu()
        if str(x.dtype) == "torch.bfloat16":
            x = x.float()
        x = x.double().numpy()
    return np.asarray(x, dtype=np.float64)


def _ints(x):
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.asarray(x, dtype=np.int64)


def attention(q, k, v, kv_len, scale):
    """Verify-form attention (draft form when T == 1).

    q: [B, T, Hq, D]; k, v: [B, Hkv, L_cap, D]; kv_len: [B] (T <= kv_len[b] <= L_cap).
    Returns (out [B, T, Hq, D] float64, lse [B, T, Hq] float64), lse in natural log.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    kv_len = _ints(kv_len)
    B, T, Hq, D = q.shape
    Hkv = k.shape[1]
    assert Hq % Hkv == 0, "query heads must be a multiple of KV heads"
    G = Hq // Hkv
    out = np.zeros((B, T, Hq, D), dtype=np.float64)
    lse = np.zeros((B, T, Hq), dtype=np.float64)
    for b in range(B):
        L = int(kv_len[b])
        assert T <= L <= k.shape[2], "need T <= kv_len <= capacity"
        for h in range(Hq):
            hk = h // G
            for t in range(T):
                n_vis = L - T + t + 1          # keys 0 .. L-T+t
                keys = k[b, hk, :n_vis, :]
                vals = v[b, hk, :n_vis, :]
                s = (keys @ q[b, t, h, :]) * scale
                m = np.max(s)
                e = np.exp(s - m)
                Z = np.sum(e)
                out[b, t, h, :] = (e @ vals) / Z
                lse[b, t, h] = m + np.log(Z)
    return out, lse


def draft_attention(q, k_draft, v_draft, draft_len, scale):
    """Draft-form attention: one query row per sequence over the compacted cache.

    q: [B, 1, Hq, D]; k_draft, v_draft: [B, Hkv, K_cap, D]; draft_len: [B].
    Identical to ``attention`` with T = 1 (no mask: every stored row is visible).
    """
    q = _f64(q)
    assert q.shape[1] == 1, "the draft pass has one query row"
    return attention(q, k_draft, v_draft, draft_len, scale)


def merge_lse(parts):
    """Combine partial attention results computed over disjoint key sets.

    parts: list of (out_s [..., D], lse_s [...]) float64, one per key subset.
    With lse = log sum_s exp(lse_s) the merged output is
    sum_s exp(lse_s - lse) * out_s.  An empty subset (lse_s = -inf) adds nothing.
    """
    lses = np.stack([np.asarray(p[1], dtype=np.float64) for p in parts])   # [S, ...]
    outs = np.stack([np.asarray(p[0], dtype=np.float64) for p in parts])   # [S, ..., D]
    m = np.max(lses, axis=0)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(lses - m_safe)                                           # [S, ...]
    total = np.sum(w, axis=0)
    lse = m_safe + np.log(total)
    out = np.sum(w[..., None] * outs, axis=0) / total[..., None]
    return out, lse
