"""Oracle: StreamingLLM-style draft cache (attention sinks + recent window).

TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__.py``.  Pins live in
``tests/test_oracle_streaming.py``.

MagicDec notes, section 5.1 (the end-to-end runs draft with a StreamingLLM-style
sparse KV) and section 5.2 (SnapKV beats it): a static selection with no
scoring at all.  The pages do not define it; the reading used here is the
usual one for StreamingLLM: keep the first `sink` positions (attention sinks)
and the most recent positions, K_eff = min(K, L) rows in total:

    kept = [0, s) followed by [L - (K_eff - s), L),   s = min(sink, K_eff),

in ascending order (the two ranges cannot overlap because K_eff <= L), and
gather those K / V rows into the compacted draft cache; draft_len = K_eff.
"""
import numpy as np

from .attention import _ints


def streaming_indices(L, sink, K):
    K_eff = min(K, L)
    s = min(sink, K_eff)
    return np.concatenate([np.arange(s), np.arange(L - (K_eff - s), L)]).astype(np.int64)


def streaming_select(k, v, kv_len, sink, K):
    """Returns dict(sel_idx [B, Hkv, K] (-1 padded), k_draft, v_draft [B, Hkv, K, D], draft_len [B])."""
    k = np.asarray(k) if not hasattr(k, "detach") else k.detach().cpu().numpy()
    v = np.asarray(v) if not hasattr(v, "detach") else v.detach().cpu().numpy()
    kv_len = _ints(kv_len)
    B, Hkv, _, D = k.shape
    sel = -np.ones((B, Hkv, K), dtype=np.int64)
    kd = np.zeros((B, Hkv, K, D), dtype=k.dtype)
    vd = np.zeros((B, Hkv, K, D), dtype=v.dtype)
    dl = np.zeros(B, dtype=np.int64)
    for b in range(B):
        idx = streaming_indices(int(kv_len[b]), sink, K)
        n = len(idx)
        dl[b] = n
        for h in range(Hkv):
            sel[b, h, :n] = idx
            kd[b, h, :n] = k[b, h, idx]
            vd[b, h, :n] = v[b, h, idx]
    return dict(sel_idx=sel, k_draft=kd, v_draft=vd, draft_len=dl)
