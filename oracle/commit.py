"""Oracle: cache bookkeeping after a verification round (commit and rollback).

TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__.py``.  Pins live in
``tests/test_oracle_commit.py``.

"Wann beschleunigt spekulatives Decoding das LLM-Serving?", "Eine
Verifizierungsrunde verstehen": after the first rejection the later candidates
are discarded.  MagicDec notes, appendix A.1: the compressed KV built at
prefill is what the draft reads; the tokens produced afterwards must reach the
draft too.  The pages give no layout, so this is the plain reading, consistent
with the verify reading (kv_len counts the T = gamma + 1 verify rows):

  * before the call, sequence b holds T verify rows at positions
    kv_len[b] - T .. kv_len[b] - 1: the last committed token followed by the
    gamma draft tokens;
  * with n = num_accepted[b] accepted drafts, rows 0 .. n of that block are
    kept and rows n + 1 .. gamma are rolled back:
    kv_len[b] <- kv_len[b] - T + n + 1 (the correction or bonus token is the
    first verify row of the next round);
  * the n + 1 kept rows (K and V, every KV head) are appended to the draft
    cache at draft_len[b] .. draft_len[b] + n, and draft_len[b] += n + 1.

A sequence whose values are out of range (n outside [0, gamma], kv_len < T,
or a draft cache that would overflow draft_cap) is left unchanged and flagged.
"""
import numpy as np

from .attention import _ints


def commit_round(kv_len, num_accepted, gamma, k, v, k_draft, v_draft, draft_len):
    """Returns (kv_len', k_draft', v_draft', draft_len', bad) as new arrays (inputs untouched).

    k, v: [B, Hkv, kv_cap, D]; k_draft, v_draft: [B, Hkv, draft_cap, D] (any dtype, copied exactly).
    """
    kv_len = _ints(kv_len).copy()
    n_acc = _ints(num_accepted)
    draft_len = _ints(draft_len).copy()
    k = np.asarray(k) if not hasattr(k, "detach") else k.detach().cpu().numpy()
    v = np.asarray(v) if not hasattr(v, "detach") else v.detach().cpu().numpy()
    kd = (np.asarray(k_draft) if not hasattr(k_draft, "detach") else k_draft.detach().cpu().numpy()).copy()
    vd = (np.asarray(v_draft) if not hasattr(v_draft, "detach") else v_draft.detach().cpu().numpy()).copy()
    T = gamma + 1
    draft_cap = kd.shape[2]
    bad = np.zeros(len(kv_len), dtype=bool)
    for b in range(len(kv_len)):
        n = int(n_acc[b])
        L = int(kv_len[b])
        dl = int(draft_len[b])
        if not (0 <= n <= gamma) or L < T or dl < 0 or dl + n + 1 > draft_cap:
            bad[b] = True
            continue
        first = L - T
        for i in range(n + 1):
            kd[b, :, dl + i] = k[b, :, first + i]
            vd[b, :, dl + i] = v[b, :, first + i]
        kv_len[b] = L - T + n + 1
        draft_len[b] = dl + n + 1
    return kv_len, kd, vd, draft_len, bad
