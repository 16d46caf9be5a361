"""Pins for the dynamic top-K drafting oracle (CPU only).

Checked against a hand-derived example with a tie (tests/golden/topk_hand.json),
the take-everything case (equals plain decode attention, pinned on its own),
the one-row budget (only the query's own row), an O(n^2) rank definition of
the selection on tie-heavy inputs, and the composition of the separately
pinned SnapKV (one-row window, no pooling) and draft-attention oracles.
"""
import json
import os

import numpy as np
import pytest

from oracle.attention import attention, draft_attention
from oracle.snapkv import snapkv_select
from oracle.topk import topk_attention

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "topk_hand.json")))
    w = np.array(g["weights"], dtype=np.float64)
    L = len(w)
    k = np.zeros((1, 1, L, 2))
    k[0, 0, :, 0] = np.log(w)
    v = np.zeros((1, 1, L, 2))
    v[0, 0, :, 0] = np.arange(L)
    v[0, 0, :, 1] = 1.0
    q = np.array([[[1.0, 0.0]]])
    for case in g["cases"]:
        K = case["K"]
        res = topk_attention(q, k, v, np.array([L]), K, 1.0)
        n = int(res["draft_len"][0])
        assert n == min(K, L)
        assert list(res["sel_idx"][0, 0, :n]) == case["kept"]
        assert np.all(res["sel_idx"][0, 0, n:] == -1)
        np.testing.assert_allclose(res["out"][0, 0], [case["out0_num"] / case["S"], 1.0], rtol=1e-14)
        np.testing.assert_allclose(res["lse"][0, 0], np.log(case["S"]), rtol=1e-14)


def _rand(B, Hq, Hkv, D, L_cap, seed, ties=False):
    rng = np.random.default_rng(seed)
    if ties:  # small integer logits: many equal scores
        q = rng.integers(-1, 2, size=(B, Hq, D)).astype(np.float64)
        k = rng.integers(-1, 2, size=(B, Hkv, L_cap, D)).astype(np.float64)
    else:
        q = rng.standard_normal((B, Hq, D))
        k = rng.standard_normal((B, Hkv, L_cap, D))
    v = rng.standard_normal((B, Hkv, L_cap, D))
    return q, k, v


@pytest.mark.parametrize("seed", [0, 1])
def test_budget_covering_the_context_is_plain_decode_attention(seed):
    B, Hq, Hkv, D, cap = 3, 8, 2, 16, 40
    q, k, v = _rand(B, Hq, Hkv, D, cap, seed)
    L = np.array([40, 17, 1])
    res = topk_attention(q, k, v, L, 64, 0.25)
    ref, ref_lse = attention(q[:, None], k, v, L, 0.25)   # T = 1: the query at position L - 1
    np.testing.assert_allclose(res["out"], ref[:, 0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(res["lse"], ref_lse[:, 0], rtol=1e-12, atol=1e-12)
    for b in range(B):
        assert list(res["sel_idx"][b, 0, : L[b]]) == list(range(L[b]))


def test_one_row_budget_keeps_only_the_querys_own_row():
    B, Hq, Hkv, D, cap = 2, 4, 1, 8, 30
    q, k, v = _rand(B, Hq, Hkv, D, cap, 3)
    L = np.array([30, 9])
    res = topk_attention(q, k, v, L, 1, 0.3)
    for b in range(B):
        assert list(res["sel_idx"][b, 0]) == [L[b] - 1]
        for h in range(Hq):
            np.testing.assert_allclose(res["out"][b, h], v[b, 0, L[b] - 1], rtol=1e-14)
            np.testing.assert_allclose(res["lse"][b, h], 0.3 * (q[b, h] @ k[b, 0, L[b] - 1]), rtol=1e-12)


@pytest.mark.parametrize("K", [2, 5, 11])
def test_selection_matches_the_rank_definition_on_ties(K):
    B, Hq, Hkv, D, cap = 2, 6, 2, 4, 24
    q, k, v = _rand(B, Hq, Hkv, D, cap, 7 + K, ties=True)
    L = np.array([24, 13])
    res = topk_attention(q, k, v, L, K, 0.5)
    G = Hq // Hkv
    for b in range(B):
        n = int(L[b])
        for hk in range(Hkv):
            # scores straight from the definition, then ranks by pairwise comparison
            sc = np.zeros(n - 1)
            for g in range(G):
                lg = 0.5 * (k[b, hk, :n] @ q[b, hk * G + g])
                p = np.exp(lg - lg.max())
                sc += (p / p.sum())[: n - 1]
            np.testing.assert_allclose(res["score"][b, hk, : n - 1], sc, rtol=1e-13)
            rank = [sum(1 for i in range(n - 1) if sc[i] > sc[j] or (sc[i] == sc[j] and i < j)) for j in range(n - 1)]
            want = sorted(j for j in range(n - 1) if rank[j] < min(K, n) - 1) + [n - 1]
            got = list(res["sel_idx"][b, hk, : int(res["draft_len"][b])])
            assert got == want


@pytest.mark.parametrize("K", [3, 16])
def test_equals_one_row_window_snapkv_then_draft_attention(K):
    B, Hq, Hkv, D, cap = 3, 8, 2, 16, 50
    q, k, v = _rand(B, Hq, Hkv, D, cap, 11)
    L = np.array([50, 20, 4])
    res = topk_attention(q, k, v, L, K, 0.2)
    sel = snapkv_select(q[:, None], k, v, L, 1, 1, K, 0.2)
    np.testing.assert_array_equal(res["sel_idx"], sel["sel_idx"])
    np.testing.assert_array_equal(res["draft_len"], sel["draft_len"])
    out, lse = draft_attention(q[:, None], sel["k_draft"], sel["v_draft"], sel["draft_len"], 0.2)
    np.testing.assert_allclose(res["out"], out[:, 0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(res["lse"], lse[:, 0], rtol=1e-12, atol=1e-13)
