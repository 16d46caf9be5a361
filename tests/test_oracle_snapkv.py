"""Pins for the SnapKV selection oracle (CPU only).

Checked against a hand-derived worked example, a closed form for equal keys,
an O(n^2) rank definition of top-K (a different route than the oracle's sort),
max-pool support properties, the take-everything case and a planted heavy
hitter.
"""
import json
import os

import numpy as np
import pytest

from oracle.snapkv import max_pool, select_indices, snapkv_select, window_scores

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _hand_inputs(g, G=1):
    L, W = g["L"], g["W"]
    k = np.zeros((1, 1, L, 2))
    k[0, 0, :, 0] = np.log(np.array(g["weights"], dtype=np.float64))
    qw = np.zeros((1, W, G, 2))
    qw[..., 0] = 1.0
    return qw, k


def test_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "snapkv_hand.json")))
    L, W = g["L"], g["W"]
    qw, k = _hand_inputs(g)
    s = window_scores(qw, k, np.array([L]), W, g["scale"])
    np.testing.assert_allclose(s[0, 0, : L - W] * 156.0, g["expected_scores_x156"], atol=1e-12)
    for case in g["cases"]:
        res = snapkv_select(qw, k, k, np.array([L]), W, case["P"], case["K"], g["scale"])
        n = int(res["draft_len"][0])
        assert n == min(case["K"], L)
        assert list(res["sel_idx"][0, 0, :n]) == case["expected_idx"]
        np.testing.assert_array_equal(res["k_draft"][0, 0, :n], k[0, 0, case["expected_idx"]])


def test_group_heads_are_summed():
    g = json.load(open(os.path.join(GOLDEN, "snapkv_hand.json")))
    qw, k = _hand_inputs(g, G=3)
    s = window_scores(qw, k, np.array([g["L"]]), g["W"], 1.0)
    np.testing.assert_allclose(s[0, 0, :6] * 156.0, 3 * np.array(g["expected_scores_x156"]), atol=1e-12)


def test_equal_keys_closed_form():
    """All keys equal: each window query spreads 1/(visible count) on every key."""
    B, Hq, Hkv, D, L, W = 1, 4, 2, 8, 40, 6
    rng = np.random.default_rng(0)
    k = np.broadcast_to(rng.standard_normal(D), (B, Hkv, L, D)).copy()
    qw = rng.standard_normal((B, W, Hq, D))
    s = window_scores(qw, k, np.array([L]), W, 0.3)
    expect = 2 * sum(1.0 / (L - W + w + 1) for w in range(W))   # G = 2 heads per KV head
    np.testing.assert_allclose(s[0, :, : L - W], expect, rtol=1e-13)
    assert np.all(s[0, :, L - W:] == 0.0)


def _rank_select(pooled, n_pre, n_top):
    """Top-n_top by rank definition: j is kept iff fewer than n_top positions beat it."""
    keep = []
    for j in range(n_pre):
        beats = sum(1 for i in range(n_pre)
                    if pooled[i] > pooled[j] or (pooled[i] == pooled[j] and i < j))
        if beats < n_top:
            keep.append(j)
    return keep


@pytest.mark.parametrize("seed", range(6))
def test_selection_matches_rank_definition(seed):
    rng = np.random.default_rng(100 + seed)
    L = int(rng.integers(8, 64))
    W = int(rng.integers(1, min(8, L) + 1))
    K = int(rng.integers(W, L + 3))
    # a coarse grid of scores makes ties frequent
    pooled = rng.integers(0, 6, size=L).astype(np.float64)
    idx = select_indices(pooled, L, W, K)
    n_top = min(K, L) - W
    expect = _rank_select(pooled, L - W, n_top) + list(range(L - W, L))
    assert list(idx) == expect


def test_pool_one_is_plain_top_k_of_scores():
    B, Hq, D, L, W, K = 1, 2, 8, 50, 4, 14
    rng = np.random.default_rng(1)
    qw, k = rng.standard_normal((B, W, Hq, D)), rng.standard_normal((B, 1, L, D))
    res = snapkv_select(qw, k, k, np.array([L]), W, 1, K, 0.35)
    s = res["scores"][0, 0]
    np.testing.assert_array_equal(res["pooled"][0, 0, : L - W], s[: L - W])
    expect = _rank_select(s, L - W, K - W) + list(range(L - W, L))
    assert list(res["sel_idx"][0, 0, :K]) == expect


def test_max_pool_support():
    n, P = 30, 7
    r = P // 2
    for p in (0, 1, 5, 29):
        row = np.zeros(n)
        row[p] = 1.0
        pooled = max_pool(row, n, P)
        expect = np.array([1.0 if abs(j - p) <= r else 0.0 for j in range(n)])
        np.testing.assert_array_equal(pooled, expect)
    rng = np.random.default_rng(2)
    row = rng.random(n)
    pooled = max_pool(row, n, P)
    assert np.all(pooled >= row)
    for j in range(n):
        assert pooled[j] in set(row[max(0, j - r): j + r + 1])


def test_budget_at_least_context_keeps_everything():
    B, Hq, D, W = 2, 2, 8, 3
    rng = np.random.default_rng(3)
    kv_len = np.array([9, 5])
    k = rng.standard_normal((B, 1, 9, D))
    res = snapkv_select(rng.standard_normal((B, W, Hq, D)), k, k, kv_len, W, 3, 9, 0.3)
    assert list(res["draft_len"]) == [9, 5]
    assert list(res["sel_idx"][0, 0]) == list(range(9))
    assert list(res["sel_idx"][1, 0, :5]) == list(range(5)) and np.all(res["sel_idx"][1, 0, 5:] == -1)


def test_planted_heavy_hitter_is_kept():
    B, Hq, D, L, W, K = 1, 4, 16, 200, 8, 24
    rng = np.random.default_rng(4)
    qw = rng.standard_normal((B, W, Hq, D))
    k = rng.standard_normal((B, 1, L, D))
    hot = [17, 101, 150]
    for j in hot:
        k[0, 0, j] = 2.0 * qw[0].sum(axis=(0, 1)) / np.sqrt(D)
    res = snapkv_select(qw, k, k, np.array([L]), W, 5, K, 1.0 / np.sqrt(D))
    sel = set(res["sel_idx"][0, 0, :K].tolist())
    assert set(hot) <= sel
    assert set(range(L - W, L)) <= sel
    assert list(res["sel_idx"][0, 0, :K]) == sorted(sel)
