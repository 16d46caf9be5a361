"""Pins for the attention oracle (CPU only).

Each check is independent of the oracle's own formula: a hand-derived worked
example, high-precision brute force, closed forms (single key, equal keys),
structural invariants (causal extent, GQA mapping, permutation, linearity) and
the split/merge identity that the split-KV kernels rely on.
"""
import json
import os

import numpy as np
import pytest

from oracle.attention import attention, draft_attention, merge_lse

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "attention_hand.json")))
    out, lse = attention(np.array(g["q"]), np.array(g["k"]), np.array(g["v"]),
                         np.array(g["kv_len"]), g["scale"])
    np.testing.assert_allclose(out, np.array(g["expected_out"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, np.array(g["expected_lse"]), rtol=0, atol=1e-13)


def test_mpmath_brute_force():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    B, T, Hq, Hkv, D, Lcap = 2, 3, 4, 2, 5, 9
    q, k, v = _rand((B, T, Hq, D), 1), _rand((B, Hkv, Lcap, D), 2), _rand((B, Hkv, Lcap, D), 3)
    kv_len = np.array([7, 3])
    scale = 0.37
    out, lse = attention(q, k, v, kv_len, scale)
    G = Hq // Hkv
    for b in range(B):
        for t in range(T):
            for h in range(Hq):
                hk = h // G
                n = int(kv_len[b]) - T + t + 1
                sc = [mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(q[b, t, h, d]) * mpmath.mpf(k[b, hk, j, d])
                                                      for d in range(D)) for j in range(n)]
                w = [mpmath.exp(s) for s in sc]
                Z = mpmath.fsum(w)
                assert abs(float(mpmath.log(Z)) - lse[b, t, h]) < 1e-12
                for d in range(D):
                    o = mpmath.fsum(w[j] * mpmath.mpf(v[b, hk, j, d]) for j in range(n)) / Z
                    assert abs(float(o) - out[b, t, h, d]) < 1e-12


def test_single_key_returns_its_value():
    q, k, v = _rand((1, 1, 2, 8), 4), _rand((1, 1, 1, 8), 5), _rand((1, 1, 1, 8), 6)
    out, lse = attention(q, k, v, np.array([1]), 0.5)
    for h in range(2):
        np.testing.assert_allclose(out[0, 0, h], v[0, 0, 0], atol=1e-15)
        np.testing.assert_allclose(lse[0, 0, h], 0.5 * q[0, 0, h] @ k[0, 0, 0], atol=1e-14)


def test_equal_keys_give_mean_value_and_log_count():
    B, T, Hq, D, L = 1, 4, 2, 6, 10
    q = _rand((B, T, Hq, D), 7)
    krow = _rand(D, 8)
    k = np.broadcast_to(krow, (B, 1, L, D)).copy()
    v = _rand((B, 1, L, D), 9)
    out, lse = attention(q, k, v, np.array([L]), 0.3)
    for t in range(T):
        n = L - T + t + 1
        for h in range(Hq):
            np.testing.assert_allclose(out[0, t, h], v[0, 0, :n].mean(axis=0), atol=1e-14)
            np.testing.assert_allclose(lse[0, t, h], 0.3 * q[0, t, h] @ krow + np.log(n), atol=1e-13)


def test_causal_extent_of_each_verify_row():
    """Row t sees exactly keys 0..L-T+t: changing key L-T+t+1 moves rows > t only."""
    B, T, Hq, D, L = 1, 4, 1, 8, 12
    q, k, v = _rand((B, T, Hq, D), 10), _rand((B, 1, L, D), 11), _rand((B, 1, L, D), 12)
    base, _ = attention(q, k, v, np.array([L]), 0.4)
    for t in range(T - 1):
        j = L - T + t + 1
        k2, v2 = k.copy(), v.copy()
        k2[0, 0, j] += 3.0
        v2[0, 0, j] += 5.0
        pert, _ = attention(q, k2, v2, np.array([L]), 0.4)
        np.testing.assert_array_equal(pert[0, : t + 1], base[0, : t + 1])
        assert np.all(np.abs(pert[0, t + 1:] - base[0, t + 1:]).max(axis=-1) > 1e-6)


def test_gqa_mapping_uses_contiguous_groups():
    """Query head h reads KV head h // G: give every KV head a constant value vector."""
    B, T, Hq, Hkv, D, L = 1, 2, 8, 4, 4, 6
    q, k = _rand((B, T, Hq, D), 13), _rand((B, Hkv, L, D), 14)
    v = np.zeros((B, Hkv, L, D))
    for hk in range(Hkv):
        v[0, hk] = 10.0 * hk + np.arange(D)
    out, _ = attention(q, k, v, np.array([L]), 1.0)
    for h in range(Hq):
        np.testing.assert_allclose(out[0, :, h], np.broadcast_to(10.0 * (h // 2) + np.arange(D), (T, D)), atol=1e-12)


def test_probabilities_sum_to_one_and_linearity_in_v():
    B, T, Hq, D, L = 2, 3, 2, 8, 16
    q, k = _rand((B, T, Hq, D), 15), _rand((B, 1, L, D), 16)
    kv_len = np.array([16, 5])
    ones, _ = attention(q, k, np.ones((B, 1, L, D)), kv_len, 0.5)
    np.testing.assert_allclose(ones, 1.0, atol=1e-14)
    v1, v2 = _rand((B, 1, L, D), 17), _rand((B, 1, L, D), 18)
    o1, _ = attention(q, k, v1, kv_len, 0.5)
    o2, _ = attention(q, k, v2, kv_len, 0.5)
    o12, _ = attention(q, k, 2.0 * v1 - v2, kv_len, 0.5)
    np.testing.assert_allclose(o12, 2.0 * o1 - o2, atol=1e-13)


def test_permutation_invariance_without_mask():
    B, Hq, D, L = 1, 2, 8, 20
    q, k, v = _rand((B, 1, Hq, D), 19), _rand((B, 1, L, D), 20), _rand((B, 1, L, D), 21)
    perm = np.random.default_rng(22).permutation(L)
    a, la = attention(q, k, v, np.array([L]), 0.5)
    b_, lb = attention(q, k[:, :, perm], v[:, :, perm], np.array([L]), 0.5)
    np.testing.assert_allclose(a, b_, atol=1e-14)
    np.testing.assert_allclose(la, lb, atol=1e-14)


def test_split_invariance_of_lse_merge():
    """Attention over disjoint key subsets merged by merge_lse equals the unsplit result."""
    B, Hq, Hkv, D, L = 2, 4, 2, 16, 37
    q, k, v = _rand((B, 1, Hq, D), 23), _rand((B, Hkv, L, D), 24), _rand((B, Hkv, L, D), 25)
    full, lfull = attention(q, k, v, np.array([L, L]), 0.25)
    for cuts in ([0, 5, 37], [0, 1, 2, 20, 36, 37], [0, 16, 32, 37]):
        parts = []
        for a, b in zip(cuts[:-1], cuts[1:]):
            parts.append(attention(q, k[:, :, a:b], v[:, :, a:b], np.array([b - a, b - a]), 0.25))
        out, lse = merge_lse(parts)
        np.testing.assert_allclose(out, full, atol=1e-12)
        np.testing.assert_allclose(lse, lfull, atol=1e-12)
    # one part is the identity; an empty part (lse = -inf) adds nothing
    out, lse = merge_lse([(full, lfull)])
    np.testing.assert_allclose(out, full, atol=1e-15)
    out, lse = merge_lse([(full, lfull), (np.zeros_like(full), np.full_like(lfull, -np.inf))])
    np.testing.assert_allclose(out, full, atol=1e-15)
    np.testing.assert_allclose(lse, lfull, atol=1e-15)


def test_merge_is_order_independent():
    rng = np.random.default_rng(26)
    parts = [(rng.standard_normal((3, 5)), rng.standard_normal(3) * 4) for _ in range(4)]
    a = merge_lse(parts)
    b = merge_lse(parts[::-1])
    c = merge_lse([merge_lse(parts[:2]), merge_lse(parts[2:])])
    for x in (b, c):
        np.testing.assert_allclose(x[0], a[0], atol=1e-13)
        np.testing.assert_allclose(x[1], a[1], atol=1e-13)


def test_draft_over_all_rows_equals_last_verify_row():
    B, T, Hq, Hkv, D, L = 2, 4, 4, 1, 8, 11
    q, k, v = _rand((B, T, Hq, D), 27), _rand((B, Hkv, L, D), 28), _rand((B, Hkv, L, D), 29)
    kv_len = np.array([11, 6])
    ver, lver = attention(q, k, v, kv_len, 0.5)
    dr, ldr = draft_attention(q[:, T - 1:], k, v, kv_len, 0.5)
    np.testing.assert_allclose(dr[:, 0], ver[:, T - 1], atol=1e-14)
    np.testing.assert_allclose(ldr[:, 0], lver[:, T - 1], atol=1e-14)


def test_sharp_scale_picks_argmax_value():
    B, Hq, D, L = 1, 1, 4, 9
    q, k, v = _rand((B, 1, Hq, D), 30), _rand((B, 1, L, D), 31), _rand((B, 1, L, D), 32)
    s = k[0, 0] @ q[0, 0, 0]
    out, _ = attention(q, k, v, np.array([L]), 1e4)
    np.testing.assert_allclose(out[0, 0, 0], v[0, 0, np.argmax(s)], atol=1e-9)
