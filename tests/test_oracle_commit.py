"""Pins for the commit/rollback oracle (CPU only): a hand-worked case, the
length invariants, the copied rows, the all-accepted and overflow cases, and
agreement with the rejection-sampling oracle on how many tokens a round
commits."""
import numpy as np

from oracle.commit import commit_round
from oracle.sampling import draft_draw, rejection_sample


def _caches(B=2, Hkv=2, cap=16, dcap=8, D=4, seed=0):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((B, Hkv, cap, D))
    v = rng.standard_normal((B, Hkv, cap, D))
    kd = rng.standard_normal((B, Hkv, dcap, D))
    vd = rng.standard_normal((B, Hkv, dcap, D))
    return k, v, kd, vd


def test_hand_worked_case():
    # gamma = 3: verify rows at positions 6..9 of a 10-row cache; one draft accepted ->
    # rows 6 (last committed token) and 7 (accepted draft) stay, kv_len 10 -> 8, both
    # appended to the draft cache at positions 3 and 4.
    k, v, kd, vd = _caches(B=1)
    L, dl = np.array([10]), np.array([3])
    kv2, kd2, vd2, dl2, bad = commit_round(L, np.array([1]), 3, k, v, kd, vd, dl)
    assert list(kv2) == [8] and list(dl2) == [5] and not bad.any()
    np.testing.assert_array_equal(kd2[0, :, 3], k[0, :, 6])
    np.testing.assert_array_equal(kd2[0, :, 4], k[0, :, 7])
    np.testing.assert_array_equal(vd2[0, :, 4], v[0, :, 7])
    np.testing.assert_array_equal(kd2[0, :, :3], kd[0, :, :3])
    np.testing.assert_array_equal(kd2[0, :, 5:], kd[0, :, 5:])


def test_invariants_over_random_rounds():
    rng = np.random.default_rng(1)
    for _ in range(20):
        gamma = int(rng.integers(1, 6))
        B = 3
        k, v, kd, vd = _caches(B=B, cap=20, dcap=12, seed=int(rng.integers(1000)))
        L = rng.integers(gamma + 1, 21, size=B)
        dl = rng.integers(0, 12 - gamma - 1, size=B)
        n = rng.integers(0, gamma + 1, size=B)
        kv2, kd2, vd2, dl2, bad = commit_round(L, n, gamma, k, v, kd, vd, dl)
        assert not bad.any()
        np.testing.assert_array_equal(kv2, L - (gamma - n))
        np.testing.assert_array_equal(dl2, dl + n + 1)
        for b in range(B):
            first = L[b] - gamma - 1
            np.testing.assert_array_equal(kd2[b, :, dl[b]:dl[b] + n[b] + 1], k[b, :, first:first + n[b] + 1])
            np.testing.assert_array_equal(vd2[b, :, dl[b]:dl[b] + n[b] + 1], v[b, :, first:first + n[b] + 1])


def test_all_accepted_rolls_nothing_back_and_overflow_is_refused():
    k, v, kd, vd = _caches(B=2, dcap=8)
    kv2, _, _, dl2, bad = commit_round(np.array([12, 12]), np.array([3, 3]), 3, k, v, kd, vd, np.array([0, 5]))
    assert kv2[0] == 12 and dl2[0] == 4 and not bad[0]
    assert bad[1] and kv2[1] == 12 and dl2[1] == 5          # 5 + 4 > 8: unchanged
    _, _, _, _, bad = commit_round(np.array([3, 12]), np.array([0, 4]), 3, k, v, kd, vd, np.array([0, 0]))
    assert bad[0] and bad[1]                                 # kv_len < T; n > gamma


def test_rows_committed_equal_tokens_emitted_by_the_round():
    rng = np.random.default_rng(2)
    B, gamma, V = 64, 4, 30
    tl = rng.standard_normal((B, gamma + 1, V))
    dl_ = tl[:, :gamma] + 0.7 * rng.standard_normal((B, gamma, V))
    u = rng.random((B, gamma + 1, 3))
    x, _ = draft_draw(dl_, u)
    res = rejection_sample(tl, dl_, x, u)
    emitted = (res["out_tokens"] >= 0).sum(axis=1)
    k, v, kd, vd = _caches(B=B, cap=20, dcap=10)
    L = np.full(B, 20)
    kv2, _, _, dl2, bad = commit_round(L, res["num_accepted"], gamma, k, v, kd, vd, np.zeros(B, dtype=int))
    assert not bad.any()
    # every emitted token but the last becomes a kept verify row; the last opens the next block
    np.testing.assert_array_equal(dl2, emitted)
    np.testing.assert_array_equal(L - kv2, gamma + 1 - emitted)
