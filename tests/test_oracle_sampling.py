"""Pins for the sampling oracle (CPU only).

  * hand-derived rounds (tests/golden/rejection_hand.json);
  * the identity P(first output = x) = p(x) checked by integrating over a fine
    grid of uniforms (brute force over the randomness, no sampling noise);
  * chi-square over 10^6 draws at vocab 16 (first output and draft draw);
  * the closed form Omega(gamma, alpha) = (1 - alpha^(gamma+1)) / (1 - alpha)
    for the mean tokens per round at constant acceptance alpha (MagicDec notes,
    section 3.1, citing Leviathan et al.);
  * special cases: p == q accepts everything and emits the bonus; a draft
    token with p(x) = 0 is always rejected and the correction follows p.
"""
import json
import os

import numpy as np
import pytest

from oracle.sampling import draft_draw, inverse_cdf, rejection_sample, softmax

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
CHI2_15DOF_P1E3 = 37.697


def test_hand_worked_rounds():
    g = json.load(open(os.path.join(GOLDEN, "rejection_hand.json")))
    tl = np.log(np.array(g["p"]))[None]
    dl = np.log(np.array(g["q"]))[None]
    for c in g["cases"]:
        res = rejection_sample(tl, dl, np.array([c["x"]]), np.array([c["u"]]))
        assert list(res["out_tokens"][0]) == c["out"]
        assert res["num_accepted"][0] == c["num_accepted"]


def test_inverse_cdf_grid_frequencies_and_edges():
    r = np.array([0.0, 0.5, 0.0, 2.0, 1.5, 0.0])
    N = 20000
    u = (np.arange(N) + 0.5) / N
    tok, _ = inverse_cdf(np.broadcast_to(r, (N, r.size)), u)
    freq = np.bincount(tok, minlength=r.size) / N
    np.testing.assert_allclose(freq, r / r.sum(), atol=2.0 / N)
    t0, _ = inverse_cdf(r[None], np.array([0.0]))
    assert t0[0] == 1                              # u = 0 -> first index with r > 0
    t1, _ = inverse_cdf(r[None], np.array([np.nextafter(1.0, 0.0)]))
    assert t1[0] == 4                              # u -> 1 -> last index with r > 0
    V = 10
    uu = np.array([0.05, 0.15, 0.55, 0.95])
    tok, _ = inverse_cdf(np.ones((4, V)), uu)
    assert list(tok) == [0, 1, 5, 9]               # uniform weights -> floor(u V)


def _dist(rng, V, alpha=None):
    return rng.dirichlet(np.ones(V))


def test_first_output_is_target_distribution_by_grid_integration():
    """Sum over draft tokens x0 and a grid over (u1, u2): P(first output = x) = p(x)."""
    rng = np.random.default_rng(5)
    V = 4
    p0, q0 = _dist(rng, V), _dist(rng, V)
    p1, q1, p2 = _dist(rng, V), _dist(rng, V), _dist(rng, V)
    N = 600
    grid = (np.arange(N) + 0.5) / N
    u1, u2 = np.meshgrid(grid, grid, indexing="ij")
    n = N * N
    prob = np.zeros(V)
    for x0 in range(V):
        tl = np.log(np.broadcast_to(np.stack([p0, p1, p2]), (n, 3, V)))
        dl = np.log(np.broadcast_to(np.stack([q0, q1]), (n, 2, V)))
        toks = np.tile(np.array([x0, 0]), (n, 1))
        u = np.zeros((n, 3, 3))
        u[:, 0, 1] = u1.ravel()
        u[:, 0, 2] = u2.ravel()
        u[:, 1, 1] = 0.5
        u[:, 1, 2] = 0.5
        u[:, 2, 2] = 0.5
        res = rejection_sample(tl, dl, toks, u)
        prob += q0[x0] * np.bincount(res["out_tokens"][:, 0], minlength=V) / n
    np.testing.assert_allclose(prob, p0, atol=4.0 / N)


def _chi2(counts, probs):
    n = counts.sum()
    e = n * probs
    return float(np.sum((counts - e) ** 2 / e))


@pytest.mark.slow
def test_chi_square_first_output_and_draft_draw():
    V, gamma, n_total, chunk = 16, 2, 1_000_000, 100_000
    rng = np.random.default_rng(6)
    tl = rng.standard_normal((gamma + 1, V)) * 1.5
    dl = tl[:gamma] + rng.standard_normal((gamma, V))
    p0 = softmax(tl[0])
    q0 = softmax(dl[0])
    c_out = np.zeros(V)
    c_draft = np.zeros(V)
    for _ in range(n_total // chunk):
        u = rng.random((chunk, gamma + 1, 3))
        dlb = np.broadcast_to(dl, (chunk, gamma, V))
        toks, _ = draft_draw(dlb, u)
        res = rejection_sample(np.broadcast_to(tl, (chunk, gamma + 1, V)), dlb, toks, u)
        c_out += np.bincount(res["out_tokens"][:, 0], minlength=V)
        c_draft += np.bincount(toks[:, 0], minlength=V)
    assert _chi2(c_out, p0) < CHI2_15DOF_P1E3
    assert _chi2(c_draft, q0) < CHI2_15DOF_P1E3
    # the same counts are far from the draft distribution (the test has power)
    assert _chi2(c_out, q0) > 10 * CHI2_15DOF_P1E3


def _overlap_pair(rng, V, alpha):
    """p, q with sum_x min(p, q) = alpha: common mass alpha plus disjoint remainders."""
    c = rng.dirichlet(np.ones(V)) * alpha
    half = V // 2
    a = np.zeros(V)
    b = np.zeros(V)
    a[:half] = rng.dirichlet(np.ones(half))
    b[half:] = rng.dirichlet(np.ones(V - half))
    return c + (1 - alpha) * a, c + (1 - alpha) * b


@pytest.mark.slow
@pytest.mark.parametrize("alpha", [0.5, 0.8, 0.9])
@pytest.mark.parametrize("gamma", [2, 3, 4])
def test_omega_closed_form(alpha, gamma):
    V, n = 16, 1_000_000
    rng = np.random.default_rng(int(alpha * 100) * 10 + gamma)
    ps, qs = zip(*[_overlap_pair(rng, V, alpha) for _ in range(gamma + 1)])
    assert all(abs(np.minimum(p, q).sum() - alpha) < 1e-12 for p, q in zip(ps, qs))
    tl = np.log(np.stack(ps))
    dl = np.log(np.stack(qs[:gamma]))
    tokens = []
    chunk = 250_000
    for _ in range(n // chunk):
        u = rng.random((chunk, gamma + 1, 3))
        dlb = np.broadcast_to(dl, (chunk, gamma, V))
        x, _ = draft_draw(dlb, u)
        res = rejection_sample(np.broadcast_to(tl, (chunk, gamma + 1, V)), dlb, x, u)
        tokens.append(res["num_accepted"] + 1)
    t = np.concatenate(tokens).astype(np.float64)
    omega = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    se = t.std() / np.sqrt(n)
    assert abs(t.mean() - omega) < 4 * se


def test_equal_distributions_accept_all_and_draw_bonus():
    rng = np.random.default_rng(7)
    B, gamma, V = 64, 3, 50
    tl = rng.standard_normal((B, gamma + 1, V))
    u = rng.random((B, gamma + 1, 3))
    x, _ = draft_draw(tl[:, :gamma], u)
    res = rejection_sample(tl, tl[:, :gamma], x, u)
    assert np.all(res["num_accepted"] == gamma)
    np.testing.assert_array_equal(res["out_tokens"][:, :gamma], x)
    bonus, _ = inverse_cdf(softmax(tl[:, gamma]), u[:, gamma, 2])
    np.testing.assert_array_equal(res["out_tokens"][:, gamma], bonus)


def test_zero_target_mass_rejects_and_follows_p():
    rng = np.random.default_rng(8)
    B, V = 4000, 8
    p = rng.dirichlet(np.ones(V))
    p[3] = 0.0
    p /= p.sum()
    with np.errstate(divide="ignore"):
        tl = np.log(np.broadcast_to(np.stack([p, p]), (B, 2, V)))
    dl = np.full((B, 1, V), -50.0)
    dl[:, 0, 3] = 50.0                              # q one-hot on token 3
    u = rng.random((B, 2, 3))
    res = rejection_sample(tl, dl, np.full((B, 1), 3), u)
    assert np.all(res["num_accepted"] == 0)
    assert np.all(res["out_tokens"][:, 1] == -1)
    freq = np.bincount(res["out_tokens"][:, 0], minlength=V) / B
    assert freq[3] == 0.0
    np.testing.assert_allclose(freq, p, atol=0.03)
