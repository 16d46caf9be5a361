"""GPU parity of the draft draw and of modified rejection sampling against the
float64 oracle, plus the distribution identities checked directly on GPU draws.

Decisions are compared per sequence and must be identical, except for
sequences where the oracle reports a tested acceptance with |u*q - p| < 1e-6
or a draw whose target u*Z lies within 1e-6*Z of a bucket edge.  For those,
the decisions before the first position inside the band must still agree.
At vocab 128256 the drafted tokens have p, q of order 1e-4, so the absolute
1e-6 band holds about 1-2 % of the tests per position.  Which sequences fall
in the band is fixed by the inputs and the oracle alone:
tests/golden/sampling_check_fraction.json holds the fully compared fraction
of each case (computed with oracle/ only), and each test asserts that it
compares that fraction, within two points."""
import json
import os

import numpy as np
import pytest
import torch

from _parity import SAMPLE_BAND, Guarded, check_guards, gpu_or_skip
from long_context_speculative_split_gb300 import mgd, ops
from long_context_speculative_split_gb300 import workloads as wl
from oracle.sampling import draft_draw as ref_draw
from oracle.sampling import rejection_sample as ref_reject
from oracle.sampling import softmax

pytestmark = pytest.mark.gpu
CHI2_15DOF_P1E3 = 37.697
with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "sampling_check_fraction.json")) as _f:
    CHECK_FRACTION = {k: v["fraction"] for k, v in json.load(_f)["cases"].items()}
FRACTION_SLACK = 0.02


def _compare_round(t, d, u, dev, case=None, min_frac=0.75, reuse=False):
    """Compare one round with the oracle; returns (num_accepted, fully compared fraction).
    With `case`, the fraction must equal the oracle-only value stored for that case
    (within FRACTION_SLACK); otherwise it must reach `min_frac`.  With `reuse`, the draws
    and the rejection sample share one workspace and the rejection sample takes the draft
    rows' normalisers from the draws (MGD_VERIFY_DRAWN)."""
    B, gp1, V = t.shape
    gamma = gp1 - 1
    # outputs between poisoned guard regions (checked after each call)
    g = dict(draft_tokens=Guarded((B, gamma), torch.int32, dev), out_tokens=Guarded((B, gp1), torch.int32, dev),
             num_accepted=Guarded((B,), torch.int32, dev))
    ws = ops.workspace(mgd.mgd_spec_workspace_size(B, gamma, V), dev) if reuse else None
    if reuse:  # one draft position per call, as a round's draft steps make them
        for s in range(gamma):
            ops.draft_draw(d.to(dev), u.to(dev), draft_tokens=g["draft_tokens"].t, row=s, ws=ws)
        tok = g["draft_tokens"].t
    else:
        tok = ops.draft_draw(d.to(dev), u.to(dev), draft_tokens=g["draft_tokens"].t)
    rtok, rmarg = ref_draw(d, u)
    tok_c = tok.cpu().numpy()
    ok_draw = rmarg >= SAMPLE_BAND
    assert np.array_equal(tok_c[ok_draw], rtok[ok_draw])
    # the verify step reads the oracle's draft tokens, on both sides (no GPU output is an oracle input)
    rtok_d = torch.from_numpy(np.ascontiguousarray(rtok, dtype=np.int32)).to(dev)
    out, nacc = ops.rejection_sample(t.to(dev), d.to(dev), rtok_d, u.to(dev), ws=ws, out_tokens=g["out_tokens"].t,
                                     num_accepted=g["num_accepted"].t, reuse_draft_stats=reuse)
    torch.cuda.synchronize()
    check_guards(**g)
    if reuse:
        assert mgd.mgd_workspace_errors(ws) == 0
    tok_c = rtok
    ref = ref_reject(t, d, rtok, u)
    out_c, nacc_c = out.cpu().numpy(), nacc.cpu().numpy()
    with np.errstate(invalid="ignore"):
        ambiguous = ref["accept_margin"] < SAMPLE_BAND          # [B, gamma], False where untested
    first_amb = np.where(ambiguous.any(axis=1), ambiguous.argmax(axis=1), gamma + 1)
    full = first_amb > gamma
    # every sequence: identical decisions up to the first position inside the band
    pre_ref = np.minimum(ref["num_accepted"], first_amb)
    pre_gpu = np.minimum(nacc_c, first_amb)
    assert np.array_equal(pre_gpu, pre_ref)
    # sequences without an ambiguous test: identical acceptance count, identical
    # correction / bonus token unless that draw itself lies inside the band
    assert np.array_equal(nacc_c[full], ref["num_accepted"][full])
    draw_ok = full & ~(ref["draw_margin"] < SAMPLE_BAND)
    assert np.array_equal(out_c[draw_ok], ref["out_tokens"][draw_ok])
    frac = float(draw_ok.mean())
    print("fully compared sequences: %.4f (%d of %d)" % (frac, int(draw_ok.sum()), B))
    if case is not None:
        assert abs(frac - CHECK_FRACTION[case]) <= FRACTION_SLACK, (frac, CHECK_FRACTION[case])
    else:
        assert frac >= min_frac
    # structure holds everywhere: accepted drafts copied, then one token, then -1
    for b in range(B):
        n = nacc_c[b]
        assert np.array_equal(out_c[b, :n], tok_c[b, :n])
        assert 0 <= out_c[b, n] < V
        assert np.all(out_c[b, n + 1:] == -1)
    return nacc_c, frac


@pytest.mark.parametrize("reuse", [False, True], ids=["own_stats", "draws_stats"])
@pytest.mark.parametrize("name", ["tiny_b2", "b32_ctx8k", "b128_ctx32k", "ragged_b256_ctx4k_64k"])
def test_round_matches_oracle(name, reuse):
    """Every configuration's round (the ragged one: batch 256, gamma 2, vocab 128256), with the
    rejection sample computing every row's statistics, and taking the draft rows' from the draws."""
    dev = gpu_or_skip()
    c = wl.WORKLOADS[name]
    t, d = wl.logits(c, "cpu")
    u = wl.uniforms(c, "cpu")
    _compare_round(t, d, u, dev, case=name, reuse=reuse)


def test_reuse_without_draws_raises_device_flag():
    """MGD_VERIFY_DRAWN on a workspace whose draft rows were not all drawn raises
    MGD_DEVERR_NOT_DRAWN; a rejection sample forgets the draws, so the next round must draw
    again; a complete round afterwards raises nothing."""
    dev = gpu_or_skip()
    c = dict(wl.WORKLOADS["b32_ctx8k"], B=8, V=5000)
    t, d = wl.logits(c, dev, seed=12)
    u = wl.uniforms(c, dev, seed=12)
    B, g, V = c["B"], c["gamma"], c["V"]
    ws = ops.workspace(mgd.mgd_spec_workspace_size(B, g, V), dev)
    tok = ops.draft_draw(d, u)  # drawn on another workspace
    ops.rejection_sample(t, d, tok, u, ws=ws, reuse_draft_stats=True)
    assert mgd.mgd_workspace_errors(ws) & mgd.MGD_DEVERR_NOT_DRAWN
    for s in range(g - 1):  # one position short
        ops.draft_draw(d, u, draft_tokens=tok, row=s, ws=ws)
    ops.rejection_sample(t, d, tok, u, ws=ws, reuse_draft_stats=True)
    assert mgd.mgd_workspace_errors(ws) & mgd.MGD_DEVERR_NOT_DRAWN
    ops.draft_draw(d, u, draft_tokens=tok, ws=ws)  # every position
    ops.rejection_sample(t, d, tok, u, ws=ws)  # the verify that computes its own statistics forgets them too
    assert mgd.mgd_workspace_errors(ws) == 0
    ops.rejection_sample(t, d, tok, u, ws=ws, reuse_draft_stats=True)
    assert mgd.mgd_workspace_errors(ws) & mgd.MGD_DEVERR_NOT_DRAWN
    ops.draft_draw(d, u, draft_tokens=tok, ws=ws)
    out, nacc = ops.rejection_sample(t, d, tok, u, ws=ws, reuse_draft_stats=True)
    assert mgd.mgd_workspace_errors(ws) == 0
    out_ref, nacc_ref = ops.rejection_sample(t, d, tok, u)
    torch.cuda.synchronize()
    # the two verify modes differ only in the rounding of the draft normalisers
    assert (nacc == nacc_ref).float().mean().item() >= 0.75


@pytest.mark.parametrize("reuse", [False, True], ids=["own_stats", "draws_stats"])
def test_odd_vocab_and_many_sequences(reuse):
    dev = gpu_or_skip()
    c = dict(wl.WORKLOADS["b32_ctx8k"], B=300, V=4099, gamma=5, sigma=2.0, sigma_n=1.0)
    t, d = wl.logits(c, "cpu", seed=4)
    u = wl.uniforms(c, "cpu", seed=4)
    _compare_round(t, d, u, dev, case="odd_vocab_b300", reuse=reuse)


@pytest.mark.parametrize("reuse", [False, True], ids=["own_stats", "draws_stats"])
def test_masked_vocabulary(reuse):
    """60 % of each sequence's vocabulary at -inf in every row, and 2 % more in the target rows
    only: masked entries weigh nothing, a drafted token the target forbids is always rejected."""
    dev = gpu_or_skip()
    c = dict(wl.WORKLOADS["b32_ctx8k"], B=64, V=32000, mask_frac=0.6)
    t, d = wl.logits(c, "cpu", seed=6)
    u = wl.uniforms(c, "cpu", seed=6)
    assert bool(torch.isinf(t).any()) and bool(torch.isinf(d).any())
    _compare_round(t, d, u, dev, case="masked_vocab_b64", reuse=reuse)


@pytest.mark.parametrize("reuse", [False, True], ids=["own_stats", "draws_stats"])
@pytest.mark.parametrize("case,gamma,B,seed", [("gamma1_b40", 1, 40, 7), ("gamma16_b24", 16, 24, 8)])
def test_gamma_extremes(case, gamma, B, seed, reuse):
    """One draft position, and the largest number the library takes (16: 33 rows per sequence)."""
    dev = gpu_or_skip()
    c = dict(wl.WORKLOADS["b32_ctx8k"], B=B, V=5000, gamma=gamma)
    t, d = wl.logits(c, "cpu", seed=seed)
    u = wl.uniforms(c, "cpu", seed=seed)
    _compare_round(t, d, u, dev, case=case, reuse=reuse)


@pytest.mark.parametrize("reuse", [False, True], ids=["own_stats", "draws_stats"])
def test_vocab_over_eight_chunks(reuse):
    """Vocabulary 152064 (the Qwen2.5 models' of the MagicDec notes' model ablation): ten
    16384-entry chunks per row, more than one thread-block cluster takes, so the draw and the
    decision kernel hand their sub-range records over through the workspace tickets."""
    dev = gpu_or_skip()
    c = dict(wl.WORKLOADS["b32_ctx8k"], B=48, V=152064)
    t, d = wl.logits(c, "cpu", seed=9)
    u = wl.uniforms(c, "cpu", seed=9)
    _compare_round(t, d, u, dev, case="qwen_vocab_b48", reuse=reuse)


@pytest.mark.parametrize("case,B,V,seed", [("odd_vocab_five_chunks_b100", 100, 65539, 10),
                                           ("odd_vocab_ten_chunks_b50", 50, 147459, 11)],
                         ids=["cluster_rows", "ticket_rows"])
@pytest.mark.parametrize("reuse", [False, True], ids=["stream_rows", "reuse_draws"])
def test_unaligned_vocab_in_two_round_draws(case, B, V, seed, reuse):
    """A vocabulary that is not a multiple of 4 (scalar loads) in grids of 500 CTAs, more than
    the one-round draw keeps resident on a 152-SM part, so every lane streams its sub-range in
    two rounds: rows of five chunks draw inside a cluster, rows of ten through the tickets."""
    dev = gpu_or_skip()
    c = dict(wl.WORKLOADS["b32_ctx8k"], B=B, V=V)
    t, d = wl.logits(c, "cpu", seed=seed)
    u = wl.uniforms(c, "cpu", seed=seed)
    _compare_round(t, d, u, dev, case=case, reuse=reuse)


def test_single_row_draft_draw():
    dev = gpu_or_skip()
    c = wl.WORKLOADS["b32_ctx8k"]
    _, d = wl.logits(c, "cpu", seed=1)
    u = wl.uniforms(c, "cpu", seed=1)
    tok = torch.full((c["B"], c["gamma"]), -7, dtype=torch.int32, device=dev)
    ops.draft_draw(d.to(dev), u.to(dev), draft_tokens=tok, row=1)
    rt, rm = ref_draw(d, u)
    tc = tok.cpu().numpy()
    assert np.all(tc[:, 0] == -7) and np.all(tc[:, 2] == -7)
    ok = rm[:, 1] >= SAMPLE_BAND
    assert np.array_equal(tc[ok, 1], rt[ok, 1])


def _chi2(counts, probs):
    e = counts.sum() * probs
    return float(np.sum((counts - e) ** 2 / e))


def test_chi_square_first_output_is_target():
    dev = gpu_or_skip()
    V, gamma, n = 16, 2, 1_000_000
    g = torch.Generator().manual_seed(11)
    tl = torch.randn((gamma + 1, V), generator=g) * 1.5
    dl = tl[:gamma] + torch.randn((gamma, V), generator=g)
    T = tl.expand(n, gamma + 1, V).contiguous().to(dev)
    Dd = dl.expand(n, gamma, V).contiguous().to(dev)
    u = torch.rand((n, gamma + 1, 3), generator=g).to(dev)
    tok = ops.draft_draw(Dd, u)
    out, _ = ops.rejection_sample(T, Dd, tok, u)
    c_out = np.bincount(out[:, 0].cpu().numpy(), minlength=V).astype(np.float64)
    c_dr = np.bincount(tok[:, 0].cpu().numpy(), minlength=V).astype(np.float64)
    assert _chi2(c_out, softmax(tl[0].double().numpy())) < CHI2_15DOF_P1E3
    assert _chi2(c_dr, softmax(dl[0].double().numpy())) < CHI2_15DOF_P1E3
    assert _chi2(c_out, softmax(dl[0].double().numpy())) > 10 * CHI2_15DOF_P1E3


def test_omega_closed_form_on_gpu():
    dev = gpu_or_skip()
    V, gamma, n, alpha = 16, 3, 1_000_000, 0.9
    rng = np.random.default_rng(12)
    ps, qs = [], []
    for _ in range(gamma + 1):
        c = rng.dirichlet(np.ones(V)) * alpha
        a = np.zeros(V)
        b = np.zeros(V)
        a[:8] = rng.dirichlet(np.ones(8))
        b[8:] = rng.dirichlet(np.ones(8))
        ps.append(c + (1 - alpha) * a)
        qs.append(c + (1 - alpha) * b)
    tl = torch.tensor(np.log(np.stack(ps)), dtype=torch.float32)
    dl = torch.tensor(np.log(np.stack(qs[:gamma])), dtype=torch.float32)
    T = tl.expand(n, gamma + 1, V).contiguous().to(dev)
    Dd = dl.expand(n, gamma, V).contiguous().to(dev)
    u = torch.rand((n, gamma + 1, 3), generator=torch.Generator().manual_seed(13)).to(dev)
    tok = ops.draft_draw(Dd, u)
    _, nacc = ops.rejection_sample(T, Dd, tok, u)
    x = nacc.double().cpu().numpy() + 1
    omega = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    assert abs(x.mean() - omega) < 4 * x.std() / np.sqrt(n)


def test_equal_distributions_accept_everything():
    dev = gpu_or_skip()
    c = dict(wl.WORKLOADS["b32_ctx8k"], B=64, V=5000)
    t, _ = wl.logits(c, "cpu", seed=2)
    d = t[:, :c["gamma"]].contiguous()
    u = wl.uniforms(c, "cpu", seed=2)
    nacc, _ = _compare_round(t, d, u, dev)
    assert np.all(nacc == c["gamma"])


def test_invalid_draft_token_raises_device_flag():
    dev = gpu_or_skip()
    c = dict(wl.WORKLOADS["tiny_b2"], B=4, V=100)
    t, d = wl.logits(c, dev)
    u = wl.uniforms(c, dev)
    tok = torch.tensor([[0, 1, 2], [5, 100, 1], [-1, 0, 0], [3, 3, 3]], dtype=torch.int32, device=dev)
    ws = ops.workspace(mgd.mgd_spec_workspace_size(4, 3, 100), dev)
    out, nacc = ops.rejection_sample(t, d, tok, u, ws=ws)
    assert mgd.mgd_workspace_errors(ws) & mgd.MGD_DEVERR_TOKEN
    n = nacc.cpu().numpy()
    assert n[1] <= 1 and n[2] == 0
    o = out.cpu().numpy()
    for b in range(4):
        assert 0 <= o[b, n[b]] < 100
