"""GPU parity of the full 32-layer speculation round (batch 32, context 16384,
gamma 3, draft budget 512, vocab 128256, 68.7 GB of KV) against the float64
oracle, over two consecutive rounds that each end with the commit / rollback
step: sampled layers and (sequence, KV head) pairs of the draft and verify
attention, the SnapKV draft caches of a sampled layer, every draft token and
the round's acceptance decisions, the lengths and the rows appended to the
draft cache after each round (bit-exact), and the second round's attention
over the committed state; plus identical results from a CUDA-graph replay and
the expected acceptance level (draft noise calibrated with the oracle so that
the mean acceptance is 0.9).

The oracle's commit is fed the oracle's own acceptance counts, never the
GPU's.  Sequences whose decisions the oracle reports as unambiguous (no test or
draw inside the 1e-6 band) must get the same count on the GPU; the commit state
is then compared on every sequence whose GPU count equals the oracle's in every
round so far (the commit depends on the count alone)."""
import math

import numpy as np
import pytest
import torch

from _parity import SAMPLE_BAND, assert_attention_close, assert_index_sets_match, gpu_or_skip
from long_context_speculative_split_gb300 import workloads as wl
from long_context_speculative_split_gb300.round import SpeculationRound
from oracle.attention import attention as ref_attention
from oracle.attention import draft_attention as ref_draft
from oracle.commit import commit_round as ref_commit
from oracle.sampling import draft_draw as ref_draw
from oracle.sampling import rejection_sample as ref_reject
from oracle.snapkv import max_pool, select_indices, window_scores

pytestmark = pytest.mark.gpu

LC = 5  # the layer whose caches are compared after each commit


def _snap(r):
    return dict(vout=r.vout.clone(), dout=r.dout.clone(), tok=r.tok.clone(), out_tok=r.out_tok.clone(),
                nacc=r.nacc.clone(), lengths=r.lengths.clone(), u=r.u.clone(),
                kd=r.sel[LC]["k_draft"].clone(), vd=r.sel[LC]["v_draft"].clone())


@pytest.fixture(scope="module")
def rnd():
    dev = gpu_or_skip()
    r = SpeculationRound(wl.WORKLOADS["round_b32_ctx16k_32layers"], dev).prepare()
    r.pre = [_snap(r)]          # state before round i, i = 0, 1, 2
    r.post = []                 # outputs of round i
    u_next = wl.uniforms(r.cfg, dev, seed=1)
    for i in range(2):
        if i == 1:
            r.u.copy_(u_next)   # the second round draws with fresh uniforms
        r.propose()
        r.verify_and_sample()
        torch.cuda.synchronize()
        r.post.append(_snap(r))
        r.commit()
        torch.cuda.synchronize()
        r.pre.append(_snap(r))
    yield r
    del r
    torch.cuda.empty_cache()


def _oracle_round(r, i):
    """The oracle's draft tokens and decisions of round i (its own draws), and the sequences
    whose decisions are unambiguous."""
    t, d, u = r.t.cpu(), r.d.cpu(), r.post[i]["u"].cpu()
    rtok, rmarg = ref_draw(d, u)
    ref = ref_reject(t, d, rtok, u)
    with np.errstate(invalid="ignore"):
        amb = ref["accept_margin"] < SAMPLE_BAND
    clear = ~amb.any(axis=1) & ~(ref["draw_margin"] < SAMPLE_BAND) & np.all(rmarg >= SAMPLE_BAND, axis=1)
    return rtok, ref, clear


def _oracle_selection(r, layer, b, h):
    """The oracle's SnapKV selection for one (layer, sequence, KV head) of the round's inputs:
    (kept positions, pooled scores, score of the lowest-ranked kept prefix position)."""
    G = r.Hq // r.Hkv
    L = int(r.kv_len[b])
    qw = wl.window_queries(r.cfg, r.dev, r.seed, layer=layer)
    s = window_scores(qw[b:b + 1, :, h * G:(h + 1) * G], r.k[layer][b:b + 1, h:h + 1, :L], r.kv_len[b:b + 1], r.W,
                      1.0 / math.sqrt(r.D))[0, 0]
    pooled = np.zeros(L)
    pooled[:L - r.W] = max_pool(s, L - r.W, r.P)
    ref_idx = select_indices(pooled, L, r.W, r.K)
    kth = np.min(pooled[ref_idx[:r.K - r.W]])
    return ref_idx, pooled, kth


def _oracle_draft_cache(r, layer, b, h, ref_idx):
    sel = torch.from_numpy(np.asarray(ref_idx, dtype=np.int64))
    return r.k[layer][b, h].cpu()[sel][None, None], r.v[layer][b, h].cpu()[sel][None, None]


def test_round_attention_matches_oracle(rnd):
    r = rnd
    G, D = r.Hq // r.Hkv, r.D
    scale = 1.0 / math.sqrt(D)
    o = r.post[0]
    for layer, b, h in [(0, 0, 0), (31, 31, 7), (17, 5, 3)]:
        L = int(r.kv_len[b])
        ref, _ = ref_attention(r.q[layer][b:b + 1, :, h * G:(h + 1) * G], r.k[layer][b:b + 1, h:h + 1, :L],
                               r.v[layer][b:b + 1, h:h + 1, :L], r.kv_len[b:b + 1], scale)
        assert_attention_close(o["vout"][layer, b:b + 1, :, h * G:(h + 1) * G], ref, "verify l%d" % layer)
        # draft attention over the oracle's own selection (where the GPU kept the same rows)
        ref_idx, pooled, kth = _oracle_selection(r, layer, b, h)
        got = r.sel[layer]["sel_idx"][b, h].cpu().numpy()[:r.K]
        assert_index_sets_match(got, ref_idx, pooled, kth)
        if set(got.tolist()) != set(np.asarray(ref_idx).tolist()):
            continue
        kd, vd = _oracle_draft_cache(r, layer, b, h, ref_idx)
        for s in range(r.gamma):
            rd, _ = ref_draft(r.qd[layer][s][b:b + 1, None, h * G:(h + 1) * G], kd, vd,
                              torch.tensor([len(ref_idx)]), scale)
            assert_attention_close(o["dout"][layer, s, b:b + 1, h * G:(h + 1) * G], rd[:, 0],
                                   "draft l%d s%d" % (layer, s))


def test_round_draft_cache_selection(rnd):
    r = rnd
    layer, b, h = 9, 12, 2
    ref_idx, pooled, kth = _oracle_selection(r, layer, b, h)
    got = r.sel[layer]["sel_idx"][b, h].cpu().numpy()
    assert_index_sets_match(got[:r.K], ref_idx, pooled, kth)


@pytest.mark.parametrize("i", [0, 1], ids=["round1", "round2"])
def test_round_tokens_match_oracle(rnd, i):
    r = rnd
    o = r.post[i]
    t, d, u = r.t.cpu(), r.d.cpu(), o["u"].cpu()
    tok = o["tok"].cpu().numpy()
    rt, rm = ref_draw(d, u)
    ok = rm >= SAMPLE_BAND
    assert np.array_equal(tok[ok], rt[ok])
    # the oracle verifies its own draft tokens; compared on the sequences where the GPU drew the same
    ref = ref_reject(t, d, rt, u)
    drew_same = np.all(tok == rt, axis=1)
    assert drew_same.mean() > 0.9
    nacc, out = o["nacc"].cpu().numpy(), o["out_tok"].cpu().numpy()
    with np.errstate(invalid="ignore"):
        amb = ref["accept_margin"] < SAMPLE_BAND
    first = np.where(amb.any(axis=1), amb.argmax(axis=1), r.gamma + 1)
    assert np.array_equal(np.minimum(nacc, first)[drew_same], np.minimum(ref["num_accepted"], first)[drew_same])
    full = (first > r.gamma) & ~(ref["draw_margin"] < SAMPLE_BAND) & drew_same
    assert np.array_equal(out[full], ref["out_tokens"][full])
    # mean acceptance 0.9 by construction: tokens per round near Omega(3, 0.9) = 3.439
    x = nacc + 1.0
    assert abs(x.mean() - 3.439) < 4 * max(x.std(), 0.5) / np.sqrt(len(x))


def test_commit_over_two_rounds_matches_oracle(rnd):
    """kv_len, draft_len and the draft-cache rows appended to layer LC after each of two
    consecutive rounds equal the oracle's commit applied to the oracle's own decisions, from the
    oracle's own starting lengths (bit-exact; every layer's lengths move together).  The selected
    rows before the appended ones stay as the selection wrote them."""
    r = rnd
    i16 = lambda x: x.cpu().view(torch.int16).numpy()  # noqa: E731  (bf16 bytes, compared exactly)
    k, v = i16(r.k[LC]), i16(r.v[LC])
    pre = r.pre[0]
    lens = r.kv_len.numpy().astype(np.int64)                  # the inputs
    dlen = np.minimum(r.K, lens)                              # K_eff: the selection's length
    assert np.array_equal(pre["lengths"][LC, 0].cpu().numpy(), lens)
    assert np.array_equal(pre["lengths"][LC, 1].cpu().numpy(), dlen)
    kd = np.zeros(tuple(pre["kd"].shape), dtype=np.int16)   # the oracle appends into its own cache
    vd = np.zeros_like(kd)
    sel_k, sel_v = i16(pre["kd"]), i16(pre["vd"])
    clear = np.ones(r.B, dtype=bool)
    for i in range(2):
        _, ref, c = _oracle_round(r, i)
        gpu_nacc = r.post[i]["nacc"].cpu().numpy()
        assert np.array_equal(gpu_nacc[c], ref["num_accepted"][c])   # unambiguous decisions agree
        clear &= gpu_nacc == ref["num_accepted"]
        assert clear.mean() >= 0.9, clear.mean()
        lens, kd, vd, dlen, bad = ref_commit(lens, ref["num_accepted"], r.gamma, k, v, kd, vd, dlen)
        assert not bad.any()
        after = r.pre[i + 1]
        g = after["lengths"].cpu().numpy()                    # [layers, 2, B]
        assert np.array_equal(g[:, :, :], np.broadcast_to(g[LC], g.shape))
        assert np.array_equal(g[LC, 0][clear], lens[clear])
        assert np.array_equal(g[LC, 1][clear], dlen[clear])
        gk, gv = i16(after["kd"]), i16(after["vd"])
        for b in np.nonzero(clear)[0]:
            lo = int(min(r.K, int(r.kv_len[b])))
            hi = int(dlen[b])
            assert np.array_equal(gk[b, :, lo:hi], kd[b, :, lo:hi]) and np.array_equal(gv[b, :, lo:hi], vd[b, :, lo:hi])
            assert np.array_equal(gk[b, :, :lo], sel_k[b, :, :lo]) and np.array_equal(gv[b, :, :lo], sel_v[b, :, :lo])


def test_second_round_attention_over_committed_state(rnd):
    """Round 2 reads what round 1 committed: verify over the rolled-back cache, draft attention
    over the draft cache with the kept rows appended.  Compared with the oracle on the oracle's
    committed state (lengths and draft rows), for sequences whose round-1 count the GPU shares."""
    r = rnd
    G, D = r.Hq // r.Hkv, r.D
    scale = 1.0 / math.sqrt(D)
    _, ref1, _ = _oracle_round(r, 0)
    clear = r.post[0]["nacc"].cpu().numpy() == ref1["num_accepted"]
    lens0 = r.kv_len.numpy()
    bs = [b for b in (0, 7, 31) if clear[b]]
    assert bs
    o = r.post[1]
    for b in bs:
        n = int(ref1["num_accepted"][b])
        L1 = int(lens0[b]) - (r.gamma - n)          # the oracle's rollback of round 1
        first = int(lens0[b]) - r.T
        for h in (0, r.Hkv - 1):
            hs = slice(h * G, (h + 1) * G)
            ref, ref_lse = ref_attention(r.q[LC][b:b + 1, :, hs], r.k[LC][b:b + 1, h:h + 1, :L1],
                                         r.v[LC][b:b + 1, h:h + 1, :L1], torch.tensor([L1]), scale)
            assert_attention_close(o["vout"][LC, b:b + 1, :, hs], ref, "round-2 verify b%d h%d" % (b, h))
            # the draft cache of round 2: the oracle's selected rows, then the n + 1 rows round 1
            # kept (compared where the GPU kept the same rows)
            ref_idx, pooled, kth = _oracle_selection(r, LC, b, h)
            got = r.sel[LC]["sel_idx"][b, h].cpu().numpy()[:r.K]
            if set(got.tolist()) != set(np.asarray(ref_idx).tolist()):
                continue
            k_sel, v_sel = _oracle_draft_cache(r, LC, b, h, ref_idx)
            dl = len(ref_idx)
            kd = torch.cat([k_sel[0, 0], r.k[LC][b, h, first:first + n + 1].cpu()])[None, None]
            vd = torch.cat([v_sel[0, 0], r.v[LC][b, h, first:first + n + 1].cpu()])[None, None]
            for s in range(r.gamma):
                rd, rl = ref_draft(r.qd[LC][s][b:b + 1, None, hs], kd, vd, torch.tensor([dl + n + 1]), scale)
                assert_attention_close(o["dout"][LC, s, b:b + 1, hs], rd[:, 0], "round-2 draft b%d s%d" % (b, s))


def test_round_graph_replay_is_identical(rnd):
    """A CUDA graph of the round that first restores the lengths replays round 1 exactly."""
    r = rnd
    r.u.copy_(r.post[0]["u"])
    ref = r.post[0]
    r.capture(restore=True)
    r.vout.zero_()
    r.out_tok.fill_(-9)
    r.replay()
    torch.cuda.synchronize()
    assert torch.equal(r.out_tok, ref["out_tok"]) and torch.equal(r.nacc, ref["nacc"])
    assert torch.equal(r.lengths, r.pre[1]["lengths"])
    # the 4-warp merge inside a CTA adds in shared memory in arrival order: equal up to rounding
    torch.testing.assert_close(r.vout, ref["vout"], rtol=1e-5, atol=1e-6)
    torch.testing.assert_close(r.dout, ref["dout"], rtol=1e-5, atol=1e-6)
    r.replay()
    torch.cuda.synchronize()
    assert torch.equal(r.out_tok, ref["out_tok"]) and torch.equal(r.lengths, r.pre[1]["lengths"])


def test_programmatic_launch_round_equals_plain_launch_round(rnd):
    """The same round (from the same restored state) with kernels launched with programmatic
    stream serialization (the default) and plainly gives the same tokens, lengths and committed
    draft rows, and attention outputs equal up to the arrival-order rounding of a CTA's merge."""
    from long_context_speculative_split_gb300 import mgd
    r = rnd
    r.u.copy_(r.post[0]["u"])
    outs = []
    for pdl in (True, False):
        mgd.mgd_set_programmatic_launch(pdl)
        try:
            r.restore()
            r.run()
            torch.cuda.synchronize()
        finally:
            mgd.mgd_set_programmatic_launch(True)
        outs.append(_snap(r))
    a, b = outs
    for name in ("tok", "out_tok", "nacc", "lengths", "kd", "vd"):
        assert torch.equal(a[name], b[name]), name
    assert torch.equal(a["out_tok"], r.post[0]["out_tok"])
    torch.testing.assert_close(a["vout"], b["vout"], rtol=1e-5, atol=1e-6)
    torch.testing.assert_close(a["dout"], b["dout"], rtol=1e-5, atol=1e-6)
