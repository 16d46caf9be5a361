"""GPU parity of verify and draft attention (C ABI via the binding) against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

from _parity import Guarded, assert_attention_close, assert_lse_close, check_guards, gpu_or_skip, poison_, to64
from long_context_speculative_split_gb300 import mgd, ops
from long_context_speculative_split_gb300 import workloads as wl
from oracle.attention import attention as ref_attention
from oracle.attention import draft_attention as ref_draft

pytestmark = pytest.mark.gpu


def _case(B, T, Hq, Hkv, D, lens, cap, seed, dtype=torch.bfloat16, hh=True, poison_pad=False):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, T, Hq, D), generator=g).to(dtype)
    k = torch.randn((B, Hkv, cap, D), generator=g)
    v = torch.randn((B, Hkv, cap, D), generator=g)
    if hh:  # a few heavy-hitter keys per head
        for b in range(B):
            idx = torch.randperm(lens[b], generator=g)[: max(1, lens[b] // 100)]
            k[b, :, idx] *= 8
    k, v = k.to(dtype), v.to(dtype)
    if poison_pad:  # rows past each sequence's length hold NaN: no result may ever see them
        for b in range(B):
            poison_(k[b, :, lens[b]:])
            poison_(v[b, :, lens[b]:])
    return q, k, v, torch.tensor(lens, dtype=torch.int32)


def _guarded_attention(fn, q, B, T, Hq, D, dev, **kw):
    """Run an attention call with its out and lse between poisoned guard regions; checks the
    guards and that every element was written."""
    o = Guarded((B, T, Hq, D) if T else (B, Hq, D), torch.float32, dev)
    l = Guarded((B, T, Hq) if T else (B, Hq), torch.float32, dev)
    out, lse = fn(out=o.t, lse=l.t, **kw)
    torch.cuda.synchronize()
    check_guards(out=o, lse=l)
    assert bool(torch.isfinite(o.t).all()) and bool(torch.isfinite(l.t).all()), "an output element was not written"
    return out, lse


CASES = [
    # B, T, Hq, Hkv, D, lens, cap  (few pairs: one wave of whole-sequence units)
    (2, 4, 32, 8, 128, [1000, 77], 1000),          # G*T = 16 rows
    (3, 5, 32, 8, 128, [4101, 64, 129], 4101),     # 20 rows, ragged tails, one-tile and tile+1
    (2, 1, 8, 2, 128, [513, 1], 513),              # draft form, a single key
    (2, 3, 32, 8, 64, [300, 3], 300),              # head_dim 64, kv_len == T
    (1, 8, 16, 4, 128, [2000], 2048),              # 32 rows (four n8 tiles)
    (2, 5, 64, 8, 128, [700, 650], 700),           # 40 rows -> two row groups
    (2, 2, 4, 4, 128, [5000, 4999], 5000),         # MHA (G=1)
    (1, 4, 32, 8, 128, [64], 64),                  # exactly one tile
    (1, 4, 32, 8, 128, [65], 128),                 # one key into the second tile
    (2, 17, 32, 8, 128, [900, 17], 900),           # gamma 16: 68 rows -> three row groups (32, 32, 4)
    (2, 1, 8, 2, 64, [513, 1], 513),               # head_dim 64: one row tile
    (2, 5, 32, 8, 64, [1000, 333], 1000),          # head_dim 64: 20 rows, P V in float16
    (1, 8, 16, 4, 64, [2000], 2048),               # head_dim 64: 32 rows (four n8 tiles)
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%d_T%d_G%d_D%d_L%s" % (c[0], c[1], c[2] // c[3], c[4],
                                                                                  "-".join(map(str, c[5]))))
def test_verify_bf16_matches_oracle(case):
    dev = gpu_or_skip()
    B, T, Hq, Hkv, D, lens, cap = case
    q, k, v, kv_len = _case(B, T, Hq, Hkv, D, lens, cap, seed=sum(lens) + T, poison_pad=True)
    out, lse = _guarded_attention(lambda **kw: ops.verify_attn(q.to(dev), k.to(dev), v.to(dev), kv_len.to(dev), **kw),
                                  q, B, T, Hq, D, dev)
    ref, ref_lse = ref_attention(q, k, v, kv_len, 1.0 / math.sqrt(D))
    assert_attention_close(out, ref)
    assert_lse_close(lse, ref_lse)


@pytest.mark.parametrize("B,T,Hq,Hkv", [(40, 4, 32, 8), (82, 2, 4, 4)], ids=["G4_T4_320pairs", "MHA_T2_328pairs"])
def test_verify_split_units_and_merges_match_oracle(B, T, Hq, Hkv):
    """More (sequence, KV head) pairs than CTA slots on a 152-SM part: short units of 256 keys,
    several per sequence (ragged lengths, ragged last units), merged by the last CTA of each
    sequence; every output is compared with the oracle."""
    dev = gpu_or_skip()
    D, cap = 128, 1000
    g = torch.Generator().manual_seed(B)
    lens = torch.randint(T, cap + 1, (B,), generator=g).tolist()
    lens[0] = cap
    q, k, v, kv_len = _case(B, T, Hq, Hkv, D, lens, cap, seed=B + T, poison_pad=True)
    out, lse = _guarded_attention(lambda **kw: ops.verify_attn(q.to(dev), k.to(dev), v.to(dev), kv_len.to(dev), **kw),
                                  q, B, T, Hq, D, dev)
    ref, ref_lse = ref_attention(q, k, v, kv_len, 1.0 / math.sqrt(D))
    assert_attention_close(out, ref)
    assert_lse_close(lse, ref_lse)


@pytest.mark.parametrize("vmax", [1e-3, 6.0e4], ids=["tiny_V", "V_near_f16_max"])
def test_verify_many_rows_across_the_float16_range_of_v(vmax):
    """With more than 16 query rows a KV head the P V product runs in float16: V entries of
    any magnitude the header allows (down to the float16 subnormals, up to 60000 of the
    65504 limit) still meet the tolerance, relative to the largest |V|."""
    dev = gpu_or_skip()
    B, T, Hq, Hkv, D, lens, cap = 2, 5, 32, 8, 128, [3000, 777], 3000
    q, k, v, kv_len = _case(B, T, Hq, Hkv, D, lens, cap, seed=41)
    v = (v.float() * (vmax / v.float().abs().max())).to(torch.bfloat16)
    out, _ = ops.verify_attn(q.to(dev), k.to(dev), v.to(dev), kv_len.to(dev))
    torch.cuda.synchronize()
    ref, _ = ref_attention(q, k, v, kv_len, 1.0 / math.sqrt(D))
    g = to64(out)
    assert np.all(np.isfinite(g))
    scale = float(v.float().abs().max())
    assert np.abs(g - ref).max() <= 2e-2 * scale / 4.0
    assert np.linalg.norm(g - ref) / np.linalg.norm(ref) <= 1e-3


def _nonfinite_cells(out):
    return {tuple(i) for i in torch.nonzero(~torch.isfinite(out.cpu())).tolist()}


@pytest.mark.parametrize("B,lens,cap", [(2, [3000, 777], 3000), (40, None, 1000)],
                         ids=["whole_sequence_units", "split_units_merged"])
def test_v_beyond_float16_range_is_confined_to_the_outputs_that_read_it(B, lens, cap):
    """The float16 P V path (G = 4, T = 5: 20 rows a KV head) needs |v| <= 65504.  One V entry
    past it makes exactly the outputs that sum it non-finite (the G heads of that KV head, that
    dimension, every verify row), both where a unit covers the whole sequence and where the last
    CTA merges partials; every other output still matches the oracle."""
    dev = gpu_or_skip()
    T, Hq, Hkv, D = 5, 32, 8, 128
    G = Hq // Hkv
    if lens is None:
        g = torch.Generator().manual_seed(3)
        lens = torch.randint(T, cap + 1, (B,), generator=g).tolist()
        lens[1] = cap  # four 256-key units on a 152-SM part
    q, k, v, kv_len = _case(B, T, Hq, Hkv, D, lens, cap, seed=B + 100)
    b, h, j, d = 1, 3, 2, 7
    v_bad = v.clone()
    v_bad[b, h, j, d] = 1.0e5  # a bfloat16 value; float16 tops out at 65504
    out, _ = ops.verify_attn(q.to(dev), k.to(dev), v_bad.to(dev), kv_len.to(dev))
    expect = {(b, t, hq, d) for t in range(T) for hq in range(h * G, (h + 1) * G)}
    assert _nonfinite_cells(out) == expect
    ref, _ = ref_attention(q, k, v, kv_len, 1.0 / math.sqrt(D))
    keep = torch.ones(out.shape, dtype=torch.bool)
    keep[b, :, h * G:(h + 1) * G] = False
    assert_attention_close(out.cpu()[keep], ref[keep.numpy()])


def test_v_beyond_float16_range_is_finite_on_the_bfloat16_path():
    """At 16 or fewer rows a KV head (here T = 4, G = 4) P V stays in bfloat16 hi + lo parts,
    which hold a V entry of 1e5: the outputs are finite and match the oracle."""
    dev = gpu_or_skip()
    B, T, Hq, Hkv, D, lens, cap = 2, 4, 32, 8, 128, [3000, 777], 3000
    q, k, v, kv_len = _case(B, T, Hq, Hkv, D, lens, cap, seed=104)
    v[1, 3, 2, 7] = 1.0e5
    out, _ = ops.verify_attn(q.to(dev), k.to(dev), v.to(dev), kv_len.to(dev))
    ref, _ = ref_attention(q, k, v, kv_len, 1.0 / math.sqrt(D))
    g = to64(out)
    assert np.all(np.isfinite(g))
    # error relative to the largest |V| (the P V sum carries it)
    assert np.abs(g - ref).max() <= 2e-2 * 1.0e5 / 4.0


def test_verify_bf16_output_dtype():
    dev = gpu_or_skip()
    q, k, v, kv_len = _case(2, 4, 32, 8, 128, [900, 333], 900, seed=5)
    out, _ = ops.verify_attn(q.to(dev), k.to(dev), v.to(dev), kv_len.to(dev), out_dtype=torch.bfloat16)
    ref, _ = ref_attention(q, k, v, kv_len, 1.0 / math.sqrt(128))
    g = to64(out)
    # bf16 output adds its own rounding (2^-9 relative): checked against that bound
    assert np.abs(g - ref).max() <= 2e-2
    assert np.linalg.norm(g - ref) / np.linalg.norm(ref) <= 5e-3


def test_verify_float32_tiny_config_full():
    dev = gpu_or_skip()
    c = wl.WORKLOADS["tiny_b2"]
    kv_len = wl.lengths(c)
    k, v = wl.kv_cache(c, dev, kv_len=kv_len)
    q = wl.queries(c, dev)
    out, lse = ops.verify_attn(q, k, v, kv_len.to(dev))
    ref, ref_lse = ref_attention(q, k, v, kv_len, 1.0 / math.sqrt(c["D"]))
    assert_attention_close(out, ref)
    assert_lse_close(lse, ref_lse)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32_out", "bf16_out"])
def test_verify_float32_head_dim_128(out_dtype):
    """The float32 CUDA-core kernel at head_dim 128, 20 rows a KV head (three passes of 8 rows),
    ragged lengths down to kv_len = T + 4, both output types."""
    dev = gpu_or_skip()
    B, T, Hq, Hkv, D, lens, cap = 2, 5, 32, 8, 128, [700, 9], 700
    q, k, v, kv_len = _case(B, T, Hq, Hkv, D, lens, cap, seed=77, dtype=torch.float32)
    out, lse = ops.verify_attn(q.to(dev), k.to(dev), v.to(dev), kv_len.to(dev), out_dtype=out_dtype)
    ref, ref_lse = ref_attention(q, k, v, kv_len, 1.0 / math.sqrt(D))
    if out_dtype == torch.float32:
        assert_attention_close(out, ref)
    else:  # bf16 output adds its own rounding (2^-9 relative)
        g = to64(out)
        assert np.abs(g - ref).max() <= 2e-2 and np.linalg.norm(g - ref) / np.linalg.norm(ref) <= 5e-3
    assert_lse_close(lse, ref_lse)


def test_draft_float32_tiny_config_full():
    dev = gpu_or_skip()
    c = wl.WORKLOADS["tiny_b2"]
    kv_len = wl.lengths(c)
    k, v = wl.kv_cache(c, dev, kv_len=kv_len)
    qd = wl.draft_queries(c, dev)
    dlen = torch.tensor([64, 37], dtype=torch.int32)
    kd, vd = k[:, :, :64].contiguous(), v[:, :, :64].contiguous()
    out, lse = ops.draft_attn(qd, kd, vd, dlen.to(dev))
    ref, ref_lse = ref_draft(qd, kd, vd, dlen, 1.0 / math.sqrt(c["D"]))
    assert_attention_close(out, ref[:, 0])
    assert_lse_close(lse, ref_lse[:, 0])


@pytest.mark.parametrize("lens,cap,D", [([1024, 700, 1], 1024, 128), ([516, 512, 64, 65], 516, 128),
                                        ([516, 512, 64, 65], 516, 64)])
def test_draft_bf16_matches_oracle(lens, cap, D):
    dev = gpu_or_skip()
    B = len(lens)
    q, k, v, dlen = _case(B, 1, 32, 8, D, lens, cap, seed=cap + D, poison_pad=True)
    out, lse = _guarded_attention(lambda **kw: ops.draft_attn(q.to(dev), k.to(dev), v.to(dev), dlen.to(dev), **kw),
                                  q, B, 0, 32, D, dev)
    ref, ref_lse = ref_draft(q, k, v, dlen, 1.0 / math.sqrt(D))
    assert_attention_close(out, ref[:, 0])
    assert_lse_close(lse, ref_lse[:, 0])


def test_empty_batch_is_a_noop():
    dev = gpu_or_skip()
    q = torch.empty((0, 4, 32, 128), dtype=torch.bfloat16, device=dev)
    k = torch.empty((0, 8, 64, 128), dtype=torch.bfloat16, device=dev)
    out, _ = ops.verify_attn(q, k, k, torch.empty(0, dtype=torch.int32, device=dev))
    assert out.shape == (0, 4, 32, 128)


def test_out_of_range_length_raises_device_flag_and_spares_others():
    dev = gpu_or_skip()
    q, k, v, kv_len = _case(2, 4, 32, 8, 128, [500, 500], 500, seed=9)
    bad = torch.tensor([500, 9999], dtype=torch.int32)
    ws = ops.workspace(mgd.mgd_verify_workspace_size(2, 4, 32, 8, 128, 500), dev)
    out, _ = ops.verify_attn(q.to(dev), k.to(dev), v.to(dev), bad.to(dev), ws=ws)
    flags = mgd.mgd_workspace_errors(ws)
    assert flags & mgd.MGD_DEVERR_KV_LEN
    ref, _ = ref_attention(q[:1], k[:1], v[:1], kv_len[:1], 1.0 / math.sqrt(128))
    assert_attention_close(out[:1], ref)
    # a clean call clears the word
    ops.verify_attn(q.to(dev), k.to(dev), v.to(dev), kv_len.to(dev), ws=ws)
    assert mgd.mgd_workspace_errors(ws) == 0


def _sampled_pairs(kv_len, Hkv, n=3, seed=0):
    L = kv_len.numpy()
    rng = np.random.default_rng(seed)
    # longest, shortest, and the last sequence (the end of the persistent unit order)
    bs = {int(np.argmax(L)), int(np.argmin(L)), len(L) - 1}
    while len(bs) < n:
        bs.add(int(rng.integers(len(L))))
    return [(b, int(rng.integers(Hkv))) for b in sorted(bs)]


@pytest.mark.parametrize("name", ["b32_ctx8k", "b128_ctx32k", "ragged_b256_ctx4k_64k"])
def test_verify_full_size_sampled(name):
    """Full-size workload in the benchmark's launch configuration; sampled (sequence, KV head) pairs."""
    dev = gpu_or_skip()
    c = wl.WORKLOADS[name]
    kv_len = wl.lengths(c)
    k, v = wl.kv_cache(c, dev, kv_len=kv_len)
    q = wl.queries(c, dev)
    out, lse = ops.verify_attn(q, k, v, kv_len.to(dev))
    torch.cuda.synchronize()
    assert bool(torch.isfinite(out).all()) and bool(torch.isfinite(lse).all())
    G, D = c["Hq"] // c["Hkv"], c["D"]
    for b, h in _sampled_pairs(kv_len, c["Hkv"]):
        L = int(kv_len[b])
        ref, ref_lse = ref_attention(q[b:b + 1, :, h * G:(h + 1) * G], k[b:b + 1, h:h + 1, :L],
                                     v[b:b + 1, h:h + 1, :L], kv_len[b:b + 1], 1.0 / math.sqrt(D))
        assert_attention_close(out[b:b + 1, :, h * G:(h + 1) * G], ref, "out[b=%d,h=%d]" % (b, h))
        assert_lse_close(lse[b:b + 1, :, h * G:(h + 1) * G], ref_lse)
    del k, v
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["b32_ctx8k", "b128_ctx32k"])
def test_draft_full_size_sampled(name):
    dev = gpu_or_skip()
    c = wl.WORKLOADS[name]
    K = c["K"]
    dlen = torch.full((c["B"],), K, dtype=torch.int32)
    kd, vd = wl.kv_cache(c, dev, kv_len=dlen, cap=K, layer=7)
    qd = wl.draft_queries(c, dev)
    out, lse = ops.draft_attn(qd, kd, vd, dlen.to(dev))
    torch.cuda.synchronize()
    assert bool(torch.isfinite(out).all())
    G, D = c["Hq"] // c["Hkv"], c["D"]
    for b, h in _sampled_pairs(dlen, c["Hkv"]):
        ref, ref_lse = ref_draft(qd[b:b + 1, :, h * G:(h + 1) * G], kd[b:b + 1, h:h + 1], vd[b:b + 1, h:h + 1],
                                 dlen[b:b + 1], 1.0 / math.sqrt(D))
        assert_attention_close(out[b:b + 1, h * G:(h + 1) * G], ref[:, 0])
        assert_lse_close(lse[b:b + 1, h * G:(h + 1) * G], ref_lse[:, 0])


def test_verify_five_rows_split_units():
    """The batch-128 x 32k verify shape (gamma 4: 20 rows per KV head, three n8 row tiles, every
    sequence split into units with an in-kernel merge) at batch 64 x 16k (2.1 GB of KV), sampled
    pairs against the oracle.  Also the small case the verify kernel's counters are captured on."""
    dev = gpu_or_skip()
    c = dict(wl.WORKLOADS["b128_ctx32k"], B=64, lens=16384)
    kv_len = wl.lengths(c)
    k, v = wl.kv_cache(c, dev, kv_len=kv_len)
    q = wl.queries(c, dev)
    plan_units = mgd.mgd_verify_workspace_size(c["B"], c["gamma"] + 1, c["Hq"], c["Hkv"], c["D"], 16384)
    assert plan_units > 256  # split plan: partials in the workspace
    out, lse = ops.verify_attn(q, k, v, kv_len.to(dev))
    torch.cuda.synchronize()
    assert bool(torch.isfinite(out).all()) and bool(torch.isfinite(lse).all())
    G, D = c["Hq"] // c["Hkv"], c["D"]
    for b, h in _sampled_pairs(kv_len, c["Hkv"], n=4, seed=5):
        ref, ref_lse = ref_attention(q[b:b + 1, :, h * G:(h + 1) * G], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1],
                                     kv_len[b:b + 1], 1.0 / math.sqrt(D))
        assert_attention_close(out[b:b + 1, :, h * G:(h + 1) * G], ref, "out[b=%d,h=%d]" % (b, h))
        assert_lse_close(lse[b:b + 1, :, h * G:(h + 1) * G], ref_lse)
    del k, v
    torch.cuda.empty_cache()


def _torch_attention(q, k, v, L, scale):
    """Float32 torch math on the GPU for one sequence: q [T, Hq, D], k/v [Hkv, L, D] -> [T, Hq, D]."""
    T, Hq, D = q.shape
    Hkv = k.shape[0]
    G = Hq // Hkv
    kk = k[:, :L].float().repeat_interleave(G, dim=0)          # [Hq, L, D]
    vv = v[:, :L].float().repeat_interleave(G, dim=0)
    s = torch.einsum("thd,hld->htl", q.float(), kk) * scale     # [Hq, T, L]
    pos = torch.arange(L, device=q.device)
    lim = L - T + torch.arange(T, device=q.device)
    s = s.masked_fill(pos[None, None, :] > lim[None, :, None], float("-inf"))
    return torch.einsum("htl,hld->thd", torch.softmax(s, dim=-1), vv)


def test_verify_ragged_every_sequence():
    """Ragged batch 256 x U[4096, 65536] (the benchmark's launch configuration): every
    sequence is compared with the float64 oracle on one of its KV heads (head b % Hkv, so all
    heads are covered across the batch), so no unit of the persistent schedule can go missing
    unnoticed.  As an extra, every head of every sequence is checked against float32 torch
    math on the GPU."""
    dev = gpu_or_skip()
    c = wl.WORKLOADS["ragged_b256_ctx4k_64k"]
    kv_len = wl.lengths(c)
    k, v = wl.kv_cache(c, dev, kv_len=kv_len)
    q = wl.queries(c, dev)
    out, lse = ops.verify_attn(q, k, v, kv_len.to(dev))
    torch.cuda.synchronize()
    scale = 1.0 / math.sqrt(c["D"])
    G, Hkv = c["Hq"] // c["Hkv"], c["Hkv"]
    worst_abs, num, den = 0.0, 0.0, 0.0
    for b in range(c["B"]):
        L, h = int(kv_len[b]), b % Hkv
        hs = slice(h * G, (h + 1) * G)
        ref, ref_lse = ref_attention(q[b:b + 1, :, hs], k[b:b + 1, h:h + 1, :L], v[b:b + 1, h:h + 1, :L],
                                     kv_len[b:b + 1], scale)
        assert_attention_close(out[b:b + 1, :, hs], ref, "out[b=%d,h=%d]" % (b, h))
        assert_lse_close(lse[b:b + 1, :, hs], ref_lse)
        t = _torch_attention(q[b], k[b], v[b], L, scale)
        d = (out[b] - t).double()
        worst_abs = max(worst_abs, float(d.abs().max()))
        num += float((d ** 2).sum())
        den += float((t.double() ** 2).sum())
    assert worst_abs <= 2e-2 and (num / den) ** 0.5 <= 1e-3, (worst_abs, (num / den) ** 0.5)
    del k, v
    torch.cuda.empty_cache()


def test_draft_split_units_match_oracle():
    """512 (sequence, KV head) pairs with 2048-row draft caches: on a 152-SM part the planner
    cuts every pair into two 1024-key units whose partials are merged (ragged second units of
    176..1024 keys); every output is compared with the oracle."""
    dev = gpu_or_skip()
    B, Hq, Hkv, D, cap = 64, 32, 8, 128, 2048
    g = torch.Generator().manual_seed(77)
    lens = torch.randint(1200, cap + 1, (B,), generator=g).tolist()
    q, k, v, dlen = _case(B, 1, Hq, Hkv, D, lens, cap, seed=78, poison_pad=True)
    out, lse = _guarded_attention(lambda **kw: ops.draft_attn(q.to(dev), k.to(dev), v.to(dev), dlen.to(dev), **kw),
                                  q, B, 0, Hq, D, dev)
    ref, ref_lse = ref_draft(q, k, v, dlen, 1.0 / math.sqrt(D))
    assert_attention_close(out, ref[:, 0])
    assert_lse_close(lse, ref_lse[:, 0])


def test_workspace_reused_across_shapes_and_errors():
    """The attention kernels leave the workspace header ready for the next call (no clearing
    launch): one zero-filled workspace serves, in turn, a split-sequence verify (merge tickets,
    claims past the grid), a draft, a verify that raises a device error and the first verify
    again.  Each result equals the same call on a fresh workspace bit for bit, and each call's
    error word holds its own bits only."""
    dev = gpu_or_skip()
    lens = [int(x) for x in np.random.default_rng(5).integers(1500, 4097, size=40)]
    qa, ka, va, la = (x.to(dev) for x in _case(40, 4, 32, 8, 128, lens, 4096, seed=21))
    qd, kd, vd, ld = (x.to(dev) for x in _case(4, 1, 32, 8, 128, [512, 300, 1, 511], 512, seed=22))
    bad = la.clone()
    bad[7] = 5000  # past the capacity
    need = max(mgd.mgd_verify_workspace_size(40, 4, 32, 8, 128, 4096), mgd.mgd_draft_workspace_size(4, 32, 8, 128, 512))
    ws = ops.workspace(need, dev)

    def verify(kv_len, w):
        return ops.verify_attn(qa, ka, va, kv_len, ws=w)

    def draft(w):
        return ops.draft_attn(qd[:, 0], kd, vd, ld, ws=w)

    fresh_v = verify(la, ops.workspace(need, dev))
    fresh_d = draft(ops.workspace(need, dev))
    fresh_bad = verify(bad, ops.workspace(need, dev))
    torch.cuda.synchronize()
    for _ in range(2):
        out = verify(la, ws)
        assert mgd.mgd_workspace_errors(ws) == 0
        assert torch.equal(out[0], fresh_v[0]) and torch.equal(out[1], fresh_v[1])
        out = draft(ws)
        assert mgd.mgd_workspace_errors(ws) == 0
        assert torch.equal(out[0], fresh_d[0]) and torch.equal(out[1], fresh_d[1])
        out = verify(bad, ws)
        assert mgd.mgd_workspace_errors(ws) == mgd.MGD_DEVERR_KV_LEN
        keep = torch.arange(40, device=dev) != 7
        assert torch.equal(out[0][keep], fresh_bad[0][keep])
    ref, _ = ref_attention(qa[:3].cpu(), ka[:3].cpu(), va[:3].cpu(), la[:3].cpu(), 1.0 / math.sqrt(128))
    assert_attention_close(fresh_v[0][:3], ref)


def test_stale_workspace_is_detected():
    """The attention calls do not clear their workspace header; a header that is not ready
    (not zero-filled, or last used as SnapKV scratch) is detected at the end of the call and
    raises MGD_DEVERR_STALE_WS.  The shape has more (sequence, KV head) pairs than CTA slots,
    so units past the first wave come from the header's work counter."""
    dev = gpu_or_skip()
    lens = [int(x) for x in np.random.default_rng(6).integers(500, 1001, size=40)]
    q, k, v, kv_len = (x.to(dev) for x in _case(40, 4, 32, 8, 128, lens, 1000, seed=31))
    qw = torch.randn((40, 32, 32, 128), generator=torch.Generator().manual_seed(32)).to(torch.bfloat16).to(dev)
    need = max(mgd.mgd_verify_workspace_size(40, 4, 32, 8, 128, 1000),
               mgd.mgd_snapkv_workspace_size(40, 32, 8, 128, 1000, 32))
    fresh = ops.verify_attn(q, k, v, kv_len, ws=ops.workspace(need, dev))
    ws = ops.workspace(need, dev)
    # err[0], err[1], next_unit, next_unit2, seq, claimed, then the 64-bit check-in word (low: id sum,
    # high: id-sum bits 32..39 and the check-in count << 8)
    hdr = ws[:256].view(torch.int32)
    # a stale work counter (small, past every unit); a stale check-in count; stale sums
    for field, value in ((2, 5), (2, 100000), (7, 3 << 8), (7, 1 << 8), (5, 2), (6, 9)):
        ws.zero_()
        hdr[field] = value
        ops.verify_attn(q, k, v, kv_len, ws=ws)
        assert mgd.mgd_workspace_errors(ws) & mgd.MGD_DEVERR_STALE_WS, (field, value)
    # zero-filled again, the same buffer gives the fresh result with no error bits
    ws.zero_()
    out = ops.verify_attn(q, k, v, kv_len, ws=ws)
    assert mgd.mgd_workspace_errors(ws) == 0
    assert torch.equal(out[0], fresh[0]) and torch.equal(out[1], fresh[1])
    # the selection call leaves its header ready too, and checks it the same way
    ws.zero_()
    hdr[2] = 3
    ops.snapkv_select(qw, k, v, kv_len, 32, 7, 128, ws=ws)
    assert mgd.mgd_workspace_errors(ws) & mgd.MGD_DEVERR_STALE_WS
    ws.zero_()
    # a buffer last used by a SnapKV call: detected if its counters were left nonzero,
    # otherwise the call is clean
    ops.snapkv_select(qw, k, v, kv_len, 32, 7, 128, ws=ws)
    torch.cuda.synchronize()
    dirty = bool(hdr[2:4].any()) or bool(hdr[5:8].any())
    out = ops.verify_attn(q, k, v, kv_len, ws=ws)
    flags = mgd.mgd_workspace_errors(ws)
    if dirty:
        assert flags & mgd.MGD_DEVERR_STALE_WS
    else:
        assert flags == 0
        assert torch.equal(out[0], fresh[0]) and torch.equal(out[1], fresh[1])
    ref, _ = ref_attention(q[:2].cpu(), k[:2].cpu(), v[:2].cpu(), kv_len[:2].cpu(), 1.0 / math.sqrt(128))
    assert_attention_close(fresh[0][:2], ref)
