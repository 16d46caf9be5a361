"""Host logic of the synthetic workload generators (CPU only)."""
import torch

from long_context_speculative_split_gb300 import workloads as wl


def test_configs_have_llama_shapes():
    for name in ("b32_ctx8k", "b128_ctx32k", "ragged_b256_ctx4k_64k", "round_b32_ctx16k_32layers"):
        c = wl.WORKLOADS[name]
        assert (c["Hq"], c["Hkv"], c["D"], c["V"]) == (32, 8, 128, 128256)
    assert wl.WORKLOADS["b128_ctx32k"]["B"] == 128 and wl.WORKLOADS["b128_ctx32k"]["lens"] == 32768 and wl.WORKLOADS["b128_ctx32k"]["gamma"] == 4


def test_ragged_lengths_are_seeded_and_in_range():
    c = wl.WORKLOADS["ragged_b256_ctx4k_64k"]
    a, b = wl.lengths(c, 0), wl.lengths(c, 0)
    assert torch.equal(a, b)
    assert int(a.min()) >= 4096 and int(a.max()) <= 65536 and a.numel() == 256
    assert not torch.equal(a, wl.lengths(c, 1))


def test_heavy_hitters_exact_count_and_scale():
    c = dict(wl.WORKLOADS["b32_ctx8k"], B=3, Hkv=2, lens=(300, 900), hh=0.01, D=64)
    kv_len = wl.lengths(c, 0)
    cap = 900
    k, v = wl.kv_cache(c, "cpu", kv_len=kv_len, cap=cap)
    c0 = dict(c, hh=0.0)
    k0, v0 = wl.kv_cache(c0, "cpu", kv_len=kv_len, cap=cap)
    assert torch.equal(v, v0)
    changed = (k != k0).any(dim=-1)            # [B, Hkv, cap]
    for b in range(3):
        n = int(round(0.01 * int(kv_len[b])))
        for h in range(2):
            rows = changed[b, h].nonzero().flatten()
            assert rows.numel() == n or (rows.numel() < n and n > 0)   # a zero row stays zero when scaled
            assert rows.numel() == 0 or int(rows.max()) < int(kv_len[b])
            assert torch.equal(k[b, h, rows].float(), 8 * k0[b, h, rows].float())


def test_generators_are_deterministic_and_distinct():
    c = wl.WORKLOADS["tiny_b2"]
    q1, q2 = wl.queries(c, "cpu"), wl.queries(c, "cpu")
    assert torch.equal(q1, q2) and q1.shape == (2, 4, 4, 64) and q1.dtype == torch.float32
    assert not torch.equal(wl.window_queries(c, "cpu")[:, :4], q1)
    t, d = wl.logits(c, "cpu")
    assert t.shape == (2, 4, 1000) and d.shape == (2, 3, 1000)
    u = wl.uniforms(c, "cpu")
    assert u.shape == (2, 4, 3) and float(u.min()) >= 0.0 and float(u.max()) < 1.0
    c2 = dict(wl.WORKLOADS["b32_ctx8k"], B=2, V=50)
    t2, d2 = wl.logits(c2, "cpu")
    assert float((d2 - t2[:, :3]).std()) < 0.6 and float(t2.std()) > 2.5


def test_round_sigma_matches_its_calibration():
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "round_sigma.json")))
    assert wl.WORKLOADS["round_b32_ctx16k_32layers"]["sigma_n"] == g["sigma_n"]
    assert abs(g["alpha_at_sigma_n"] - 0.9) < 1e-6
