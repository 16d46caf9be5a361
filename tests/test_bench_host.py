"""Host-side pieces of bench.py that need no GPU: the attention-only speedup model (the MagicDec
notes' quick-read summary, Eq. 2 with Eq. 3's draft cost) against its closed forms, and the rule
that a recorded DRAM-traffic figure is reported only while the kernel source it was captured on
is unchanged."""
import hashlib
import json
import os
import shutil

import pytest

import bench


def test_speedup_model_closed_forms():
    # free drafting and selection, verify as cheap as decode: the speedup is Omega itself
    out = bench.speedup_model(t_decode=2.0, t_verify=2.0, t_draft=0.0, t_select=0.0, gamma=4)
    for alpha in (0.8, 0.9):
        om = sum(alpha ** i for i in range(5))  # 1 + a + ... + a^4 = (1 - a^5) / (1 - a)
        blk = out["alpha_%.1f" % alpha]
        assert blk["omega"] == pytest.approx(om, rel=1e-12)
        assert blk["speedup_selection_amortised"] == pytest.approx(om, rel=1e-12)
        assert blk["speedup_selection_every_round"] == pytest.approx(om, rel=1e-12)
        assert blk["ms_per_token"] == pytest.approx(2.0 / om, rel=1e-12)
    # a draft step costing a decode step and a selection costing another: T_T * Omega / ((gamma + 1) T_T + T_T)
    out = bench.speedup_model(t_decode=1.0, t_verify=1.0, t_draft=1.0, t_select=1.0, gamma=3)
    om = 1 + 0.9 + 0.81 + 0.729
    assert out["alpha_0.9"]["speedup_selection_amortised"] == pytest.approx(om / 4.0, rel=1e-12)
    assert out["alpha_0.9"]["speedup_selection_every_round"] == pytest.approx(om / 5.0, rel=1e-12)
    assert out["alpha_0.9"]["round_ms"] == pytest.approx(4.0)
    assert out["T_V_over_T_T"] == 1.0 and out["T_D_over_T_T"] == 1.0


def test_recorded_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "verify_attention_traffic.json")))
    src_path = os.path.join(bench.ROOT, "long_context_speculative_split_gb300", "csrc", "attn_tc.cu")
    current = hashlib.sha256(open(src_path, "rb").read()).hexdigest()[:16] == rec["kernel_source_sha256_16"]
    assert bench.load_traffic("b128_ctx32k") == (rec["b128_ctx32k"] if current else None)
    assert rec["b128_ctx32k"] >= 17179869184  # at least the algorithmic K+V bytes of one launch
    # a copy of the tree whose kernel source differs: no traffic figure
    root = tmp_path / "repo"
    (root / "profiles").mkdir(parents=True)
    (root / "long_context_speculative_split_gb300" / "csrc").mkdir(parents=True)
    shutil.copy(os.path.join(bench.ROOT, "profiles", "verify_attention_traffic.json"), root / "profiles")
    src = open(os.path.join(bench.ROOT, "long_context_speculative_split_gb300", "csrc", "attn_tc.cu")).read()
    (root / "long_context_speculative_split_gb300" / "csrc" / "attn_tc.cu").write_text(src + "\n// changed\n")
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.load_traffic("b128_ctx32k") is None
    (root / "long_context_speculative_split_gb300" / "csrc" / "attn_tc.cu").write_text(src)
    assert bench.load_traffic("b128_ctx32k") == (rec["b128_ctx32k"] if current else None)
    assert bench.load_traffic("no_such_workload") is None
