"""The C ABI without a GPU: the library builds, loads, exports every entry point
that include/mgd.h declares, and rejects bad arguments on the host before any
launch (null pointers, shapes, alignment, workspace size)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mgd.h")

FAKE = 1 << 20  # aligned, never dereferenced: every call below fails validation first


@pytest.fixture(scope="module")
def lib():
    from long_context_speculative_split_gb300 import build, mgd
    build.build()
    return mgd.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mgd_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_four_calls():
    names = declared_functions()
    for n in ("mgd_verify_attn", "mgd_draft_attn", "mgd_snapkv_select", "mgd_spec_sample",
              "mgd_verify_workspace_size", "mgd_draft_workspace_size", "mgd_snapkv_workspace_size",
              "mgd_spec_workspace_size", "mgd_status_string", "mgd_last_error", "mgd_workspace_errors"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from long_context_speculative_split_gb300 import mgd
    raw = ctypes.CDLL(mgd.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), name
        assert name in mgd.SIGNATURES, "binding misses " + name


def test_binding_constants_match_the_header():
    """Every enum value and device error bit the header defines has the same value in the
    binding (the names the Python side passes and tests against)."""
    from long_context_speculative_split_gb300 import mgd
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    consts = {name: int(val, 0) for name, val in re.findall(r"#define\s+(MGD_DEVERR_[A-Z_]+)\s+(0x[0-9a-fA-F]+)u", text)}
    for body in re.findall(r"typedef enum \{(.*?)\}", text, flags=re.S):
        consts.update({name: int(val) for name, val in re.findall(r"(MGD_[A-Z0-9_]+)\s*=\s*(\d+)", body)})
    assert "MGD_VERIFY_DRAWN" in consts and "MGD_DEVERR_NOT_DRAWN" in consts
    for name, val in consts.items():
        if hasattr(mgd, name):
            assert getattr(mgd, name) == val, name
    for name in ("MGD_VERIFY", "MGD_DRAW_DRAFT", "MGD_VERIFY_DRAWN", "MGD_DEVERR_KV_LEN", "MGD_DEVERR_SNAP_LEN",
                 "MGD_DEVERR_TOKEN", "MGD_DEVERR_TIMEOUT", "MGD_DEVERR_COMMIT", "MGD_DEVERR_STALE_WS",
                 "MGD_DEVERR_NOT_DRAWN"):
        assert getattr(mgd, name) == consts[name], name


def test_status_strings_and_version(lib):
    from long_context_speculative_split_gb300 import mgd
    for s in range(5):
        assert mgd.mgd_status_string(s).startswith(mgd.status_name(s))
    assert mgd.mgd_version() >= 100


def test_workspace_sizes_are_deterministic_and_grow(lib):
    from long_context_speculative_split_gb300 import mgd
    a = mgd.mgd_verify_workspace_size(128, 5, 32, 8, 128, 32768)
    assert a == mgd.mgd_verify_workspace_size(128, 5, 32, 8, 128, 32768)
    assert a > mgd.mgd_verify_workspace_size(8, 5, 32, 8, 128, 32768) >= 256
    assert mgd.mgd_draft_workspace_size(128, 32, 8, 128, 1024) >= 256
    assert mgd.mgd_snapkv_workspace_size(128, 32, 8, 128, 32768, 32) > 2 * 4 * 128 * 8 * 32768
    assert mgd.mgd_spec_workspace_size(128, 4, 128256) >= 256 + 8 * 128 * 9
    assert mgd.mgd_spec_workspace_size(0, 4, 10) == 256


def _verify(mgd, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, kv_len=FAKE, B=2, T=4, Hq=8, Hkv=2, D=128, kv_cap=1024,
             kv_batch_stride=2 * 1024 * 128, kv_head_stride=1024 * 128, sm_scale=0.1, in_dtype=mgd.MGD_BF16,
             out=FAKE, out_dtype=mgd.MGD_F32, lse=None, ws=FAKE, ws_bytes=1 << 40, stream=0)
    a.update(kw)
    try:
        mgd.mgd_verify_attn(**a)
        return mgd.MGD_OK
    except mgd.MgdError as e:
        return e.status


@pytest.mark.parametrize("kw,status", [
    (dict(D=96), 2), (dict(Hq=6, Hkv=4), 1), (dict(T=0), 1), (dict(T=18), 1), (dict(q=None), 1),
    (dict(kv_len=None), 1), (dict(k=FAKE + 8), 1), (dict(kv_head_stride=100), 1), (dict(kv_batch_stride=1), 1),
    (dict(kv_head_stride=1024 * 128 + 4, kv_batch_stride=2 * (1024 * 128 + 4)), 1), (dict(in_dtype=7), 1),
    (dict(ws_bytes=16), 3), (dict(ws=None), 1), (dict(B=-1), 1)])
def test_verify_rejects_bad_arguments_on_host(lib, kw, status):
    from long_context_speculative_split_gb300 import mgd
    assert _verify(mgd, **kw) == status
    assert mgd.mgd_last_error() != ""


def test_empty_batch_is_a_noop(lib):
    from long_context_speculative_split_gb300 import mgd
    assert _verify(mgd, B=0, q=None, k=None, v=None, kv_len=None, out=None, ws=None) == mgd.MGD_OK


def test_snapkv_rejects_bad_arguments_on_host(lib):
    from long_context_speculative_split_gb300 import mgd

    def call(**kw):
        a = dict(q_win=FAKE, k=FAKE, v=FAKE, kv_len=FAKE, B=2, Hq=8, Hkv=2, D=128, kv_cap=4096,
                 kv_batch_stride=2 * 4096 * 128, kv_head_stride=4096 * 128, W=32, pool=7, K=512, sm_scale=0.1,
                 in_dtype=mgd.MGD_BF16, sel_idx=FAKE, k_draft=FAKE, v_draft=FAKE, draft_cap=512, draft_len=FAKE,
                 scores=None, ws=FAKE, ws_bytes=1 << 40, stream=0)
        a.update(kw)
        try:
            mgd.mgd_snapkv_select(**a)
            return 0
        except mgd.MgdError as e:
            return e.status
    assert call(pool=6) == 1
    assert call(pool=65) == 1
    assert call(K=16) == 1           # K < W
    assert call(draft_cap=100) == 1  # draft_cap < K
    assert call(W=0) == 2 and call(W=65) == 2
    assert call(D=80) == 2
    assert call(ws_bytes=1024) == 3
    assert call(sel_idx=None) == 1


def test_topk_draft_rejects_bad_arguments_on_host(lib):
    from long_context_speculative_split_gb300 import mgd

    def call(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, kv_len=FAKE, B=2, Hq=8, Hkv=2, D=128, kv_cap=4096,
                 kv_batch_stride=2 * 4096 * 128, kv_head_stride=4096 * 128, K=256, sm_scale=0.1,
                 in_dtype=mgd.MGD_BF16, sel_idx=FAKE, k_draft=FAKE, v_draft=FAKE, draft_cap=256, draft_len=FAKE,
                 out=FAKE, out_dtype=mgd.MGD_F32, lse=None, ws=FAKE, ws_bytes=1 << 40, stream=0)
        a.update(kw)
        try:
            mgd.mgd_topk_draft_attn(**a)
            return 0
        except mgd.MgdError as e:
            return e.status
    assert call(K=0) == 1
    assert call(draft_cap=100) == 1   # draft_cap < K
    assert call(D=80) == 2
    assert call(out=None) == 1
    assert call(ws_bytes=1024) == 3
    assert call(B=0, q=None, k=None, v=None, kv_len=None, out=None, ws=None) == 0
    small = mgd.mgd_topk_draft_workspace_size(2, 8, 2, 128, 4096, 256)
    assert small > mgd.mgd_snapkv_workspace_size(2, 8, 2, 128, 4096, 1)
    assert mgd.mgd_topk_draft_workspace_size(2, 8, 2, 128, 8192, 256) > small


def test_spec_sample_rejects_bad_arguments_on_host(lib):
    from long_context_speculative_split_gb300 import mgd

    def call(**kw):
        a = dict(target_logits=FAKE, draft_logits=FAKE, draft_tokens=FAKE, u=FAKE, B=4, gamma=3, V=1000, mode=0,
                 row=-1, out_tokens=FAKE, num_accepted=FAKE, ws=FAKE, ws_bytes=1 << 30, stream=0)
        a.update(kw)
        try:
            mgd.mgd_spec_sample(**a)
            return 0
        except mgd.MgdError as e:
            return e.status
    assert call(gamma=0) == 2 and call(gamma=17) == 2
    assert call(V=0) == 1
    assert call(mode=5) == 1 and call(mode=3) == 1
    assert call(mode=1, row=3) == 1
    assert call(target_logits=None) == 1          # verify needs the target
    assert call(out_tokens=None) == 1
    assert call(mode=2, target_logits=None) == 1  # so does the verify that reuses the draws' statistics
    assert call(mode=2, num_accepted=None) == 1
    assert call(ws_bytes=8) == 3
    assert call(B=0, draft_logits=None) == 0


def test_snapkv_budgets_rejects_bad_arguments_on_host(lib):
    from long_context_speculative_split_gb300 import mgd

    def call(**kw):
        a = dict(q_win=FAKE, k=FAKE, v=FAKE, kv_len=FAKE, B=2, Hq=8, Hkv=2, D=128, kv_cap=1024,
                 kv_batch_stride=2 * 1024 * 128, kv_head_stride=1024 * 128, W=32, pool=7, budgets=FAKE, sm_scale=0.1,
                 in_dtype=0, sel_idx=FAKE, k_draft=FAKE, v_draft=FAKE, draft_cap=256, draft_len=FAKE, scores=None,
                 ws=FAKE, ws_bytes=8, stream=0)
        a.update(kw)
        try:
            mgd.mgd_snapkv_select_budgets(**a)
            return 0
        except mgd.MgdError as e:
            return e.status
    assert call(budgets=None) == 1
    assert call(draft_cap=16) == 1               # below the window
    assert call(ws_bytes=8) == 3                 # the workspace of mgd_snapkv_select
    assert call(B=0, budgets=None) == 0


def test_selftest_rejects_bad_arguments_on_host(lib):
    from long_context_speculative_split_gb300 import mgd

    def call(which=0, ws=FAKE, ws_bytes=mgd.SELFTEST_WS_BYTES):
        try:
            mgd.mgd_selftest_bounded_wait(which, ws, ws_bytes, stream=0)
            return 0
        except mgd.MgdError as e:
            return e.status
    assert call(which=2) == 1 and call(which=-1) == 1
    assert call(ws=None) == 1
    assert call(ws_bytes=mgd.SELFTEST_WS_BYTES - 1) == 3
    assert "MGD_SELFTEST_WS_BYTES %du" % mgd.SELFTEST_WS_BYTES in open(HEADER).read()


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    from long_context_speculative_split_gb300 import mgd
    monkeypatch.setattr(mgd, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(mgd, "_lib", None)
    with pytest.raises(RuntimeError, match="not found"):
        mgd.load()


def test_workspaces_from_the_binding_start_zero_filled():
    """The attention calls do not clear their workspace per call; they rely on a zero start."""
    import torch
    from long_context_speculative_split_gb300 import ops
    ws = ops.workspace(4096 + 3, "cpu")
    assert ws.dtype == torch.uint8 and ws.numel() == 4099 and int(ws.count_nonzero()) == 0
    assert ops.workspace(0, "cpu").numel() == 256
