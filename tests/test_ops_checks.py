"""Host-side argument checks of the tensor wrappers: a tensor the C ABI would read through its
raw pointer in the wrong layout, dtype or place is refused before any library call (these
tests run without a GPU: every case fails before the first call into libmgd)."""
import pytest
import torch

from long_context_speculative_split_gb300 import ops


def _attn_args(B=2, T=3, Hq=8, Hkv=2, D=64, cap=32):
    q = torch.zeros((B, T, Hq, D), dtype=torch.bfloat16)
    k = torch.zeros((B, Hkv, cap, D), dtype=torch.bfloat16)
    v = torch.zeros_like(k)
    kv_len = torch.full((B,), cap, dtype=torch.int32)
    return q, k, v, kv_len


def test_verify_refuses_a_strided_query():
    q, k, v, kv_len = _attn_args()
    qt = q.transpose(1, 2).contiguous().transpose(1, 2)  # same shape, not packed
    assert not qt.is_contiguous()
    with pytest.raises(ValueError, match="q must be contiguous"):
        ops.verify_attn(qt, k, v, kv_len)


def test_verify_refuses_mixed_dtypes_and_int64_lengths():
    q, k, v, kv_len = _attn_args()
    with pytest.raises(TypeError, match="k has dtype"):
        ops.verify_attn(q, k.float(), v, kv_len)
    with pytest.raises(TypeError, match="kv_len must be int32"):
        ops.verify_attn(q, k, v, kv_len.long())


def test_draft_refuses_a_length_vector_elsewhere():
    q, k, v, kv_len = _attn_args(T=1)
    with pytest.raises(ValueError, match="draft_len is on meta"):
        ops.draft_attn(q, k, v, torch.empty((2,), dtype=torch.int32, device="meta"))


def test_sampling_refuses_bf16_logits_and_strided_uniforms():
    B, gamma, V = 3, 2, 100
    t = torch.zeros((B, gamma + 1, V))
    d = torch.zeros((B, gamma, V))
    tok = torch.zeros((B, gamma), dtype=torch.int32)
    u = torch.zeros((B, gamma + 1, 3))
    with pytest.raises(TypeError, match="target_logits must be float32"):
        ops.rejection_sample(t.bfloat16(), d, tok, u)
    with pytest.raises(TypeError, match="draft_tokens must be int32"):
        ops.rejection_sample(t, d, tok.long(), u)
    u_strided = torch.zeros((B, gamma + 1, 6))[:, :, ::2]
    with pytest.raises(ValueError, match="u must be contiguous"):
        ops.draft_draw(d, u_strided)


def test_commit_refuses_int64_counts():
    q, k, v, kv_len = _attn_args()
    kd, vd = torch.zeros((2, 2, 16, 64), dtype=torch.bfloat16), torch.zeros((2, 2, 16, 64), dtype=torch.bfloat16)
    dlen = torch.full((2,), 8, dtype=torch.int32)
    with pytest.raises(TypeError, match="num_accepted must be int32"):
        ops.commit_round(torch.zeros((2,), dtype=torch.int64), 2, kv_len, k, v, kd, vd, dlen)
    with pytest.raises(TypeError, match="k_draft has dtype"):
        ops.commit_round(torch.zeros((2,), dtype=torch.int32), 2, kv_len, k, v, kd.float(), vd, dlen)


def test_snapkv_refuses_a_float32_window_against_bf16_keys():
    q, k, v, kv_len = _attn_args(T=4)
    with pytest.raises(TypeError, match="k has dtype"):
        ops.snapkv_select(q.float(), k, v, kv_len, 4, 3, 8)
