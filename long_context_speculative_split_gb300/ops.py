"""Tensor-level wrappers over the C ABI: infer shapes and strides from torch
tensors, allocate outputs and workspaces with torch (device memory only) and
call ``mgd``.  No arithmetic of the method happens here.
"""
import math

import torch

from . import mgd


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return mgd.MGD_BF16
    if t.dtype == torch.float32:
        return mgd.MGD_F32
    raise TypeError("unsupported dtype %s (bfloat16 or float32)" % t.dtype)


def _check(device, dense=(), int32=(), f32=(), same=()):
    """Argument checks the C ABI cannot make on raw pointers: every tensor on `device`; the
    ones in `dense` packed row-major (the calls take them without strides); `int32` / `f32`
    of that dtype; `same` a list of tensors that must share one dtype.  Raises before any
    launch."""
    named = list(dense) + list(int32) + list(f32) + list(same)
    for name, t in named:
        if t is not None and t.device != device:
            raise ValueError("%s is on %s, expected %s" % (name, t.device, device))
    for name, t in dense:
        if t is not None and not t.is_contiguous():
            raise ValueError("%s must be contiguous (the C ABI reads it as a packed row-major array)" % name)
    for name, t in int32:
        if t is not None and t.dtype != torch.int32:
            raise TypeError("%s must be int32, got %s" % (name, t.dtype))
    for name, t in f32:
        if t is not None and t.dtype != torch.float32:
            raise TypeError("%s must be float32, got %s" % (name, t.dtype))
    if same:
        d0 = same[0][1].dtype
        for name, t in same[1:]:
            if t.dtype != d0:
                raise TypeError("%s has dtype %s, expected %s like %s" % (name, t.dtype, d0, same[0][0]))


def _kv_strides(k, v, D):
    if k.stride(3) != 1 or k.stride(2) != D or k.stride() != v.stride():
        raise ValueError("K and V must share strides with contiguous rows of D elements")
    return k.stride(0), k.stride(1)


def workspace(nbytes, device):
    """Zero-filled device scratch (calls that skip clearing it rely on a zero start)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def verify_attn(q, k, v, kv_len, sm_scale=None, out_dtype=torch.float32, ws=None, out=None, lse=None,
                stream=None):
    """q [B,T,Hq,D], k/v [B,Hkv,kv_cap,D] (same dtype), kv_len [B] int32 -> (out [B,T,Hq,D], lse [B,T,Hq])."""
    B, T, Hq, D = q.shape
    Hkv, cap = k.shape[1], k.shape[2]
    sb, sh = _kv_strides(k, v, D)
    scale = 1.0 / math.sqrt(D) if sm_scale is None else sm_scale
    if out is None:
        out = torch.empty((B, T, Hq, D), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, T, Hq), dtype=torch.float32, device=q.device)
    _check(q.device, dense=[("q", q), ("kv_len", kv_len), ("out", out), ("lse", lse)], int32=[("kv_len", kv_len)],
           f32=[("lse", lse)], same=[("q", q), ("k", k), ("v", v)])
    need = mgd.mgd_verify_workspace_size(B, T, Hq, Hkv, D, cap)
    if ws is None:
        ws = workspace(need, q.device)
    mgd.mgd_verify_attn(q, k, v, kv_len, B, T, Hq, Hkv, D, cap, sb, sh, scale, _dtype_code(q), out,
                        _dtype_code(out), lse, ws, ws.numel(), stream)
    return out, lse


def draft_attn(q, k_draft, v_draft, draft_len, sm_scale=None, out_dtype=torch.float32, ws=None, out=None,
               lse=None, stream=None):
    """q [B,Hq,D] or [B,1,Hq,D], compacted k/v [B,Hkv,k_cap,D], draft_len [B] -> (out [B,Hq,D], lse [B,Hq])."""
    if q.dim() == 4:
        q = q[:, 0]
    B, Hq, D = q.shape
    Hkv, cap = k_draft.shape[1], k_draft.shape[2]
    sb, sh = _kv_strides(k_draft, v_draft, D)
    scale = 1.0 / math.sqrt(D) if sm_scale is None else sm_scale
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    _check(q.device, dense=[("q", q), ("draft_len", draft_len), ("out", out), ("lse", lse)],
           int32=[("draft_len", draft_len)], f32=[("lse", lse)], same=[("q", q), ("k_draft", k_draft), ("v_draft", v_draft)])
    need = mgd.mgd_draft_workspace_size(B, Hq, Hkv, D, cap)
    if ws is None:
        ws = workspace(need, q.device)
    mgd.mgd_draft_attn(q, k_draft, v_draft, draft_len, B, Hq, Hkv, D, cap, sb, sh, scale, _dtype_code(q), out,
                       _dtype_code(out), lse, ws, ws.numel(), stream)
    return out, lse


def snapkv_select(q_win, k, v, kv_len, W, pool, K, draft_cap=None, sm_scale=None, ws=None, want_scores=False,
                  out=None, stream=None):
    """Returns dict(sel_idx [B,Hkv,draft_cap] int32, k_draft, v_draft [B,Hkv,draft_cap,D], draft_len [B],
    scores [B,Hkv,kv_cap] float32 or None).  K is one budget for every sequence, or an int32 device tensor
    [B] of per-sequence budgets (then draft_cap is required)."""
    B, Wq, Hq, D = q_win.shape
    assert Wq == W
    Hkv, cap = k.shape[1], k.shape[2]
    sb, sh = _kv_strides(k, v, D)
    per_seq = torch.is_tensor(K)
    if per_seq and draft_cap is None:
        raise ValueError("per-sequence budgets need an explicit draft_cap")
    cap_d = K if draft_cap is None else draft_cap
    scale = 1.0 / math.sqrt(D) if sm_scale is None else sm_scale
    dev = q_win.device
    if out is None:
        out = dict(sel_idx=torch.empty((B, Hkv, cap_d), dtype=torch.int32, device=dev),
                   k_draft=torch.zeros((B, Hkv, cap_d, D), dtype=k.dtype, device=dev),
                   v_draft=torch.zeros((B, Hkv, cap_d, D), dtype=k.dtype, device=dev),
                   draft_len=torch.empty((B,), dtype=torch.int32, device=dev),
                   scores=torch.zeros((B, Hkv, cap), dtype=torch.float32, device=dev) if want_scores else None)
    _check(dev, dense=[("q_win", q_win), ("kv_len", kv_len), ("sel_idx", out["sel_idx"]),
                       ("draft_len", out["draft_len"]), ("scores", out["scores"]), ("K", K if per_seq else None)],
           int32=[("kv_len", kv_len), ("sel_idx", out["sel_idx"]), ("draft_len", out["draft_len"]),
                  ("K", K if per_seq else None)],
           f32=[("scores", out["scores"])],
           same=[("q_win", q_win), ("k", k), ("v", v), ("k_draft", out["k_draft"]), ("v_draft", out["v_draft"])])
    need = mgd.mgd_snapkv_workspace_size(B, Hq, Hkv, D, cap, W)
    if ws is None:
        ws = workspace(need, dev)
    if per_seq:
        mgd.mgd_snapkv_select_budgets(q_win, k, v, kv_len, B, Hq, Hkv, D, cap, sb, sh, W, pool, K, scale,
                                      _dtype_code(k), out["sel_idx"], out["k_draft"], out["v_draft"], cap_d,
                                      out["draft_len"], out["scores"], ws, ws.numel(), stream)
    else:
        mgd.mgd_snapkv_select(q_win, k, v, kv_len, B, Hq, Hkv, D, cap, sb, sh, W, pool, K, scale, _dtype_code(k),
                              out["sel_idx"], out["k_draft"], out["v_draft"], cap_d, out["draft_len"], out["scores"],
                              ws, ws.numel(), stream)
    return out


def topk_draft_attn(q, k, v, kv_len, K, draft_cap=None, sm_scale=None, out_dtype=torch.float32, ws=None, out=None,
                    stream=None):
    """One dynamic top-K draft step: q [B,Hq,D] (or [B,1,Hq,D]) at position kv_len-1 selects the newest row plus
    the K-1 earlier rows it attends to most (summed over the heads of a KV head) and attends over them.
    Returns dict(out [B,Hq,D], lse [B,Hq], sel_idx, k_draft, v_draft, draft_len)."""
    if q.dim() == 4:
        q = q[:, 0]
    B, Hq, D = q.shape
    Hkv, cap = k.shape[1], k.shape[2]
    sb, sh = _kv_strides(k, v, D)
    cap_d = K if draft_cap is None else draft_cap
    scale = 1.0 / math.sqrt(D) if sm_scale is None else sm_scale
    dev = q.device
    if out is None:
        out = dict(out=torch.empty((B, Hq, D), dtype=out_dtype, device=dev),
                   lse=torch.empty((B, Hq), dtype=torch.float32, device=dev),
                   sel_idx=torch.empty((B, Hkv, cap_d), dtype=torch.int32, device=dev),
                   k_draft=torch.zeros((B, Hkv, cap_d, D), dtype=k.dtype, device=dev),
                   v_draft=torch.zeros((B, Hkv, cap_d, D), dtype=k.dtype, device=dev),
                   draft_len=torch.empty((B,), dtype=torch.int32, device=dev))
    _check(dev, dense=[("q", q), ("kv_len", kv_len), ("out", out["out"]), ("lse", out["lse"]), ("sel_idx", out["sel_idx"]),
                       ("draft_len", out["draft_len"])],
           int32=[("kv_len", kv_len), ("sel_idx", out["sel_idx"]), ("draft_len", out["draft_len"])],
           f32=[("lse", out["lse"])],
           same=[("q", q), ("k", k), ("v", v), ("k_draft", out["k_draft"]), ("v_draft", out["v_draft"])])
    need = mgd.mgd_topk_draft_workspace_size(B, Hq, Hkv, D, cap, cap_d)
    if ws is None:
        ws = workspace(need, dev)
    mgd.mgd_topk_draft_attn(q, k, v, kv_len, B, Hq, Hkv, D, cap, sb, sh, K, scale, _dtype_code(k), out["sel_idx"],
                            out["k_draft"], out["v_draft"], cap_d, out["draft_len"], out["out"],
                            _dtype_code(out["out"]), out["lse"], ws, ws.numel(), stream)
    return out


def draft_draw(draft_logits, u, draft_tokens=None, row=-1, ws=None, stream=None):
    """Fill draft_tokens [B, gamma] from softmax(draft_logits[b, s]) with u[b, s, 0] (row < 0: every s)."""
    B, gamma, V = draft_logits.shape
    if draft_tokens is None:
        draft_tokens = torch.full((B, gamma), -1, dtype=torch.int32, device=draft_logits.device)
    _check(draft_logits.device, dense=[("draft_logits", draft_logits), ("u", u), ("draft_tokens", draft_tokens)],
           int32=[("draft_tokens", draft_tokens)], f32=[("draft_logits", draft_logits), ("u", u)])
    need = mgd.mgd_spec_workspace_size(B, gamma, V)
    if ws is None:
        ws = workspace(need, draft_logits.device)
    mgd.mgd_spec_sample(None, draft_logits, draft_tokens, u, B, gamma, V, mgd.MGD_DRAW_DRAFT, row, None, None, ws,
                        ws.numel(), stream)
    return draft_tokens


def rejection_sample(target_logits, draft_logits, draft_tokens, u, ws=None, out_tokens=None, num_accepted=None,
                     stream=None, reuse_draft_stats=False):
    """-> (out_tokens [B, gamma+1] int32 (-1 padded), num_accepted [B] int32).
    reuse_draft_stats: take the draft rows' normalisers from the draws this round made with
    draft_draw on the same `ws` (MGD_VERIFY_DRAWN) instead of streaming those rows again."""
    B, gp1, V = target_logits.shape
    gamma = gp1 - 1
    dev = target_logits.device
    if out_tokens is None:
        out_tokens = torch.empty((B, gp1), dtype=torch.int32, device=dev)
    if num_accepted is None:
        num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    if reuse_draft_stats and ws is None:
        raise ValueError("reuse_draft_stats needs the workspace the draws used")
    _check(dev, dense=[("target_logits", target_logits), ("draft_logits", draft_logits), ("draft_tokens", draft_tokens),
                       ("u", u), ("out_tokens", out_tokens), ("num_accepted", num_accepted)],
           int32=[("draft_tokens", draft_tokens), ("out_tokens", out_tokens), ("num_accepted", num_accepted)],
           f32=[("target_logits", target_logits), ("draft_logits", draft_logits), ("u", u)])
    need = mgd.mgd_spec_workspace_size(B, gamma, V)
    if ws is None:
        ws = workspace(need, dev)
    mode = mgd.MGD_VERIFY_DRAWN if reuse_draft_stats else mgd.MGD_VERIFY
    mgd.mgd_spec_sample(target_logits, draft_logits, draft_tokens, u, B, gamma, V, mode, -1, out_tokens,
                        num_accepted, ws, ws.numel(), stream)
    return out_tokens, num_accepted


def commit_round(num_accepted, gamma, kv_len, k, v, k_draft, v_draft, draft_len, ws=None, stream=None):
    """Keep accepted verify rows, roll back the rest, append the kept rows to the draft cache (in place)."""
    B, Hkv, cap, D = k.shape
    if k_draft.stride(3) != 1 or k_draft.stride(2) != D or k_draft.stride() != v_draft.stride():
        raise ValueError("draft K and V must share strides with contiguous rows of D elements")
    sb, sh = _kv_strides(k, v, D)
    _check(k.device, dense=[("num_accepted", num_accepted), ("kv_len", kv_len), ("draft_len", draft_len)],
           int32=[("num_accepted", num_accepted), ("kv_len", kv_len), ("draft_len", draft_len)],
           same=[("k", k), ("v", v), ("k_draft", k_draft), ("v_draft", v_draft)])
    if ws is None:
        ws = workspace(mgd.mgd_commit_workspace_size(B), k.device)
    mgd.mgd_commit_round(num_accepted, B, gamma, Hkv, D, _dtype_code(k), kv_len, k, v, cap, sb, sh, k_draft,
                         v_draft, k_draft.shape[2], k_draft.stride(0), k_draft.stride(1), draft_len, ws, ws.numel(),
                         stream)
    return kv_len, draft_len


def streaming_select(k, v, kv_len, sink, K, draft_cap=None, out=None, stream=None):
    """StreamingLLM-style draft cache: first `sink` rows plus the most recent ones, min(K, L) in total."""
    B, Hkv, cap, D = k.shape
    sb, sh = _kv_strides(k, v, D)
    cap_d = K if draft_cap is None else draft_cap
    dev = k.device
    if out is None:
        out = dict(sel_idx=torch.empty((B, Hkv, cap_d), dtype=torch.int32, device=dev),
                   k_draft=torch.zeros((B, Hkv, cap_d, D), dtype=k.dtype, device=dev),
                   v_draft=torch.zeros((B, Hkv, cap_d, D), dtype=k.dtype, device=dev),
                   draft_len=torch.empty((B,), dtype=torch.int32, device=dev))
    _check(dev, dense=[("kv_len", kv_len), ("sel_idx", out["sel_idx"]), ("draft_len", out["draft_len"])],
           int32=[("kv_len", kv_len), ("sel_idx", out["sel_idx"]), ("draft_len", out["draft_len"])],
           same=[("k", k), ("v", v), ("k_draft", out["k_draft"]), ("v_draft", out["v_draft"])])
    mgd.mgd_streaming_select(k, v, kv_len, B, Hkv, D, cap, sb, sh, sink, K, _dtype_code(k), out["sel_idx"],
                             out["k_draft"], out["v_draft"], cap_d, out["draft_len"], stream)
    return out
