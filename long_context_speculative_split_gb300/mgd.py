"""Thin ctypes binding of libmgd.so (C ABI declared in include/mgd.h).

Every function here has the name and the argument order of the C entry point
it wraps and only marshals arguments: a pointer argument accepts a torch
tensor (its ``data_ptr()``), a plain integer address or ``None`` (NULL); the
stream argument accepts a ``torch.cuda.Stream``, a raw handle or ``None``
(the current torch stream).  All arithmetic runs in the library's CUDA
kernels.  A non-OK status raises ``MgdError``.  There is no fallback: if the
library has not been built, loading it raises.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmgd.so")

MGD_OK, MGD_ERR_INVALID_ARG, MGD_ERR_UNSUPPORTED, MGD_ERR_WORKSPACE, MGD_ERR_CUDA = range(5)
MGD_BF16, MGD_F32 = 0, 1
MGD_VERIFY, MGD_DRAW_DRAFT, MGD_VERIFY_DRAWN = 0, 1, 2
MGD_DEVERR_KV_LEN, MGD_DEVERR_SNAP_LEN, MGD_DEVERR_TOKEN, MGD_DEVERR_TIMEOUT = 0x1, 0x2, 0x4, 0x8
MGD_DEVERR_COMMIT = 0x10
MGD_DEVERR_STALE_WS = 0x20
MGD_DEVERR_NOT_DRAWN = 0x40

_vp, _i32, _i64, _f32, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t

# name -> (restype, argtypes), in the order of include/mgd.h
SIGNATURES = {
    "mgd_status_string": (ctypes.c_char_p, [_i32]),
    "mgd_last_error": (ctypes.c_char_p, []),
    "mgd_version": (_i32, []),
    "mgd_workspace_errors": (_i32, [_vp, _vp, ctypes.POINTER(ctypes.c_uint32)]),
    "mgd_selftest_bounded_wait": (_i32, [_i32, _vp, _sz, _vp]),
    "mgd_selftest_occupy": (_i32, [_i32, _i32, _i32, _vp]),
    "mgd_set_programmatic_launch": (None, [_i32]),
    "mgd_verify_workspace_size": (_sz, [_i32] * 6),
    "mgd_verify_attn": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i64, _i64, _f32, _i32,
                               _vp, _i32, _vp, _vp, _sz, _vp]),
    "mgd_draft_workspace_size": (_sz, [_i32] * 5),
    "mgd_draft_attn": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i64, _i64, _f32, _i32,
                              _vp, _i32, _vp, _vp, _sz, _vp]),
    "mgd_snapkv_workspace_size": (_sz, [_i32] * 6),
    "mgd_snapkv_select": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i64, _i64, _i32, _i32, _i32,
                                 _f32, _i32, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _sz, _vp]),
    "mgd_snapkv_select_budgets": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i64, _i64, _i32, _i32,
                                         _vp, _f32, _i32, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _sz, _vp]),
    "mgd_topk_draft_workspace_size": (_sz, [_i32] * 6),
    "mgd_topk_draft_attn": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i64, _i64, _i32, _f32, _i32,
                                   _vp, _vp, _vp, _i32, _vp, _vp, _i32, _vp, _vp, _sz, _vp]),
    "mgd_spec_workspace_size": (_sz, [_i32] * 3),
    "mgd_spec_sample": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _sz, _vp]),
    "mgd_streaming_select": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i64, _i64, _i32, _i32, _i32, _vp, _vp,
                                    _vp, _i32, _vp, _vp]),
    "mgd_commit_workspace_size": (_sz, [_i32]),
    "mgd_commit_round": (_i32, [_vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _i32, _i64, _i64, _vp, _vp, _i32,
                                _i64, _i64, _vp, _vp, _sz, _vp]),
    "mgd_spec_sample_noalloc": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp]),
}

# Bytes of the library-owned scratch array used by mgd_spec_sample_noalloc.
MGD_NOALLOC_SCRATCH_BYTES = 1 << 20

_lib = None


class MgdError(RuntimeError):
    def __init__(self, status, detail):
        self.status = status
        super().__init__("%s: %s" % (status_name(status), detail))


def load():
    """Load libmgd.so once (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libmgd.so not found at %s; build it with __graft_entry__.build() "
                               "(python -m long_context_speculative_split_gb300.build)" % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_name(s):
    return ["MGD_OK", "MGD_ERR_INVALID_ARG", "MGD_ERR_UNSUPPORTED", "MGD_ERR_WORKSPACE", "MGD_ERR_CUDA"][s] \
        if 0 <= s <= 4 else "status %d" % s


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status):
    if status != MGD_OK:
        raise MgdError(status, load().mgd_last_error().decode())


def mgd_status_string(s):
    return load().mgd_status_string(s).decode()


def mgd_last_error():
    return load().mgd_last_error().decode()


def mgd_version():
    return load().mgd_version()


def mgd_workspace_errors(ws, stream=None):
    flags = ctypes.c_uint32(0)
    _check(load().mgd_workspace_errors(_ptr(ws), _stream(stream), ctypes.byref(flags)))
    return flags.value


SELFTEST_WS_BYTES = 512


def mgd_selftest_bounded_wait(which, ws, ws_bytes=None, stream=None):
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size()
    _check(load().mgd_selftest_bounded_wait(which, _ptr(ws), ws_bytes, _stream(stream)))


def mgd_set_programmatic_launch(enable):
    """Launch later calls' kernels with programmatic stream serialization (True, the default) or plainly."""
    load().mgd_set_programmatic_launch(1 if enable else 0)


def mgd_selftest_occupy(ctas, smem_bytes, usec, stream=None):
    _check(load().mgd_selftest_occupy(ctas, smem_bytes, usec, _stream(stream)))


def mgd_verify_workspace_size(B, T, Hq, Hkv, D, kv_cap):
    return load().mgd_verify_workspace_size(B, T, Hq, Hkv, D, kv_cap)


def mgd_verify_attn(q, k, v, kv_len, B, T, Hq, Hkv, D, kv_cap, kv_batch_stride, kv_head_stride, sm_scale,
                    in_dtype, out, out_dtype, lse, ws, ws_bytes, stream=None):
    _check(load().mgd_verify_attn(_ptr(q), _ptr(k), _ptr(v), _ptr(kv_len), B, T, Hq, Hkv, D, kv_cap,
                                  kv_batch_stride, kv_head_stride, sm_scale, in_dtype, _ptr(out), out_dtype,
                                  _ptr(lse), _ptr(ws), ws_bytes, _stream(stream)))


def mgd_draft_workspace_size(B, Hq, Hkv, D, k_cap):
    return load().mgd_draft_workspace_size(B, Hq, Hkv, D, k_cap)


def mgd_draft_attn(q, k_draft, v_draft, draft_len, B, Hq, Hkv, D, k_cap, kv_batch_stride, kv_head_stride,
                   sm_scale, in_dtype, out, out_dtype, lse, ws, ws_bytes, stream=None):
    _check(load().mgd_draft_attn(_ptr(q), _ptr(k_draft), _ptr(v_draft), _ptr(draft_len), B, Hq, Hkv, D, k_cap,
                                 kv_batch_stride, kv_head_stride, sm_scale, in_dtype, _ptr(out), out_dtype,
                                 _ptr(lse), _ptr(ws), ws_bytes, _stream(stream)))


def mgd_topk_draft_workspace_size(B, Hq, Hkv, D, kv_cap, draft_cap):
    return load().mgd_topk_draft_workspace_size(B, Hq, Hkv, D, kv_cap, draft_cap)


def mgd_topk_draft_attn(q, k, v, kv_len, B, Hq, Hkv, D, kv_cap, kv_batch_stride, kv_head_stride, K, sm_scale,
                        in_dtype, sel_idx, k_draft, v_draft, draft_cap, draft_len, out, out_dtype, lse, ws, ws_bytes,
                        stream=None):
    _check(load().mgd_topk_draft_attn(_ptr(q), _ptr(k), _ptr(v), _ptr(kv_len), B, Hq, Hkv, D, kv_cap,
                                      kv_batch_stride, kv_head_stride, K, sm_scale, in_dtype, _ptr(sel_idx),
                                      _ptr(k_draft), _ptr(v_draft), draft_cap, _ptr(draft_len), _ptr(out), out_dtype,
                                      _ptr(lse), _ptr(ws), ws_bytes, _stream(stream)))


def mgd_snapkv_workspace_size(B, Hq, Hkv, D, kv_cap, W):
    return load().mgd_snapkv_workspace_size(B, Hq, Hkv, D, kv_cap, W)


def mgd_snapkv_select(q_win, k, v, kv_len, B, Hq, Hkv, D, kv_cap, kv_batch_stride, kv_head_stride, W, pool, K,
                      sm_scale, in_dtype, sel_idx, k_draft, v_draft, draft_cap, draft_len, scores, ws, ws_bytes,
                      stream=None):
    _check(load().mgd_snapkv_select(_ptr(q_win), _ptr(k), _ptr(v), _ptr(kv_len), B, Hq, Hkv, D, kv_cap,
                                    kv_batch_stride, kv_head_stride, W, pool, K, sm_scale, in_dtype,
                                    _ptr(sel_idx), _ptr(k_draft), _ptr(v_draft), draft_cap, _ptr(draft_len),
                                    _ptr(scores), _ptr(ws), ws_bytes, _stream(stream)))


def mgd_snapkv_select_budgets(q_win, k, v, kv_len, B, Hq, Hkv, D, kv_cap, kv_batch_stride, kv_head_stride, W, pool,
                              budgets, sm_scale, in_dtype, sel_idx, k_draft, v_draft, draft_cap, draft_len, scores, ws,
                              ws_bytes, stream=None):
    _check(load().mgd_snapkv_select_budgets(_ptr(q_win), _ptr(k), _ptr(v), _ptr(kv_len), B, Hq, Hkv, D, kv_cap,
                                            kv_batch_stride, kv_head_stride, W, pool, _ptr(budgets), sm_scale,
                                            in_dtype, _ptr(sel_idx), _ptr(k_draft), _ptr(v_draft), draft_cap,
                                            _ptr(draft_len), _ptr(scores), _ptr(ws), ws_bytes, _stream(stream)))


def mgd_spec_workspace_size(B, gamma, V):
    return load().mgd_spec_workspace_size(B, gamma, V)


def mgd_spec_sample(target_logits, draft_logits, draft_tokens, u, B, gamma, V, mode, row, out_tokens,
                    num_accepted, ws, ws_bytes, stream=None):
    _check(load().mgd_spec_sample(_ptr(target_logits), _ptr(draft_logits), _ptr(draft_tokens), _ptr(u), B, gamma,
                                  V, mode, row, _ptr(out_tokens), _ptr(num_accepted), _ptr(ws), ws_bytes,
                                  _stream(stream)))


def mgd_streaming_select(k, v, kv_len, B, Hkv, D, kv_cap, kv_batch_stride, kv_head_stride, sink, K, dtype, sel_idx,
                         k_draft, v_draft, draft_cap, draft_len, stream=None):
    _check(load().mgd_streaming_select(_ptr(k), _ptr(v), _ptr(kv_len), B, Hkv, D, kv_cap, kv_batch_stride,
                                       kv_head_stride, sink, K, dtype, _ptr(sel_idx), _ptr(k_draft), _ptr(v_draft),
                                       draft_cap, _ptr(draft_len), _stream(stream)))


def mgd_commit_workspace_size(B):
    return load().mgd_commit_workspace_size(B)


def mgd_commit_round(num_accepted, B, gamma, Hkv, D, dtype, kv_len, k, v, kv_cap, kv_batch_stride, kv_head_stride,
                     k_draft, v_draft, draft_cap, draft_batch_stride, draft_head_stride, draft_len, ws, ws_bytes,
                     stream=None):
    _check(load().mgd_commit_round(_ptr(num_accepted), B, gamma, Hkv, D, dtype, _ptr(kv_len), _ptr(k), _ptr(v),
                                   kv_cap, kv_batch_stride, kv_head_stride, _ptr(k_draft), _ptr(v_draft), draft_cap,
                                   draft_batch_stride, draft_head_stride, _ptr(draft_len), _ptr(ws), ws_bytes,
                                   _stream(stream)))


def mgd_spec_sample_noalloc(target_logits, draft_logits, draft_tokens, u, B, gamma, V, mode, row, out_tokens,
                            num_accepted, stream=None):
    """mgd_spec_sample without a workspace, for callers that may not allocate device memory.

    Its scratch is a fixed library-owned device array (MGD_NOALLOC_SCRATCH_BYTES) shared by
    every call, so calls that overlap on the GPU must be serialised by the caller.
    """
    _check(load().mgd_spec_sample_noalloc(_ptr(target_logits), _ptr(draft_logits), _ptr(draft_tokens), _ptr(u),
                                          B, gamma, V, mode, row, _ptr(out_tokens), _ptr(num_accepted),
                                          _stream(stream)))
