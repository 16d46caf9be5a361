"""The device error path on the GPU, without a fault: a bounded wait that nothing satisfies
(an mbarrier phase, a counter other CTAs would raise) gives up after its limit, raises
MGD_DEVERR_TIMEOUT in the workspace's error word and lets the kernel return; the context
stays usable, and a later call on the same workspace starts from a clean error word."""
import math

import pytest
import torch

from _parity import assert_attention_close, gpu_or_skip
from long_context_speculative_split_gb300 import mgd, ops
from long_context_speculative_split_gb300 import workloads as wl
from oracle.attention import attention

pytestmark = pytest.mark.gpu

MGD_DEVERR_TIMEOUT = 0x8


@pytest.mark.parametrize("which", [0, 1], ids=["mbarrier_phase", "cross_cta_counter"])
def test_wait_that_nothing_satisfies_times_out_and_the_context_survives(which):
    dev = gpu_or_skip()
    ws = ops.workspace(mgd.SELFTEST_WS_BYTES, dev)
    mgd.mgd_selftest_bounded_wait(which, ws)
    assert mgd.mgd_workspace_errors(ws) == MGD_DEVERR_TIMEOUT
    # the same context and workspace still run real work, and the call resets the error word
    cfg = dict(B=2, Hq=8, Hkv=2, D=128, dtype="bf16", lens=[300, 77], W=16, hh=0.01, gamma=1)
    kv_len = torch.tensor([300, 77], dtype=torch.int32)
    k, v = wl.kv_cache(cfg, dev, seed=9, kv_len=kv_len, cap=320)
    q = wl.queries(cfg, dev, seed=9)
    big = ops.workspace(mgd.mgd_verify_workspace_size(2, 2, 8, 2, 128, 320), dev)
    big[:ws.numel()].copy_(ws)  # start from the timed-out error word
    out, lse = ops.verify_attn(q, k, v, kv_len.to(dev), ws=big)
    assert mgd.mgd_workspace_errors(big) == 0
    ref, _ = attention(q, k, v, kv_len, 1.0 / math.sqrt(128))
    assert_attention_close(out, ref)
