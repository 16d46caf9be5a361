"""The one-read SnapKV scorer's CTAs wait for one another (a slice's pass 2 needs
the log-sum-exp over every slice of its (sequence, KV head)).  Before waiting, a
CTA claims and runs pass 1 over every slice of its pair that nobody has claimed
yet, so the waits end however few of its CTAs are resident.

This test holds all but a few SMs with a diagnostic kernel on one stream (one
CTA per SM, each holding 200 KB of shared memory, so no scorer CTA fits beside
it) while a selection whose pairs have 64 slices each -- far more than the
scorer CTAs that fit on the free SMs -- runs on a second stream.  The selection
must finish while the SMs are still held, raise no device error (no bounded
wait ran out), and give exactly the results of the same call on an idle GPU
(the scorer's arithmetic does not depend on which CTA runs which slice)."""
import math

import numpy as np
import pytest
import torch

from _parity import assert_index_sets_match, gpu_or_skip
from long_context_speculative_split_gb300 import mgd, ops
from long_context_speculative_split_gb300 import workloads as wl
from oracle.snapkv import max_pool, select_indices, window_scores

pytestmark = pytest.mark.gpu

FREE_SMS = 4
HOLD_US = 1_500_000


def test_snapkv_progress_with_most_sms_held():
    dev = gpu_or_skip()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    L = 64 * 1536                                   # 64 scoring slices per (sequence, KV head)
    cfg = dict(B=2, Hq=32, Hkv=8, D=128, dtype="bf16", lens=[L, L - 777], W=32, hh=0.01, gamma=1)
    kv_len = torch.tensor(cfg["lens"], dtype=torch.int32)
    k, v = wl.kv_cache(cfg, dev, seed=9, kv_len=kv_len, cap=L)
    qw = wl.window_queries(cfg, dev, seed=9)
    W, P, K = 32, 7, 512
    need = mgd.mgd_snapkv_workspace_size(2, 32, 8, 128, L, W)

    ws0 = ops.workspace(need, dev)
    ref = ops.snapkv_select(qw, k, v, kv_len.to(dev), W, P, K, ws=ws0, want_scores=True)
    torch.cuda.synchronize()
    assert mgd.mgd_workspace_errors(ws0) == 0

    ws1 = ops.workspace(need, dev)
    kvl = kv_len.to(dev)
    hold, work = torch.cuda.Stream(), torch.cuda.Stream()
    # every kernel launched below is launched once first: with lazy module loading the first
    # launch of a kernel can wait for the device to go idle, i.e. for the holders to end
    torch.cuda._sleep(1000)
    torch.cuda.synchronize()
    # nothing may go to the legacy default stream from here on: it would wait for the holders
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    ev[0].record(hold)
    mgd.mgd_selftest_occupy(sms - FREE_SMS, 200 * 1024, HOLD_US, stream=hold)
    ev[1].record(hold)
    with torch.cuda.stream(work):
        torch.cuda._sleep(int(2e6))                 # about a millisecond: the holders settle first
        ev[2].record(work)
        got = ops.snapkv_select(qw, k, v, kvl, W, P, K, ws=ws1, want_scores=True, stream=work)
        ev[3].record(work)
    work.synchronize()
    still_held = not hold.query()
    hold.synchronize()
    hold_ms, sel_ms, gap_ms = ev[0].elapsed_time(ev[1]), ev[2].elapsed_time(ev[3]), ev[0].elapsed_time(ev[2])
    flags = mgd.mgd_workspace_errors(ws1)
    print("held %.1f ms; selection %.2f ms, started %.2f ms after the holders; flags %#x" % (
        hold_ms, sel_ms, gap_ms, flags))
    assert flags == 0, "device error bits %#x (selection took %.1f ms)" % (flags, sel_ms)
    assert still_held and gap_ms + sel_ms < hold_ms, \
        "the holders (%.1f ms) ended before the selection (%.1f ms from %.1f ms)" % (hold_ms, sel_ms, gap_ms)
    for name in ("sel_idx", "draft_len", "k_draft", "v_draft", "scores"):
        assert torch.equal(got[name], ref[name]), name
    # and the selection itself is the oracle's, on one sampled pair
    b, h, G = 1, 5, 4
    Lb = int(kv_len[b])
    s = window_scores(qw[b:b + 1, :, h * G:(h + 1) * G], k[b:b + 1, h:h + 1, :Lb], kv_len[b:b + 1], W,
                      1.0 / math.sqrt(128))[0, 0]
    pooled = np.zeros(Lb)
    pooled[:Lb - W] = max_pool(s, Lb - W, P)
    ref_idx = select_indices(pooled, Lb, W, K)
    kth = np.min(pooled[ref_idx[:K - W]])
    assert_index_sets_match(got["sel_idx"][b, h, :K].cpu().numpy(), ref_idx, pooled, kth)
