"""GPU parity of the StreamingLLM-style draft cache (mgd_streaming_select)
against the oracle: index lists, lengths and gathered rows bit for bit."""
import numpy as np
import pytest
import torch

from _parity import gpu_or_skip
from long_context_speculative_split_gb300 import ops
from long_context_speculative_split_gb300 import workloads as wl
from oracle.streaming import streaming_select as ref_streaming


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("sink,K,lens", [(4, 64, [500, 64, 63, 1, 300]), (0, 32, [40, 32, 5]),
                                         (16, 16, [100, 10]), (4, 1024, [4096, 1000, 1030])])
def test_streaming_matches_oracle(dtype, sink, K, lens):
    dev = gpu_or_skip()
    cap = max(lens)
    g = torch.Generator().manual_seed(K + sink)
    B, Hkv, D = len(lens), 8, 128
    k = torch.randn((B, Hkv, cap, D), generator=g).to(dtype)
    v = torch.randn((B, Hkv, cap, D), generator=g).to(dtype)
    kv_len = torch.tensor(lens, dtype=torch.int32)
    res = ops.streaming_select(k.to(dev), v.to(dev), kv_len.to(dev), sink, K)
    view = (lambda t: t.view(torch.int16)) if dtype == torch.bfloat16 else (lambda t: t)
    ref = ref_streaming(view(k), view(v), kv_len, sink, K)
    np.testing.assert_array_equal(res["sel_idx"].cpu().numpy(), ref["sel_idx"])
    np.testing.assert_array_equal(res["draft_len"].cpu().numpy(), ref["draft_len"])
    for b in range(B):
        n = int(ref["draft_len"][b])
        np.testing.assert_array_equal(view(res["k_draft"][b, :, :n].cpu()).numpy(), ref["k_draft"][b, :, :n])
        np.testing.assert_array_equal(view(res["v_draft"][b, :, :n].cpu()).numpy(), ref["v_draft"][b, :, :n])


@pytest.mark.gpu
def test_streaming_full_size():
    """Benchmark shape: batch 128, context 32768, budget 1024 with 4 sinks."""
    dev = gpu_or_skip()
    c = wl.WORKLOADS["b128_ctx32k"]
    kv_len = wl.lengths(c)
    k, v = wl.kv_cache(c, dev, kv_len=kv_len)
    res = ops.streaming_select(k, v, kv_len.to(dev), 4, c["K"])
    torch.cuda.synchronize()
    idx = res["sel_idx"][5, 3].long()
    assert torch.equal(idx[:4].cpu(), torch.arange(4))
    assert torch.equal(idx[4:].cpu(), torch.arange(32768 - 1020, 32768))
    assert torch.equal(res["k_draft"][5, 3], k[5, 3, idx])
    assert torch.equal(res["v_draft"][127, 0], v[127, 0, res["sel_idx"][127, 0].long()])
