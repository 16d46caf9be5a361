"""Pins for the StreamingLLM-style selection oracle (CPU only)."""
import numpy as np

from oracle.streaming import streaming_indices, streaming_select


def test_hand_cases():
    assert list(streaming_indices(10, 2, 5)) == [0, 1, 7, 8, 9]          # 2 sinks + 3 recent
    assert list(streaming_indices(10, 0, 4)) == [6, 7, 8, 9]             # recent window only
    assert list(streaming_indices(10, 6, 4)) == [0, 1, 2, 3]             # sinks fill the budget
    assert list(streaming_indices(4, 2, 8)) == [0, 1, 2, 3]              # budget >= context


def test_properties_by_enumeration():
    for L in range(1, 40):
        for K in range(1, 45):
            for sink in range(0, 6):
                idx = streaming_indices(L, sink, K)
                assert len(idx) == min(K, L)
                assert len(set(idx.tolist())) == len(idx) and list(idx) == sorted(idx)
                assert idx.min() >= 0 and idx.max() < L
                s = min(sink, K, L)
                assert set(range(s)) <= set(idx.tolist())                     # the sinks
                tail = min(K, L) - s
                assert set(range(L - tail, L)) <= set(idx.tolist())          # the newest rows


def test_gather_copies_rows():
    rng = np.random.default_rng(0)
    k = rng.standard_normal((2, 3, 20, 8))
    v = rng.standard_normal((2, 3, 20, 8))
    res = streaming_select(k, v, np.array([20, 7]), 4, 10)
    assert list(res["draft_len"]) == [10, 7]
    np.testing.assert_array_equal(res["k_draft"][0, 1, :10], k[0, 1, [0, 1, 2, 3, 14, 15, 16, 17, 18, 19]])
    np.testing.assert_array_equal(res["v_draft"][1, 2, :7], v[1, 2, :7])
    assert np.all(res["sel_idx"][1, :, 7:] == -1)
