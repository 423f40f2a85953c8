"""Pins of the oracle's paged-KV append: a placement worked out by hand, a
round trip against a cache the input generator filled by a different route
(whole padded sequences scattered page by page), and its error cases."""
import numpy as np
import pytest

import oracle
import workloads as wl
from tests.common import oracle_on_call


def test_hand_placed_example():
    # page_size 2, one kv head of width 1.  Request 0 owns pages [3, 0] and
    # kv_len 3 (last page holds 1); its 2 new tokens are positions 1 and 2:
    # page 3 slot 1 and page 0 slot 0.  Request 1 owns page [2], kv_len 2, and
    # one new token: position 1 = page 2 slot 1.  Request 2 appends nothing.
    k = np.arange(8, dtype=np.uint16).reshape(4, 2, 1, 1) + 100
    v = k + 1000
    k_new = np.array([7, 8, 9], dtype=np.uint16).reshape(3, 1, 1)
    v_new = k_new + 50
    kc, vc = oracle.append_paged_kv(k, v, k_new, v_new, [0, 2, 3, 3], [0, 2, 3, 4],
                                    [3, 0, 2, 1], [1, 2, 1], page_size=2)
    want_k = k.copy()
    want_k[3, 1], want_k[0, 0], want_k[2, 1] = 7, 8, 9
    want_v = v.copy()
    want_v[3, 1], want_v[0, 0], want_v[2, 1] = 57, 58, 59
    assert np.array_equal(kc, want_k) and np.array_equal(vc, want_v)
    # the inputs are not modified
    assert k[3, 1, 0, 0] == 107


@pytest.mark.parametrize("P,chunk", [(1, 5), (16, 24), (16, 100), (64, 48)])
def test_round_trip_against_generated_cache(P, chunk):
    store = wl.PagedStore([wl.Sequence(300 + i, pre, new) for i, (pre, new) in
                           enumerate([(0, 130), (37, 64), (500, 3), (16, 0)])], 4, 2, 16, P,
                          "cpu", layout_seed=P)
    full_k, full_v = wl.bf16_bits(store.k_cache), wl.bf16_bits(store.v_cache)
    for call in wl.chunked_calls(store, chunk):
        k_new, v_new = wl.new_kv_rows(call)
        kc, vc = store.k_cache.clone(), store.v_cache.clone()
        wl.clear_slots(call, kc, vc, 0.0)
        # the cleared cache differs wherever the call appends
        if call.total_q:
            assert not np.array_equal(wl.bf16_bits(kc), full_k)
        got_k, got_v = oracle.append_paged_kv(
            wl.bf16_bits(kc), wl.bf16_bits(vc), wl.bf16_bits(k_new), wl.bf16_bits(v_new),
            call.qo_indptr.numpy(), call.kv_indptr.numpy(), call.kv_indices.numpy(),
            call.kv_last_page_len.numpy(), page_size=P)
        # NaN slots compare by bits
        assert np.array_equal(got_k, full_k) and np.array_equal(got_v, full_v)


def test_attention_after_append_equals_attention_on_the_full_cache():
    store = wl.PagedStore([wl.Sequence(41, 200, 60), wl.Sequence(42, 0, 90)], 8, 2, 64, 16,
                          "cpu", layout_seed=5)
    call = wl.chunked_calls(store, 40)[1]
    want_o, want_l = oracle_on_call(call)
    k_new, v_new = wl.new_kv_rows(call)
    kc, vc = store.k_cache.clone(), store.v_cache.clone()
    wl.clear_slots(call, kc, vc)  # NaN: any miss shows in the output
    got_k, got_v = oracle.append_paged_kv(
        wl.bf16_bits(kc), wl.bf16_bits(vc), wl.bf16_bits(k_new), wl.bf16_bits(v_new),
        call.qo_indptr.numpy(), call.kv_indptr.numpy(), call.kv_indices.numpy(),
        call.kv_last_page_len.numpy(), page_size=16)
    o, l = oracle.attention(wl.bf16_bits(call.q), got_k, got_v, call.qo_indptr.numpy(),
                            call.kv_indptr.numpy(), call.kv_indices.numpy(),
                            call.kv_last_page_len.numpy(), num_qo_heads=8, num_kv_heads=2,
                            head_dim=64, page_size=16)
    assert np.array_equal(o, want_o) and np.array_equal(l, want_l, equal_nan=True)


def test_errors():
    k = np.zeros((2, 4, 1, 8), np.uint16)
    new = np.zeros((3, 1, 8), np.uint16)
    with pytest.raises(ValueError):  # 3 new tokens, 2 keys
        oracle.append_paged_kv(k, k, new, new, [0, 3], [0, 1], [0], [2], page_size=4)
    with pytest.raises(ValueError):  # page 5 of a 2-page cache
        oracle.append_paged_kv(k, k, new, new, [0, 3], [0, 1], [5], [4], page_size=4)
