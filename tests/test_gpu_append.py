"""bia_append_paged_kv on the GPU against the oracle's append, bit for bit,
and append followed by an extend call against the extend on a cache that
already held the chunk."""
import numpy as np
import pytest
import torch

import invariant_paged_attention_gb300 as bia
import oracle
import workloads as wl
from tests.gpu_util import run_prefill, same_bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _append(call, kc, vc, k_new, v_new, status=None, kv_indices=None):
    st = call.store
    desc = bia.make_desc(st.num_qo_heads, st.num_kv_heads, st.head_dim, st.page_size)
    idx = call.kv_indices if kv_indices is None else kv_indices
    bia.bia_append_paged_kv(desc, k_new, v_new, kc, vc, call.qo_indptr.to(DEV),
                            call.kv_indptr.to(DEV), idx.to(DEV), call.kv_last_page_len.to(DEV),
                            call.qo_indptr, call.kv_indptr, call.kv_last_page_len, status=status)


def _oracle_append(call, kc, vc, k_new, v_new):
    return oracle.append_paged_kv(
        wl.bf16_bits(kc), wl.bf16_bits(vc), wl.bf16_bits(k_new), wl.bf16_bits(v_new),
        call.qo_indptr.numpy(), call.kv_indptr.numpy(), call.kv_indices.numpy(),
        call.kv_last_page_len.numpy(), page_size=call.store.page_size)


@pytest.mark.parametrize("Hq,Hkv,D,P,chunk", [(32, 8, 128, 1, 300), (32, 8, 128, 16, 64),
                                              (16, 2, 64, 64, 100), (8, 8, 128, 256, 1000),
                                              (32, 8, 96, 16, 64)])
def test_append_matches_oracle_bitwise(Hq, Hkv, D, P, chunk):
    store = wl.PagedStore([wl.Sequence(700 + i, pre, new) for i, (pre, new) in
                           enumerate([(0, 1000), (3000, 77), (5, 0), (129, 640), (0, 1)])],
                          Hq, Hkv, D, P, DEV, layout_seed=P + 3)
    full_k, full_v = wl.bf16_bits(store.k_cache), wl.bf16_bits(store.v_cache)
    for call in wl.chunked_calls(store, chunk):
        k_new, v_new = wl.new_kv_rows(call)
        kc, vc = store.k_cache.clone(), store.v_cache.clone()
        wl.clear_slots(call, kc, vc, 0.0)
        want_k, want_v = _oracle_append(call, kc, vc, k_new, v_new)
        status = torch.full((1,), 77, dtype=torch.int32, device=DEV)
        _append(call, kc, vc, k_new, v_new, status=status)
        torch.cuda.synchronize()
        assert np.array_equal(wl.bf16_bits(kc), want_k)
        assert np.array_equal(wl.bf16_bits(vc), want_v)
        assert np.array_equal(want_k, full_k) and np.array_equal(want_v, full_v)
        assert int(status.item()) == 0  # zeroed by the call, no bad page


def test_append_then_extend_equals_extend_on_filled_cache():
    store = wl.PagedStore([wl.Sequence(800 + i, pre, new) for i, (pre, new) in
                           enumerate([(0, 512), (1000, 256), (77, 130)])], 32, 8, 128, 16, DEV,
                          layout_seed=8)
    kc, vc = store.k_cache.clone(), store.v_cache.clone()
    for call in wl.chunked_calls(store, 128):  # 4 q tiles of 32 tokens per chunk
        wl.clear_slots(call, kc, vc)  # NaN until the append writes them
    for call in wl.chunked_calls(store, 128):
        k_new, v_new = wl.new_kv_rows(call)
        _append(call, kc, vc, k_new, v_new)
        want_o, want_l = run_prefill(call)  # on the generator's filled cache
        got_o, got_l = run_prefill(call, k_cache=kc, v_cache=vc)
        assert same_bits(got_o, want_o) and same_bits(got_l, want_l)
    assert same_bits(kc, store.k_cache) and same_bits(vc, store.v_cache)


def test_empty_calls_and_requests():
    store = wl.PagedStore([wl.Sequence(900, 40, 0), wl.Sequence(901, 0, 3)], 4, 1, 64, 16, DEV)
    call = wl.whole_prefill(store)
    kc, vc = store.k_cache.clone(), store.v_cache.clone()
    wl.clear_slots(call, kc, vc, 0.0)
    before = bia.bia_launch_count()
    k_new, v_new = wl.new_kv_rows(call)
    _append(call, kc, vc, k_new, v_new)
    assert bia.bia_launch_count() == before + 1
    assert same_bits(kc, store.k_cache) and same_bits(vc, store.v_cache)
    # nothing to append: no kernel, caches untouched, status zeroed
    none = wl.make_call(store, [(0, 0, 0), (1, 3, 3)])
    status = torch.full((1,), 5, dtype=torch.int32, device=DEV)
    k0 = torch.empty((0, 1, 64), dtype=torch.bfloat16, device=DEV)
    _append(none, kc, vc, k0, k0, status=status)
    torch.cuda.synchronize()
    assert bia.bia_launch_count() == before + 1 and int(status.item()) == 0
    assert same_bits(kc, store.k_cache)


def test_bad_page_sets_status_and_skips_only_that_token():
    store = wl.PagedStore([wl.Sequence(910, 0, 40), wl.Sequence(911, 20, 30)], 8, 2, 128, 16,
                          DEV, layout_seed=4)
    call = wl.whole_prefill(store)
    kc, vc = store.k_cache.clone(), store.v_cache.clone()
    wl.clear_slots(call, kc, vc, 0.0)
    cleared_k = kc.clone()
    bad = call.kv_indices.clone()
    bad[1] = store.num_pages + 5  # request 0, tokens 16..31
    k_new, v_new = wl.new_kv_rows(call)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    _append(call, kc, vc, k_new, v_new, status=status, kv_indices=bad)
    assert bia.bia_read_status(status) & 1
    # every other token landed, the bad page's tokens did not
    good = call.kv_indices[torch.arange(len(bad)) != 1].long()
    assert same_bits(kc[good.to(DEV)], store.k_cache[good.to(DEV)])
    assert same_bits(kc[call.kv_indices[1].long()], cleared_k[call.kv_indices[1].long()])


def test_host_validation():
    store = wl.PagedStore([wl.Sequence(920, 0, 8)], 4, 1, 64, 16, DEV)
    call = wl.whole_prefill(store)
    desc = bia.make_desc(4, 1, 64, 16)
    k_new, v_new = wl.new_kv_rows(call)
    args = [call.qo_indptr.to(DEV), call.kv_indptr.to(DEV), call.kv_indices.to(DEV),
            call.kv_last_page_len.to(DEV)]
    too_many = torch.tensor([0, 9], dtype=torch.int32)  # 9 new tokens, 8 keys
    with pytest.raises(bia.BiaError) as e:
        bia.bia_append_paged_kv(desc, k_new, v_new, store.k_cache, store.v_cache, too_many.to(DEV),
                                *args[1:], too_many, call.kv_indptr, call.kv_last_page_len)
    assert e.value.status == bia.BIA_ERR_INVALID_ARG
    with pytest.raises(bia.BiaError) as e:
        bia.bia_append_paged_kv(bia.make_desc(4, 1, 80, 16), k_new, v_new, store.k_cache,
                                store.v_cache, *args, call.qo_indptr, call.kv_indptr,
                                call.kv_last_page_len)
    assert e.value.status == bia.BIA_ERR_UNSUPPORTED


def test_full_size_extend_append():
    # 8 requests x 4096 new tokens after a 4096-token prefix, 8 kv heads of 128:
    # 32768 tokens, 2 x 64 MiB of new rows scattered into single-slot pages
    store = wl.PagedStore([wl.Sequence(950 + i, 4096, 4096) for i in range(8)], 32, 8, 128, 1,
                          DEV, layout_seed=95)
    call = wl.whole_prefill(store)
    k_new, v_new = wl.new_kv_rows(call)
    kc, vc = store.k_cache.clone(), store.v_cache.clone()
    kvi = call.kv_indices.long()
    # the new tokens' slots (page size 1: one page per position)
    new_pages = torch.cat([kvi[int(call.kv_indptr[b]) + 4096:int(call.kv_indptr[b + 1])]
                           for b in range(8)]).to(DEV)
    kc[new_pages] = 0
    vc[new_pages] = 0
    want_k, want_v = _oracle_append(call, kc, vc, k_new, v_new)
    _append(call, kc, vc, k_new, v_new)
    torch.cuda.synchronize()
    assert np.array_equal(wl.bf16_bits(kc), want_k) and np.array_equal(wl.bf16_bits(vc), want_v)
    assert same_bits(kc, store.k_cache) and same_bits(vc, store.v_cache)
    # the rows landed where the definition puts them: token t of request b at
    # page kv_indices[kv_indptr[b] + 4096 + t]
    assert same_bits(kc[new_pages].view(-1, 8, 128), k_new)
