"""bia_decode_paged_noalloc: decode for callers that cannot allocate device
memory (engine plugin hooks that may not call cudaMalloc while enqueuing
work, hosts with a fixed memory budget).  It must give what
bia_decode_paged gives with a caller workspace, call after call, although
every call shares the library's one static scratch array.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import invariant_paged_attention_gb300 as bia
import workloads as wl
from tests.common import bf16_to_f64, error_stats

MAX_ABS, MEAN_ABS = 2e-2, 2e-3  # the bf16 output tolerance used across the suite


def _decode_reference(call, desc):
    st = call.store
    dev = st.k_cache.device
    ws = torch.empty(bia.bia_decode_workspace_size(desc, call.kv_indptr, call.kv_last_page_len),
                     dtype=torch.uint8, device=dev)
    out = torch.empty_like(call.q)
    lse = torch.empty(call.total_q, st.num_qo_heads, dtype=torch.float32, device=dev)
    bia.bia_decode_paged(desc, call.q, st.k_cache, st.v_cache, call.kv_indptr.to(dev),
                         call.kv_indices.to(dev), call.kv_last_page_len.to(dev), call.kv_indptr,
                         call.kv_last_page_len, ws, out, lse)
    return out, lse


def _decode_noalloc(call, desc):
    st = call.store
    dev = st.k_cache.device
    out = torch.full_like(call.q, float("nan"))
    lse = torch.full((call.total_q, st.num_qo_heads), float("nan"), dtype=torch.float32,
                     device=dev)
    bia.bia_decode_paged_noalloc(desc, call.q, st.k_cache, st.v_cache, call.kv_indptr.to(dev),
                                 call.kv_indices.to(dev), call.kv_last_page_len.to(dev),
                                 call.kv_indptr, call.kv_last_page_len, out, lse)
    return out, lse


@pytest.mark.gpu
def test_noalloc_decode_matches_the_workspace_entry_point_twice_in_a_row():
    # two different batches back to back: the second call must not see
    # anything the first one left in the shared scratch array
    batches = [
        wl.PagedStore([wl.Sequence(7100 + i, c - 1, 1) for i, c in
                       enumerate([9000, 130, 2048, 4097, 33, 12000])], 32, 8, 128, 16, "cuda",
                      layout_seed=71),
        wl.PagedStore([wl.Sequence(7200 + i, c - 1, 1) for i, c in
                       enumerate([2049, 700, 16000])], 32, 8, 128, 1, "cuda", layout_seed=72),
    ]
    for store in batches:
        call = wl.whole_prefill(store)
        desc = bia.make_desc(store.num_qo_heads, store.num_kv_heads, store.head_dim,
                             store.page_size)
        want_o, want_l = _decode_reference(call, desc)
        got_o, got_l = _decode_noalloc(call, desc)
        torch.cuda.synchronize()
        mx, mean = error_stats(bf16_to_f64(got_o), bf16_to_f64(want_o))
        assert mx <= MAX_ABS and mean <= MEAN_ABS, (mx, mean)
        assert torch.allclose(got_l, want_l, atol=1e-3, rtol=0)
        # same kernels on the same inputs: the bits agree as well
        assert torch.equal(got_o.view(torch.int16), want_o.view(torch.int16))
        assert torch.equal(got_l, want_l)


def test_noalloc_decode_rejects_work_beyond_its_static_scratch():
    """Checked on the host before anything reaches a GPU."""
    from invariant_paged_attention_gb300 import build
    build.build()
    lib = bia.load()
    desc = bia.make_desc(32, 8, 128, 1)
    # 64 requests of 131072 keys: 64 splits each -> ~135 MB of partials
    n = 64
    kvp = torch.arange(0, (n + 1) * 131072, 131072, dtype=torch.int32)
    last = torch.ones(n, dtype=torch.int32)
    need = bia.bia_decode_workspace_size(desc, kvp, last)
    assert need > bia.BIA_DECODE_NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the call returns first
    rc = lib.bia_decode_paged_noalloc(ctypes.byref(desc), fake, fake, fake, 1 << 24, fake, fake,
                                      fake, ctypes.c_void_p(kvp.data_ptr()),
                                      ctypes.c_void_p(last.data_ptr()), n, 0, fake, None, None)
    assert rc == bia.BIA_ERR_WORKSPACE_TOO_SMALL
