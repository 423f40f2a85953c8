"""The C ABI refuses, before enqueuing anything, any buffer that is not device
memory of the current GPU: pinned host memory (which a kernel could reach
through unified addressing) is rejected with BIA_ERR_INVALID_ARG and no
kernel is launched.  The prefill kernels multicast their K/V gathers inside
thread-block clusters, which the library does for this GPU's own memory
only.  Called through the raw C entry points: the binding refuses host
tensors itself before the library sees them."""
import ctypes

import pytest
import torch

import invariant_paged_attention_gb300 as bia
import workloads as wl
from tests.gpu_util import desc_of

pytestmark = pytest.mark.gpu
DEV = "cuda"
p = ctypes.c_void_p


def ptr(t):
    return p(t.data_ptr())


def _decode_args(store, call):
    ws = torch.empty(bia.bia_decode_workspace_size(desc_of(store), call.kv_indptr,
                                                   call.kv_last_page_len),
                     dtype=torch.uint8, device=DEV)
    return dict(q=call.q, k=store.k_cache, v=store.v_cache, kvp=call.kv_indptr.to(DEV),
                idx=call.kv_indices.to(DEV), last=call.kv_last_page_len.to(DEV), ws=ws,
                out=torch.empty_like(call.q))


def _decode(lib, desc, call, a):
    return lib.bia_decode_paged(ctypes.byref(desc), ptr(a["q"]), ptr(a["k"]), ptr(a["v"]),
                                a["k"].shape[0], ptr(a["kvp"]), ptr(a["idx"]), ptr(a["last"]),
                                ptr(call.kv_indptr), ptr(call.kv_last_page_len), call.batch, 0,
                                ptr(a["ws"]), a["ws"].numel(), ptr(a["out"]), None, None)


@pytest.mark.parametrize("which", ["q", "k", "idx", "ws", "out"])
def test_decode_refuses_a_pinned_host_buffer(which):
    lib = bia.load()
    store = wl.PagedStore([wl.Sequence(9500 + i, c - 1, 1) for i, c in enumerate([700, 40])],
                          32, 8, 128, 16, DEV, layout_seed=95)
    call = wl.whole_prefill(store)
    desc = desc_of(store)
    a = _decode_args(store, call)
    assert _decode(lib, desc, call, a) == bia.BIA_OK  # the device buffers are accepted
    torch.cuda.synchronize()
    host = a[which].cpu().pin_memory()
    a[which] = host
    before = lib.bia_launch_count()
    assert _decode(lib, desc, call, a) == bia.BIA_ERR_INVALID_ARG
    assert lib.bia_launch_count() == before
    assert b"not device memory" in lib.bia_last_error()


def test_prefill_and_merge_refuse_pinned_host_buffers():
    lib = bia.load()
    store = wl.PagedStore([wl.Sequence(9600, 0, 200)], 32, 8, 128, 16, DEV, layout_seed=96)
    call = wl.whole_prefill(store)
    desc = desc_of(store)
    ws = torch.empty(bia.bia_prefill_workspace_size(desc, call.qo_indptr, call.kv_indptr,
                                                    call.kv_last_page_len),
                     dtype=torch.uint8, device=DEV)
    out = torch.empty_like(call.q)
    k_host = store.k_cache.cpu().pin_memory()
    before = lib.bia_launch_count()
    rc = lib.bia_prefill_paged(ctypes.byref(desc), ptr(call.q), ptr(k_host), ptr(store.v_cache),
                               store.k_cache.shape[0], ptr(call.qo_indptr.to(DEV)),
                               ptr(call.kv_indptr.to(DEV)), ptr(call.kv_indices.to(DEV)),
                               ptr(call.kv_last_page_len.to(DEV)), ptr(call.qo_indptr),
                               ptr(call.kv_indptr), ptr(call.kv_last_page_len), 1, 1, 0, ptr(ws),
                               ws.numel(), ptr(out), None, None)
    assert rc == bia.BIA_ERR_INVALID_ARG
    assert b"k_cache" in lib.bia_last_error()
    v = torch.zeros(4, 2, 8, 128, dtype=torch.float32).pin_memory()
    s = torch.zeros(4, 2, 8, dtype=torch.float32, device=DEV)
    mo = torch.empty(4, 8, 128, dtype=torch.bfloat16, device=DEV)
    assert lib.bia_merge_states(ptr(v), ptr(s), None, 4, 2, 8, 128, ptr(mo), None,
                                None) == bia.BIA_ERR_INVALID_ARG
    assert lib.bia_launch_count() == before
