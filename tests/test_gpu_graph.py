"""The entry points inside a CUDA graph: nothing in a call copies host data to
the device (the plan is built by a device kernel from the device index
arrays), so a prefill + decode step captured once replays with new q and K/V
values and gives the same bits as eager calls on those values."""
import pytest
import torch

import invariant_paged_attention_gb300 as bia
import workloads as wl
from tests.gpu_util import same_bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _setup(call, store, decode):
    desc = bia.make_desc(store.num_qo_heads, store.num_kv_heads, store.head_dim,
                         store.page_size)
    if decode:
        nbytes = bia.bia_decode_workspace_size(desc, call.kv_indptr, call.kv_last_page_len)
    else:
        nbytes = bia.bia_prefill_workspace_size(desc, call.qo_indptr, call.kv_indptr,
                                                call.kv_last_page_len)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    out = torch.empty_like(call.q)
    lse = torch.empty(call.total_q, store.num_qo_heads, dtype=torch.float32, device=DEV)
    idx = [call.qo_indptr.to(DEV), call.kv_indptr.to(DEV), call.kv_indices.to(DEV),
           call.kv_last_page_len.to(DEV)]

    def run(q, stream=None):
        if decode:
            bia.bia_decode_paged(desc, q, store.k_cache, store.v_cache, idx[1], idx[2], idx[3],
                                 call.kv_indptr, call.kv_last_page_len, ws, out, lse,
                                 stream=stream)
        else:
            bia.bia_prefill_paged(desc, q, store.k_cache, store.v_cache, *idx, call.qo_indptr,
                                  call.kv_indptr, call.kv_last_page_len, ws, out, lse,
                                  stream=stream)
        return out, lse
    return run


def test_captured_prefill_and_decode_replay_bit_identically():
    pstore = wl.PagedStore([wl.Sequence(8100 + i, p, n) for i, (p, n) in
                            enumerate([(0, 700), (5000, 64), (100, 33)])], 32, 8, 128, 1, DEV,
                           layout_seed=81)
    dstore = wl.PagedStore([wl.Sequence(8200 + i, c - 1, 1) for i, c in
                            enumerate([9000, 2048, 300])], 32, 8, 128, 16, DEV, layout_seed=82)
    pcall, dcall = wl.whole_prefill(pstore), wl.whole_prefill(dstore)
    prun = _setup(pcall, pstore, decode=False)
    drun = _setup(dcall, dstore, decode=True)
    pq = pcall.q.clone()
    dq = dcall.q.clone()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the capture
        prun(pq, stream=side)
        drun(dq, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        s = torch.cuda.current_stream()
        pout, plse = prun(pq, stream=s)
        dout, dlse = drun(dq, stream=s)

    for trial in range(3):
        # new inputs in the captured buffers, then replay
        pq.copy_(wl.draw_normal_bf16(pq.shape, 9000 + trial, DEV))
        dq.copy_(wl.draw_normal_bf16(dq.shape, 9100 + trial, DEV))
        graph.replay()
        torch.cuda.synchronize()
        g = [t.clone() for t in (pout, plse, dout, dlse)]
        e_pout, e_plse = prun(pq)
        e_pout, e_plse = e_pout.clone(), e_plse.clone()
        e_dout, e_dlse = drun(dq)
        torch.cuda.synchronize()
        assert same_bits(g[0], e_pout) and same_bits(g[1], e_plse)
        assert same_bits(g[2], e_dout) and same_bits(g[3], e_dlse)
        assert torch.isfinite(g[0].float()).all()
