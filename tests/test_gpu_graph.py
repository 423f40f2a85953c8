"""The entry points inside a CUDA graph: nothing in a call copies host data to
the device (the plan is built by a device kernel from the device index
arrays), so a prefill + decode step captured once replays with new q and K/V
values and gives the same bits as eager calls on those values, and matches
the oracle on them.  Replays across steps whose lengths change are covered
by the bounded calls' tests."""
import dataclasses

import pytest
import torch

import invariant_paged_attention_gb300 as bia
import workloads as wl
from tests.gpu_util import check_rows, same_bits

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
        # and the replayed values themselves against the oracle
        check_rows(dataclasses.replace(pcall, q=pq.clone()), g[0], g[1])
        check_rows(dataclasses.replace(dcall, q=dq.clone()), g[2], g[3])


def test_captured_append_extend_and_mla_replay_bit_identically():
    """An append, then an extend whose single-token q tiles run on the
    streaming kernel, then an MLA decode, captured as one graph: replays with
    new inputs match eager calls bit for bit."""
    store = wl.PagedStore([wl.Sequence(8300 + i, p, n) for i, (p, n) in
                           enumerate([(700, 33), (5000, 1), (0, 64)])], 32, 8, 128, 16, DEV,
                          layout_seed=83)
    call = wl.whole_prefill(store)
    desc = bia.make_desc(32, 8, 128, 16)
    k_new, v_new = wl.new_kv_rows(call)
    k_new, v_new = k_new.clone(), v_new.clone()
    idx = [call.qo_indptr.to(DEV), call.kv_indptr.to(DEV), call.kv_indices.to(DEV),
           call.kv_last_page_len.to(DEV)]
    ws = torch.empty(bia.bia_prefill_workspace_size(desc, call.qo_indptr, call.kv_indptr,
                                                    call.kv_last_page_len),
                     dtype=torch.uint8, device=DEV)
    out = torch.empty_like(call.q)
    lse = torch.empty(call.total_q, 32, dtype=torch.float32, device=DEV)
    q = call.q.clone()

    mst = wl.MLAStore([wl.Sequence(8400 + i, c - 1, 1) for i, c in enumerate([3000, 129, 5000])],
                      16, 512, 64, 16, DEV, layout_seed=84)
    mc = wl.mla_call(mst, [(i, 0, 1) for i in range(3)])
    mdesc = bia.make_mla_desc(16, 16)
    mws = torch.empty(bia.bia_mla_decode_workspace_size(mdesc, mc.kv_indptr, mc.kv_last_page_len),
                      dtype=torch.uint8, device=DEV)
    mout = torch.empty((3, 16, 512), dtype=torch.bfloat16, device=DEV)
    mlse = torch.empty((3, 16), dtype=torch.float32, device=DEV)
    midx = [mc.kv_indptr.to(DEV), mc.kv_indices.to(DEV), mc.kv_last_page_len.to(DEV)]
    q_nope, q_pe = mc.q_nope.clone(), mc.q_pe.clone()

    def step(stream=None):
        bia.bia_append_paged_kv(desc, k_new, v_new, store.k_cache, store.v_cache, *idx,
                                call.qo_indptr, call.kv_indptr, call.kv_last_page_len,
                                stream=stream)
        bia.bia_prefill_paged(desc, q, store.k_cache, store.v_cache, *idx, call.qo_indptr,
                              call.kv_indptr, call.kv_last_page_len, ws, out, lse, stream=stream)
        bia.bia_mla_decode_paged(mdesc, q_nope, q_pe, mst.ckv_cache, mst.kpe_cache, *midx,
                                 mc.kv_indptr, mc.kv_last_page_len, mws, mout, mlse,
                                 stream=stream)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the capture
        step(stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(stream=torch.cuda.current_stream())

    for trial in range(2):
        q.copy_(wl.draw_normal_bf16(q.shape, 9300 + trial, DEV))
        k_new.copy_(wl.draw_normal_bf16(k_new.shape, 9400 + trial, DEV))
        v_new.copy_(wl.draw_normal_bf16(v_new.shape, 9500 + trial, DEV))
        q_nope.copy_(wl.draw_normal_bf16(q_nope.shape, 9600 + trial, DEV))
        graph.replay()
        torch.cuda.synchronize()
        g = [t.clone() for t in (out, lse, mout, mlse)]
        step()
        torch.cuda.synchronize()
        assert same_bits(g[0], out) and same_bits(g[1], lse)
        assert same_bits(g[2], mout) and same_bits(g[3], mlse)
        assert torch.isfinite(g[0].float()).all() and torch.isfinite(g[2].float()).all()


def test_capture_first_on_a_fresh_thread_matches_the_forked_eager_call():
    """A prefill call with tensor-core tiles and a streamed one-token tile runs
    the streamed tile on a per-thread side stream.  A thread whose first call
    is being captured creates no side stream and keeps the call on one
    stream; its replay gives the bits of the eager (forked) call."""
    import threading
    store = wl.PagedStore([wl.Sequence(8500 + i, p, n) for i, (p, n) in
                           enumerate([(300, 97), (4000, 1), (0, 33)])], 32, 8, 128, 16, DEV,
                          layout_seed=85)
    call = wl.whole_prefill(store)
    run = _setup(call, store, decode=False)
    q = call.q.clone()
    eager_out, eager_lse = [t.clone() for t in run(q)]  # this thread: forked
    torch.cuda.synchronize()
    result = {}

    def capture_and_replay():
        try:
            torch.cuda.set_device(torch.device(DEV).index or 0)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                out, lse = run(q, stream=torch.cuda.current_stream())
            graph.replay()
            torch.cuda.synchronize()
            result["out"], result["lse"] = out.clone(), lse.clone()
        except Exception as e:  # reported on the test's thread
            result["error"] = e

    t = threading.Thread(target=capture_and_replay)
    t.start()
    t.join()
    assert "error" not in result, result.get("error")
    assert same_bits(result["out"], eager_out) and same_bits(result["lse"], eager_lse)
    check_rows(call, result["out"], result["lse"])
