"""Bounded calls (launch sized from upper bounds, index arrays read on the
device only): the same bits as the exact calls on the same inputs; lengths
beyond the bounds compute nothing and set status bit 1; and one captured
CUDA graph (append + extend, append + decode) replays across serving steps
whose lengths and page tables grow, matching eager calls bit for bit and the
oracle within tolerance, with the fixed split-KV tiles kept ("sglang PR
#10417 [POC] Support deterministic inference", Modifications: split-KV is
turned off under CUDA graphs there)."""
import pytest
import torch

import invariant_paged_attention_gb300 as bia
import workloads as wl
from tests.gpu_util import check_rows, desc_of, run_decode, run_prefill, same_bits

pytestmark = pytest.mark.gpu
DEV = "cuda"
STATUS_PLAN = 2  # bit 1 of the status word


def bounded_prefill(call, bounds, q=None, split=0):
    st = call.store
    desc = desc_of(st)
    ws = torch.empty(bia.bia_prefill_bounded_workspace_size(desc, bounds, call.batch, True, split),
                     dtype=torch.uint8, device=DEV)
    rows = max(bounds.max_total_q, call.total_q)  # room for a call beyond its bounds
    qb = torch.zeros((rows, st.num_qo_heads, st.head_dim), dtype=torch.bfloat16, device=DEV)
    qb[:call.total_q] = call.q if q is None else q
    out = torch.full_like(qb, float("nan"))
    lse = torch.full((rows, st.num_qo_heads), float("nan"), dtype=torch.float32, device=DEV)
    bia.bia_prefill_paged_bounded(desc, bounds, qb, st.k_cache, st.v_cache,
                                  call.qo_indptr.to(DEV), call.kv_indptr.to(DEV),
                                  call.kv_indices.to(DEV), call.kv_last_page_len.to(DEV), ws, out,
                                  lse, split_size=split)
    return out, lse, bia.bia_read_status(ws)


def bounded_decode(call, bounds, split=0):
    st = call.store
    desc = desc_of(st)
    ws = torch.empty(bia.bia_decode_bounded_workspace_size(desc, bounds, call.batch, split),
                     dtype=torch.uint8, device=DEV)
    out = torch.full_like(call.q, float("nan"))
    lse = torch.full((call.batch, st.num_qo_heads), float("nan"), dtype=torch.float32, device=DEV)
    bia.bia_decode_paged_bounded(desc, bounds, call.q, st.k_cache, st.v_cache,
                                 call.kv_indptr.to(DEV), call.kv_indices.to(DEV),
                                 call.kv_last_page_len.to(DEV), ws, out, lse, split_size=split)
    return out, lse, bia.bia_read_status(ws)


@pytest.mark.parametrize("page_size,split", [(1, 0), (16, 1024)])
def test_bounded_prefill_matches_the_exact_call_bit_for_bit(page_size, split):
    # prefixes and lengths spanning several split tiles, a single-token tail
    # tile (33 new tokens: 32 + 1) and a one-token extend
    store = wl.PagedStore([wl.Sequence(8600 + i, p, n) for i, (p, n) in
                           enumerate([(0, 700), (5000, 33), (3000, 1), (100, 2000)])],
                          32, 8, 128, page_size, DEV, layout_seed=86)
    call = wl.whole_prefill(store)
    want_o, want_l = run_prefill(call, split=split)
    # loose bounds: room for far more work than this call needs
    bounds = bia.make_bounds(4096, 12000, call.total_q + 500)
    got_o, got_l, status = bounded_prefill(call, bounds, split=split)
    assert status == 0
    n = call.total_q
    assert same_bits(got_o[:n], want_o) and same_bits(got_l[:n], want_l)
    assert torch.isnan(got_o[n:].float()).all()  # rows past the call stay untouched


@pytest.mark.parametrize("page_size", [1, 16])
def test_bounded_decode_matches_the_exact_call_bit_for_bit(page_size):
    store = wl.PagedStore([wl.Sequence(8700 + i, c - 1, 1) for i, c in
                           enumerate([9000, 1, 2048, 2049, 300, 17000])], 32, 8, 128, page_size,
                          DEV, layout_seed=87)
    call = wl.whole_prefill(store)
    want_o, want_l = run_decode(call)
    got_o, got_l, status = bounded_decode(call, bia.make_bounds(1, 32768, 0))
    assert status == 0
    assert same_bits(got_o, want_o) and same_bits(got_l, want_l)


def test_lengths_beyond_the_bounds_compute_nothing_and_set_the_status():
    """Nothing is computed, the status says so, and out / lse read NaN (a
    stale value would pass unnoticed under graph replay)."""
    store = wl.PagedStore([wl.Sequence(8800 + i, c - 1, 1) for i, c in enumerate([500, 3000])],
                          32, 8, 128, 16, DEV, layout_seed=88)
    call = wl.whole_prefill(store)
    st = call.store
    desc = desc_of(st)
    bd = bia.make_bounds(1, 2999, 0)
    ws = torch.empty(bia.bia_decode_bounded_workspace_size(desc, bd, call.batch),
                     dtype=torch.uint8, device=DEV)
    out = torch.zeros_like(call.q)  # zeros, not NaN: the call must overwrite them
    lse = torch.zeros((call.batch, st.num_qo_heads), dtype=torch.float32, device=DEV)
    bia.bia_decode_paged_bounded(desc, bd, call.q, st.k_cache, st.v_cache,
                                 call.kv_indptr.to(DEV), call.kv_indices.to(DEV),
                                 call.kv_last_page_len.to(DEV), ws, out, lse)
    assert bia.bia_read_status(ws) & STATUS_PLAN
    assert torch.isnan(out.float()).all() and torch.isnan(lse).all()
    pstore = wl.PagedStore([wl.Sequence(8900 + i, p, n) for i, (p, n) in
                            enumerate([(0, 300), (64, 64)])], 32, 8, 128, 16, DEV, layout_seed=89)
    pcall = wl.whole_prefill(pstore)
    for bounds in (bia.make_bounds(299, 4096, 1000),   # q_len 300 > 299
                   bia.make_bounds(300, 299, 1000),    # kv_len 300 > 299
                   bia.make_bounds(300, 4096, 363)):   # 364 tokens > 363
        out, lse, status = bounded_prefill(pcall, bounds)
        assert status & STATUS_PLAN
        assert torch.isnan(out.float()).all() and torch.isnan(lse).all()


class Replay:
    """Device index buffers sized for the last step; each step's arrays are
    copied in before a replay."""

    def __init__(self, calls):
        last = calls[-1]
        self.qo = torch.zeros(last.batch + 1, dtype=torch.int32, device=DEV)
        self.kvp = torch.zeros(last.batch + 1, dtype=torch.int32, device=DEV)
        self.idx = torch.zeros(max(len(c.kv_indices) for c in calls), dtype=torch.int32,
                               device=DEV)
        self.last = torch.zeros(last.batch, dtype=torch.int32, device=DEV)

    def load(self, call):
        self.qo.copy_(call.qo_indptr)
        self.kvp.copy_(call.kv_indptr)
        self.idx.zero_()
        self.idx[:len(call.kv_indices)].copy_(call.kv_indices)
        self.last.copy_(call.kv_last_page_len)


def _capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the capture
        fn(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn(torch.cuda.current_stream())
    return graph


def test_graph_replays_decode_steps_while_every_context_grows():
    steps = 4
    ctx0 = [9000, 2047, 4095, 300]  # two of them cross a 2048-key split tile on the way
    store = wl.PagedStore([wl.Sequence(9100 + i, c - 1, steps) for i, c in enumerate(ctx0)],
                          32, 8, 128, 16, DEV, layout_seed=91)
    calls = [wl.make_call(store, [(i, s, s + 1) for i in range(len(ctx0))]) for s in range(steps)]
    # the appends below must write the new keys: poison their slots first
    wl.clear_slots(wl.make_call(store, [(i, 0, steps) for i in range(len(ctx0))]), store.k_cache,
                   store.v_cache)
    desc = desc_of(store)
    B = len(ctx0)
    bounds = bia.make_bounds(1, max(ctx0) + steps, 0)
    ws = torch.empty(bia.bia_decode_bounded_workspace_size(desc, bounds, B), dtype=torch.uint8,
                     device=DEV)
    buf = Replay(calls)
    q = torch.empty_like(calls[0].q)
    k_new, v_new = (torch.empty((B, 8, 128), dtype=torch.bfloat16, device=DEV) for _ in range(2))
    ap = torch.arange(B + 1, dtype=torch.int32)
    ap_dev = ap.to(DEV)  # made before the capture: no host copies inside it
    out = torch.empty_like(q)
    lse = torch.empty(B, 32, dtype=torch.float32, device=DEV)

    def step(stream):
        bia.bia_append_paged_kv(desc, k_new, v_new, store.k_cache, store.v_cache, ap_dev,
                                buf.kvp, buf.idx, buf.last, ap, calls[0].kv_indptr,
                                calls[0].kv_last_page_len, stream=stream)
        bia.bia_decode_paged_bounded(desc, bounds, q, store.k_cache, store.v_cache, buf.kvp,
                                     buf.idx, buf.last, ws, out, lse, stream=stream)

    def load(s):
        buf.load(calls[s])
        q.copy_(calls[s].q)
        kn, vn = wl.new_kv_rows(calls[s])
        k_new.copy_(kn)
        v_new.copy_(vn)

    load(0)
    graph = _capture(step)
    for s in range(steps):
        load(s)
        graph.replay()
        torch.cuda.synchronize()
        assert bia.bia_read_status(ws) == 0, s
        g_o, g_l = out.clone(), lse.clone()
        e_o, e_l = run_decode(calls[s])  # eager exact call on the cache the replay appended to
        assert same_bits(g_o, e_o) and same_bits(g_l, e_l), s
        check_rows(calls[s], g_o, g_l)


def test_graph_replays_chunked_extend_steps_while_every_prefix_grows():
    steps, C = 3, 256  # chunks on the 32-token grid
    prefixes = [0, 3900, 130, 8000]  # the second crosses a 4096-key split tile mid-way
    store = wl.PagedStore([wl.Sequence(9200 + i, p, steps * C) for i, p in enumerate(prefixes)],
                          32, 8, 128, 16, DEV, layout_seed=92)
    calls = [wl.make_call(store, [(i, s * C, (s + 1) * C) for i in range(len(prefixes))])
             for s in range(steps)]
    wl.clear_slots(wl.make_call(store, [(i, 0, steps * C) for i in range(len(prefixes))]),
                   store.k_cache, store.v_cache)
    desc = desc_of(store)
    B = len(prefixes)
    bounds = bia.make_bounds(C, max(prefixes) + steps * C, B * C)
    ws = torch.empty(bia.bia_prefill_bounded_workspace_size(desc, bounds, B), dtype=torch.uint8,
                     device=DEV)
    buf = Replay(calls)
    q = torch.empty((B * C, 32, 128), dtype=torch.bfloat16, device=DEV)
    k_new, v_new = (torch.empty((B * C, 8, 128), dtype=torch.bfloat16, device=DEV)
                    for _ in range(2))
    out = torch.empty_like(q)
    lse = torch.empty(B * C, 32, dtype=torch.float32, device=DEV)

    def step(stream):
        bia.bia_append_paged_kv(desc, k_new, v_new, store.k_cache, store.v_cache, buf.qo,
                                buf.kvp, buf.idx, buf.last, calls[0].qo_indptr,
                                calls[0].kv_indptr, calls[0].kv_last_page_len, stream=stream)
        bia.bia_prefill_paged_bounded(desc, bounds, q, store.k_cache, store.v_cache, buf.qo,
                                      buf.kvp, buf.idx, buf.last, ws, out, lse, stream=stream)

    def load(s):
        buf.load(calls[s])
        q.copy_(calls[s].q)
        kn, vn = wl.new_kv_rows(calls[s])
        k_new.copy_(kn)
        v_new.copy_(vn)

    load(0)
    graph = _capture(step)
    for s in range(steps):
        load(s)
        graph.replay()
        torch.cuda.synchronize()
        assert bia.bia_read_status(ws) == 0, s
        g_o, g_l = out.clone(), lse.clone()
        e_o, e_l = run_prefill(calls[s])
        assert same_bits(g_o, e_o) and same_bits(g_l, e_l), s
        check_rows(calls[s], g_o, g_l, tokens_per_part=64, seed=s)


def test_device_arrays_that_disagree_with_the_host_mirrors_give_nan():
    """An exact call whose device index arrays differ from the host mirrors it
    was sized from: nothing is computed, status bit 1, out and lse read NaN."""
    store = wl.PagedStore([wl.Sequence(8850 + i, c - 1, 1) for i, c in enumerate([3000, 5000])],
                          32, 8, 128, 1, DEV, layout_seed=885)
    call = wl.whole_prefill(store)
    desc = desc_of(store)
    short = wl.make_call(wl.PagedStore([wl.Sequence(8850, 999, 1), wl.Sequence(8851, 4999, 1)],
                                       32, 8, 128, 1, DEV, layout_seed=885),
                         [(0, 0, 1), (1, 0, 1)])
    ws = torch.empty(bia.bia_decode_workspace_size(desc, short.kv_indptr, short.kv_last_page_len),
                     dtype=torch.uint8, device=DEV)
    out = torch.zeros_like(call.q)
    lse = torch.zeros((2, 32), dtype=torch.float32, device=DEV)
    # host mirrors of a 1000-key first request, device arrays of a 3000-key one
    bia.bia_decode_paged(desc, call.q, store.k_cache, store.v_cache, call.kv_indptr.to(DEV),
                         call.kv_indices.to(DEV), call.kv_last_page_len.to(DEV),
                         short.kv_indptr, short.kv_last_page_len, ws, out, lse)
    assert bia.bia_read_status(ws) & STATUS_PLAN
    assert torch.isnan(out.float()).all() and torch.isnan(lse).all()
