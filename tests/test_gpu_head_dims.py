"""head_dim 96 (zero-padded onto the 128-wide kernels) and 256 (its own prefill
kernel: one q tile per CTA, 64-key blocks): prefill and decode
parity with the oracle, chunked prefill on the q-tile grid and batch
composition bit-identical, and the append and masked paths at that width."""
import pytest

import workloads as wl
from tests.gpu_util import check_rows, run_decode, run_prefill, same_bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("Hq,Hkv,P,seqs,causal", [
    (32, 8, 16, [(0, 300), (700, 77), (5, 1), (129, 160)], True),
    (16, 16, 1, [(0, 130), (4100, 40)], True),
    (32, 8, 16, [(10, 90), (0, 33)], False),
])
def test_prefill_d96_matches_oracle(Hq, Hkv, P, seqs, causal):
    store = wl.PagedStore([wl.Sequence(1600 + i, p, n) for i, (p, n) in enumerate(seqs)],
                          Hq, Hkv, 96, P, DEV, layout_seed=21)
    call = wl.whole_prefill(store)
    out, lse = run_prefill(call, causal=causal)
    check_rows(call, out, lse, causal=causal)


def test_decode_d96_matches_oracle():
    store = wl.PagedStore([wl.Sequence(1700 + i, c - 1, 1) for i, c in
                           enumerate([1, 100, 2048, 2049, 9000])], 32, 8, 96, 1, DEV,
                          layout_seed=22)
    call = wl.whole_prefill(store)
    out, lse = run_decode(call)
    check_rows(call, out, lse)


def test_d96_chunked_prefill_and_batch_invariance():
    store = wl.PagedStore([wl.Sequence(1800 + i, p, n) for i, (p, n) in
                           enumerate([(0, 256), (300, 200)])], 32, 8, 96, 16, DEV, layout_seed=23)
    whole = wl.whole_prefill(store)
    ref_o, ref_l = run_prefill(whole)
    # chunks of 32 tokens: the 128-row q-tile grid at G = 4
    for c in wl.chunked_calls(store, 32):
        o, l = run_prefill(c)
        for k, (si, a, b) in enumerate(c.parts):
            base = int(whole.qo_indptr[si])
            ca, cb = int(c.qo_indptr[k]), int(c.qo_indptr[k + 1])
            assert same_bits(o[ca:cb], ref_o[base + a:base + b])
            assert same_bits(l[ca:cb], ref_l[base + a:base + b])
    # request 1 alone
    solo = wl.make_call(store, [(1, 0, 200)])
    so, sl = run_prefill(solo)
    a, b = int(whole.qo_indptr[1]), int(whole.qo_indptr[2])
    assert same_bits(so, ref_o[a:b]) and same_bits(sl, ref_l[a:b])


@pytest.mark.parametrize("Hq,Hkv,P,seqs,causal", [
    (16, 8, 16, [(0, 300), (700, 77), (5, 1), (129, 160)], True),
    (8, 1, 1, [(0, 130), (4100, 70)], True),
    (32, 4, 16, [(10, 90), (0, 33)], False),
    (16, 8, 16, [(4000, 300), (0, 4200), (31, 17)], True),
    (16, 8, 32, [(1000, 250), (4090, 20)], True),
])
def test_prefill_d256_matches_oracle(Hq, Hkv, P, seqs, causal):
    store = wl.PagedStore([wl.Sequence(1900 + i, p, n) for i, (p, n) in enumerate(seqs)],
                          Hq, Hkv, 256, P, DEV, layout_seed=31)
    call = wl.whole_prefill(store)
    out, lse = run_prefill(call, causal=causal)
    check_rows(call, out, lse, causal=causal)


def test_decode_d256_matches_oracle():
    store = wl.PagedStore([wl.Sequence(2000 + i, c - 1, 1) for i, c in
                           enumerate([1, 100, 2048, 2049, 9000])], 16, 8, 256, 1, DEV,
                          layout_seed=32)
    call = wl.whole_prefill(store)
    out, lse = run_decode(call)
    check_rows(call, out, lse)


def test_d256_chunked_prefill_and_batch_invariance():
    # G = 2: the q-tile grid is 64 tokens
    store = wl.PagedStore([wl.Sequence(2100 + i, p, n) for i, (p, n) in
                           enumerate([(0, 256), (4000, 192)])], 16, 8, 256, 16, DEV,
                          layout_seed=33)
    whole = wl.whole_prefill(store)
    ref_o, ref_l = run_prefill(whole)
    for c in wl.chunked_calls(store, 64):
        o, l = run_prefill(c)
        for k, (si, a, b) in enumerate(c.parts):
            base = int(whole.qo_indptr[si])
            ca, cb = int(c.qo_indptr[k]), int(c.qo_indptr[k + 1])
            assert same_bits(o[ca:cb], ref_o[base + a:base + b])
            assert same_bits(l[ca:cb], ref_l[base + a:base + b])
    solo = wl.make_call(store, [(1, 0, 192)])
    so, sl = run_prefill(solo)
    a, b = int(whole.qo_indptr[1]), int(whole.qo_indptr[2])
    assert same_bits(so, ref_o[a:b]) and same_bits(sl, ref_l[a:b])


@pytest.mark.parametrize("Hq,Hkv", [(64, 8), (8, 8), (32, 16)])
def test_decode_d256_other_group_sizes(Hq, Hkv):
    """Group sizes 8, 1 and 2 at head_dim 256 (a chunk's lazy-rescale decision
    is taken per 2-step sub-chunk at G=8, per chunk otherwise)."""
    store = wl.PagedStore([wl.Sequence(2200 + i, c - 1, 1) for i, c in
                           enumerate([1, 3000, 4097, 200])], Hq, Hkv, 256, 16, DEV,
                          layout_seed=34)
    call = wl.whole_prefill(store)
    out, lse = run_decode(call)
    check_rows(call, out, lse)


@pytest.mark.parametrize("P", [16, 32, 256])
def test_d256_prefill_bits_do_not_depend_on_the_page_size(P):
    """With pages of 16+ keys a CTA's keys arrive as tiled boxes of whole page
    runs (rows past the sequence still gathered); at page 1 every row is
    gathered.  The shared-memory tiles and so the results are the same bits."""
    seqs = [wl.Sequence(2300 + i, p, n) for i, (p, n) in enumerate([(0, 700), (4100, 90),
                                                                    (33, 250)])]
    ref_o, ref_l = run_prefill(wl.whole_prefill(wl.PagedStore(seqs, 16, 8, 256, 1, DEV,
                                                              layout_seed=34)))
    o, l = run_prefill(wl.whole_prefill(wl.PagedStore(seqs, 16, 8, 256, P, DEV,
                                                      layout_seed=35)))
    assert same_bits(o, ref_o) and same_bits(l, ref_l)
