"""Single-token q tiles of a prefill call (one-token extends, and the
one-token tail tile of a longer request) run on the streaming kernel with the
prefill split size.  Parity with the oracle at every head dim and group size,
across split tiles, causal and not; bits that do not depend on the batch; and
a request chunked on the q-tile grid (its last chunk a single token)
bit-identical to the unchunked run, whose tail tile is streamed the same
way."""
import pytest

import invariant_paged_attention_gb300 as bia
import workloads as wl
from tests.gpu_util import check_rows, run_prefill, same_bits

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [  # (Hq, Hkv, D, P, [(prefix, new)], causal)
    # G = 4 (32-token tiles): 33 and 65 end in a one-token tile; 8193 keys
    # span three split tiles of 4096
    (32, 8, 128, 16, [(0, 1), (4095, 1), (8192, 1), (31, 33), (100, 65), (5000, 1)], True),
    (32, 8, 128, 1, [(0, 1), (8192, 1), (31, 33), (4000, 97)], False),
    # G = 1 (128-token tiles)
    (16, 16, 64, 16, [(0, 129), (300, 1), (9000, 257)], True),
    # G = 8 (16-token tiles), head_dim 96 on the 128-wide layout
    (32, 4, 96, 16, [(0, 17), (70, 1), (4000, 33)], True),
    # G = 2 (64-token tiles), head_dim 256
    (16, 8, 256, 1, [(0, 65), (5000, 1), (4100, 129)], True),
]


@pytest.mark.parametrize("Hq,Hkv,D,P,seqs,causal", CASES)
def test_streamed_tiles_match_oracle(Hq, Hkv, D, P, seqs, causal):
    store = wl.PagedStore([wl.Sequence(2400 + i, p, n) for i, (p, n) in enumerate(seqs)],
                          Hq, Hkv, D, P, DEV, layout_seed=41)
    call = wl.whole_prefill(store)
    out, lse = run_prefill(call, causal=causal)
    check_rows(call, out, lse, causal=causal)


def test_streamed_tile_other_split_size():
    store = wl.PagedStore([wl.Sequence(2500 + i, p, n) for i, (p, n) in
                           enumerate([(3000, 1), (700, 33)])], 32, 8, 128, 16, DEV,
                          layout_seed=42)
    call = wl.whole_prefill(store)
    out, lse = run_prefill(call, split=1024)
    check_rows(call, out, lse)


def test_one_token_tail_chunked_on_the_grid_is_bit_identical():
    # G = 4: the grid is 32 tokens; 65 new tokens end in a one-token tile,
    # which the unchunked call and the chunked calls both stream
    store = wl.PagedStore([wl.Sequence(2600 + i, p, n) for i, (p, n) in
                           enumerate([(100, 65), (5000, 33)])], 32, 8, 128, 16, DEV,
                          layout_seed=43)
    assert bia.bia_q_tile_tokens(4) == 32
    whole = wl.whole_prefill(store)
    ref_o, ref_l = run_prefill(whole)
    for chunk in (32, 64):
        for c in wl.chunked_calls(store, chunk):
            o, l = run_prefill(c)
            for k, (si, a, b) in enumerate(c.parts):
                base = int(whole.qo_indptr[si])
                ca, cb = int(c.qo_indptr[k]), int(c.qo_indptr[k + 1])
                assert same_bits(o[ca:cb], ref_o[base + a:base + b]), (chunk, si, a, b)
                assert same_bits(l[ca:cb], ref_l[base + a:base + b]), (chunk, si, a, b)


def test_streamed_tiles_do_not_depend_on_the_batch():
    seqs = [(8192, 1), (31, 33), (700, 300), (12000, 1), (0, 1)]
    store = wl.PagedStore([wl.Sequence(2700 + i, p, n) for i, (p, n) in enumerate(seqs)],
                          32, 8, 128, 16, DEV, layout_seed=44)
    full = wl.whole_prefill(store)
    out, lse = run_prefill(full)
    for i in range(len(seqs)):
        solo = wl.whole_prefill(wl.PagedStore([store.seqs[i]], 32, 8, 128, 16, DEV,
                                              layout_seed=50 + i, spare_pages=3))
        o, l = run_prefill(solo)
        a, b = int(full.qo_indptr[i]), int(full.qo_indptr[i + 1])
        assert same_bits(o, out[a:b]) and same_bits(l, lse[a:b]), i
    rev = wl.PagedStore([store.seqs[i] for i in reversed(range(len(seqs)))], 32, 8, 128, 16,
                        DEV, layout_seed=60)
    o, l = run_prefill(wl.whole_prefill(rev))
    pos = 0
    for i in reversed(range(len(seqs))):
        a, b = int(full.qo_indptr[i]), int(full.qo_indptr[i + 1])
        assert same_bits(o[pos:pos + b - a], out[a:b]) and same_bits(l[pos:pos + b - a], lse[a:b])
        pos += b - a
