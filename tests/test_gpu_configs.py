"""The five workloads at full size on the GPU: oracle parity and bit-identity
across batch sizes, batch composition, page placement and q-tile-aligned
chunking.  Off-grid chunking is checked against the oracle only: it may
differ from the unchunked run.

Parity coverage: the tiny prefill, the batched prefill and every decode
batch are compared on every row of every request; the long prefix extend
and the mixed batch's 4096-token chunk on every request, all rows of its
first and last q tile plus a seeded sample of 128 tokens (4096 rows), and
both chunked runs (on and off the grid) also on the first and last token of
every chunk.
Rows are checked a few requests at a time so the oracle's host copies stay
small."""
import pytest
import torch

import workloads as wl
from tests.gpu_util import check_rows, run_decode, run_prefill, same_bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


def assemble(whole: wl.Call, calls, results):
    """Places the rows of chunked calls where the unchunked call has them."""
    o0, l0 = results[0]
    out = torch.full((whole.total_q,) + tuple(o0.shape[1:]), float("nan"), dtype=o0.dtype,
                     device=o0.device)
    lse = torch.full((whole.total_q,) + tuple(l0.shape[1:]), float("nan"), dtype=l0.dtype,
                     device=l0.device)
    start = {si: int(whole.qo_indptr[k]) for k, (si, _, _) in enumerate(whole.parts)}
    for call, (o, l) in zip(calls, results):
        for k, (si, a, b) in enumerate(call.parts):
            c0, c1 = int(call.qo_indptr[k]), int(call.qo_indptr[k + 1])
            out[start[si] + a:start[si] + b] = o[c0:c1]
            lse[start[si] + a:start[si] + b] = l[c0:c1]
    return out, lse


def test_cfg1_tiny_prefill_and_grid_chunks():
    store = wl.cfg1_tiny(DEV)
    whole = wl.whole_prefill(store)
    out, lse = run_prefill(whole)
    check_rows(whole, out, lse)
    calls = wl.chunked_calls(store, 32)
    assert len(calls) == 8
    o, l = assemble(whole, calls, [run_prefill(c) for c in calls])
    assert same_bits(o, out) and same_bits(l, lse)


def check_groups(call, out, lse, group, **kw):
    """check_rows over the parts `group` at a time; returns (max, mean, rows)."""
    mx = tot = n = 0.0
    for g in range(0, call.batch, group):
        m, mean, rows = check_rows(call, out, lse, part_ids=range(g, min(call.batch, g + group)),
                                   **kw)
        mx, tot, n = max(mx, m), tot + mean * rows, n + rows
    return mx, tot / max(n, 1), int(n)


def test_cfg2_batched_prefill_matches_oracle_and_solo_runs(capsys):
    store = wl.cfg2_prefill(DEV)
    call = wl.whole_prefill(store)
    out, lse = run_prefill(call)
    mx, mean, n = check_groups(call, out, lse, 1)  # every row of every request
    with capsys.disabled():
        print(f"\n[cfg2] oracle rows {n} (all): max {mx:.3e} mean {mean:.3e}")
    for i, s in enumerate(store.seqs):
        solo = wl.whole_prefill(wl.PagedStore([s], 32, 8, 128, 1, DEV, layout_seed=800 + i))
        o, l = run_prefill(solo)
        a, b = int(call.qo_indptr[i]), int(call.qo_indptr[i + 1])
        assert same_bits(o, out[a:b]) and same_bits(l, lse[a:b]), f"request {i}"


def test_cfg3_chunked_prefill_with_prefix(capsys):
    store = wl.cfg3_prefix(DEV)
    whole = wl.whole_prefill(store)
    out, lse = run_prefill(whole)
    mx, mean, n = check_rows(whole, out, lse, tokens_per_part=128)
    # chunks of 256 tokens start on the 32-token grid: bit-identical, so the
    # first and last token of every chunk are checked on the unchunked rows
    calls = wl.chunked_calls(store, 256)
    assert len(calls) == 64
    o, l = assemble(whole, calls, [run_prefill(c) for c in calls])
    assert same_bits(o, out) and same_bits(l, lse)
    grid_edges = sorted({t for c in range(64) for t in (256 * c, 256 * c + 255)})
    for i in range(whole.batch):
        check_rows(whole, out, lse, part_ids=[i], tokens=grid_edges)
    # chunks of 100 tokens leave the grid: held to the oracle only, on a
    # sample and on the first and last token of every chunk
    calls = wl.chunked_calls(store, 100)
    assert len(calls) == 164
    o, l = assemble(whole, calls, [run_prefill(c) for c in calls])
    mx2, mean2, n2 = check_rows(whole, o, l, tokens_per_part=128, seed=1)
    edges = sorted({t for c in range(164) for t in (100 * c, min(16384, 100 * c + 100) - 1)})
    for i in range(whole.batch):
        check_rows(whole, o, l, part_ids=[i], tokens=edges)
    with capsys.disabled():
        print(f"\n[cfg3] oracle rows {n}: max {mx:.3e} mean {mean:.3e}; off-grid (100) rows "
              f"{n2}: max {mx2:.3e} mean {mean2:.3e}, bit-identical to unchunked: "
              f"{same_bits(o, out)}")


def test_cfg4_decode_sweep_request0_identical_across_batch_sizes(capsys):
    first = None
    for B in (1, 8, 64, 256):
        store = wl.cfg4_decode(DEV, B)
        call = wl.whole_prefill(store)
        out, lse = run_decode(call)
        mx, mean, n = check_groups(call, out, lse, 32)  # every request
        with capsys.disabled():
            print(f"\n[cfg4 B={B}] oracle rows {n} (all): max {mx:.3e} mean {mean:.3e}")
        got = (out[0].clone(), lse[0].clone())
        if first is None:
            first = got
        else:
            assert same_bits(got[0], first[0]) and same_bits(got[1], first[1]), B
        del store, call, out, lse
        torch.cuda.empty_cache()


def test_cfg5_mixed_batch_every_request_matches_its_solo_run():
    pstore, dstore = wl.cfg5_mixed(DEV)
    pcall = wl.whole_prefill(pstore)
    out, lse = run_prefill(pcall)
    check_rows(pcall, out, lse, tokens_per_part=128)
    for i, s in enumerate(pstore.seqs):
        solo = wl.whole_prefill(wl.PagedStore([s], 32, 8, 128, 16, DEV, layout_seed=900 + i))
        o, l = run_prefill(solo)
        a, b = int(pcall.qo_indptr[i]), int(pcall.qo_indptr[i + 1])
        assert same_bits(o, out[a:b]) and same_bits(l, lse[a:b]), f"prefill request {i}"
    dcall = wl.whole_prefill(dstore)
    dout, dlse = run_decode(dcall)
    check_groups(dcall, dout, dlse, 4)  # all 32 decodes
    for i, s in enumerate(dstore.seqs):
        solo = wl.whole_prefill(wl.PagedStore([s], 32, 8, 128, 16, DEV, layout_seed=950 + i))
        o, l = run_decode(solo)
        assert same_bits(o[0], dout[i]) and same_bits(l[0], dlse[i]), f"decode request {i}"
