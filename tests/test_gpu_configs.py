"""The five workloads at full size on the GPU: oracle parity on sampled rows
(every request; all rows of the first and last q tile plus a seeded sample),
and bit-identity across batch sizes, batch composition, page placement and
q-tile-aligned chunking.  Off-grid chunking is checked against the oracle
only: it may differ from the unchunked run."""
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


def test_cfg2_batched_prefill_matches_oracle_and_solo_runs():
    store = wl.cfg2_prefill(DEV)
    call = wl.whole_prefill(store)
    out, lse = run_prefill(call)
    mx, mean, n = check_rows(call, out, lse, tokens_per_part=64)
    print(f"\n[cfg2] oracle rows {n}: max {mx:.3e} mean {mean:.3e}")
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
    # chunks of 256 tokens start on the 32-token grid: bit-identical
    calls = wl.chunked_calls(store, 256)
    assert len(calls) == 64
    o, l = assemble(whole, calls, [run_prefill(c) for c in calls])
    assert same_bits(o, out) and same_bits(l, lse)
    # chunks of 100 tokens leave the grid: held to the oracle only
    calls = wl.chunked_calls(store, 100)
    assert len(calls) == 164
    o, l = assemble(whole, calls, [run_prefill(c) for c in calls])
    mx2, mean2, n2 = check_rows(whole, o, l, tokens_per_part=128, seed=1)
    with capsys.disabled():
        print(f"\n[cfg3] oracle rows {n}: max {mx:.3e} mean {mean:.3e}; off-grid (100) rows "
              f"{n2}: max {mx2:.3e} mean {mean2:.3e}, bit-identical to unchunked: "
              f"{same_bits(o, out)}")


def test_cfg4_decode_sweep_request0_identical_across_batch_sizes():
    first = None
    for B in (1, 8, 64, 256):
        store = wl.cfg4_decode(DEV, B)
        call = wl.whole_prefill(store)
        out, lse = run_decode(call)
        check_rows(call, out, lse, part_ids=sorted({0, B // 2, B - 1}))
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
    check_rows(dcall, dout, dlse, part_ids=[0, 31])
    for i, s in enumerate(dstore.seqs):
        solo = wl.whole_prefill(wl.PagedStore([s], 32, 8, 128, 16, DEV, layout_seed=950 + i))
        o, l = run_decode(solo)
        assert same_bits(o[0], dout[i]) and same_bits(l[0], dlse[i]), f"decode request {i}"
