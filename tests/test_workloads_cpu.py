"""The seeded input generator both sides use (workloads.py): a request's q,
K and V bits depend only on its own seed, never on the batch around it or the
page layout; unused cache slots hold NaN; calls describe the pages and
lengths they claim.  The GPU bit-identity tests compare runs on different
batches and rely on these properties.  CPU only."""
import numpy as np
import torch

import workloads as wl


def bits(t):
    return t.contiguous().view(torch.int16)


def gathered(store, i):
    """Sequence i's K and V rows in key order, through its page list."""
    s, pages = store.seqs[i], store.pages[i].long()
    Hkv, D = store.num_kv_heads, store.head_dim
    k = store.k_cache[pages].reshape(-1, Hkv, D)[: s.length]
    v = store.v_cache[pages].reshape(-1, Hkv, D)[: s.length]
    return k, v


def seqs3():
    return [wl.Sequence(11, 5, 30), wl.Sequence(12, 0, 17), wl.Sequence(13, 40, 1)]


def test_request_bits_do_not_depend_on_the_batch_or_the_layout():
    big = wl.PagedStore(seqs3(), 8, 2, 32, 4, "cpu", layout_seed=1)
    for i, s in enumerate(seqs3()):
        solo = wl.PagedStore([s], 8, 2, 32, 4, "cpu", layout_seed=50 + i)
        assert torch.equal(bits(solo.q[0]), bits(big.q[i]))
        for a, b in zip(gathered(solo, 0), gathered(big, i)):
            assert torch.equal(bits(a), bits(b))
            assert not torch.isnan(a.float()).any()


def test_pages_are_disjoint_and_unused_slots_hold_nan():
    st = wl.PagedStore(seqs3(), 8, 2, 32, 4, "cpu", layout_seed=2)
    ids = torch.cat(st.pages).tolist()
    assert len(ids) == len(set(ids)) and all(0 <= p < st.num_pages for p in ids)
    finite = (~torch.isnan(st.k_cache.float())).all(-1).all(-1)  # [pages, slots]
    assert int(finite.sum()) == sum(s.length for s in st.seqs)
    for i, s in enumerate(st.seqs):
        n = len(st.pages[i])
        slots = finite[st.pages[i].long()].reshape(-1)
        assert slots[: s.length].all() and not slots[s.length: n * st.page_size].any()


def test_uniform_lengths_keep_their_prefix_and_range():
    a = wl.uniform_lengths(8, 100, 200, 77)
    assert a[:3] == wl.uniform_lengths(3, 100, 200, 77)
    assert all(100 <= x <= 200 for x in a)


def test_chunked_calls_cover_the_whole_prefill():
    st = wl.PagedStore(seqs3(), 8, 2, 32, 4, "cpu", layout_seed=3)
    whole = wl.whole_prefill(st)
    got = {i: [] for i in range(len(st.seqs))}
    for call in wl.chunked_calls(st, 7):
        qo = call.qo_indptr.tolist()
        kvp = call.kv_indptr.tolist()
        for j, (si, a, b) in enumerate(call.parts):
            got[si].append(call.q[qo[j]:qo[j + 1]])
            s = st.seqs[si]
            assert call.kv_lens[j] == s.prefix + b and call.q_lens[j] == b - a
            n_pages = kvp[j + 1] - kvp[j]
            last = int(call.kv_last_page_len[j])
            assert 1 <= last <= st.page_size
            assert (n_pages - 1) * st.page_size + last == s.prefix + b
            assert torch.equal(call.kv_indices[kvp[j]:kvp[j + 1]], st.pages[si][:n_pages])
    qo = whole.qo_indptr.tolist()
    for i in range(len(st.seqs)):
        assert torch.equal(bits(torch.cat(got[i])), bits(whole.q[qo[i]:qo[i + 1]]))


def test_new_kv_rows_are_the_cache_rows_at_the_new_positions():
    st = wl.PagedStore(seqs3(), 8, 2, 32, 4, "cpu", layout_seed=4)
    call = wl.make_call(st, [(0, 3, 20), (2, 0, 1), (1, 0, 17)])
    k_new, v_new = wl.new_kv_rows(call)
    rows_k, rows_v, at = [], [], 0
    for (si, a, b) in call.parts:
        k, v = gathered(st, si)
        p = st.seqs[si].prefix
        rows_k.append(k[p + a:p + b])
        rows_v.append(v[p + a:p + b])
        at += b - a
    assert k_new.shape[0] == at
    assert torch.equal(bits(k_new), bits(torch.cat(rows_k)))
    assert torch.equal(bits(v_new), bits(torch.cat(rows_v)))


def test_custom_mask_bits_unpack_to_the_dense_matrices():
    st = wl.PagedStore(seqs3(), 8, 2, 32, 4, "cpu", layout_seed=5)
    call = wl.whole_prefill(st)
    packed, offs, dense = wl.custom_mask(call, seed=9, density=0.4, causal_part=True)
    flat = np.unpackbits(packed, bitorder="little")
    for j, m in enumerate(dense):
        ql, kl = call.q_lens[j], call.kv_lens[j]
        assert offs[j + 1] - offs[j] == ql * kl
        assert np.array_equal(flat[offs[j]:offs[j + 1]].reshape(ql, kl).astype(bool), m)
        pos = kl - ql + np.arange(ql)
        assert not (m & (np.arange(kl)[None, :] > pos[:, None])).any()  # causal part


def test_mla_request_bits_do_not_depend_on_the_batch():
    seqs = [wl.Sequence(21, 9, 3), wl.Sequence(22, 0, 5)]
    big = wl.MLAStore(seqs, 4, 32, 8, 4, "cpu", layout_seed=6)
    solo = wl.MLAStore(seqs[1:], 4, 32, 8, 4, "cpu", layout_seed=7)
    assert torch.equal(bits(big.q_nope[1]), bits(solo.q_nope[0]))
    assert torch.equal(bits(big.q_pe[1]), bits(solo.q_pe[0]))
    for cache in ("ckv_cache", "kpe_cache"):
        a = getattr(big, cache)[big.pages[1].long()].reshape(-1, getattr(big, cache).shape[-1])
        b = getattr(solo, cache)[solo.pages[0].long()].reshape(-1, getattr(solo, cache).shape[-1])
        assert torch.equal(bits(a[:5]), bits(b[:5]))
