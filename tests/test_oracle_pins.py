"""Pins for the CPU oracle: each check ties it to something other than itself
(brute force with numpy, closed forms, invariants, a hand-derived example) so
that a dropped term, a wrong sign, a wrong index or a transposed operand in
the oracle fails at least one of them.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.common import oracle_on_call

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def dense_kv(call: wl.Call):
    """Gather each request's keys/values into dense [kv_len, Hkv, D] fp64
    arrays with numpy fancy indexing (a different route from the oracle's)."""
    st = call.store
    k = st.k_cache.float().numpy().astype(np.float64)
    v = st.v_cache.float().numpy().astype(np.float64)
    out = []
    for b in range(call.batch):
        pages = call.kv_indices[call.kv_indptr[b]:call.kv_indptr[b + 1]].numpy()
        kk = k[pages].reshape(-1, st.num_kv_heads, st.head_dim)[: call.kv_lens[b]]
        vv = v[pages].reshape(-1, st.num_kv_heads, st.head_dim)[: call.kv_lens[b]]
        out.append((kk, vv))
    return out


def brute_force(call: wl.Call, causal=True, scale=None):
    """softmax(Q K^T * scale + mask) V per request and head, as dense matrices."""
    st = call.store
    G = st.num_qo_heads // st.num_kv_heads
    scale = 1.0 / math.sqrt(st.head_dim) if scale is None else scale
    q = call.q.float().numpy().astype(np.float64)
    outs, lses = [], []
    for b, (kk, vv) in enumerate(dense_kv(call)):
        qb = q[call.qo_indptr[b]:call.qo_indptr[b + 1]]
        ql, kl = qb.shape[0], kk.shape[0]
        ob = np.zeros((ql, st.num_qo_heads, st.head_dim))
        lb = np.full((ql, st.num_qo_heads), -np.inf)
        pos = kl - ql + np.arange(ql)
        vis = (np.arange(kl)[None, :] <= pos[:, None]) if causal else np.ones((ql, kl), bool)
        for h in range(st.num_qo_heads):
            S = (qb[:, h, :] @ kk[:, h // G, :].T) * scale
            S = np.where(vis, S, -np.inf)
            m = S.max(axis=1, keepdims=True)
            ok = np.isfinite(m[:, 0])
            E = np.exp(np.where(ok[:, None], S - np.where(ok[:, None], m, 0), -np.inf))
            den = E.sum(axis=1, keepdims=True)
            ob[ok, h] = (E[ok] / den[ok]) @ vv[:, h // G, :]
            lb[ok, h] = (m[ok] + np.log(den[ok]))[:, 0]
        outs.append(ob)
        lses.append(lb)
    return np.concatenate(outs), np.concatenate(lses)


SMALL = [
    # (Hq, Hkv, D, page, [(prefix, new)], causal)
    (4, 1, 64, 16, [(0, 40)], True),
    (4, 2, 16, 1, [(0, 17), (5, 9), (30, 33)], True),
    (2, 2, 16, 4, [(3, 1), (0, 64), (12, 7)], True),
    (8, 2, 16, 3, [(10, 20), (0, 5)], False),
    (4, 4, 64, 2, [(63, 1), (0, 1)], True),
]


@pytest.mark.parametrize("Hq,Hkv,D,P,seqs,causal", SMALL)
def test_matches_dense_brute_force(Hq, Hkv, D, P, seqs, causal):
    store = wl.PagedStore([wl.Sequence(50 + i, p, n) for i, (p, n) in enumerate(seqs)],
                          Hq, Hkv, D, P, "cpu", layout_seed=11)
    call = wl.whole_prefill(store)
    out, lse = oracle_on_call(call, causal=causal)
    ref_out, ref_lse = brute_force(call, causal=causal)
    assert np.max(np.abs(out - ref_out)) <= 1e-12
    assert np.max(np.abs(lse - ref_lse)) <= 1e-12


def test_probabilities_form_a_distribution_and_respect_the_mask():
    store = wl.PagedStore([wl.Sequence(61, 9, 23)], 4, 2, 16, 4, "cpu")
    call = wl.whole_prefill(store)
    st = store
    for t in (0, 5, 22):
        for h in (0, 3):
            p = oracle.row_probs(wl.bf16_bits(call.q), wl.bf16_bits(st.k_cache),
                                 wl.bf16_bits(st.v_cache), call.qo_indptr.numpy(),
                                 call.kv_indptr.numpy(), call.kv_indices.numpy(),
                                 call.kv_last_page_len.numpy(), token=t, head=h,
                                 num_qo_heads=4, num_kv_heads=2, head_dim=16, page_size=4)
            pos = 9 + t
            assert p.shape == (32,)
            assert abs(p.sum() - 1.0) <= 1e-12
            assert np.all(p[: pos + 1] > 0.0)
            assert np.all(p[pos + 1:] == 0.0)


@pytest.mark.parametrize("Hq,Hkv,D,P,seqs,causal", SMALL)
def test_probabilities_equal_the_dense_softmax_weights(Hq, Hkv, D, P, seqs, causal):
    """Values of oracle_row_probs against numpy's dense softmax(q K^T * scale
    + mask) row (keys gathered by fancy indexing, a different route): every
    weight to 1e-12, and the weights times the dense V give the brute-force
    output row.  A wrong scale, kv head, q row or mask offset fails here."""
    store = wl.PagedStore([wl.Sequence(50 + i, p, n) for i, (p, n) in enumerate(seqs)],
                          Hq, Hkv, D, P, "cpu", layout_seed=11)
    call = wl.whole_prefill(store)
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(D)
    q = call.q.float().numpy().astype(np.float64)
    ref_out, _ = brute_force(call, causal=causal)
    rng = np.random.default_rng(7)
    for b, (kk, vv) in enumerate(dense_kv(call)):
        q0, q1 = int(call.qo_indptr[b]), int(call.qo_indptr[b + 1])
        if q1 == q0:
            continue
        kl = kk.shape[0]
        for t in sorted({q0, q1 - 1, int(rng.integers(q0, q1))}):
            for h in sorted({0, Hq - 1, int(rng.integers(0, Hq))}):
                got = oracle.row_probs(
                    wl.bf16_bits(call.q), wl.bf16_bits(store.k_cache), wl.bf16_bits(store.v_cache),
                    call.qo_indptr.numpy(), call.kv_indptr.numpy(), call.kv_indices.numpy(),
                    call.kv_last_page_len.numpy(), token=t, head=h, num_qo_heads=Hq,
                    num_kv_heads=Hkv, head_dim=D, page_size=P, causal=causal)
                pos = kl - (q1 - q0) + (t - q0)
                s = (kk[:, h // G, :] @ q[t, h, :]) * scale
                vis = np.arange(kl) <= pos if causal else np.ones(kl, bool)
                e = np.where(vis, np.exp(s - s[vis].max()), 0.0)
                want = e / e.sum()
                assert got.shape == (kl,)
                assert np.max(np.abs(got - want)) <= 1e-12
                assert np.max(np.abs(got @ vv[:, h // G, :] - ref_out[t, h])) <= 1e-12


def test_masked_keys_do_not_reach_a_row():
    """Overwrite every key/value after position p with huge values and NaN:
    row p must not change by a single bit."""
    store = wl.PagedStore([wl.Sequence(71, 6, 30)], 4, 1, 16, 1, "cpu")
    call = wl.whole_prefill(store)
    t = 10
    p = 6 + t
    rows = [(t, h) for h in range(4)]
    before = oracle_on_call(call, rows=rows)
    pages = call.kv_indices.long()
    store.k_cache[pages[p + 1:]] = 3.0e38
    store.v_cache[pages[p + 1:]] = float("nan")
    after = oracle_on_call(call, rows=rows)
    assert np.array_equal(before[0], after[0]) and np.array_equal(before[1], after[1])
    assert np.all(np.isfinite(after[0]))


def test_single_visible_key_returns_its_value():
    """First token of a causal prefill with no prefix sees only key 0."""
    store = wl.PagedStore([wl.Sequence(81, 0, 12)], 8, 2, 64, 16, "cpu")
    call = wl.whole_prefill(store)
    out, lse = oracle_on_call(call)
    v0 = store.v_cache[call.kv_indices[0].item(), 0].float().numpy().astype(np.float64)
    k0 = store.k_cache[call.kv_indices[0].item(), 0].float().numpy().astype(np.float64)
    q0 = call.q[0].float().numpy().astype(np.float64)
    for h in range(8):
        assert np.array_equal(out[0, h], v0[h // 4])
        assert lse[0, h] == pytest.approx(float(q0[h] @ k0[h // 4]) / 8.0, abs=1e-12)


@pytest.mark.parametrize("split", [1, 7, 16, 64, 4096])
def test_split_then_merge_equals_unsplit(split):
    store = wl.PagedStore([wl.Sequence(91, 40, 50), wl.Sequence(92, 0, 70)], 4, 2, 16, 1,
                          "cpu")
    call = wl.whole_prefill(store)
    full_out, full_lse = oracle_on_call(call)
    n_splits = -(-max(call.kv_lens) // split)
    parts_o, parts_l = [], []
    for s in range(n_splits):
        o, l = oracle_on_call(call, key_window=(s * split, (s + 1) * split))
        parts_o.append(o.astype(np.float32))
        parts_l.append(l.astype(np.float32))
    # the partial states are fp32 (as the library stores them): compare the
    # merge against the oracle evaluated in fp64 on the same fp32 states
    v = np.stack(parts_o, 1)  # [tokens, S, H, D]
    s = np.stack(parts_l, 1)  # [tokens, S, H]
    out, lse = oracle.merge_states(v, s)
    assert np.max(np.abs(out - full_out)) <= 2e-7
    assert np.max(np.abs(lse - full_lse)) <= 2e-6
    # exact-precision version: fp64 partials merged in fp64 by the definition
    o64 = np.stack([oracle_on_call(call, key_window=(i * split, (i + 1) * split))[0]
                    for i in range(n_splits)], 1)
    l64 = np.stack([oracle_on_call(call, key_window=(i * split, (i + 1) * split))[1]
                    for i in range(n_splits)], 1)
    m = np.max(l64, axis=1)
    tot = m + np.log(np.sum(np.exp(l64 - m[:, None]), axis=1))
    mixed = np.sum(np.exp(l64 - tot[:, None])[..., None] * o64, axis=1)
    assert np.max(np.abs(mixed - full_out)) <= 1e-12
    assert np.max(np.abs(tot - full_lse)) <= 1e-12


def test_empty_split_window_gives_neg_inf():
    store = wl.PagedStore([wl.Sequence(93, 0, 20)], 4, 1, 16, 1, "cpu")
    call = wl.whole_prefill(store)
    o, l = oracle_on_call(call, key_window=(12, 16))
    for t in range(20):
        if t < 12:
            assert np.all(l[t] == -np.inf) and np.all(o[t] == 0.0)
        else:
            assert np.all(np.isfinite(l[t]))


def test_page_placement_does_not_change_bits():
    seqs = [wl.Sequence(101, 13, 29), wl.Sequence(102, 0, 44)]
    a = wl.whole_prefill(wl.PagedStore(seqs, 4, 2, 16, 4, "cpu", layout_seed=1))
    b = wl.whole_prefill(wl.PagedStore(seqs, 4, 2, 16, 4, "cpu", layout_seed=2, spare_pages=5))
    assert not torch.equal(a.kv_indices, b.kv_indices)
    oa, la = oracle_on_call(a)
    ob, lb = oracle_on_call(b)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


def test_equal_keys_give_the_mean_of_visible_values():
    store = wl.PagedStore([wl.Sequence(111, 5, 11)], 4, 1, 16, 2, "cpu")
    store.k_cache[:] = 0.25
    call = wl.whole_prefill(store)
    out, lse = oracle_on_call(call)
    vdense = []
    for j in range(16):
        page = call.kv_indices[j // 2].item()
        vdense.append(store.v_cache[page, j % 2, 0].float().numpy().astype(np.float64))
    vdense = np.stack(vdense)
    q = call.q.float().numpy().astype(np.float64)
    for t in range(11):
        n = 5 + t + 1
        for h in range(4):
            assert np.max(np.abs(out[t, h] - vdense[:n].mean(0))) <= 1e-12
            s = 0.25 * q[t, h].sum() / 4.0
            assert lse[t, h] == pytest.approx(s + math.log(n), abs=1e-12)


def test_gqa_head_grouping():
    """kv head g holds value g+1 everywhere: q head h must read h // G + 1."""
    store = wl.PagedStore([wl.Sequence(121, 3, 9)], 8, 2, 16, 1, "cpu")
    store.v_cache[:, :, 0] = 1.0
    store.v_cache[:, :, 1] = 2.0
    out, _ = oracle_on_call(wl.whole_prefill(store))
    for h in range(8):
        assert np.max(np.abs(out[:, h] - float(h // 4 + 1))) <= 1e-12


def test_sm_scale_and_noncausal_closed_form():
    """Two keys with scores a, b: out = sigma(a-b) v0 + sigma(b-a) v1."""
    store = wl.PagedStore([wl.Sequence(131, 0, 2)], 1, 1, 16, 1, "cpu")
    call = wl.whole_prefill(store)
    p0, p1 = call.kv_indices[0].item(), call.kv_indices[1].item()
    store.k_cache[:] = 0.0
    store.k_cache[p0, 0, 0, 0] = 1.0
    store.k_cache[p1, 0, 0, 0] = -2.0
    call.q[:] = 0.0
    call.q[:, 0, 0] = 1.5
    for scale in (0.25, 1.0, 3.0):
        out, lse = oracle_on_call(call, causal=False, sm_scale=scale)
        a, b = 1.5 * scale, -3.0 * scale
        w0 = 1.0 / (1.0 + math.exp(b - a))
        v0 = store.v_cache[p0, 0, 0].double().numpy()
        v1 = store.v_cache[p1, 0, 0].double().numpy()
        for t in range(2):
            assert np.max(np.abs(out[t, 0] - (w0 * v0 + (1 - w0) * v1))) <= 1e-12
            assert lse[t, 0] == pytest.approx(math.log(math.exp(a) + math.exp(b)), abs=1e-12)


def test_hand_derived_example():
    with open(os.path.join(GOLDEN, "hand_example.json")) as f:
        ex = json.load(f)
    q = torch.tensor(ex["q"], dtype=torch.bfloat16)
    k_cache = torch.full((2, 2, 1, 4), float("nan"), dtype=torch.bfloat16)
    v_cache = torch.full_like(k_cache, float("nan"))
    for j, (kr, vr) in enumerate(zip(ex["keys"], ex["values"])):
        page = ex["kv_indices"][j // 2]
        k_cache[page, j % 2, 0] = torch.tensor(kr, dtype=torch.bfloat16)
        v_cache[page, j % 2, 0] = torch.tensor(vr, dtype=torch.bfloat16)
    out, lse = oracle.attention(wl.bf16_bits(q), wl.bf16_bits(k_cache), wl.bf16_bits(v_cache),
                                ex["qo_indptr"], ex["kv_indptr"], ex["kv_indices"],
                                ex["kv_last_page_len"], num_qo_heads=2, num_kv_heads=1,
                                head_dim=4, page_size=2, causal=True)
    values = np.array(ex["values"], np.float64)
    for key, scores in ex["expected_scores"].items():
        if key == "comment":
            continue
        t, h = int(key[1]), int(key[4])
        e = np.exp(np.array(scores))
        want = (e / e.sum()) @ values[: len(scores)]
        assert np.max(np.abs(out[t, h] - want)) <= 1e-15
        assert lse[t, h] == pytest.approx(math.log(e.sum()), abs=1e-15)
    assert out[2, 0] == pytest.approx([0.0900305731703805, 0.2447284710547976,
                                       0.6652409557748219, 0.0], abs=1e-15)
    assert lse[2, 0] == pytest.approx(2.4076059644443806, abs=1e-15)


def test_unused_page_slots_are_never_read():
    """Slots past kv_len in the last page hold NaN (workload fill)."""
    store = wl.PagedStore([wl.Sequence(141, 2, 13), wl.Sequence(142, 0, 3)], 4, 1, 16, 8, "cpu")
    call = wl.whole_prefill(store)
    assert torch.isnan(store.k_cache.float()).any()
    out, lse = oracle_on_call(call, causal=False)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))


def test_rows_without_keys_and_requests_without_queries():
    """Non-causal row of a request with no key: out 0, lse -inf; a request
    with no query contributes no row and leaves its neighbours alone."""
    store = wl.PagedStore([wl.Sequence(151, 0, 5), wl.Sequence(152, 4, 0),
                           wl.Sequence(153, 0, 6)], 4, 1, 16, 2, "cpu")
    call = wl.whole_prefill(store)
    assert call.q_lens == [5, 0, 6]
    out, lse = oracle_on_call(call)
    solo0 = oracle_on_call(wl.make_call(store, [(0, 0, 5)]))
    solo2 = oracle_on_call(wl.make_call(store, [(2, 0, 6)]))
    assert np.array_equal(out[:5], solo0[0]) and np.array_equal(out[5:], solo2[0])
    # no keys at all: zero pages for a request queried non-causally
    st = wl.PagedStore([wl.Sequence(154, 0, 0)], 4, 1, 16, 2, "cpu")
    q = wl.draw_normal_bf16((2, 4, 16), 9, "cpu")
    o, l = oracle.attention(wl.bf16_bits(q), wl.bf16_bits(st.k_cache), wl.bf16_bits(st.v_cache),
                            [0, 2], [0, 0], [0], [0], num_qo_heads=4, num_kv_heads=1,
                            head_dim=16, page_size=2, causal=False)
    assert np.all(o == 0.0) and np.all(l == -np.inf)


def test_merge_closed_forms():
    rng = np.random.default_rng(5)
    v = rng.standard_normal((3, 4, 2, 8)).astype(np.float32)
    s = rng.standard_normal((3, 4, 2)).astype(np.float32)
    # identical states: out = v, lse = l + ln S
    vs = np.repeat(v[:, :1], 4, axis=1)
    ss = np.repeat(s[:, :1], 4, axis=1)
    out, lse = oracle.merge_states(vs, ss)
    assert np.max(np.abs(out - v[:, 0])) <= 1e-7
    assert np.max(np.abs(lse - (s[:, 0] + math.log(4)))) <= 1e-6
    # -inf states carry no weight, NaN payload included
    s2 = s.copy()
    v2 = v.copy()
    s2[:, 1] = -np.inf
    v2[:, 1] = np.nan
    o2, l2 = oracle.merge_states(v2, s2)
    keep = [0, 2, 3]
    o3, l3 = oracle.merge_states(v[:, keep], s[:, keep])
    assert np.array_equal(o2, o3) and np.array_equal(l2, l3)
    # two states: sigmoid weights
    o4, l4 = oracle.merge_states(v[:, :2], s[:, :2])
    w = 1.0 / (1.0 + np.exp(s[:, 1].astype(np.float64) - s[:, 0]))
    want = w[..., None] * v[:, 0] + (1 - w[..., None]) * v[:, 1]
    assert np.max(np.abs(o4 - want)) <= 1e-6
    # num_states limits the fold; zero states -> 0 / -inf
    o5, l5 = oracle.merge_states(v, s, num_states=[2, 0, 4])
    assert np.array_equal(o5[0], o4[0]) and np.all(o5[1] == 0) and np.all(l5[1] == -np.inf)


def test_merge_is_order_free_associative_and_shift_stable():
    """What the log-sum-exp merge fixes mathematically: the result does not
    depend on the order of the states, merging merged groups gives the merge
    of all, and shifting every lse by c shifts the result's lse by c and
    leaves the output alone (no overflow at large lse)."""
    rng = np.random.default_rng(11)
    n, S, H, D = 5, 7, 3, 16
    v = rng.standard_normal((n, S, H, D)).astype(np.float32)
    s = (rng.integers(-24, 24, (n, S, H)) / 8.0).astype(np.float32)  # exact in fp32
    out, lse = oracle.merge_states(v, s)
    perm = rng.permutation(S)
    po, pl = oracle.merge_states(v[:, perm], s[:, perm])
    assert np.max(np.abs(po - out)) <= 1e-12 and np.max(np.abs(pl - lse)) <= 1e-12
    # two groups merged first (their states rounded to fp32), then merged
    ao, al = oracle.merge_states(v[:, :3], s[:, :3])
    bo, bl = oracle.merge_states(v[:, 3:], s[:, 3:])
    gv = np.stack([ao, bo], 1).astype(np.float32)
    gs = np.stack([al, bl], 1).astype(np.float32)
    go, gl = oracle.merge_states(gv, gs)
    assert np.max(np.abs(go - out)) <= 1e-6 and np.max(np.abs(gl - lse)) <= 1e-6
    # every lse shifted by 4096 (exact in fp32 for these values)
    so, sl = oracle.merge_states(v, s + np.float32(4096.0))
    assert np.all(np.isfinite(so)) and np.max(np.abs(so - out)) <= 1e-12
    assert np.max(np.abs(sl - (lse + 4096.0))) <= 1e-9


def test_key_shift_and_value_affine_invariance():
    """Softmax ignores a score offset that every key of a row shares: adding
    one vector c to every key leaves the output alone and moves lse by
    scale * <q, c>.  The output is affine in the values (the weights sum to
    one): V -> 2 V + b gives 2 out + b.  Small integers keep every input exact
    in bf16."""
    Hq, Hkv, D, P = 4, 2, 16, 4
    G = Hq // Hkv
    store = wl.PagedStore([wl.Sequence(70, 5, 9), wl.Sequence(71, 0, 12)], Hq, Hkv, D, P, "cpu",
                          layout_seed=13)
    call = wl.whole_prefill(store)
    g = torch.Generator().manual_seed(3)

    def rint(shape, lo=-3, hi=4):
        return torch.randint(lo, hi, tuple(shape), generator=g).to(torch.bfloat16)
    call.q = rint(call.q.shape)
    store.k_cache = rint(store.k_cache.shape)
    store.v_cache = rint(store.v_cache.shape)
    out, lse = oracle_on_call(call)

    c = rint((Hkv, D))
    k0 = store.k_cache
    store.k_cache = (k0.float() + c.float()).to(torch.bfloat16)  # |values| <= 6: exact
    so, sl = oracle_on_call(call)
    store.k_cache = k0
    q = call.q.float().numpy().astype(np.float64)
    cq = np.stack([q[:, h] @ c.float().numpy()[h // G] for h in range(Hq)], 1)
    assert np.max(np.abs(so - out)) <= 1e-12
    assert np.max(np.abs(sl - (lse + cq / math.sqrt(D)))) <= 1e-12

    b = rint((Hkv, D))
    store.v_cache = (2 * store.v_cache.float() + b.float()).to(torch.bfloat16)
    ao, al = oracle_on_call(call)
    bb = np.stack([b.float().numpy()[h // G] for h in range(Hq)], 0)
    assert np.max(np.abs(ao - (2 * out + bb[None]))) <= 1e-12
    assert np.array_equal(al, lse)
