"""Pins of the oracle's custom mask: dense brute force with the mask applied
as -inf, the causal pattern given as a mask, an all-ones mask, rows that see
nothing, and masked keys that never reach a row."""
import math

import numpy as np
import pytest

import oracle
import workloads as wl
from tests.test_oracle_pins import dense_kv


def masked_oracle(call, bits, indptr, causal):
    st = call.store
    return oracle.attention(
        wl.bf16_bits(call.q), wl.bf16_bits(st.k_cache), wl.bf16_bits(st.v_cache),
        call.qo_indptr.numpy(), call.kv_indptr.numpy(), call.kv_indices.numpy(),
        call.kv_last_page_len.numpy(), num_qo_heads=st.num_qo_heads,
        num_kv_heads=st.num_kv_heads, head_dim=st.head_dim, page_size=st.page_size,
        causal=causal, mask=bits, mask_indptr=indptr)


def brute_force_masked(call, dense_masks, causal):
    st = call.store
    G = st.num_qo_heads // st.num_kv_heads
    scale = 1.0 / math.sqrt(st.head_dim)
    q = call.q.float().numpy().astype(np.float64)
    outs, lses = [], []
    for b, (kk, vv) in enumerate(dense_kv(call)):
        qb = q[call.qo_indptr[b]:call.qo_indptr[b + 1]]
        ql, kl = qb.shape[0], kk.shape[0]
        vis = dense_masks[b].copy()
        if causal:
            pos = kl - ql + np.arange(ql)
            vis &= np.arange(kl)[None, :] <= pos[:, None]
        ob = np.zeros((ql, st.num_qo_heads, st.head_dim))
        lb = np.full((ql, st.num_qo_heads), -np.inf)
        for h in range(st.num_qo_heads):
            S = np.where(vis, (qb[:, h, :] @ kk[:, h // G, :].T) * scale, -np.inf)
            m = S.max(axis=1, keepdims=True)
            ok = np.isfinite(m[:, 0])
            E = np.exp(np.where(ok[:, None], S - np.where(ok[:, None], m, 0), -np.inf))
            den = E.sum(axis=1, keepdims=True)
            ob[ok, h] = (E[ok] / den[ok]) @ vv[:, h // G, :]
            lb[ok, h] = (m[ok] + np.log(den[ok]))[:, 0]
        outs.append(ob)
        lses.append(lb)
    return np.concatenate(outs), np.concatenate(lses)


def small_call(seqs, Hq=4, Hkv=2, D=16, P=4, seed=0):
    store = wl.PagedStore([wl.Sequence(70 + seed + i, p, n) for i, (p, n) in enumerate(seqs)],
                          Hq, Hkv, D, P, "cpu", layout_seed=13 + seed)
    return wl.whole_prefill(store)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("density", [0.05, 0.5, 0.95])
def test_matches_masked_brute_force(causal, density):
    call = small_call([(0, 23), (9, 14), (40, 3), (5, 0)], seed=int(density * 100))
    bits, indptr, dense = wl.custom_mask(call, seed=7, density=density)
    out, lse = masked_oracle(call, bits, indptr, causal)
    ref_out, ref_lse = brute_force_masked(call, dense, causal)
    assert np.max(np.abs(out - ref_out)) <= 1e-12
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(lse))
    assert np.max(np.abs(lse[fin] - ref_lse[fin]), initial=0.0) <= 1e-12
    assert np.all(out[~fin] == 0.0)


def test_causal_pattern_as_mask_equals_causal():
    call = small_call([(0, 31), (17, 6)], seed=3)
    bits, indptr, _ = wl.custom_mask(call, seed=1, density=1.0, causal_part=True)
    out_m, lse_m = masked_oracle(call, bits, indptr, causal=False)
    out_c, lse_c = masked_oracle(call, None, None, causal=True)
    assert np.array_equal(out_m, out_c) and np.array_equal(lse_m, lse_c)


def test_all_ones_mask_is_no_mask():
    call = small_call([(3, 12), (0, 20)], seed=4)
    bits, indptr, _ = wl.custom_mask(call, seed=2, density=1.0)
    for causal in (False, True):
        a = masked_oracle(call, bits, indptr, causal)
        b = masked_oracle(call, None, None, causal)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_rows_without_visible_keys_and_masked_keys_never_read():
    call = small_call([(0, 8)], seed=5)
    bits, indptr, dense = wl.custom_mask(call, seed=3, density=0.5)
    # row 2 sees nothing; key 5 is hidden from every row
    dense[0][2, :] = False
    dense[0][:, 5] = False
    flat = np.concatenate([d.reshape(-1) for d in dense])
    bits = np.concatenate([np.packbits(flat, bitorder="little"), np.zeros(4, np.uint8)])
    out, lse = masked_oracle(call, bits, indptr, causal=False)
    assert np.all(out[2] == 0.0) and np.all(np.isneginf(lse[2]))
    # poison key 5's K and V: no row changes
    st = call.store
    page = int(call.kv_indices[5 // st.page_size])
    st.k_cache[page, 5 % st.page_size] = float("nan")
    st.v_cache[page, 5 % st.page_size] = 1e30
    out2, lse2 = masked_oracle(call, bits, indptr, causal=False)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)
