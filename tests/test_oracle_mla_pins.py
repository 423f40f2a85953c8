"""Pins of the oracle's multi-head latent attention: the same numbers as the
(already pinned) GQA oracle run as one 576-wide kv head whose value rows are
the latent rows padded with zeros; dense numpy brute force; split-then-merge
equal to the unsplit result; a single visible key returns its latent row."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl


def run_mla(call, causal=True, key_window=None, sm_scale=None):
    st = call.store
    scale = 1.0 / math.sqrt(st.dc + st.dp) if sm_scale is None else sm_scale
    return oracle.mla(wl.bf16_bits(call.q_nope), wl.bf16_bits(call.q_pe),
                      wl.bf16_bits(st.ckv_cache), wl.bf16_bits(st.kpe_cache),
                      call.qo_indptr.numpy(), call.kv_indptr.numpy(), call.kv_indices.numpy(),
                      call.kv_last_page_len.numpy(), page_size=st.page_size, sm_scale=scale,
                      causal=causal, key_window=key_window)


def small(seqs, H=4, dc=32, dp=8, P=4, seed=0):
    store = wl.MLAStore([wl.Sequence(90 + seed + i, p, n) for i, (p, n) in enumerate(seqs)],
                        H, dc, dp, P, "cpu", layout_seed=3 + seed)
    return wl.mla_call(store, [(i, 0, s.new) for i, s in enumerate(store.seqs)])


@pytest.mark.parametrize("causal", [True, False])
def test_equals_gqa_oracle_as_one_wide_kv_head(causal):
    call = small([(0, 9), (13, 4), (5, 1)], H=8, dc=32, dp=8, P=4)
    st = call.store
    out, lse = run_mla(call, causal=causal)
    # K = [ckv | kpe], V = [ckv | 0], q = [q_nope | q_pe], one kv head
    k = torch.cat([st.ckv_cache, st.kpe_cache], -1).unsqueeze(2)
    v = torch.cat([st.ckv_cache, torch.zeros_like(st.kpe_cache)], -1).unsqueeze(2)
    q = torch.cat([call.q_nope, call.q_pe], -1)
    ref_o, ref_l = oracle.attention(
        wl.bf16_bits(q), wl.bf16_bits(k), wl.bf16_bits(v), call.qo_indptr.numpy(),
        call.kv_indptr.numpy(), call.kv_indices.numpy(), call.kv_last_page_len.numpy(),
        num_qo_heads=8, num_kv_heads=1, head_dim=40, page_size=4, causal=causal,
        sm_scale=1.0 / math.sqrt(40))
    assert np.max(np.abs(out - ref_o[..., :32])) <= 1e-12
    assert np.max(np.abs(lse - ref_l)) <= 1e-12
    assert np.all(ref_o[..., 32:] == 0.0)


def test_matches_dense_brute_force():
    call = small([(0, 7), (20, 3)], H=2, dc=16, dp=4, P=1, seed=2)
    st = call.store
    out, lse = run_mla(call)
    scale = 1.0 / math.sqrt(20)
    for b in range(2):
        pages = call.kv_indices[call.kv_indptr[b]:call.kv_indptr[b + 1]].numpy()
        kvl = call.kv_lens[b]
        ckv = st.ckv_cache.float().numpy().astype(np.float64)[pages].reshape(-1, 16)[:kvl]
        kpe = st.kpe_cache.float().numpy().astype(np.float64)[pages].reshape(-1, 4)[:kvl]
        a, e = int(call.qo_indptr[b]), int(call.qo_indptr[b + 1])
        qn = call.q_nope.float().numpy().astype(np.float64)[a:e]
        qp = call.q_pe.float().numpy().astype(np.float64)[a:e]
        ql = e - a
        pos = kvl - ql + np.arange(ql)
        vis = np.arange(kvl)[None, :] <= pos[:, None]
        for h in range(2):
            S = (qn[:, h] @ ckv.T + qp[:, h] @ kpe.T) * scale
            S = np.where(vis, S, -np.inf)
            m = S.max(1, keepdims=True)
            E = np.exp(S - m)
            ref = (E / E.sum(1, keepdims=True)) @ ckv
            assert np.max(np.abs(out[a:e, h] - ref)) <= 1e-12
            assert np.max(np.abs(lse[a:e, h] - (m[:, 0] + np.log(E.sum(1))))) <= 1e-12


def test_split_then_merge_equals_unsplit():
    call = small([(40, 1), (70, 2)], H=4, dc=32, dp=8, P=2, seed=3)
    out, lse = run_mla(call)
    split = 16
    n_splits = (max(call.kv_lens) + split - 1) // split
    parts_o, parts_l = [], []
    for s in range(n_splits):
        o, l = run_mla(call, key_window=(s * split, (s + 1) * split))
        parts_o.append(o)
        parts_l.append(l)
    v = np.stack(parts_o, 1).astype(np.float32)       # [T, S, H, dc]
    l = np.stack(parts_l, 1).astype(np.float32)       # [T, S, H]
    mo, ml = oracle.merge_states(v, l)
    assert np.max(np.abs(mo - out)) <= 2e-6 and np.max(np.abs(ml - lse)) <= 2e-6


def test_single_visible_key_returns_its_latent_row():
    call = small([(0, 3)], H=2, dc=16, dp=4, P=4, seed=4)
    out, lse = run_mla(call)
    st = call.store
    page = int(call.kv_indices[0])
    assert np.array_equal(out[0, 0], st.ckv_cache[page, 0].double().numpy())
    assert np.array_equal(out[0, 1], st.ckv_cache[page, 0].double().numpy())
