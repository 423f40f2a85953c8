"""GPU-side test plumbing: run the library's entry points on workload calls,
cut a call down to a few requests for the oracle, and compare bits.  Layout
manipulation only; no attention arithmetic."""
from __future__ import annotations

import numpy as np
import torch

import invariant_paged_attention_gb300 as bia
import workloads as wl
from tests.common import bf16_to_f64, error_stats, oracle_on_call

MAX_ABS, MEAN_ABS = 2e-2, 2e-3  # bf16 output tolerance against the fp64 oracle
LSE_TOL = 1e-3                  # |lse_gpu - lse_oracle| <= LSE_TOL * max(1, |lse|)


def desc_of(store, sm_scale=0.0):
    return bia.make_desc(store.num_qo_heads, store.num_kv_heads, store.head_dim,
                         store.page_size, sm_scale)


def run_prefill(call: wl.Call, causal=True, split=0, sm_scale=0.0, k_cache=None, v_cache=None):
    st = call.store
    dev = st.k_cache.device
    k_cache = st.k_cache if k_cache is None else k_cache
    v_cache = st.v_cache if v_cache is None else v_cache
    desc = desc_of(st, sm_scale)
    nbytes = bia.bia_prefill_workspace_size(desc, call.qo_indptr, call.kv_indptr,
                                            call.kv_last_page_len, causal, split)
    assert nbytes > 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = torch.full_like(call.q, float("nan"))
    lse = torch.full((call.total_q, st.num_qo_heads), float("nan"), dtype=torch.float32,
                     device=dev)
    bia.bia_prefill_paged(desc, call.q, k_cache, v_cache, call.qo_indptr.to(dev),
                          call.kv_indptr.to(dev), call.kv_indices.to(dev),
                          call.kv_last_page_len.to(dev), call.qo_indptr, call.kv_indptr,
                          call.kv_last_page_len, ws, out, lse, causal=causal, split_size=split)
    assert bia.bia_read_status(ws) == 0
    return out, lse


def run_decode(call: wl.Call, split=0, sm_scale=0.0):
    st = call.store
    dev = st.k_cache.device
    assert all(n == 1 for n in call.q_lens)
    desc = desc_of(st, sm_scale)
    nbytes = bia.bia_decode_workspace_size(desc, call.kv_indptr, call.kv_last_page_len, split)
    assert nbytes > 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = torch.full_like(call.q, float("nan"))
    lse = torch.full((call.total_q, st.num_qo_heads), float("nan"), dtype=torch.float32,
                     device=dev)
    bia.bia_decode_paged(desc, call.q, st.k_cache, st.v_cache, call.kv_indptr.to(dev),
                         call.kv_indices.to(dev), call.kv_last_page_len.to(dev), call.kv_indptr,
                         call.kv_last_page_len, ws, out, lse, split_size=split)
    assert bia.bia_read_status(ws) == 0
    return out, lse


def bits(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def same_bits(a: torch.Tensor, b: torch.Tensor) -> bool:
    return a.shape == b.shape and torch.equal(bits(a), bits(b))


def compact(call: wl.Call, part_ids) -> wl.Call:
    """The same call restricted to parts `part_ids`, over a compact CPU copy
    of just their pages (page placement does not change results)."""
    st = call.store
    pages, qs, kvp, qo, last, parts, q_lens, kv_lens = [], [], [0], [0], [], [], [], []
    for i in part_ids:
        a, b = int(call.kv_indptr[i]), int(call.kv_indptr[i + 1])
        pages.append(call.kv_indices[a:b])
        kvp.append(kvp[-1] + (b - a))
        qa, qb = int(call.qo_indptr[i]), int(call.qo_indptr[i + 1])
        qs.append(call.q[qa:qb])
        qo.append(qo[-1] + (qb - qa))
        last.append(int(call.kv_last_page_len[i]))
        parts.append(call.parts[i])
        q_lens.append(call.q_lens[i])
        kv_lens.append(call.kv_lens[i])
    idx = torch.cat(pages).long()
    sub = wl.PagedStore.__new__(wl.PagedStore)
    sub.seqs, sub.num_qo_heads, sub.num_kv_heads = st.seqs, st.num_qo_heads, st.num_kv_heads
    sub.head_dim, sub.page_size, sub.device = st.head_dim, st.page_size, "cpu"
    sub.k_cache = st.k_cache[idx.to(st.k_cache.device)].cpu()
    sub.v_cache = st.v_cache[idx.to(st.v_cache.device)].cpu()
    sub.q, sub.pages = None, None
    return wl.Call(sub, parts, torch.cat(qs).cpu(), torch.tensor(qo, dtype=torch.int32),
                   torch.tensor(kvp, dtype=torch.int32),
                   torch.arange(len(idx), dtype=torch.int32),
                   torch.tensor(last, dtype=torch.int32), q_lens, kv_lens)


def check_rows(call: wl.Call, out, lse, part_ids=None, tokens_per_part=None, seed=0,
               causal=True, sm_scale=None, threads=None, tokens=None):
    """Compares GPU rows with the oracle.  part_ids: which parts (default all);
    tokens_per_part: None = every token, else a seeded sample of that many
    tokens per part, always including the first and last q tile; tokens: an
    explicit list of in-part token indices instead (those inside each part).
    Returns (max_abs, mean_abs, rows_checked)."""
    part_ids = list(range(call.batch)) if part_ids is None else list(part_ids)
    sub = compact(call, part_ids)
    st = call.store
    G = st.num_qo_heads // st.num_kv_heads
    T = 128 // G
    rng = np.random.default_rng(seed)
    tok_rows, gpu_idx = [], []
    for k, i in enumerate(part_ids):
        n = call.q_lens[i]
        if n == 0:
            continue
        toks = np.arange(n)
        if tokens is not None:
            toks = np.array(sorted(t for t in set(tokens) if 0 <= t < n), dtype=np.int64)
            if toks.size == 0:
                continue
        elif tokens_per_part is not None and n > tokens_per_part:
            edge = np.concatenate([np.arange(min(T, n)), np.arange(max(0, n - T), n)])
            pick = rng.choice(n, size=tokens_per_part, replace=False)
            toks = np.unique(np.concatenate([edge, pick]))
        tok_rows.append(int(sub.qo_indptr[k]) + toks)
        gpu_idx.append(int(call.qo_indptr[i]) + toks)
    sub_tokens = np.concatenate(tok_rows)
    gpu_tokens = torch.from_numpy(np.concatenate(gpu_idx)).to(out.device)
    H = st.num_qo_heads
    rows = np.stack([np.repeat(sub_tokens, H), np.tile(np.arange(H), len(sub_tokens))], 1)
    o_ref, l_ref = oracle_on_call(sub, causal=causal, rows=rows, sm_scale=sm_scale,
                                  threads=threads)
    got = bf16_to_f64(out[gpu_tokens]).reshape(-1, st.head_dim)
    got_l = lse[gpu_tokens].double().cpu().numpy().reshape(-1)
    mx, mean = error_stats(got, o_ref)
    assert np.all(np.isfinite(got)), "non-finite output"
    assert mx <= MAX_ABS and mean <= MEAN_ABS, (mx, mean)
    fin = np.isfinite(l_ref)
    assert np.array_equal(fin, np.isfinite(got_l))
    dl = np.abs(got_l[fin] - l_ref[fin]) / np.maximum(1.0, np.abs(l_ref[fin]))
    assert dl.size == 0 or dl.max() <= LSE_TOL, float(dl.max())
    return mx, mean, rows.shape[0]
