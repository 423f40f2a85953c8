"""Test plumbing shared by the CPU and GPU suites: run the oracle on a
workload call, and compare results.  No attention arithmetic lives here."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as wl


def oracle_on_call(call: wl.Call, causal=True, rows=None, key_window=None, sm_scale=None,
                   threads=None):
    st = call.store
    return oracle.attention(
        wl.bf16_bits(call.q), wl.bf16_bits(st.k_cache), wl.bf16_bits(st.v_cache),
        call.qo_indptr.numpy(), call.kv_indptr.numpy(), call.kv_indices.numpy(),
        call.kv_last_page_len.numpy(), num_qo_heads=st.num_qo_heads,
        num_kv_heads=st.num_kv_heads, head_dim=st.head_dim, page_size=st.page_size,
        causal=causal, rows=rows, key_window=key_window, sm_scale=sm_scale, threads=threads)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def error_stats(got: np.ndarray, want: np.ndarray):
    d = np.abs(np.asarray(got, np.float64) - np.asarray(want, np.float64))
    return float(d.max(initial=0.0)), float(d.mean()) if d.size else 0.0
