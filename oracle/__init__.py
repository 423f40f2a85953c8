"""CPU fp64 oracle for batch-invariant paged-KV GQA attention.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the
benchmark's CPU-baseline leg are the only callers.  The product library never
imports, links or runs anything here, and this package imports nothing from
the product package.

The arithmetic lives in ``bia_oracle.c`` (plain C, fp64, one loop per term of
the definition); this module compiles it with gcc and marshals numpy arrays.
bf16 tensors are passed as their raw 16-bit patterns (``numpy.uint16``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bia_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libbia_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libbia_oracle.so`` (gcc, -O2).

    ``-ffp-contract=off`` keeps the fp64 arithmetic identical on x86 and Arm.
    """
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32, i64, f64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.oracle_attention_rows.argtypes = [i32, i32, i32, i32, f64, i32, vp, vp, vp, vp,
                                                  vp, vp, vp, i32, i64, i64, vp, i64, vp, vp,
                                                  i32]
            lib.oracle_attention_rows.restype = i32
            lib.oracle_attention_rows_masked.argtypes = [i32, i32, i32, i32, f64, i32, vp, vp,
                                                         vp, vp, vp, vp, vp, i32, i64, i64, vp,
                                                         vp, vp, i64, vp, vp, i32]
            lib.oracle_attention_rows_masked.restype = i32
            lib.oracle_mla.argtypes = [i32, i32, i32, i32, f64, i32, vp, vp, vp, vp, vp, vp, vp,
                                       vp, i32, i64, i64, vp, vp]
            lib.oracle_mla.restype = i32
            lib.oracle_row_probs.argtypes = [i32, i32, i32, i32, f64, i32, vp, vp, vp, vp, vp,
                                             vp, vp, i32, i64, i32, vp, i64]
            lib.oracle_row_probs.restype = i32
            lib.oracle_merge_states.argtypes = [vp, vp, vp, i64, i32, i32, i32, vp, vp]
            lib.oracle_merge_states.restype = i32
            _lib = lib
    return _lib


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"bf16 data must be passed as uint16 bit patterns, got {a.dtype}")
    return a


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def attention(q, k_cache, v_cache, qo_indptr, kv_indptr, kv_indices, kv_last_page_len, *,
              num_qo_heads, num_kv_heads, head_dim, page_size, causal=True, sm_scale=None,
              rows=None, key_window=None, threads=None, mask=None, mask_indptr=None):
    """Paged GQA attention in fp64.

    q: [total_q, Hq, D] uint16 (bf16 bits); k_cache / v_cache:
    [num_pages, page_size, Hkv, D] uint16.  ``rows`` is an optional int64
    array of (global q token, q head) pairs; without it every row is computed.
    ``key_window=(lo, hi)`` restricts visible keys to [lo, hi) (a split-KV
    partial).  ``mask`` (uint8, little-endian bit order) with ``mask_indptr``
    (int64 bit offsets, [batch+1]) is a custom mask: bit
    mask_indptr[b] + t*kv_len + j lets in-call token t of request b see key j
    (together with the causal rule when causal).  Returns (out [n, D]
    float64, lse [n] float64); with rows=None the shapes are
    [total_q, Hq, D] and [total_q, Hq].
    """
    lib = _load()
    q, k_cache, v_cache = _u16(q), _u16(k_cache), _u16(v_cache)
    qo, kvp, kvi, last = _i32(qo_indptr), _i32(kv_indptr), _i32(kv_indices), _i32(kv_last_page_len)
    if kvi.size == 0:
        kvi = np.zeros(1, np.int32)
    batch = len(qo) - 1
    scale = 1.0 / np.sqrt(head_dim) if sm_scale is None else float(sm_scale)
    lo, hi = (0, np.iinfo(np.int64).max) if key_window is None else key_window
    if rows is None:
        n = int(qo[-1]) * num_qo_heads
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 2))
        n = rows_arr.shape[0]
    out = np.zeros((max(n, 1), head_dim), np.float64)
    lse = np.zeros(max(n, 1), np.float64)
    if mask is not None:
        mask_arr = np.ascontiguousarray(np.asarray(mask, dtype=np.uint8))
        if mask_arr.size == 0:
            mask_arr = np.zeros(1, np.uint8)
        mip = np.ascontiguousarray(np.asarray(mask_indptr, dtype=np.int64))
    rc = lib.oracle_attention_rows_masked(
        num_qo_heads, num_kv_heads, head_dim, page_size, scale, int(bool(causal)), _ptr(q),
        _ptr(k_cache), _ptr(v_cache), _ptr(qo), _ptr(kvp), _ptr(kvi), _ptr(last), batch, int(lo),
        int(hi), None if mask is None else _ptr(mask_arr), None if mask is None else _ptr(mip),
        None if rows_arr is None else _ptr(rows_arr), n, _ptr(out), _ptr(lse),
        threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_attention_rows failed with {rc}")
    out, lse = out[:n], lse[:n]
    if rows is None:
        total_q = int(qo[-1])
        return out.reshape(total_q, num_qo_heads, head_dim), lse.reshape(total_q, num_qo_heads)
    return out, lse


def row_probs(q, k_cache, v_cache, qo_indptr, kv_indptr, kv_indices, kv_last_page_len, *,
              token, head, num_qo_heads, num_kv_heads, head_dim, page_size, causal=True,
              sm_scale=None):
    """Attention weights of one row over keys 0..kv_len-1 (fp64)."""
    lib = _load()
    q, k_cache, v_cache = _u16(q), _u16(k_cache), _u16(v_cache)
    qo, kvp, kvi, last = _i32(qo_indptr), _i32(kv_indptr), _i32(kv_indices), _i32(kv_last_page_len)
    batch = len(qo) - 1
    b = int(np.searchsorted(qo, token, side="right") - 1)
    pages = int(kvp[b + 1] - kvp[b])
    kv_len = 0 if pages == 0 else (pages - 1) * page_size + int(last[b])
    probs = np.zeros(max(kv_len, 1), np.float64)
    scale = 1.0 / np.sqrt(head_dim) if sm_scale is None else float(sm_scale)
    rc = lib.oracle_row_probs(num_qo_heads, num_kv_heads, head_dim, page_size, scale,
                              int(bool(causal)), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                              _ptr(qo), _ptr(kvp), _ptr(kvi), _ptr(last), batch, int(token),
                              int(head), _ptr(probs), probs.size)
    if rc != 0:
        raise ValueError(f"oracle_row_probs failed with {rc}")
    return probs[:kv_len]


def merge_states(v, lse, num_states=None):
    """Closed-form log-sum-exp merge.  v: [n, S, H, D] fp32, lse: [n, S, H]
    fp32.  Returns (out [n, H, D] float64, lse [n, H] float64)."""
    lib = _load()
    v = np.ascontiguousarray(v, dtype=np.float32)
    s = np.ascontiguousarray(lse, dtype=np.float32)
    n, S, H, D = v.shape
    ns = None if num_states is None else _i32(num_states)
    out = np.zeros((max(n, 1), H, D), np.float64)
    lo = np.zeros((max(n, 1), H), np.float64)
    rc = lib.oracle_merge_states(_ptr(v), _ptr(s), None if ns is None else _ptr(ns), n, S, H, D,
                                 _ptr(out), _ptr(lo))
    if rc != 0:
        raise ValueError(f"oracle_merge_states failed with {rc}")
    return out[:n], lo[:n]


def append_paged_kv(k_cache, v_cache, k_new, v_new, append_indptr, kv_indptr, kv_indices,
                    kv_last_page_len, *, page_size):
    """Paged-KV append, by its definition: the write that puts a chunk's K/V
    into the cache before that chunk attends to it ("sglang PR #43612",
    Summary: a chunked prefill reads a cache that already holds the chunk; the
    pages leave the write itself implicit).  Reading: request b's page table
    already spans its n_new new tokens as its LAST n_new keys (the same
    convention as the q tokens of a prefill call), so new token t of request b
    lands at position p = kv_len - n_new + (t - append_indptr[b]), i.e. page
    kv_indices[kv_indptr[b] + p // page_size], slot p % page_size, all kv
    heads.  Returns updated copies of the caches (uint16 bf16 bit patterns,
    [num_pages, page_size, Hkv, D]); the inputs are left as they are.
    Raises ValueError on a page index outside the cache or n_new > kv_len."""
    kc = np.array(_u16(k_cache), copy=True)
    vc = np.array(_u16(v_cache), copy=True)
    kn, vn = _u16(k_new), _u16(v_new)
    ap, kvp = _i32(append_indptr), _i32(kv_indptr)
    idx, last = _i32(kv_indices), _i32(kv_last_page_len)
    num_pages = kc.shape[0]
    for b in range(len(ap) - 1):
        n_new = int(ap[b + 1] - ap[b])
        n_pages = int(kvp[b + 1] - kvp[b])
        kv_len = (n_pages - 1) * page_size + int(last[b]) if n_pages > 0 else 0
        if n_new > kv_len:
            raise ValueError(f"request {b}: {n_new} new tokens but only {kv_len} keys")
        for i in range(n_new):
            p = kv_len - n_new + i
            page = int(idx[kvp[b] + p // page_size])
            if not 0 <= page < num_pages:
                raise ValueError(f"request {b}: page index {page} outside the cache")
            kc[page, p % page_size] = kn[ap[b] + i]
            vc[page, p % page_size] = vn[ap[b] + i]
    return kc, vc


def mla(q_nope, q_pe, ckv_cache, kpe_cache, qo_indptr, kv_indptr, kv_indices, kv_last_page_len,
        *, page_size, sm_scale, causal=True, key_window=None):
    """Multi-head latent attention over a paged latent cache, fp64: every q
    head attends to the shared rows [ckv | kpe] with scores
    sm_scale * (<q_nope, ckv> + <q_pe, kpe>) and takes the ckv rows as values.
    q_nope [total_q, H, Dc], q_pe [total_q, H, Dp], ckv_cache
    [num_pages, P, Dc], kpe_cache [num_pages, P, Dp] as bf16 bit patterns.
    Returns (out [total_q, H, Dc], lse [total_q, H]) float64."""
    lib = _load()
    qn, qp = _u16(q_nope), _u16(q_pe)
    ckv, kpe = _u16(ckv_cache), _u16(kpe_cache)
    qo, kvp, kvi, last = _i32(qo_indptr), _i32(kv_indptr), _i32(kv_indices), _i32(kv_last_page_len)
    if kvi.size == 0:
        kvi = np.zeros(1, np.int32)
    total_q, H, dc = qn.shape
    dp = qp.shape[2]
    lo, hi = (0, np.iinfo(np.int64).max) if key_window is None else key_window
    out = np.zeros((max(total_q, 1), H, dc), np.float64)
    lse = np.zeros((max(total_q, 1), H), np.float64)
    rc = lib.oracle_mla(H, dc, dp, page_size, float(sm_scale), int(bool(causal)), _ptr(qn),
                        _ptr(qp), _ptr(ckv), _ptr(kpe), _ptr(qo), _ptr(kvp), _ptr(kvi), _ptr(last),
                        len(qo) - 1, int(lo), int(hi), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_mla failed with {rc}")
    return out[:total_q], lse[:total_q]
