"""The C ABI on the host: the library builds for sm_103a, loads, exports every
symbol bia.h declares, and rejects bad arguments before enqueuing any work
(so these calls are safe without a GPU: fake, never-dereferenced device
pointers are passed)."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bia.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and
                                not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available")


@pytest.fixture(scope="module")
def bia():
    from invariant_paged_attention_gb300 import build
    build.build()
    import invariant_paged_attention_gb300 as m
    m.load()
    return m


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"BIA_API[^;(]*?\b(bia_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    syms = declared_symbols()
    for name in ("bia_prefill_paged", "bia_decode_paged", "bia_merge_states"):
        assert name in syms


def test_library_exports_every_declared_symbol(bia):
    lib = bia.load()
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert sorted(bia.EXPORTS) == declared_symbols()
    nm = shutil.which("nm")
    if nm:
        out = subprocess.run([nm, "-D", "--defined-only", bia.LIB_PATH], capture_output=True,
                             text=True).stdout
        exported = set(re.findall(r"\b(bia_\w+)\b", out))
        assert exported == set(declared_symbols())


def test_q_tile_grid(bia):
    assert bia.bia_q_tile_tokens(4) == 32
    assert bia.bia_q_tile_tokens(1) == 128
    assert bia.bia_q_tile_tokens(8) == 16
    assert bia.bia_q_tile_tokens(3) == 0
    assert bia.bia_q_tile_tokens(0) == 0


def test_status_strings(bia):
    assert bia.status_string(0) == "ok"
    assert "workspace" in bia.status_string(-3)
    assert bia.status_string(12345) == "unknown status"


QWEN = dict(num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=1)


def test_workspace_size_counts_split_partials(bia):
    desc = bia.make_desc(**QWEN)
    qo = torch.tensor([0, 5000], dtype=torch.int32)
    kvp = torch.tensor([0, 5000], dtype=torch.int32)
    last = torch.tensor([1], dtype=torch.int32)
    one_split = bia.bia_prefill_workspace_size(desc, qo, kvp, last, True, 8192)
    two_splits = bia.bia_prefill_workspace_size(desc, qo, kvp, last, True, 4096)
    assert one_split > 0
    # rows that need a merge: all 5000 tokens x 2 splits x 32 heads x (128+1) fp32
    assert two_splits - one_split >= 5000 * 2 * 32 * 129 * 4
    # bad inputs answer 0
    assert bia.bia_prefill_workspace_size(desc, qo, kvp, last, True, 100) == 0
    assert bia.bia_prefill_workspace_size(bia.make_desc(32, 8, 80, 1), qo, kvp, last) == 0
    assert bia.bia_decode_workspace_size(desc, kvp, last) > 0


FAKE = 1 << 20  # a 256-byte aligned address that is never dereferenced


def call_prefill(bia, desc, qo, kvp, last, *, causal=1, split=0, ws_bytes=1 << 30, ws=FAKE,
                 num_pages=1 << 20, lse=None, kv_indices=FAKE):
    lib = bia.load()
    qo = torch.tensor(qo, dtype=torch.int32)
    kvp = torch.tensor(kvp, dtype=torch.int32)
    last = torch.tensor(last, dtype=torch.int32)
    p = ctypes.c_void_p
    return lib.bia_prefill_paged(ctypes.byref(desc), p(FAKE), p(FAKE), p(FAKE), num_pages,
                                 p(FAKE), p(FAKE), p(kv_indices), p(FAKE), p(qo.data_ptr()),
                                 p(kvp.data_ptr()), p(last.data_ptr()), len(qo) - 1, causal,
                                 split, p(ws), ws_bytes, p(FAKE), None if lse is None else p(lse),
                                 None)


def test_prefill_rejects_bad_arguments_on_the_host(bia):
    d = bia.make_desc(**QWEN)
    inv, uns, small = bia.BIA_ERR_INVALID_ARG, bia.BIA_ERR_UNSUPPORTED, bia.BIA_ERR_WORKSPACE_TOO_SMALL
    assert call_prefill(bia, d, [0, 10, 5], [0, 10, 20], [1, 1]) == inv  # qo not monotone
    assert call_prefill(bia, d, [1, 10], [0, 10], [1]) == inv  # qo_indptr[0] != 0
    assert call_prefill(bia, d, [0, 10], [0, 5], [1]) == inv  # q_len > kv_len (causal)
    assert call_prefill(bia, d, [0, 10], [0, 10], [0]) == inv  # last page length 0
    assert call_prefill(bia, d, [0, 10], [0, 10], [1], split=100) == uns
    assert call_prefill(bia, bia.make_desc(32, 8, 80, 1), [0, 10], [0, 10], [1]) == uns
    assert call_prefill(bia, bia.make_desc(32, 6, 128, 1), [0, 10], [0, 10], [1]) == uns
    assert call_prefill(bia, bia.make_desc(48, 3, 128, 1), [0, 10], [0, 10], [1]) == uns
    assert call_prefill(bia, bia.make_desc(32, 8, 128, 3), [0, 10], [0, 10], [1]) == uns
    assert call_prefill(bia, d, [0, 10], [0, 10], [1], ws_bytes=300) == small
    assert call_prefill(bia, d, [0, 10], [0, 10], [1], ws=FAKE + 16) == inv  # unaligned
    assert call_prefill(bia, d, [0, 10], [0, 10], [1], num_pages=0) == inv
    assert call_prefill(bia, d, [0, 10], [0, 10], [1], lse=FAKE + 2) == inv  # unaligned lse
    assert call_prefill(bia, d, [0, 10], [0, 10], [1], kv_indices=FAKE + 1) == inv
    lib = bia.load()
    args = [None] * 20
    args[4], args[12], args[13], args[14], args[16] = 0, 0, 0, 0, 0
    assert lib.bia_prefill_paged(*args) == inv


def test_decode_and_merge_reject_bad_arguments_on_the_host(bia):
    lib = bia.load()
    d = bia.make_desc(**QWEN)
    p = ctypes.c_void_p
    kvp = torch.tensor([0, 0], dtype=torch.int32)  # a request with no key
    last = torch.tensor([1], dtype=torch.int32)
    rc = lib.bia_decode_paged(ctypes.byref(d), p(FAKE), p(FAKE), p(FAKE), 1 << 20, p(FAKE),
                              p(FAKE), p(FAKE), p(kvp.data_ptr()), p(last.data_ptr()), 1, 0,
                              p(FAKE), 1 << 30, p(FAKE), None, None)
    assert rc == bia.BIA_ERR_INVALID_ARG
    assert lib.bia_merge_states(p(FAKE), p(FAKE), None, 4, 2, 8, 130, p(FAKE), None,
                                None) == bia.BIA_ERR_UNSUPPORTED
    assert lib.bia_merge_states(p(FAKE + 4), p(FAKE), None, 4, 2, 8, 128, p(FAKE), None,
                                None) == bia.BIA_ERR_INVALID_ARG
    assert lib.bia_merge_states(p(FAKE), p(FAKE + 2), None, 4, 2, 8, 128, p(FAKE), None,
                                None) == bia.BIA_ERR_INVALID_ARG  # unaligned lse of the states
    assert lib.bia_merge_states(p(FAKE), p(FAKE), p(FAKE + 1), 4, 2, 8, 128, p(FAKE), None,
                                None) == bia.BIA_ERR_INVALID_ARG  # unaligned counts
    assert lib.bia_merge_states(None, None, None, 0, 2, 8, 128, None, None, None) == bia.BIA_OK


def test_append_rejects_bad_arguments_on_the_host(bia):
    lib = bia.load()
    p = ctypes.c_void_p

    def call(desc, ap, kvp, last, k_new=FAKE, status=None):
        ap, kvp, last = (torch.tensor(x, dtype=torch.int32) for x in (ap, kvp, last))
        return lib.bia_append_paged_kv(ctypes.byref(desc), p(k_new), p(FAKE), p(FAKE), p(FAKE),
                                       1 << 20, p(FAKE), p(FAKE), p(FAKE), p(FAKE),
                                       p(ap.data_ptr()), p(kvp.data_ptr()), p(last.data_ptr()),
                                       len(ap) - 1, None if status is None else p(status), None)
    d = bia.make_desc(32, 8, 128, 16)
    inv = bia.BIA_ERR_INVALID_ARG
    assert call(d, [0, 17], [0, 1], [16]) == inv  # 17 new tokens, 16 keys
    assert call(d, [1, 2], [0, 1], [16]) == inv  # append_indptr[0] != 0
    assert call(d, [0, 2, 1], [0, 1, 2], [16, 16]) == inv  # decreasing append_indptr
    assert call(d, [0, 1], [0, 1], [0]) == inv  # last page length 0
    assert call(d, [0, 1], [0, 1], [1], k_new=FAKE + 8) == inv  # unaligned rows
    assert call(d, [0, 1], [0, 1], [1], status=FAKE + 2) == inv  # unaligned status word
    assert call(bia.make_desc(32, 8, 80, 16), [0, 1], [0, 1], [1]) == bia.BIA_ERR_UNSUPPORTED
    # nothing to write and no status word: returns before touching the device
    assert call(d, [0, 0, 0], [0, 1, 3], [5, 2]) == bia.BIA_OK


def test_binding_fails_loudly_without_the_library(tmp_path):
    import invariant_paged_attention_gb300 as m
    saved = m._lib
    m._lib = None
    try:
        with pytest.raises(RuntimeError, match="not built"):
            m.load(str(tmp_path / "missing.so"))
    finally:
        m._lib = saved


def test_mla_extend_rejects_bad_arguments_on_the_host(bia):
    lib = bia.load()
    p = ctypes.c_void_p

    def call(desc, qo, kvp, last, split=0, ws_bytes=1 << 30, qo_host=True):
        qo, kvp, last = (torch.tensor(x, dtype=torch.int32) for x in (qo, kvp, last))
        return lib.bia_mla_prefill_paged(
            ctypes.byref(desc), p(FAKE), p(FAKE), p(FAKE), p(FAKE), 1 << 20, p(FAKE), p(FAKE),
            p(FAKE), p(FAKE), p(qo.data_ptr()) if qo_host else None, p(kvp.data_ptr()),
            p(last.data_ptr()), len(kvp) - 1, split, p(FAKE), ws_bytes, p(FAKE), None, None)
    d = bia.make_mla_desc(16, 16)
    inv = bia.BIA_ERR_INVALID_ARG
    assert call(d, [0, 17], [0, 1], [16]) == inv  # 17 q tokens, 16 keys
    assert call(d, [1, 2], [0, 1], [16]) == inv  # qo_indptr[0] != 0
    assert call(d, [0, 3, 2], [0, 1, 2], [16, 16]) == inv  # decreasing qo_indptr
    assert call(d, [0, 1], [0, 1], [16], qo_host=False) == inv
    assert call(d, [0, 1], [0, 1], [16], split=100) == bia.BIA_ERR_UNSUPPORTED
    assert call(bia.make_mla_desc(12, 16), [0, 1], [0, 1], [16]) == bia.BIA_ERR_UNSUPPORTED
    assert call(d, [0, 1], [0, 1], [16], ws_bytes=16) == bia.BIA_ERR_WORKSPACE_TOO_SMALL
    # no q token anywhere: nothing is enqueued
    assert call(d, [0, 0, 0], [0, 1, 3], [5, 2]) == bia.BIA_OK


def test_mla_extend_workspace_counts_token_partials(bia):
    d = bia.make_mla_desc(16, 16)
    # 20 tokens at positions 4090..4109: none reaches a second 8192-key split
    # tile; with the default 4096 the last 14 do, so the request has 2 splits
    one = bia.bia_mla_prefill_workspace_size(d, [0, 20], [0, 257], [14], 8192)
    two = bia.bia_mla_prefill_workspace_size(d, [0, 20], [0, 257], [14])
    # partial rows: 20 tokens x 2 splits x 16 heads x (512 + 1) fp32
    assert two - one >= 20 * 2 * 16 * 513 * 4
    assert bia.bia_mla_prefill_workspace_size(d, [0, 20], [0, 257], [14], 100) == 0
    assert bia.bia_mla_prefill_workspace_size(d, [0, 20], [0, 1], [14]) == 0  # 20 > 14 keys


def test_sizes_past_the_32_bit_limits_are_refused_on_the_host(bia):
    """The limits include/bia.h states: keys per request below 2^30, and for
    the prefill / MLA tensor maps fewer than 2^31 key rows; refused before
    anything is enqueued (the pointers here are never dereferenced)."""
    d = bia.make_desc(32, 8, 128, 1)
    uns = bia.BIA_ERR_UNSUPPORTED
    # one request of 2^30 + 1 keys
    assert call_prefill(bia, d, [0, 1], [0, (1 << 30) + 1], [1]) == uns
    # 2^28 pages x 1 key x 8 kv heads = 2^31 rows of the K/V tensor maps
    assert call_prefill(bia, d, [0, 10], [0, 10], [1], num_pages=1 << 28) == uns
    lib = bia.load()
    p = ctypes.c_void_p
    md = bia.make_mla_desc(16, 1)
    kvp = torch.tensor([0, 10], dtype=torch.int32)
    last = torch.tensor([1], dtype=torch.int32)
    rc = lib.bia_mla_decode_paged(ctypes.byref(md), p(FAKE), p(FAKE), p(FAKE), p(FAKE), 1 << 31,
                                  p(FAKE), p(FAKE), p(FAKE), p(kvp.data_ptr()),
                                  p(last.data_ptr()), 1, 0, p(FAKE), 1 << 30, p(FAKE), None,
                                  None)
    assert rc == uns


def test_binding_constants_match_the_header(bia):
    """The numbers the binding mirrors from include/bia.h (split sizes, the
    q-tile height, status codes, MLA widths, the static decode scratch)."""
    import re
    text = open(HEADER).read()
    defines = {m.group(1): m.group(2) for m in
               re.finditer(r"#define (BIA_[A-Z0-9_]+) (.+)", text)}
    assert int(defines["BIA_Q_TILE_ROWS"]) == bia.BIA_Q_TILE_ROWS
    assert int(defines["BIA_PREFILL_SPLIT"]) == bia.BIA_PREFILL_SPLIT
    assert int(defines["BIA_DECODE_SPLIT"]) == bia.BIA_DECODE_SPLIT
    assert int(defines["BIA_MLA_CKV_DIM"]) == bia.MLA_CKV_DIM
    assert int(defines["BIA_MLA_KPE_DIM"]) == bia.MLA_KPE_DIM
    assert defines["BIA_DECODE_NOALLOC_SCRATCH_BYTES"].strip() == "((size_t)64 << 20)"
    assert bia.BIA_DECODE_NOALLOC_SCRATCH_BYTES == 64 << 20
    codes = dict(re.findall(r"(BIA_(?:OK|ERR_[A-Z_]+)) = (-?\d+)", text))
    assert {k: int(v) for k, v in codes.items()} == {
        "BIA_OK": bia.BIA_OK, "BIA_ERR_INVALID_ARG": bia.BIA_ERR_INVALID_ARG,
        "BIA_ERR_UNSUPPORTED": bia.BIA_ERR_UNSUPPORTED,
        "BIA_ERR_WORKSPACE_TOO_SMALL": bia.BIA_ERR_WORKSPACE_TOO_SMALL,
        "BIA_ERR_CUDA": bia.BIA_ERR_CUDA}


def test_noalloc_decode_reports_the_regular_status_codes(bia):
    """The static-scratch decode runs every host-side check of the regular
    decode first, so a bad split or a request without keys gets the same
    status, before anything touches a GPU."""
    lib = bia.load()
    p = ctypes.c_void_p
    d = bia.make_desc(**QWEN)
    kvp = torch.tensor([0, 10], dtype=torch.int32)
    last = torch.tensor([1], dtype=torch.int32)

    def call(split, kvp=kvp):
        return lib.bia_decode_paged_noalloc(ctypes.byref(d), p(FAKE), p(FAKE), p(FAKE), 1 << 20,
                                            p(FAKE), p(FAKE), p(FAKE), p(kvp.data_ptr()),
                                            p(last.data_ptr()), 1, split, p(FAKE), None, None)
    assert call(100) == bia.BIA_ERR_UNSUPPORTED  # not a multiple of 128
    assert call(0, torch.tensor([0, 0], dtype=torch.int32)) == bia.BIA_ERR_INVALID_ARG


def test_host_pointers_are_refused_before_any_launch(bia):
    """A call whose every argument is valid but whose buffers live in host
    memory returns an error and launches nothing (without a GPU the residency
    check itself cannot run and the call fails with BIA_ERR_CUDA)."""
    lib = bia.load()
    p = ctypes.c_void_p
    d = bia.make_desc(32, 8, 128, 16)
    kvp = torch.tensor([0, 2], dtype=torch.int32)
    last = torch.tensor([5], dtype=torch.int32)
    idx = torch.tensor([0, 1], dtype=torch.int32)
    k = torch.zeros(2, 16, 8, 128, dtype=torch.bfloat16)
    q = torch.zeros(1, 32, 128, dtype=torch.bfloat16)
    out = torch.zeros_like(q)
    ws = torch.zeros(1 << 20, dtype=torch.uint8)
    wsp = (ws.data_ptr() + 255) // 256 * 256
    before = lib.bia_launch_count()
    rc = lib.bia_decode_paged(ctypes.byref(d), p(q.data_ptr()), p(k.data_ptr()), p(k.data_ptr()),
                              2, p(kvp.data_ptr()), p(idx.data_ptr()), p(last.data_ptr()),
                              p(kvp.data_ptr()), p(last.data_ptr()), 1, 0, p(wsp), 1 << 19,
                              p(out.data_ptr()), None, None)
    assert rc in (bia.BIA_ERR_INVALID_ARG, bia.BIA_ERR_CUDA)
    assert lib.bia_launch_count() == before


def test_bounded_workspace_covers_every_call_within_the_bounds(bia):
    """A bounded call's workspace holds the plan of any call within its
    bounds: never smaller than the exact size of a random such call."""
    import numpy as np
    rng = np.random.default_rng(5)
    for Hq, Hkv, D, P in [(32, 8, 128, 1), (32, 8, 128, 16), (16, 8, 256, 1), (8, 8, 64, 4)]:
        d = bia.make_desc(Hq, Hkv, D, P)
        for _ in range(20):
            B = int(rng.integers(1, 9))
            max_q, max_kv = int(rng.integers(1, 3000)), int(rng.integers(1, 20000))
            max_kv = max(max_kv, max_q)
            total = int(rng.integers(max_q, B * max_q + 1))
            bd = bia.make_bounds(max_q, max_kv, total)
            cap = bia.bia_prefill_bounded_workspace_size(d, bd, B)
            dcap = bia.bia_decode_bounded_workspace_size(d, bd, B)
            assert cap > 0 and dcap > 0
            # a random call inside the bounds
            kv = rng.integers(1, max_kv + 1, B)
            q = np.minimum(rng.integers(0, max_q + 1, B), kv)
            while q.sum() > total:
                q[int(np.argmax(q))] -= 1
            pages = -(-kv // P)
            qo = torch.tensor(np.concatenate([[0], np.cumsum(q)]), dtype=torch.int32)
            kvp = torch.tensor(np.concatenate([[0], np.cumsum(pages)]), dtype=torch.int32)
            last = torch.tensor(kv - (pages - 1) * P, dtype=torch.int32)
            assert bia.bia_prefill_workspace_size(d, qo, kvp, last) <= cap
            assert bia.bia_decode_workspace_size(d, kvp, last) <= dcap


def test_bounded_calls_reject_bad_arguments_on_the_host(bia):
    lib = bia.load()
    p = ctypes.c_void_p
    d = bia.make_desc(**QWEN)

    def prefill(bounds, split=0, ws_bytes=1 << 30, batch=2):
        return lib.bia_prefill_paged_bounded(
            ctypes.byref(d), None if bounds is None else ctypes.byref(bounds), p(FAKE), p(FAKE),
            p(FAKE), 1 << 20, p(FAKE), p(FAKE), p(FAKE), p(FAKE), batch, 1, split, p(FAKE),
            ws_bytes, p(FAKE), None, None)

    def decode(bounds, split=0):
        return lib.bia_decode_paged_bounded(
            ctypes.byref(d), None if bounds is None else ctypes.byref(bounds), p(FAKE), p(FAKE),
            p(FAKE), 1 << 20, p(FAKE), p(FAKE), p(FAKE), 4, split, p(FAKE), 1 << 30, p(FAKE),
            None, None)
    inv = bia.BIA_ERR_INVALID_ARG
    assert prefill(None) == inv
    assert prefill(bia.make_bounds(100, -1, 200)) == inv
    assert prefill(bia.make_bounds(-1, 100, 200)) == inv
    assert prefill(bia.make_bounds(100, 1000, 200), batch=0) == inv
    assert prefill(bia.make_bounds(100, 1000, 200), split=100) == bia.BIA_ERR_UNSUPPORTED
    assert prefill(bia.make_bounds(100, 1 << 30, 200)) == bia.BIA_ERR_UNSUPPORTED
    assert prefill(bia.make_bounds(100, 1000, 200), ws_bytes=64) == \
        bia.BIA_ERR_WORKSPACE_TOO_SMALL
    assert decode(None) == inv
    assert decode(bia.make_bounds(1, 0, 0)) == inv  # a decode request owns at least one key
    assert decode(bia.make_bounds(1, 1000, 0), split=100) == bia.BIA_ERR_UNSUPPORTED
    assert bia.bia_decode_bounded_workspace_size(d, bia.make_bounds(1, 0, 0), 4) == 0
    assert bia.bia_prefill_bounded_workspace_size(d, bia.make_bounds(1, 10, -1), 4) == 0
