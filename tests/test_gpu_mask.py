"""bia_prefill_paged_mask on the GPU: parity with the oracle's custom mask,
the causal pattern as a mask and an all-ones mask bit-identical to the
unmasked calls, rows left without keys, and batch invariance."""
import numpy as np
import pytest
import torch

import invariant_paged_attention_gb300 as bia
import oracle
import workloads as wl
from tests.common import bf16_to_f64, error_stats
from tests.gpu_util import LSE_TOL, MAX_ABS, MEAN_ABS, desc_of, run_prefill, same_bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_masked(call, bits, indptr, causal=True, split=0):
    st = call.store
    desc = desc_of(st)
    ws = torch.empty(bia.bia_prefill_workspace_size(desc, call.qo_indptr, call.kv_indptr,
                                                    call.kv_last_page_len, causal, split),
                     dtype=torch.uint8, device=DEV)
    out = torch.full_like(call.q, float("nan"))
    lse = torch.full((call.total_q, st.num_qo_heads), float("nan"), dtype=torch.float32,
                     device=DEV)
    mask_d = torch.from_numpy(bits).to(DEV)
    ip = torch.from_numpy(indptr)
    bia.bia_prefill_paged_mask(desc, call.q, st.k_cache, st.v_cache, call.qo_indptr.to(DEV),
                               call.kv_indptr.to(DEV), call.kv_indices.to(DEV),
                               call.kv_last_page_len.to(DEV), call.qo_indptr, call.kv_indptr,
                               call.kv_last_page_len, mask_d, ip.to(DEV), ip, ws, out, lse,
                               causal=causal, split_size=split)
    torch.cuda.synchronize()
    assert bia.bia_read_status(ws) == 0
    return out, lse


def oracle_masked(call, bits, indptr, causal):
    st = call.store
    return oracle.attention(
        wl.bf16_bits(call.q), wl.bf16_bits(st.k_cache), wl.bf16_bits(st.v_cache),
        call.qo_indptr.numpy(), call.kv_indptr.numpy(), call.kv_indices.numpy(),
        call.kv_last_page_len.numpy(), num_qo_heads=st.num_qo_heads,
        num_kv_heads=st.num_kv_heads, head_dim=st.head_dim, page_size=st.page_size,
        causal=causal, mask=bits, mask_indptr=indptr)


def check(call, out, lse, ref_out, ref_lse):
    got = bf16_to_f64(out).reshape(ref_out.shape)
    got_l = lse.double().cpu().numpy().reshape(ref_lse.shape)
    mx, mean = error_stats(got, ref_out)
    assert np.all(np.isfinite(got))
    assert mx <= MAX_ABS and mean <= MEAN_ABS, (mx, mean)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(got_l))
    assert np.all(got[~fin] == 0.0)
    dl = np.abs(got_l[fin] - ref_lse[fin]) / np.maximum(1.0, np.abs(ref_lse[fin]))
    assert dl.size == 0 or dl.max() <= LSE_TOL


SHAPES = [  # (Hq, Hkv, D, P, [(prefix, new)])
    (32, 8, 128, 16, [(0, 300), (700, 77), (5, 1), (0, 0), (129, 160)]),
    (4, 1, 64, 1, [(0, 256), (33, 100)]),
    (32, 8, 96, 16, [(0, 130), (4090, 20)]),
    (16, 8, 256, 16, [(0, 200), (4090, 30)]),
]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("density", [0.05, 0.5, 0.95])
@pytest.mark.parametrize("shape", range(len(SHAPES)))
def test_mask_matches_oracle(shape, density, causal):
    Hq, Hkv, D, P, seqs = SHAPES[shape]
    store = wl.PagedStore([wl.Sequence(1100 + i, p, n) for i, (p, n) in enumerate(seqs)],
                          Hq, Hkv, D, P, DEV, layout_seed=3 + shape)
    call = wl.whole_prefill(store)
    bits, indptr, _ = wl.custom_mask(call, seed=int(density * 100) + shape, density=density)
    out, lse = run_masked(call, bits, indptr, causal)
    ref_out, ref_lse = oracle_masked(call, bits, indptr, causal)
    check(call, out, lse, ref_out, ref_lse)


def test_mask_across_split_tiles():
    # a 6000-key request: q tiles past key 4096 touch two split tiles
    store = wl.PagedStore([wl.Sequence(1200, 5000, 1000)], 32, 8, 128, 16, DEV, layout_seed=9)
    call = wl.whole_prefill(store)
    bits, indptr, _ = wl.custom_mask(call, seed=12, density=0.3)
    out, lse = run_masked(call, bits, indptr, causal=True)
    ref_out, ref_lse = oracle_masked(call, bits, indptr, True)
    check(call, out, lse, ref_out, ref_lse)


def test_causal_pattern_and_all_ones_masks_match_unmasked_bits():
    store = wl.PagedStore([wl.Sequence(1300 + i, p, n) for i, (p, n) in
                           enumerate([(0, 200), (4500, 90), (31, 33)])], 32, 8, 128, 16, DEV,
                          layout_seed=5)
    call = wl.whole_prefill(store)
    ref_c = run_prefill(call, causal=True)
    ref_n = run_prefill(call, causal=False)
    bits, indptr, _ = wl.custom_mask(call, seed=1, density=1.0, causal_part=True)
    o, l = run_masked(call, bits, indptr, causal=False)
    assert same_bits(o, ref_c[0]) and same_bits(l, ref_c[1])
    ones, indptr1, _ = wl.custom_mask(call, seed=2, density=1.0)
    for causal, ref in ((True, ref_c), (False, ref_n)):
        o, l = run_masked(call, ones, indptr1, causal=causal)
        assert same_bits(o, ref[0]) and same_bits(l, ref[1])


def test_rows_without_keys_and_batch_invariance():
    seqs = [(10, 70), (0, 150), (300, 40)]
    store = wl.PagedStore([wl.Sequence(1400 + i, p, n) for i, (p, n) in enumerate(seqs)],
                          32, 8, 128, 16, DEV, layout_seed=6)
    call = wl.whole_prefill(store)
    bits, indptr, dense = wl.custom_mask(call, seed=4, density=0.4)
    dense[1][7, :] = False  # request 1, token 7 sees nothing
    flat = np.concatenate([d.reshape(-1) for d in dense])
    bits = np.concatenate([np.packbits(flat, bitorder="little"), np.zeros(4, np.uint8)])
    out, lse = run_masked(call, bits, indptr, causal=True)
    row = int(call.qo_indptr[1]) + 7
    assert torch.all(out[row].float() == 0) and torch.all(torch.isneginf(lse[row]))
    # request 1 alone, with its own mask bits: the same bits
    solo = wl.make_call(store, [(1, 0, 150)])
    sflat = dense[1].reshape(-1)
    sbits = np.concatenate([np.packbits(sflat, bitorder="little"), np.zeros(4, np.uint8)])
    so, sl = run_masked(solo, sbits, np.array([0, sflat.size], np.int64), causal=True)
    a, b = int(call.qo_indptr[1]), int(call.qo_indptr[2])
    assert same_bits(so, out[a:b]) and same_bits(sl, lse[a:b])


def test_mask_validation():
    store = wl.PagedStore([wl.Sequence(1500, 0, 64)], 32, 8, 128, 16, DEV)
    call = wl.whole_prefill(store)
    bits, indptr, _ = wl.custom_mask(call, seed=5)
    with pytest.raises(bia.BiaError) as e:  # buffer shorter than q_len * kv_len bits
        run_masked(call, bits[:100], indptr)
    assert e.value.status == bia.BIA_ERR_INVALID_ARG
    with pytest.raises(bia.BiaError) as e:  # negative offset
        run_masked(call, bits, np.array([-8, 64 * 64 - 8], np.int64))
    assert e.value.status == bia.BIA_ERR_INVALID_ARG
