"""bia_mla_decode_paged on the GPU: parity with the oracle's multi-head latent
attention (8, 16 and 128 heads, pages of 1 and 16, contexts across split
tiles), bit-identical results for a request alone and in a batch, and the
host checks."""
import math

import numpy as np
import pytest
import torch

import invariant_paged_attention_gb300 as bia
import oracle
import workloads as wl
from tests.common import bf16_to_f64, error_stats
from tests.gpu_util import LSE_TOL, MAX_ABS, MEAN_ABS, same_bits

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCALE = 1.0 / math.sqrt(192)  # the pre-absorption q.k width of DeepSeek-style MLA


def run_mla(call, split=0):
    st = call.store
    desc = bia.make_mla_desc(st.num_heads, st.page_size, SCALE)
    nbytes = bia.bia_mla_decode_workspace_size(desc, call.kv_indptr, call.kv_last_page_len, split)
    assert nbytes > 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    B = len(call.q_lens)
    out = torch.full((B, st.num_heads, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, st.num_heads), float("nan"), dtype=torch.float32, device=DEV)
    bia.bia_mla_decode_paged(desc, call.q_nope, call.q_pe, st.ckv_cache, st.kpe_cache,
                             call.kv_indptr.to(DEV), call.kv_indices.to(DEV),
                             call.kv_last_page_len.to(DEV), call.kv_indptr,
                             call.kv_last_page_len, ws, out, lse, split_size=split)
    torch.cuda.synchronize()
    return out, lse, bia.bia_read_status(ws)


def oracle_mla(call):
    st = call.store
    return oracle.mla(wl.bf16_bits(call.q_nope), wl.bf16_bits(call.q_pe),
                      wl.bf16_bits(st.ckv_cache), wl.bf16_bits(st.kpe_cache),
                      call.qo_indptr.numpy(), call.kv_indptr.numpy(), call.kv_indices.numpy(),
                      call.kv_last_page_len.numpy(), page_size=st.page_size, sm_scale=SCALE)


def decode_store(ctxs, H, P, seed):
    return wl.MLAStore([wl.Sequence(seed + i, c - 1, 1) for i, c in enumerate(ctxs)], H, 512, 64,
                       P, DEV, layout_seed=seed)


@pytest.mark.parametrize("H,P", [(16, 1), (8, 16), (128, 1), (16, 64), (32, 256)])
def test_mla_decode_matches_oracle(H, P):
    st = decode_store([1, 100, 2048, 2049, 9000], H, P, seed=3000 + H + P)
    call = wl.mla_call(st, [(i, 0, 1) for i in range(len(st.seqs))])
    out, lse, status = run_mla(call)
    assert status == 0
    ref_o, ref_l = oracle_mla(call)
    got = bf16_to_f64(out)
    assert np.all(np.isfinite(got))
    mx, mean = error_stats(got, ref_o)
    assert mx <= MAX_ABS and mean <= MEAN_ABS, (mx, mean)
    got_l = lse.double().cpu().numpy()
    dl = np.abs(got_l - ref_l) / np.maximum(1.0, np.abs(ref_l))
    assert dl.max() <= LSE_TOL


def test_mla_decode_split_sizes_and_batch_invariance():
    st = decode_store([5000, 300, 12000, 2048], 16, 1, seed=3100)
    call = wl.mla_call(st, [(i, 0, 1) for i in range(4)])
    ref_o, ref_l = oracle_mla(call)
    for split in (0, 1024, 128):
        out, lse, status = run_mla(call, split)
        assert status == 0
        mx, mean = error_stats(bf16_to_f64(out), ref_o)
        assert mx <= MAX_ABS and mean <= MEAN_ABS, (split, mx, mean)
    out, lse, _ = run_mla(call)
    for i in range(4):
        solo = wl.mla_call(st, [(i, 0, 1)])
        so, sl, _ = run_mla(solo)
        assert same_bits(so, out[i:i + 1]) and same_bits(sl, lse[i:i + 1])
    # the batch in reverse order
    rev = wl.mla_call(st, [(i, 0, 1) for i in reversed(range(4))])
    ro, rl, _ = run_mla(rev)
    assert same_bits(ro.flip(0), out) and same_bits(rl.flip(0), lse)


def test_mla_bad_page_and_host_checks():
    st = decode_store([100, 50], 16, 16, seed=3200)
    call = wl.mla_call(st, [(0, 0, 1), (1, 0, 1)])
    call.kv_indices = call.kv_indices.clone()
    call.kv_indices[0] = 10_000
    _, _, status = run_mla(call)
    assert status & 1
    with pytest.raises(bia.BiaError) as e:  # 12 heads: not a multiple of 8
        desc = bia.make_mla_desc(12, 16)
        ws = torch.empty(1 << 20, dtype=torch.uint8, device=DEV)
        out = torch.empty((2, 12, 512), dtype=torch.bfloat16, device=DEV)
        bia.bia_mla_decode_paged(desc, out, out, st.ckv_cache, st.kpe_cache,
                                 call.kv_indptr.to(DEV), call.kv_indices.to(DEV),
                                 call.kv_last_page_len.to(DEV), call.kv_indptr,
                                 call.kv_last_page_len, ws, out)
    assert e.value.status == bia.BIA_ERR_UNSUPPORTED
