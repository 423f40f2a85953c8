"""bia_mla_prefill_paged on the GPU: causal multi-head latent attention extend
against the oracle, and its invariance.  Each q token runs as its own query,
so its bits are the same in any batch, under any chunking of the extend (on
the q-tile grid or off it), and equal to a decode of that position with the
same split size."""
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
SCALE = 1.0 / math.sqrt(192)


def run_extend(call, split=0):
    st = call.store
    desc = bia.make_mla_desc(st.num_heads, st.page_size, SCALE)
    nbytes = bia.bia_mla_prefill_workspace_size(desc, call.qo_indptr, call.kv_indptr,
                                                call.kv_last_page_len, split)
    assert nbytes > 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    T = int(call.qo_indptr[-1])
    out = torch.full((T, st.num_heads, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((T, st.num_heads), float("nan"), dtype=torch.float32, device=DEV)
    bia.bia_mla_prefill_paged(desc, call.q_nope, call.q_pe, st.ckv_cache, st.kpe_cache,
                              call.qo_indptr.to(DEV), call.kv_indptr.to(DEV),
                              call.kv_indices.to(DEV), call.kv_last_page_len.to(DEV),
                              call.qo_indptr, call.kv_indptr, call.kv_last_page_len, ws, out, lse,
                              split_size=split)
    torch.cuda.synchronize()
    return out, lse, bia.bia_read_status(ws)


def run_decode(call, split):
    st = call.store
    desc = bia.make_mla_desc(st.num_heads, st.page_size, SCALE)
    ws = torch.empty(bia.bia_mla_decode_workspace_size(desc, call.kv_indptr,
                                                       call.kv_last_page_len, split),
                     dtype=torch.uint8, device=DEV)
    B = len(call.q_lens)
    out = torch.empty((B, st.num_heads, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((B, st.num_heads), dtype=torch.float32, device=DEV)
    bia.bia_mla_decode_paged(desc, call.q_nope, call.q_pe, st.ckv_cache, st.kpe_cache,
                             call.kv_indptr.to(DEV), call.kv_indices.to(DEV),
                             call.kv_last_page_len.to(DEV), call.kv_indptr,
                             call.kv_last_page_len, ws, out, lse, split_size=split)
    torch.cuda.synchronize()
    return out, lse


def oracle_mla(call):
    st = call.store
    return oracle.mla(wl.bf16_bits(call.q_nope), wl.bf16_bits(call.q_pe),
                      wl.bf16_bits(st.ckv_cache), wl.bf16_bits(st.kpe_cache),
                      call.qo_indptr.numpy(), call.kv_indptr.numpy(), call.kv_indices.numpy(),
                      call.kv_last_page_len.numpy(), page_size=st.page_size, sm_scale=SCALE)


def check_parity(call, out, lse):
    ref_o, ref_l = oracle_mla(call)
    got = bf16_to_f64(out)
    assert np.all(np.isfinite(got))
    mx, mean = error_stats(got, ref_o)
    assert mx <= MAX_ABS and mean <= MEAN_ABS, (mx, mean)
    got_l = lse.double().cpu().numpy()
    assert np.max(np.abs(got_l - ref_l) / np.maximum(1.0, np.abs(ref_l))) <= LSE_TOL


# (prefix, new tokens): a prompt from key 0, short extends, one that crosses
# the 4096-key split boundary inside the extend, a long prefix, an empty one
SEQS = [(0, 37), (3000, 5), (4090, 20), (9000, 3), (100, 0)]


def extend_store(H, P, seed, seqs=SEQS):
    return wl.MLAStore([wl.Sequence(seed + i, p, n) for i, (p, n) in enumerate(seqs)], H, 512, 64,
                       P, DEV, layout_seed=seed)


@pytest.mark.parametrize("H,P", [(16, 16), (8, 1), (128, 16)])
def test_mla_extend_matches_oracle(H, P):
    st = extend_store(H, P, seed=5000 + H + P)
    call = wl.mla_call(st, [(i, 0, s.new) for i, s in enumerate(st.seqs)])
    out, lse, status = run_extend(call)
    assert status == 0
    check_parity(call, out, lse)


@pytest.mark.parametrize("split", [128, 1024])
def test_mla_extend_small_splits_match_oracle(split):
    st = extend_store(16, 1, seed=5200)
    call = wl.mla_call(st, [(i, 0, s.new) for i, s in enumerate(st.seqs)])
    out, lse, status = run_extend(call, split)
    assert status == 0
    check_parity(call, out, lse)


def test_mla_extend_batch_chunk_and_decode_invariance():
    st = extend_store(16, 16, seed=5300)
    parts = [(i, 0, s.new) for i, s in enumerate(st.seqs)]
    out, lse, _ = run_extend(wl.mla_call(st, parts))
    qo = wl.mla_call(st, parts).qo_indptr.tolist()
    # each request alone
    for i, s in enumerate(st.seqs):
        if s.new == 0:
            continue
        so, sl, _ = run_extend(wl.mla_call(st, [(i, 0, s.new)]))
        assert same_bits(so, out[qo[i]:qo[i + 1]]) and same_bits(sl, lse[qo[i]:qo[i + 1]])
    # request 2 (crossing the split boundary) in chunks of 7 tokens, off any grid,
    # each chunk batched with a one-token extend of request 1
    i, n = 2, st.seqs[2].new
    for a in range(0, n, 7):
        b = min(n, a + 7)
        co, cl, _ = run_extend(wl.mla_call(st, [(1, 4, 5), (i, a, b)]))
        assert same_bits(co[1:], out[qo[i] + a:qo[i] + b])
        assert same_bits(cl[1:], lse[qo[i] + a:qo[i] + b])
    # a token of the extend equals a decode of its position at the same split
    for t in (0, 5, 6, 19):
        do, dl = run_decode(wl.mla_call(st, [(i, t, t + 1)]), bia.BIA_PREFILL_SPLIT)
        assert same_bits(do[0], out[qo[i] + t]) and same_bits(dl[0], lse[qo[i] + t])
