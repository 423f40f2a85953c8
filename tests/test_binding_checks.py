"""The Python binding checks the tensors it is given before the library sees
their addresses: dtype, contiguity, the shapes it takes sizes from, and last
that they are CUDA tensors.  These cases run on CPU tensors; the library is
replaced by a stub that fails the test if any call reaches it."""
import pytest
import torch

import invariant_paged_attention_gb300 as bia

BF16, F32, I32 = torch.bfloat16, torch.float32, torch.int32


@pytest.fixture(autouse=True)
def no_library(monkeypatch):
    def reached(*a, **k):
        raise AssertionError("the library was called before the binding's checks failed")
    monkeypatch.setattr(bia, "load", reached)


def prefill_args(**over):
    """Well-formed CPU arguments of one prefill call: 2 requests, 4 q heads
    over 1 kv head of 64, pages of 16."""
    a = dict(desc=bia.make_desc(4, 1, 64, 16), q=torch.zeros(10, 4, 64, dtype=BF16),
             k_cache=torch.zeros(3, 16, 1, 64, dtype=BF16),
             v_cache=torch.zeros(3, 16, 1, 64, dtype=BF16),
             qo_indptr=torch.tensor([0, 6, 10], dtype=I32),
             kv_indptr=torch.tensor([0, 1, 3], dtype=I32),
             kv_indices=torch.tensor([0, 1, 2], dtype=I32),
             kv_last_page_len=torch.tensor([6, 4], dtype=I32),
             qo_indptr_host=[0, 6, 10], kv_indptr_host=[0, 1, 3], kv_last_page_len_host=[6, 4],
             workspace=torch.zeros(1024, dtype=torch.uint8), out=torch.zeros(10, 4, 64, dtype=BF16),
             lse=torch.zeros(10, 4, dtype=F32))
    a.update(over)
    return a


def decode_args(**over):
    a = prefill_args(q=torch.zeros(2, 4, 64, dtype=BF16), out=torch.zeros(2, 4, 64, dtype=BF16),
                     lse=torch.zeros(2, 4, dtype=F32))
    for k in ("qo_indptr", "qo_indptr_host"):
        del a[k]
    a.update(over)
    return a


def test_well_formed_host_tensors_stop_at_the_device_check():
    with pytest.raises(ValueError, match="q must be a CUDA tensor"):
        bia.bia_prefill_paged(**prefill_args())
    with pytest.raises(ValueError, match="q must be a CUDA tensor"):
        bia.bia_decode_paged(**decode_args())
    a = decode_args()
    del a["workspace"]
    with pytest.raises(ValueError, match="q must be a CUDA tensor"):
        bia.bia_decode_paged_noalloc(**a)


@pytest.mark.parametrize("name,bad", [
    ("q", torch.zeros(10, 4, 64, dtype=torch.float16)),
    ("k_cache", torch.zeros(3, 16, 1, 64, dtype=F32)),
    ("kv_indices", torch.tensor([0, 1, 2], dtype=torch.int64)),
    ("lse", torch.zeros(10, 4, dtype=torch.float64)),
])
def test_wrong_dtype(name, bad):
    with pytest.raises(TypeError, match=f"{name} must be"):
        bia.bia_prefill_paged(**prefill_args(**{name: bad}))


def test_strided_views_and_missing_tensors():
    strided = torch.zeros(3, 16, 2, 64, dtype=BF16)[:, :, :1]
    with pytest.raises(ValueError, match="v_cache must be contiguous"):
        bia.bia_prefill_paged(**prefill_args(v_cache=strided))
    with pytest.raises(TypeError, match="out is required"):
        bia.bia_prefill_paged(**prefill_args(out=None))
    with pytest.raises(TypeError, match="must be a torch.Tensor"):
        bia.bia_prefill_paged(**prefill_args(kv_indptr=[0, 1, 3]))
    # lse is optional: without it the next failure is the device check
    with pytest.raises(ValueError, match="CUDA tensor"):
        bia.bia_prefill_paged(**prefill_args(lse=None))


def test_shapes_the_sizes_come_from():
    with pytest.raises(ValueError, match="out has shape"):
        bia.bia_prefill_paged(**prefill_args(out=torch.zeros(10, 4, 32, dtype=BF16)))
    with pytest.raises(ValueError, match="lse must hold"):
        bia.bia_decode_paged(**decode_args(lse=torch.zeros(2, 3, dtype=F32)))
    with pytest.raises(ValueError, match="k_cache and v_cache"):
        bia.bia_prefill_paged(**prefill_args(v_cache=torch.zeros(2, 16, 1, 64, dtype=BF16)))
    with pytest.raises(ValueError, match="k_cache and v_cache"):
        bia.bia_decode_paged(**decode_args(k_cache=torch.zeros(3, 16, 64, dtype=BF16),
                                           v_cache=torch.zeros(3, 16, 64, dtype=BF16)))


def test_mask_and_append_checks():
    a = prefill_args()
    a.update(mask=torch.zeros(16, dtype=I32), mask_indptr=torch.tensor([0, 36, 86]),
             mask_indptr_host=[0, 36, 86])
    with pytest.raises(TypeError, match="mask must be"):
        bia.bia_prefill_paged_mask(**a)
    a.update(mask=torch.zeros(16, dtype=torch.uint8), mask_indptr=torch.tensor([0, 36, 86],
                                                                                dtype=I32))
    with pytest.raises(TypeError, match="mask_indptr must be"):
        bia.bia_prefill_paged_mask(**a)

    p = prefill_args()
    app = dict(desc=p["desc"], k_new=torch.zeros(10, 1, 64, dtype=BF16),
               v_new=torch.zeros(9, 1, 64, dtype=BF16), k_cache=p["k_cache"],
               v_cache=p["v_cache"], append_indptr=p["qo_indptr"], kv_indptr=p["kv_indptr"],
               kv_indices=p["kv_indices"], kv_last_page_len=p["kv_last_page_len"],
               append_indptr_host=[0, 6, 10], kv_indptr_host=[0, 1, 3],
               kv_last_page_len_host=[6, 4])
    with pytest.raises(ValueError, match="v_new has shape"):
        bia.bia_append_paged_kv(**app)
    app["v_new"] = torch.zeros(10, 1, 64, dtype=BF16)
    with pytest.raises(TypeError, match="status must be"):
        bia.bia_append_paged_kv(**app, status=torch.zeros(1, dtype=torch.int64))
    with pytest.raises(ValueError, match="CUDA tensor"):
        bia.bia_append_paged_kv(**app)


def test_merge_checks():
    v, s = torch.zeros(5, 3, 2, 128), torch.zeros(5, 3, 2)
    out, lse = torch.zeros(5, 2, 128, dtype=BF16), torch.zeros(5, 2)
    with pytest.raises(ValueError, match="v must be"):
        bia.bia_merge_states(v[0], s, out, lse)
    with pytest.raises(ValueError, match="s must be"):
        bia.bia_merge_states(v, torch.zeros(5, 2, 2), out, lse)
    with pytest.raises(ValueError, match="out_lse must be"):
        bia.bia_merge_states(v, s, out, torch.zeros(2, 5))
    with pytest.raises(ValueError, match="num_states must hold"):
        bia.bia_merge_states(v, s, out, lse, torch.zeros(4, dtype=I32))
    with pytest.raises(TypeError, match="v must be"):
        bia.bia_merge_states(v.double(), s, out, lse)
    with pytest.raises(ValueError, match="CUDA tensor"):
        bia.bia_merge_states(v, s, out, lse, torch.zeros(5, dtype=I32))


def test_mla_checks():
    args = dict(desc=bia.make_mla_desc(16, 16), q_nope=torch.zeros(2, 16, 512, dtype=BF16),
                q_pe=torch.zeros(2, 16, 64, dtype=BF16),
                ckv_cache=torch.zeros(4, 16, 512, dtype=BF16),
                kpe_cache=torch.zeros(3, 16, 64, dtype=BF16),
                kv_indptr=torch.tensor([0, 1, 2], dtype=I32),
                kv_indices=torch.tensor([0, 1], dtype=I32),
                kv_last_page_len=torch.tensor([3, 5], dtype=I32), kv_indptr_host=[0, 1, 2],
                kv_last_page_len_host=[3, 5], workspace=torch.zeros(256, dtype=torch.uint8),
                out=torch.zeros(2, 16, 512, dtype=BF16))
    with pytest.raises(ValueError, match="same number of pages"):
        bia.bia_mla_decode_paged(**args)
    args["kpe_cache"] = torch.zeros(4, 16, 64, dtype=BF16)
    with pytest.raises(ValueError, match="out has shape"):
        bia.bia_mla_decode_paged(**{**args, "out": torch.zeros(2, 16, 64, dtype=BF16)})
    with pytest.raises(ValueError, match="CUDA tensor"):
        bia.bia_mla_decode_paged(**args)


def test_read_status_wants_a_device_workspace():
    with pytest.raises(ValueError, match="workspace must be a CUDA tensor"):
        bia.bia_read_status(torch.zeros(256, dtype=torch.uint8))


def test_mla_extend_checks():
    args = dict(desc=bia.make_mla_desc(16, 16), q_nope=torch.zeros(5, 16, 512, dtype=BF16),
                q_pe=torch.zeros(5, 16, 64, dtype=BF16),
                ckv_cache=torch.zeros(4, 16, 512, dtype=BF16),
                kpe_cache=torch.zeros(4, 16, 64, dtype=BF16),
                qo_indptr=torch.tensor([0, 2, 5], dtype=I32),
                kv_indptr=torch.tensor([0, 1, 2], dtype=I32),
                kv_indices=torch.tensor([0, 1], dtype=I32),
                kv_last_page_len=torch.tensor([3, 5], dtype=I32), qo_indptr_host=[0, 2, 5],
                kv_indptr_host=[0, 1, 2], kv_last_page_len_host=[3, 5],
                workspace=torch.zeros(256, dtype=torch.uint8),
                out=torch.zeros(5, 16, 512, dtype=BF16), lse=torch.zeros(5, 16))
    with pytest.raises(TypeError, match="qo_indptr must be"):
        bia.bia_mla_prefill_paged(**{**args, "qo_indptr": torch.tensor([0, 2, 5])})
    with pytest.raises(ValueError, match="lse must hold"):
        bia.bia_mla_prefill_paged(**{**args, "lse": torch.zeros(2, 16)})
    with pytest.raises(ValueError, match="CUDA tensor"):
        bia.bia_mla_prefill_paged(**args)


def test_tensors_must_sit_on_the_launch_device(monkeypatch):
    from types import SimpleNamespace as NS
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    on = lambda i: NS(device=torch.device("cuda", i))  # noqa: E731
    bia._check_cuda([("q", on(0)), ("out", on(0))])  # the current device: fine
    with pytest.raises(ValueError, match="the other arguments on cuda:0"):
        bia._check_cuda([("q", on(0)), ("out", on(1))])
    with pytest.raises(ValueError, match="would run on cuda:0"):
        bia._check_cuda([("q", on(1)), ("out", on(1))])
    # a stream of device 1 takes the work there
    bia._check_cuda([("q", on(1))], stream=NS(device=torch.device("cuda", 1)))
    with pytest.raises(ValueError, match="would run on cuda:1"):
        bia._check_cuda([("q", on(0))], stream=NS(device=torch.device("cuda", 1)))
    # a raw stream handle belongs to the current device
    bia._check_cuda([("q", on(0))], stream=12345)
