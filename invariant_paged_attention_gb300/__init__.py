"""Python binding of libbia.so: batch-invariant paged-KV GQA attention on
GB300 (sm_103a).

Argument marshalling only.  Every step of the computation runs in the CUDA
kernels of libbia.so; PyTorch supplies device memory and streams.  There is
no fallback: if the library is missing or fails to load, every call raises.

The functions carry the C names of ``include/bia.h`` and take torch tensors:
device tensors for the data and the device copies of the index arrays, CPU
int32 tensors for the host mirrors.  Before a call reaches the library, its
device tensors are checked for dtype, contiguity, the shapes the passed sizes
come from and the CUDA device the call enqueues on (TypeError / ValueError);
everything else (descriptor, index arrays, workspace size) is checked by the
library itself, which raises BiaError with its status code.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbia.so")

BIA_OK = 0
BIA_ERR_INVALID_ARG = -1
BIA_ERR_UNSUPPORTED = -2
BIA_ERR_WORKSPACE_TOO_SMALL = -3
BIA_ERR_CUDA = -4
BIA_Q_TILE_ROWS = 128
BIA_PREFILL_SPLIT = 4096
BIA_DECODE_SPLIT = 2048

# every symbol include/bia.h exports
EXPORTS = ("bia_prefill_paged", "bia_prefill_workspace_size", "bia_decode_paged",
           "bia_decode_workspace_size", "bia_merge_states", "bia_q_tile_tokens",
           "bia_status_string", "bia_read_status", "bia_set_profile_events",
           "bia_launch_count", "bia_last_error", "bia_decode_paged_noalloc",
           "bia_append_paged_kv", "bia_prefill_paged_mask", "bia_mla_decode_paged",
           "bia_mla_decode_workspace_size", "bia_mla_prefill_paged",
           "bia_mla_prefill_workspace_size", "bia_prefill_paged_bounded",
           "bia_prefill_bounded_workspace_size", "bia_decode_paged_bounded",
           "bia_decode_bounded_workspace_size")


class BiaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = ""
        if status == BIA_ERR_CUDA:
            detail = ": " + load().bia_last_error().decode()
        super().__init__(f"{where} failed: {status_string(status)} ({status}){detail}")


class AttnDesc(ctypes.Structure):
    _fields_ = [("num_qo_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("sm_scale", ctypes.c_float)]


_lib = None


class MlaDesc(ctypes.Structure):
    _fields_ = [("num_heads", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("sm_scale", ctypes.c_float)]


MLA_CKV_DIM, MLA_KPE_DIM = 512, 64


class Bounds(ctypes.Structure):
    _fields_ = [("max_q_len", ctypes.c_int32), ("max_kv_len", ctypes.c_int32),
                ("max_total_q", ctypes.c_int64)]


def load(path: str = LIB_PATH):
    """Loads libbia.so (built by ``build.build()``); raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libbia.so not built at {path}: run "
                           "`python -m invariant_paged_attention_gb300.build`")
    lib = ctypes.CDLL(path)
    i32, i64, vp, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
    dp = ctypes.POINTER(AttnDesc)
    lib.bia_prefill_paged.argtypes = [dp, vp, vp, vp, i64, vp, vp, vp, vp, vp, vp, vp, i32, i32,
                                      i32, vp, sz, vp, vp, vp]
    lib.bia_prefill_paged.restype = ctypes.c_int
    lib.bia_prefill_workspace_size.argtypes = [dp, vp, vp, vp, i32, i32, i32]
    lib.bia_prefill_workspace_size.restype = sz
    lib.bia_decode_paged.argtypes = [dp, vp, vp, vp, i64, vp, vp, vp, vp, vp, i32, i32, vp, sz,
                                     vp, vp, vp]
    lib.bia_decode_paged.restype = ctypes.c_int
    lib.bia_decode_workspace_size.argtypes = [dp, vp, vp, i32, i32]
    lib.bia_decode_workspace_size.restype = sz
    lib.bia_merge_states.argtypes = [vp, vp, vp, i64, i32, i32, i32, vp, vp, vp]
    lib.bia_merge_states.restype = ctypes.c_int
    lib.bia_q_tile_tokens.argtypes = [i32]
    lib.bia_q_tile_tokens.restype = i32
    lib.bia_status_string.argtypes = [ctypes.c_int]
    lib.bia_status_string.restype = ctypes.c_char_p
    lib.bia_read_status.argtypes = [vp, ctypes.POINTER(i32), vp]
    lib.bia_read_status.restype = ctypes.c_int
    lib.bia_set_profile_events.argtypes = [vp, vp]
    lib.bia_set_profile_events.restype = None
    lib.bia_launch_count.argtypes = []
    lib.bia_launch_count.restype = ctypes.c_uint64
    lib.bia_last_error.argtypes = []
    lib.bia_last_error.restype = ctypes.c_char_p
    lib.bia_decode_paged_noalloc.argtypes = [dp, vp, vp, vp, i64, vp, vp, vp, vp, vp, i32, i32,
                                             vp, vp, vp]
    lib.bia_decode_paged_noalloc.restype = ctypes.c_int
    lib.bia_append_paged_kv.argtypes = [dp, vp, vp, vp, vp, i64, vp, vp, vp, vp, vp, vp, vp, i32,
                                        vp, vp]
    lib.bia_append_paged_kv.restype = ctypes.c_int
    lib.bia_prefill_paged_mask.argtypes = [dp, vp, vp, vp, i64, vp, vp, vp, vp, vp, vp, vp, i32,
                                           i32, i32, vp, sz, vp, vp, vp, sz, vp, vp, vp]
    lib.bia_prefill_paged_mask.restype = ctypes.c_int
    mp = ctypes.POINTER(MlaDesc)
    lib.bia_mla_decode_paged.argtypes = [mp, vp, vp, vp, vp, i64, vp, vp, vp, vp, vp, i32, i32,
                                         vp, sz, vp, vp, vp]
    lib.bia_mla_decode_paged.restype = ctypes.c_int
    lib.bia_mla_decode_workspace_size.argtypes = [mp, vp, vp, i32, i32]
    lib.bia_mla_decode_workspace_size.restype = sz
    lib.bia_mla_prefill_paged.argtypes = [mp, vp, vp, vp, vp, i64, vp, vp, vp, vp, vp, vp, vp,
                                          i32, i32, vp, sz, vp, vp, vp]
    lib.bia_mla_prefill_paged.restype = ctypes.c_int
    lib.bia_mla_prefill_workspace_size.argtypes = [mp, vp, vp, vp, i32, i32]
    lib.bia_mla_prefill_workspace_size.restype = sz
    bp = ctypes.POINTER(Bounds)
    lib.bia_prefill_paged_bounded.argtypes = [dp, bp, vp, vp, vp, i64, vp, vp, vp, vp, i32, i32,
                                              i32, vp, sz, vp, vp, vp]
    lib.bia_prefill_paged_bounded.restype = ctypes.c_int
    lib.bia_prefill_bounded_workspace_size.argtypes = [dp, bp, i32, i32, i32]
    lib.bia_prefill_bounded_workspace_size.restype = sz
    lib.bia_decode_paged_bounded.argtypes = [dp, bp, vp, vp, vp, i64, vp, vp, vp, i32, i32, vp,
                                             sz, vp, vp, vp]
    lib.bia_decode_paged_bounded.restype = ctypes.c_int
    lib.bia_decode_bounded_workspace_size.argtypes = [dp, bp, i32, i32]
    lib.bia_decode_bounded_workspace_size.restype = sz
    _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


BF16, F32, I32, I64, U8 = torch.bfloat16, torch.float32, torch.int32, torch.int64, torch.uint8


# The library sees only the addresses of the device tensors: a host tensor, a
# strided view or a tensor of another dtype would be read as a dense device
# array of the stated type.  So every call checks its tensors first: dtype and
# layout (_check_types), the shapes the sizes it passes are taken from, and
# last that all of them live on one CUDA device (_check_cuda).


def _check_types(*specs):
    """Each spec is (name, tensor, dtype[, optional]): dtype None takes any
    dtype (a byte buffer); an optional argument may be None.  Returns the
    (name, tensor) pairs that were given."""
    given = []
    for spec in specs:
        name, t, dtype = spec[:3]
        if t is None:
            if len(spec) > 3 and spec[3]:
                continue
            raise TypeError(f"{name} is required")
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor, got {type(t).__name__}")
        if dtype is not None and t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        given.append((name, t))
    return given


def _launch_device(stream) -> torch.device:
    """The device the library enqueues on: a torch stream's own device, else
    the current one (a raw cudaStream_t handle is taken to belong to it)."""
    dev = getattr(stream, "device", None)
    if isinstance(dev, torch.device) and dev.type == "cuda":
        return torch.device("cuda", dev.index if dev.index is not None else
                            torch.cuda.current_device())
    return torch.device("cuda", torch.cuda.current_device())


def _check_cuda(given, stream=None):
    device = None
    for name, t in given:
        if t.device.type != "cuda":
            raise ValueError(f"{name} must be a CUDA tensor, got one on {t.device}")
        if device is None:
            device = t.device
        elif t.device != device:
            raise ValueError(f"{name} is on {t.device}, the other arguments on {device}")
    if device is not None:
        want = _launch_device(stream)
        have = torch.device("cuda", device.index if device.index is not None else want.index)
        if have != want:
            raise ValueError(f"the tensors are on {have} but the work would run on {want}")


def _check_rows(q, out, lse, qname="q"):
    """out has q's shape; lse, when given, one float per (token, head) of q."""
    if tuple(out.shape) != tuple(q.shape):
        raise ValueError(f"out has shape {tuple(out.shape)}, {qname} {tuple(q.shape)}")
    if lse is not None and (q.dim() < 2 or lse.numel() != q.shape[0] * q.shape[1]):
        raise ValueError(f"lse must hold {qname}.shape[0] x {qname}.shape[1] floats")


def _check_caches(k_cache, v_cache):
    if tuple(v_cache.shape) != tuple(k_cache.shape) or k_cache.dim() != 4:
        raise ValueError(f"k_cache and v_cache must both be [num_pages, page_size, "
                         f"num_kv_heads, head_dim], got {tuple(k_cache.shape)} and "
                         f"{tuple(v_cache.shape)}")


def _host_i32(t) -> torch.Tensor:
    t = torch.as_tensor(t, dtype=torch.int32)
    if t.device.type != "cpu":
        raise ValueError("host mirrors must be CPU tensors")
    return t.contiguous()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def make_desc(num_qo_heads, num_kv_heads, head_dim, page_size, sm_scale=0.0) -> AttnDesc:
    return AttnDesc(num_qo_heads, num_kv_heads, head_dim, page_size, float(sm_scale))


def status_string(status: int) -> str:
    return load().bia_status_string(int(status)).decode()


def bia_q_tile_tokens(gqa_group: int) -> int:
    return int(load().bia_q_tile_tokens(int(gqa_group)))


def bia_prefill_workspace_size(desc, qo_indptr_host, kv_indptr_host, kv_last_page_len_host,
                               causal=True, split_size=0) -> int:
    qo, kvp, last = (_host_i32(qo_indptr_host), _host_i32(kv_indptr_host),
                     _host_i32(kv_last_page_len_host))
    return int(load().bia_prefill_workspace_size(ctypes.byref(desc), _ptr(qo), _ptr(kvp),
                                                 _ptr(last), len(qo) - 1, int(bool(causal)),
                                                 int(split_size)))


def bia_decode_workspace_size(desc, kv_indptr_host, kv_last_page_len_host, split_size=0) -> int:
    kvp, last = _host_i32(kv_indptr_host), _host_i32(kv_last_page_len_host)
    return int(load().bia_decode_workspace_size(ctypes.byref(desc), _ptr(kvp), _ptr(last),
                                                len(kvp) - 1, int(split_size)))


def bia_prefill_paged(desc, q, k_cache, v_cache, qo_indptr, kv_indptr, kv_indices,
                      kv_last_page_len, qo_indptr_host, kv_indptr_host, kv_last_page_len_host,
                      workspace, out, lse=None, causal=True, split_size=0, stream=None):
    ts = _check_types(("q", q, BF16), ("k_cache", k_cache, BF16), ("v_cache", v_cache, BF16),
                      ("qo_indptr", qo_indptr, I32), ("kv_indptr", kv_indptr, I32),
                      ("kv_indices", kv_indices, I32), ("kv_last_page_len", kv_last_page_len, I32),
                      ("workspace", workspace, None), ("out", out, BF16), ("lse", lse, F32, True))
    _check_caches(k_cache, v_cache)
    _check_rows(q, out, lse)
    _check_cuda(ts, stream)
    qo, kvp, last = (_host_i32(qo_indptr_host), _host_i32(kv_indptr_host),
                     _host_i32(kv_last_page_len_host))
    rc = load().bia_prefill_paged(
        ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
        _ptr(qo_indptr), _ptr(kv_indptr), _ptr(kv_indices), _ptr(kv_last_page_len), _ptr(qo),
        _ptr(kvp), _ptr(last), len(qo) - 1, int(bool(causal)), int(split_size), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse), _stream(stream))
    if rc != BIA_OK:
        raise BiaError(rc, "bia_prefill_paged")


def bia_prefill_paged_mask(desc, q, k_cache, v_cache, qo_indptr, kv_indptr, kv_indices,
                           kv_last_page_len, qo_indptr_host, kv_indptr_host,
                           kv_last_page_len_host, mask, mask_indptr, mask_indptr_host,
                           workspace, out, lse=None, causal=True, split_size=0, stream=None):
    """bia_prefill_paged with a custom mask: ``mask`` a device uint8 tensor of
    little-endian bits, ``mask_indptr`` its device int64 [batch+1] bit
    offsets (include/bia.h states the rule)."""
    ts = _check_types(("q", q, BF16), ("k_cache", k_cache, BF16), ("v_cache", v_cache, BF16),
                      ("qo_indptr", qo_indptr, I32), ("kv_indptr", kv_indptr, I32),
                      ("kv_indices", kv_indices, I32), ("kv_last_page_len", kv_last_page_len, I32),
                      ("mask", mask, U8), ("mask_indptr", mask_indptr, I64),
                      ("workspace", workspace, None), ("out", out, BF16), ("lse", lse, F32, True))
    _check_caches(k_cache, v_cache)
    _check_rows(q, out, lse)
    _check_cuda(ts, stream)
    qo, kvp, last = (_host_i32(qo_indptr_host), _host_i32(kv_indptr_host),
                     _host_i32(kv_last_page_len_host))
    mih = torch.as_tensor(mask_indptr_host, dtype=torch.int64).contiguous()
    if mih.device.type != "cpu":
        raise ValueError("host mirrors must be CPU tensors")
    rc = load().bia_prefill_paged_mask(
        ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
        _ptr(qo_indptr), _ptr(kv_indptr), _ptr(kv_indices), _ptr(kv_last_page_len), _ptr(qo),
        _ptr(kvp), _ptr(last), len(qo) - 1, int(bool(causal)), int(split_size), _ptr(mask),
        mask.numel() * mask.element_size(), _ptr(mask_indptr), _ptr(mih), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse), _stream(stream))
    if rc != BIA_OK:
        raise BiaError(rc, "bia_prefill_paged_mask")


def bia_decode_paged(desc, q, k_cache, v_cache, kv_indptr, kv_indices, kv_last_page_len,
                     kv_indptr_host, kv_last_page_len_host, workspace, out, lse=None,
                     split_size=0, stream=None):
    ts = _check_types(("q", q, BF16), ("k_cache", k_cache, BF16), ("v_cache", v_cache, BF16),
                      ("kv_indptr", kv_indptr, I32), ("kv_indices", kv_indices, I32),
                      ("kv_last_page_len", kv_last_page_len, I32), ("workspace", workspace, None),
                      ("out", out, BF16), ("lse", lse, F32, True))
    _check_caches(k_cache, v_cache)
    _check_rows(q, out, lse)
    _check_cuda(ts, stream)
    kvp, last = _host_i32(kv_indptr_host), _host_i32(kv_last_page_len_host)
    rc = load().bia_decode_paged(
        ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
        _ptr(kv_indptr), _ptr(kv_indices), _ptr(kv_last_page_len), _ptr(kvp), _ptr(last),
        len(kvp) - 1, int(split_size), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse), _stream(stream))
    if rc != BIA_OK:
        raise BiaError(rc, "bia_decode_paged")


def make_bounds(max_q_len=1, max_kv_len=1, max_total_q=0) -> Bounds:
    return Bounds(int(max_q_len), int(max_kv_len), int(max_total_q))


def bia_prefill_bounded_workspace_size(desc, bounds, batch, causal=True, split_size=0) -> int:
    return int(load().bia_prefill_bounded_workspace_size(ctypes.byref(desc), ctypes.byref(bounds),
                                                         int(batch), int(bool(causal)),
                                                         int(split_size)))


def bia_decode_bounded_workspace_size(desc, bounds, batch, split_size=0) -> int:
    return int(load().bia_decode_bounded_workspace_size(ctypes.byref(desc), ctypes.byref(bounds),
                                                        int(batch), int(split_size)))


def bia_prefill_paged_bounded(desc, bounds, q, k_cache, v_cache, qo_indptr, kv_indptr,
                              kv_indices, kv_last_page_len, workspace, out, lse=None,
                              causal=True, split_size=0, stream=None):
    """bia_prefill_paged sized from `bounds` (a Bounds): the index arrays are
    read on the device only, so a captured call replays while they change.
    q / out / lse hold bounds.max_total_q token rows."""
    ts = _check_types(("q", q, BF16), ("k_cache", k_cache, BF16), ("v_cache", v_cache, BF16),
                      ("qo_indptr", qo_indptr, I32), ("kv_indptr", kv_indptr, I32),
                      ("kv_indices", kv_indices, I32), ("kv_last_page_len", kv_last_page_len, I32),
                      ("workspace", workspace, None), ("out", out, BF16), ("lse", lse, F32, True))
    _check_caches(k_cache, v_cache)
    _check_rows(q, out, lse)
    if q.shape[0] < bounds.max_total_q:
        raise ValueError(f"q holds {q.shape[0]} token rows, bounds.max_total_q is "
                         f"{bounds.max_total_q}")
    _check_cuda(ts, stream)
    rc = load().bia_prefill_paged_bounded(
        ctypes.byref(desc), ctypes.byref(bounds), _ptr(q), _ptr(k_cache), _ptr(v_cache),
        k_cache.shape[0], _ptr(qo_indptr), _ptr(kv_indptr), _ptr(kv_indices),
        _ptr(kv_last_page_len), qo_indptr.numel() - 1, int(bool(causal)), int(split_size),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse),
        _stream(stream))
    if rc != BIA_OK:
        raise BiaError(rc, "bia_prefill_paged_bounded")


def bia_decode_paged_bounded(desc, bounds, q, k_cache, v_cache, kv_indptr, kv_indices,
                             kv_last_page_len, workspace, out, lse=None, split_size=0,
                             stream=None):
    """bia_decode_paged sized from `bounds` (max_kv_len): the index arrays are
    read on the device only, so a captured decode replays step after step."""
    ts = _check_types(("q", q, BF16), ("k_cache", k_cache, BF16), ("v_cache", v_cache, BF16),
                      ("kv_indptr", kv_indptr, I32), ("kv_indices", kv_indices, I32),
                      ("kv_last_page_len", kv_last_page_len, I32), ("workspace", workspace, None),
                      ("out", out, BF16), ("lse", lse, F32, True))
    _check_caches(k_cache, v_cache)
    _check_rows(q, out, lse)
    if q.shape[0] != kv_indptr.numel() - 1:
        raise ValueError(f"q holds {q.shape[0]} rows for {kv_indptr.numel() - 1} requests")
    _check_cuda(ts, stream)
    rc = load().bia_decode_paged_bounded(
        ctypes.byref(desc), ctypes.byref(bounds), _ptr(q), _ptr(k_cache), _ptr(v_cache),
        k_cache.shape[0], _ptr(kv_indptr), _ptr(kv_indices), _ptr(kv_last_page_len),
        kv_indptr.numel() - 1, int(split_size), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse), _stream(stream))
    if rc != BIA_OK:
        raise BiaError(rc, "bia_decode_paged_bounded")


BIA_DECODE_NOALLOC_SCRATCH_BYTES = 64 << 20


def bia_decode_paged_noalloc(desc, q, k_cache, v_cache, kv_indptr, kv_indices, kv_last_page_len,
                             kv_indptr_host, kv_last_page_len_host, out, lse=None, split_size=0,
                             stream=None):
    """bia_decode_paged for callers that cannot allocate device memory: no
    workspace argument; the library's static scratch array is used instead
    (see include/bia.h for its size, first-call and concurrency rules)."""
    ts = _check_types(("q", q, BF16), ("k_cache", k_cache, BF16), ("v_cache", v_cache, BF16),
                      ("kv_indptr", kv_indptr, I32), ("kv_indices", kv_indices, I32),
                      ("kv_last_page_len", kv_last_page_len, I32), ("out", out, BF16),
                      ("lse", lse, F32, True))
    _check_caches(k_cache, v_cache)
    _check_rows(q, out, lse)
    _check_cuda(ts, stream)
    kvp, last = _host_i32(kv_indptr_host), _host_i32(kv_last_page_len_host)
    rc = load().bia_decode_paged_noalloc(
        ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
        _ptr(kv_indptr), _ptr(kv_indices), _ptr(kv_last_page_len), _ptr(kvp), _ptr(last),
        len(kvp) - 1, int(split_size), _ptr(out), _ptr(lse), _stream(stream))
    if rc != BIA_OK:
        raise BiaError(rc, "bia_decode_paged_noalloc")


def bia_append_paged_kv(desc, k_new, v_new, k_cache, v_cache, append_indptr, kv_indptr,
                        kv_indices, kv_last_page_len, append_indptr_host, kv_indptr_host,
                        kv_last_page_len_host, status=None, stream=None):
    """Write the new tokens' K/V rows [total_new, Hkv, D] into the last
    n_new positions of each request's pages (include/bia.h states the rule);
    `status` is an optional 1-element device int32 tensor."""
    ts = _check_types(("k_new", k_new, BF16), ("v_new", v_new, BF16), ("k_cache", k_cache, BF16),
                      ("v_cache", v_cache, BF16), ("append_indptr", append_indptr, I32),
                      ("kv_indptr", kv_indptr, I32), ("kv_indices", kv_indices, I32),
                      ("kv_last_page_len", kv_last_page_len, I32), ("status", status, I32, True))
    _check_caches(k_cache, v_cache)
    if tuple(v_new.shape) != tuple(k_new.shape):
        raise ValueError(f"v_new has shape {tuple(v_new.shape)}, k_new {tuple(k_new.shape)}")
    _check_cuda(ts, stream)
    ap, kvp, last = (_host_i32(append_indptr_host), _host_i32(kv_indptr_host),
                     _host_i32(kv_last_page_len_host))
    rc = load().bia_append_paged_kv(
        ctypes.byref(desc), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
        k_cache.shape[0], _ptr(append_indptr), _ptr(kv_indptr), _ptr(kv_indices),
        _ptr(kv_last_page_len), _ptr(ap), _ptr(kvp), _ptr(last), len(ap) - 1, _ptr(status),
        _stream(stream))
    if rc != BIA_OK:
        raise BiaError(rc, "bia_append_paged_kv")


def bia_merge_states(v, s, out, out_lse=None, num_states=None, stream=None):
    """v [n, S, H, D] fp32, s [n, S, H] fp32 -> out [n, H, D] bf16, out_lse [n, H]."""
    ts = _check_types(("v", v, F32), ("s", s, F32), ("out", out, BF16),
                      ("out_lse", out_lse, F32, True), ("num_states", num_states, I32, True))
    if v.dim() != 4:
        raise ValueError(f"v must be [n, S, H, D], got shape {tuple(v.shape)}")
    n, S, H, D = v.shape
    if tuple(s.shape) != (n, S, H) or tuple(out.shape) != (n, H, D):
        raise ValueError(f"s must be {(n, S, H)} and out {(n, H, D)}, got "
                         f"{tuple(s.shape)} and {tuple(out.shape)}")
    if out_lse is not None and tuple(out_lse.shape) != (n, H):
        raise ValueError(f"out_lse must be {(n, H)}, got {tuple(out_lse.shape)}")
    if num_states is not None and num_states.numel() != n:
        raise ValueError(f"num_states must hold {n} counts, got {num_states.numel()}")
    _check_cuda(ts, stream)
    rc = load().bia_merge_states(_ptr(v), _ptr(s), _ptr(num_states), n, S, H, D, _ptr(out),
                                 _ptr(out_lse), _stream(stream))
    if rc != BIA_OK:
        raise BiaError(rc, "bia_merge_states")


def bia_read_status(workspace, stream=None) -> int:
    ts = _check_types(("workspace", workspace, None))
    _check_cuda(ts, stream)
    st = ctypes.c_int32(0)
    rc = load().bia_read_status(_ptr(workspace), ctypes.byref(st), _stream(stream))
    if rc != BIA_OK:
        raise BiaError(rc, "bia_read_status")
    return int(st.value)


def bia_set_profile_events(begin=None, end=None):
    """Record torch.cuda.Event `begin` / `end` (created with enable_timing)
    around the attention kernel of every later prefill / decode call
    (None, None: off)."""
    def handle(e):
        if e is None:
            return None
        if not e.cuda_event:  # torch creates the CUDA event on first record
            e.record()
        return ctypes.c_void_p(e.cuda_event)
    load().bia_set_profile_events(handle(begin), handle(end))


def bia_launch_count() -> int:
    return int(load().bia_launch_count())


def make_mla_desc(num_heads, page_size, sm_scale=0.0) -> MlaDesc:
    return MlaDesc(num_heads, page_size, float(sm_scale))


def bia_mla_decode_workspace_size(desc, kv_indptr_host, kv_last_page_len_host,
                                  split_size=0) -> int:
    kvp, last = _host_i32(kv_indptr_host), _host_i32(kv_last_page_len_host)
    return int(load().bia_mla_decode_workspace_size(ctypes.byref(desc), _ptr(kvp), _ptr(last),
                                                    len(kvp) - 1, int(split_size)))


def bia_mla_decode_paged(desc, q_nope, q_pe, ckv_cache, kpe_cache, kv_indptr, kv_indices,
                         kv_last_page_len, kv_indptr_host, kv_last_page_len_host, workspace,
                         out, lse=None, split_size=0, stream=None):
    """Multi-head latent attention decode (include/bia.h states the layouts)."""
    ts = _check_types(("q_nope", q_nope, BF16), ("q_pe", q_pe, BF16), ("ckv_cache", ckv_cache, BF16),
                      ("kpe_cache", kpe_cache, BF16), ("kv_indptr", kv_indptr, I32),
                      ("kv_indices", kv_indices, I32), ("kv_last_page_len", kv_last_page_len, I32),
                      ("workspace", workspace, None), ("out", out, BF16), ("lse", lse, F32, True))
    if kpe_cache.dim() < 1 or ckv_cache.dim() < 1 or kpe_cache.shape[0] != ckv_cache.shape[0]:
        raise ValueError("ckv_cache and kpe_cache must have the same number of pages")
    _check_rows(q_nope, out, lse, "q_nope")
    _check_cuda(ts, stream)
    kvp, last = _host_i32(kv_indptr_host), _host_i32(kv_last_page_len_host)
    rc = load().bia_mla_decode_paged(
        ctypes.byref(desc), _ptr(q_nope), _ptr(q_pe), _ptr(ckv_cache), _ptr(kpe_cache),
        ckv_cache.shape[0], _ptr(kv_indptr), _ptr(kv_indices), _ptr(kv_last_page_len),
        _ptr(kvp), _ptr(last), len(kvp) - 1, int(split_size), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse), _stream(stream))
    if rc != BIA_OK:
        raise BiaError(rc, "bia_mla_decode_paged")


def bia_mla_prefill_workspace_size(desc, qo_indptr_host, kv_indptr_host, kv_last_page_len_host,
                                   split_size=0) -> int:
    qo, kvp, last = (_host_i32(qo_indptr_host), _host_i32(kv_indptr_host),
                     _host_i32(kv_last_page_len_host))
    return int(load().bia_mla_prefill_workspace_size(ctypes.byref(desc), _ptr(qo), _ptr(kvp),
                                                     _ptr(last), len(qo) - 1, int(split_size)))


def bia_mla_prefill_paged(desc, q_nope, q_pe, ckv_cache, kpe_cache, qo_indptr, kv_indptr,
                          kv_indices, kv_last_page_len, qo_indptr_host, kv_indptr_host,
                          kv_last_page_len_host, workspace, out, lse=None, split_size=0,
                          stream=None):
    """Causal multi-head latent attention extend: q_nope / q_pe / out hold
    total_q token rows (include/bia.h states the layouts and the rule)."""
    ts = _check_types(("q_nope", q_nope, BF16), ("q_pe", q_pe, BF16),
                      ("ckv_cache", ckv_cache, BF16), ("kpe_cache", kpe_cache, BF16),
                      ("qo_indptr", qo_indptr, I32), ("kv_indptr", kv_indptr, I32),
                      ("kv_indices", kv_indices, I32), ("kv_last_page_len", kv_last_page_len, I32),
                      ("workspace", workspace, None), ("out", out, BF16), ("lse", lse, F32, True))
    if kpe_cache.dim() < 1 or ckv_cache.dim() < 1 or kpe_cache.shape[0] != ckv_cache.shape[0]:
        raise ValueError("ckv_cache and kpe_cache must have the same number of pages")
    _check_rows(q_nope, out, lse, "q_nope")
    _check_cuda(ts, stream)
    qo, kvp, last = (_host_i32(qo_indptr_host), _host_i32(kv_indptr_host),
                     _host_i32(kv_last_page_len_host))
    rc = load().bia_mla_prefill_paged(
        ctypes.byref(desc), _ptr(q_nope), _ptr(q_pe), _ptr(ckv_cache), _ptr(kpe_cache),
        ckv_cache.shape[0], _ptr(qo_indptr), _ptr(kv_indptr), _ptr(kv_indices),
        _ptr(kv_last_page_len), _ptr(qo), _ptr(kvp), _ptr(last), len(qo) - 1, int(split_size),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse),
        _stream(stream))
    if rc != BIA_OK:
        raise BiaError(rc, "bia_mla_prefill_paged")
