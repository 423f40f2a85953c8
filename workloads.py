"""Seeded synthetic inputs for paged-KV attention: the one module that both the
CPU oracle's tests and the GPU path use.

It holds no attention arithmetic: it draws bf16 tensors, lays key/value rows
out in a paged cache under a seeded random page permutation, and writes the
CSR arrays (qo_indptr, kv_indptr, kv_indices, kv_last_page_len) that describe
a call.  Every sequence draws its own values from its own seeds, so a request
has the same bits whether it runs alone or inside any batch, and whatever
physical pages it lands on.

Terms: a *sequence* has ``prefix`` cached tokens followed by ``new`` tokens;
its key/value rows cover prefix+new positions and its queries cover the new
tokens.  A *call* is a list of parts (sequence, q_start, q_end): the part's
queries are new tokens q_start..q_end-1 and it sees the first
prefix+q_end keys.  Decode is a call whose parts each carry one query.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

BF16 = torch.bfloat16


@dataclass(frozen=True)
class Sequence:
    seed: int
    prefix: int
    new: int

    @property
    def length(self) -> int:
        return self.prefix + self.new


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def draw_normal_bf16(shape, seed: int, device) -> torch.Tensor:
    """i.i.d. N(0, 1) values rounded to bf16 (round-to-nearest-even)."""
    t = torch.randn(shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    return t.to(BF16)


def uniform_lengths(n: int, lo: int, hi: int, seed: int) -> list[int]:
    """n integers uniform in [lo, hi]; value i comes from its own seed
    (seed + i), so the first values do not depend on n."""
    out = []
    for i in range(n):
        g = _gen(seed + i, "cpu")
        out.append(int(torch.randint(lo, hi + 1, (1,), generator=g).item()))
    return out


@dataclass
class PagedStore:
    """Key/value rows of a set of sequences in one paged cache pair.

    k_cache / v_cache: [num_pages, page_size, num_kv_heads, head_dim] bf16.
    pages[i]: physical page ids of sequence i in order.  Slots past the end of
    a sequence's last page are filled with NaN so that any read of them shows.
    """
    seqs: list
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    device: str
    layout_seed: int = 7
    spare_pages: int = 0
    k_cache: torch.Tensor = field(init=False)
    v_cache: torch.Tensor = field(init=False)
    q: list = field(init=False)
    pages: list = field(init=False)

    def __post_init__(self):
        P, Hkv, D, Hq = self.page_size, self.num_kv_heads, self.head_dim, self.num_qo_heads
        counts = [-(-s.length // P) for s in self.seqs]
        num_pages = sum(counts) + self.spare_pages
        perm = torch.randperm(max(num_pages, 1), generator=_gen(self.layout_seed, "cpu"))
        self.k_cache = torch.full((max(num_pages, 1), P, Hkv, D), float("nan"), dtype=BF16,
                                  device=self.device)
        self.v_cache = torch.full_like(self.k_cache, float("nan"))
        self.q, self.pages = [], []
        start = 0
        for s, c in zip(self.seqs, counts):
            ids = perm[start:start + c].to(torch.int32)
            start += c
            self.pages.append(ids)
            base = 4 * int(s.seed)
            self.q.append(draw_normal_bf16((s.new, Hq, D), base + 1, self.device))
            if c == 0:
                continue
            for cache, sub in ((self.k_cache, 2), (self.v_cache, 3)):
                rows = draw_normal_bf16((s.length, Hkv, D), base + sub, self.device)
                padded = torch.full((c * P, Hkv, D), float("nan"), dtype=BF16, device=self.device)
                padded[: s.length] = rows
                cache[ids.to(self.device).long()] = padded.view(c, P, Hkv, D)

    @property
    def num_pages(self) -> int:
        return self.k_cache.shape[0]


@dataclass
class Call:
    """One prefill/extend or decode call: what the library entry points take."""
    store: PagedStore
    parts: list  # (sequence index, q_start, q_end)
    q: torch.Tensor
    qo_indptr: torch.Tensor  # int32, CPU
    kv_indptr: torch.Tensor  # int32, CPU
    kv_indices: torch.Tensor  # int32, CPU
    kv_last_page_len: torch.Tensor  # int32, CPU
    q_lens: list
    kv_lens: list

    @property
    def batch(self) -> int:
        return len(self.parts)

    @property
    def total_q(self) -> int:
        return int(self.qo_indptr[-1])


def make_call(store: PagedStore, parts) -> Call:
    """Assemble the CSR description of a call over ``store``."""
    P = store.page_size
    qs, q_lens, kv_lens, idx, last = [], [], [], [], []
    qo, kvp = [0], [0]
    for (si, a, b) in parts:
        s = store.seqs[si]
        if not (0 <= a <= b <= s.new):
            raise ValueError(f"part {(si, a, b)} outside sequence of {s.new} new tokens")
        kv_len = s.prefix + b
        n_pages = -(-kv_len // P)
        qs.append(store.q[si][a:b])
        q_lens.append(b - a)
        kv_lens.append(kv_len)
        idx.append(store.pages[si][:n_pages])
        last.append(kv_len - (n_pages - 1) * P if n_pages > 0 else 0)
        qo.append(qo[-1] + (b - a))
        kvp.append(kvp[-1] + n_pages)
    Hq, D = store.num_qo_heads, store.head_dim
    q = torch.cat(qs, 0) if qs else torch.zeros((0, Hq, D), dtype=BF16, device=store.device)
    kv_indices = torch.cat(idx) if idx else torch.zeros(0, dtype=torch.int32)
    return Call(store, list(parts), q.contiguous(), torch.tensor(qo, dtype=torch.int32),
                torch.tensor(kvp, dtype=torch.int32), kv_indices.to(torch.int32).cpu(),
                torch.tensor(last, dtype=torch.int32), q_lens, kv_lens)


def whole_prefill(store: PagedStore) -> Call:
    """Every sequence extended by all its new tokens in one call."""
    return make_call(store, [(i, 0, s.new) for i, s in enumerate(store.seqs)])


def chunked_calls(store: PagedStore, chunk: int) -> list:
    """Step c extends every sequence by its new tokens [c*chunk, (c+1)*chunk)."""
    steps = max((-(-s.new // chunk)) for s in store.seqs)
    calls = []
    for c in range(steps):
        parts = []
        for i, s in enumerate(store.seqs):
            a = c * chunk
            if a < s.new:
                parts.append((i, a, min(s.new, a + chunk)))
        calls.append(make_call(store, parts))
    return calls


def new_kv_rows(call: Call):
    """K/V rows [total_q, Hkv, D] of a call's new tokens, in call order: the
    same seeded rows the store holds at those positions (for append)."""
    st = call.store
    ks, vs = [], []
    for (si, a, b) in call.parts:
        s = st.seqs[si]
        base = 4 * int(s.seed)
        for rows, sub in ((ks, 2), (vs, 3)):
            full = draw_normal_bf16((s.length, st.num_kv_heads, st.head_dim), base + sub,
                                    st.device)
            rows.append(full[s.prefix + a:s.prefix + b])
    empty = torch.zeros((0, st.num_kv_heads, st.head_dim), dtype=BF16, device=st.device)
    k = torch.cat(ks, 0) if ks else empty
    v = torch.cat(vs, 0) if vs else empty
    return k.contiguous(), v.contiguous()


def clear_slots(call: Call, k_cache: torch.Tensor, v_cache: torch.Tensor, value=float("nan")):
    """Overwrite the cache slots of a call's new tokens with `value`."""
    P = call.store.page_size
    for (si, a, b), pages in zip(call.parts, _part_pages(call)):
        s = call.store.seqs[si]
        for p in range(s.prefix + a, s.prefix + b):
            page = int(pages[p // P])
            k_cache[page, p % P] = value
            v_cache[page, p % P] = value


def _part_pages(call: Call):
    kvp = call.kv_indptr.tolist()
    return [call.kv_indices[kvp[i]:kvp[i + 1]] for i in range(call.batch)]


@dataclass
class MLAStore:
    """Latent rows of a set of sequences in one paged latent cache (multi-head
    latent attention): ckv_cache [num_pages, page_size, dc] and kpe_cache
    [num_pages, page_size, dp] bf16, q_nope [new, H, dc] / q_pe [new, H, dp]
    per sequence.  Slots past a sequence's end hold NaN."""
    seqs: list
    num_heads: int
    dc: int
    dp: int
    page_size: int
    device: str
    layout_seed: int = 7
    ckv_cache: torch.Tensor = field(init=False)
    kpe_cache: torch.Tensor = field(init=False)
    q_nope: list = field(init=False)
    q_pe: list = field(init=False)
    pages: list = field(init=False)

    def __post_init__(self):
        P = self.page_size
        counts = [-(-s.length // P) for s in self.seqs]
        num_pages = max(sum(counts), 1)
        perm = torch.randperm(num_pages, generator=_gen(self.layout_seed, "cpu"))
        self.ckv_cache = torch.full((num_pages, P, self.dc), float("nan"), dtype=BF16,
                                    device=self.device)
        self.kpe_cache = torch.full((num_pages, P, self.dp), float("nan"), dtype=BF16,
                                    device=self.device)
        self.q_nope, self.q_pe, self.pages = [], [], []
        start = 0
        for s, c in zip(self.seqs, counts):
            ids = perm[start:start + c].to(torch.int32)
            start += c
            self.pages.append(ids)
            base = 4 * int(s.seed)
            self.q_nope.append(draw_normal_bf16((s.new, self.num_heads, self.dc), base + 1,
                                                self.device))
            self.q_pe.append(draw_normal_bf16((s.new, self.num_heads, self.dp), base + 2,
                                              self.device))
            if c == 0:
                continue
            for cache, sub, width in ((self.ckv_cache, 3, self.dc), (self.kpe_cache, 0, self.dp)):
                rows = draw_normal_bf16((s.length, width), base + sub, self.device)
                padded = torch.full((c * P, width), float("nan"), dtype=BF16, device=self.device)
                padded[: s.length] = rows
                cache[ids.to(self.device).long()] = padded.view(c, P, width)


@dataclass
class MLACall:
    store: MLAStore
    q_nope: torch.Tensor
    q_pe: torch.Tensor
    qo_indptr: torch.Tensor  # int32, CPU
    kv_indptr: torch.Tensor
    kv_indices: torch.Tensor
    kv_last_page_len: torch.Tensor
    q_lens: list
    kv_lens: list


def mla_call(store: MLAStore, parts) -> MLACall:
    """CSR description of an MLA call; parts are (sequence, q_start, q_end)."""
    P = store.page_size
    qn, qp, q_lens, kv_lens, idx, last, qo, kvp = [], [], [], [], [], [], [0], [0]
    for (si, a, b) in parts:
        s = store.seqs[si]
        kv_len = s.prefix + b
        n_pages = -(-kv_len // P)
        qn.append(store.q_nope[si][a:b])
        qp.append(store.q_pe[si][a:b])
        q_lens.append(b - a)
        kv_lens.append(kv_len)
        idx.append(store.pages[si][:n_pages])
        last.append(kv_len - (n_pages - 1) * P if n_pages > 0 else 0)
        qo.append(qo[-1] + (b - a))
        kvp.append(kvp[-1] + n_pages)
    return MLACall(store, torch.cat(qn, 0).contiguous(), torch.cat(qp, 0).contiguous(),
                   torch.tensor(qo, dtype=torch.int32), torch.tensor(kvp, dtype=torch.int32),
                   torch.cat(idx).to(torch.int32).cpu(), torch.tensor(last, dtype=torch.int32),
                   q_lens, kv_lens)


def custom_mask(call: Call, seed: int, density: float = 0.7, causal_part: bool = False):
    """A seeded custom mask for a call: per request a [q_len, kv_len] boolean
    matrix (True = the token may see the key), i.i.d. Bernoulli(density), and
    optionally AND-ed with the bottom-right causal pattern.  Returns
    (bits uint8 [little-endian bit order], indptr int64 [batch+1] bit offsets,
    list of the dense matrices)."""
    import numpy as np
    rng = np.random.default_rng(seed)
    dense, flat, offs = [], [], [0]
    for ql, kl in zip(call.q_lens, call.kv_lens):
        m = rng.random((ql, kl)) < density
        if causal_part:
            pos = kl - ql + np.arange(ql)
            m &= np.arange(kl)[None, :] <= pos[:, None]
        dense.append(m)
        flat.append(m.reshape(-1))
        offs.append(offs[-1] + ql * kl)
    bits = np.concatenate(flat) if flat else np.zeros(0, bool)
    packed = np.packbits(bits, bitorder="little")
    # four spare bytes so that 32-bit reads of the last word stay in bounds
    packed = np.concatenate([packed, np.zeros(4, np.uint8)])
    return packed, np.asarray(offs, np.int64), dense


def bf16_bits(t: torch.Tensor):
    """Raw bf16 bit patterns of a tensor as a CPU numpy uint16 array."""
    import numpy as np
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------
# The five workloads (Qwen3-8B shapes: 32 q heads, 8 kv heads, head_dim 128).

QWEN = dict(num_qo_heads=32, num_kv_heads=8, head_dim=128)


def cfg1_tiny(device) -> PagedStore:
    """1 request, q_len = kv_len = 256, 4 q / 1 kv head, head_dim 64, page 16."""
    return PagedStore([Sequence(1000, 0, 256)], 4, 1, 64, 16, device, layout_seed=1999)


def cfg2_prefill(device, batch: int = 8, first: int = 0) -> PagedStore:
    """Batched prefill: lengths uniform in [512, 8192], page 1.  ``first``
    selects requests first..first+batch-1 of the same seeded population."""
    lens = uniform_lengths(first + batch, 512, 8192, 2000)[first:]
    seqs = [Sequence(2000 + first + i, 0, L) for i, L in enumerate(lens)]
    return PagedStore(seqs, page_size=1, device=device, layout_seed=2999 + first, **QWEN)


def cfg3_prefix(device, new: int = 16384, prefixes=(1, 511, 2048, 4097)) -> PagedStore:
    """Chunked prefill with cached prefixes 1/511/2048/4097 + 16384 new tokens."""
    seqs = [Sequence(3000 + i, p, new) for i, p in enumerate(prefixes)]
    return PagedStore(seqs, page_size=1, device=device, layout_seed=3999, **QWEN)


def cfg4_decode(device, batch: int, lo: int = 1024, hi: int = 32768) -> PagedStore:
    """Decode: contexts uniform in [1024, 32768]; the last context token is the
    query, so each sequence has ctx-1 cached tokens and 1 new token."""
    lens = uniform_lengths(batch, lo, hi, 4000)
    seqs = [Sequence(4000 + i, L - 1, 1) for i, L in enumerate(lens)]
    return PagedStore(seqs, page_size=1, device=device, layout_seed=4999 + batch, **QWEN)


def wide_prefill(device, batch: int = 8, page_size: int = 1) -> PagedStore:
    """cfg2's lengths (uniform in [512, 8192], same seed) with head_dim 256:
    16 q heads / 8 kv heads (a Gemma-style layout), page 1 by default."""
    lens = uniform_lengths(batch, 512, 8192, 2000)
    seqs = [Sequence(7000 + i, 0, L) for i, L in enumerate(lens)]
    return PagedStore(seqs, 16, 8, 256, page_size, device, layout_seed=7999)


def wide_decode(device, B: int = 64) -> PagedStore:
    """cfg4-style decode (contexts uniform in [1024, 32768]) at head_dim 256,
    16 q heads / 8 kv heads, page 1."""
    ctx = uniform_lengths(B, 1024, 32768, 4000)
    seqs = [Sequence(7500 + i, c - 1, 1) for i, c in enumerate(ctx)]
    return PagedStore(seqs, 16, 8, 256, 1, device, layout_seed=7998)


def cfg5_mixed(device, n_extend: int = 64, n_decode: int = 32, decode_ctx: int = 131072,
               chunk: int = 4096, chunk_prefix: int = 4096):
    """Mixed serving batch, page 16: one prefill chunk (prefix 4096 + 4096 new),
    one-token extends (contexts uniform in [1024, 32768]) and decodes at
    131072 context.  Returns (prefill store, decode store)."""
    ext = uniform_lengths(n_extend, 1024, 32768, 5100)
    pre = [Sequence(5000, chunk_prefix, chunk)] + [
        Sequence(5100 + i, L - 1, 1) for i, L in enumerate(ext)]
    dec = [Sequence(5500 + i, decode_ctx - 1, 1) for i in range(n_decode)]
    return (PagedStore(pre, page_size=16, device=device, layout_seed=5999, **QWEN),
            PagedStore(dec, page_size=16, device=device, layout_seed=5998, **QWEN))
