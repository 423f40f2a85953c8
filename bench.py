#!/usr/bin/env python3
"""Benchmark of the batch-invariant paged attention path on GB300.

A step is one pass of the whole path over one synthetic batch: a causal
prefill call on the Qwen3-8B-shaped batch (8 requests, lengths uniform in
[512, 8192], 32 q / 8 kv heads, head_dim 128, page size 1, split-KV 4096)
followed by a decode call on the decode sweep's largest batch (256 requests,
contexts uniform in [1024, 32768], page size 1, split-KV 2048).  Each call
runs the device planner, the attention kernel and the split merge.

Printed (one JSON line): prefill algorithmic TFLOP/s as `value`
(causal-exact flops 4*D*sum(visible keys) over the prefill call time),
decode K+V GB/s under `decode`, the attention kernels' rooflines against
the measured peaks, end-to-end numbers of both calls through host buffers,
clocks sampled during the timed region, the number of kernel launches, the
CPU oracle timed on a bounded sample as a baseline, and under `configs` the
other workloads (the prefix extend unchunked and in 256-token chunks, the
mixed serving batch's prefill and decode calls, decode batches of 1, 8 and
64), each call timed on its own with its kernel's roofline.

The library drives one GPU per process: with --gpus other than 1, or under
torchrun with several ranks, rank 0 prints a one-line `unavailable` record
and no rank touches a GPU.

  python bench.py [--gpus 1] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "prefill attn TFLOPS & decode KV GB/s (batch-invariant) on 1 GB300, % roofline"
WORKLOAD = ("Qwen3-8B-shaped batched causal prefill: 8 requests, lengths U[512,8192], "
            "32 q / 8 kv heads, head_dim 128, page_size 1, split-KV 4096; then decode: "
            "256 requests, context U[1024,32768], split-KV 2048")
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true",
                   help="skip the oracle CPU baseline (quick runs)")
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer e2e legs")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the other workloads' legs (cfg3, cfg5, decode batches 1/8/64)")
    p.add_argument("--cpu-seconds", type=float, default=20.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--only", choices=["both", "prefill", "decode"], default="both",
                   help="run one of the two calls (profiling captures of a small case)")
    p.add_argument("--decode-batch", type=int, default=256,
                   help="decode requests (the decode sweep's largest batch by default)")
    p.add_argument("--sweep", action="store_true",
                   help="time every workload (one JSON line each) instead of the default step")
    p.add_argument("--sweep-only", default="",
                   help="comma list of sweep groups to run (tiny,cfg2,append,cfg3,cfg5,d256,"
                        "mla,cfg4); empty: all")
    return p.parse_args()


# ----------------------------------------------------------------- helpers
def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            raw = json.load(f)
        flat = {}

        def walk(d):
            for k, v in d.items():
                if isinstance(v, dict):
                    walk(v)
                elif isinstance(v, (int, float)):
                    flat.setdefault(k, float(v))
        walk(raw)
        if all(k in flat for k in ("bf16_tflops", "hbm_gbs")):
            flat.setdefault("bf16_tflops_sustained", flat["bf16_tflops"])
            return flat, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def prefill_flops(call: wl.Call, D: int, Hq: int) -> int:
    """Causal-exact algorithmic flops: 4*D per (row, visible key)."""
    total = 0
    for q_len, kv_len in zip(call.q_lens, call.kv_lens):
        first = kv_len - q_len + 1  # keys visible to the first new token
        total += q_len * first + q_len * (q_len - 1) // 2
    return 4 * D * Hq * total


def kv_bytes(call: wl.Call, Hkv: int, D: int) -> int:
    return sum(call.kv_lens) * Hkv * D * 2 * 2


def source_hash(*files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_from_profiles(kernel: str, src: list, units_now: float):
    """DRAM bytes per launch from the committed ncu counters, scaled to this
    launch's units; None if absent or captured on different kernel source."""
    path = os.path.join(ROOT, "profiles", "counters.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel)
    if not rec or rec.get("source_sha") != source_hash(*src):
        return None
    return rec["dram_bytes_per_launch"] * units_now / rec["units_per_launch"]


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"bia_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_median": statistics.median(power), "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------- oracle baseline
def oracle_sample_rate(call: wl.Call, target_s: float, seed: int = 0):
    """Times the CPU oracle on a seeded sample of rows of `call` sized to take
    about target_s seconds; returns (TFLOP/s, cores, description)."""
    import oracle

    st = call.store
    H, D = st.num_qo_heads, st.head_dim
    cores = host_cores()
    rng = np.random.default_rng(seed)
    cpu_call = wl.Call(st, call.parts, call.q.cpu(), call.qo_indptr, call.kv_indptr,
                       call.kv_indices, call.kv_last_page_len, call.q_lens, call.kv_lens)
    k_bits, v_bits = wl.bf16_bits(st.k_cache), wl.bf16_bits(st.v_cache)
    q_bits = wl.bf16_bits(cpu_call.q)
    total_q = call.total_q
    owner = np.repeat(np.arange(call.batch), call.q_lens)
    qo = call.qo_indptr.numpy()

    def visible(tokens):
        b = owner[tokens]
        t = tokens - qo[b]
        return np.array(call.kv_lens)[b] - np.array(call.q_lens)[b] + t + 1

    def run(n_rows):
        toks = rng.integers(0, total_q, n_rows)
        heads = rng.integers(0, H, n_rows)
        rows = np.stack([toks, heads], 1)
        t0 = time.perf_counter()
        oracle.attention(q_bits, k_bits, v_bits, call.qo_indptr.numpy(),
                         call.kv_indptr.numpy(), call.kv_indices.numpy(),
                         call.kv_last_page_len.numpy(), num_qo_heads=H,
                         num_kv_heads=st.num_kv_heads, head_dim=D, page_size=st.page_size,
                         rows=rows, threads=cores)
        dt = time.perf_counter() - t0
        return 4.0 * D * float(visible(toks).sum()), dt

    flops, dt = run(max(cores * 4, 64))
    per_row = dt / max(cores * 4, 64)
    n = int(max(cores * 4, min(2_000_000, target_s / max(per_row, 1e-7))))
    flops, dt = run(n)
    desc = (f"{n} (token, q head) rows drawn uniformly from the same batch, all their "
            f"visible keys; {flops / 1e9:.1f} GFLOP algorithmic in {dt:.1f} s")
    return flops / dt / 1e12, cores, desc, dt


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on this workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    store = wl.cfg2_prefill("cpu")
    call = wl.whole_prefill(store)
    per_step = max(1.0, min(6.0, 150.0 / (args.steps + args.warmup)))
    vals = []
    descs = []
    for i in range(args.warmup + args.steps):
        v, cores, desc, dt = oracle_sample_rate(call, per_step, seed=100 + i)
        if i >= args.warmup:
            vals.append(v)
            descs.append(dt)
    value = float(statistics.median(vals))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * statistics.median(descs), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD.split("; then")[0],
                       "note": "CPU fp64 oracle on a bounded row sample per step"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- our arm
def run_sweep(args):
    """One JSON line per workload: each call timed with CUDA events on its
    stream (median of --steps after --warmup, L2 flushed before each, calls
    enqueued back to back), kernel time from the library's profile events.
    For tables; not the driver's single-line contract."""
    import invariant_paged_attention_gb300 as bia
    from invariant_paged_attention_gb300 import build as bia_build
    bia_build.build()
    bia.load()
    dev = "cuda:0"
    stream = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    peaks, peak_kind = load_peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def dev_idx(call):
        return [call.qo_indptr.to(dev), call.kv_indptr.to(dev), call.kv_indices.to(dev),
                call.kv_last_page_len.to(dev)]

    def time_calls(fns):
        for _ in range(args.warmup):
            for f in fns:
                f(None)
        evs = []
        for _ in range(args.steps):  # enqueued back to back: the GPU's time per call
            flush.zero_()  # L2 (129 MB) flushed before every timed call
            a0, a1, k0, k1 = ev(), ev(), ev(), ev()
            a0.record(stream)
            for f in fns:
                f((k0, k1) if len(fns) == 1 else None)
            a1.record(stream)
            evs.append((a0, a1, k0, k1))
        torch.cuda.synchronize()
        bia.bia_set_profile_events(None, None)
        call_ms = [a0.elapsed_time(a1) for a0, a1, _, _ in evs]
        kern_ms = [k0.elapsed_time(k1) for _, _, k0, k1 in evs] if len(fns) == 1 else []
        return statistics.median(call_ms), (statistics.median(kern_ms) if kern_ms else None)

    def prefill_fn(store, call):
        st = store
        desc = bia.make_desc(st.num_qo_heads, st.num_kv_heads, st.head_dim, st.page_size)
        qo, kvp, idx, last = dev_idx(call)
        ws = torch.empty(bia.bia_prefill_workspace_size(desc, call.qo_indptr, call.kv_indptr,
                                                        call.kv_last_page_len),
                         dtype=torch.uint8, device=dev)
        out = torch.empty_like(call.q)
        lse = torch.empty(call.total_q, st.num_qo_heads, dtype=torch.float32, device=dev)

        def f(evs):
            if evs:
                bia.bia_set_profile_events(*evs)
            bia.bia_prefill_paged(desc, call.q, st.k_cache, st.v_cache, qo, kvp, idx, last,
                                  call.qo_indptr, call.kv_indptr, call.kv_last_page_len, ws, out,
                                  lse, stream=stream)
            if evs:
                bia.bia_set_profile_events(None, None)
        return f

    def decode_fn(store, call):
        st = store
        desc = bia.make_desc(st.num_qo_heads, st.num_kv_heads, st.head_dim, st.page_size)
        _, kvp, idx, last = dev_idx(call)
        ws = torch.empty(bia.bia_decode_workspace_size(desc, call.kv_indptr,
                                                       call.kv_last_page_len),
                         dtype=torch.uint8, device=dev)
        out = torch.empty_like(call.q)
        lse = torch.empty(call.total_q, st.num_qo_heads, dtype=torch.float32, device=dev)

        def f(evs):
            if evs:
                bia.bia_set_profile_events(*evs)
            bia.bia_decode_paged(desc, call.q, st.k_cache, st.v_cache, kvp, idx, last,
                                 call.kv_indptr, call.kv_last_page_len, ws, out, lse,
                                 stream=stream)
            if evs:
                bia.bia_set_profile_events(None, None)
        return f

    def append_fn(store, call, k_new, v_new):
        st = store
        desc = bia.make_desc(st.num_qo_heads, st.num_kv_heads, st.head_dim, st.page_size)
        ap, kvp, idx, last = dev_idx(call)

        def f(evs):
            if evs:
                evs[0].record(stream)
            bia.bia_append_paged_kv(desc, k_new, v_new, st.k_cache, st.v_cache, ap, kvp, idx,
                                    last, call.qo_indptr, call.kv_indptr, call.kv_last_page_len,
                                    stream=stream)
            if evs:
                evs[1].record(stream)
        return f

    def emit(name, kind, work, call_ms, kern_ms, extra=None):
        if kind == "prefill":
            v, u, pk = work / call_ms / 1e9, "TFLOP/s", peaks["bf16_tflops"]
            kv = work / kern_ms / 1e9 if kern_ms else None
        else:
            v, u, pk = work / call_ms / 1e6, "GB/s", peaks["hbm_gbs"]
            kv = work / kern_ms / 1e6 if kern_ms else None
        line = {"workload": name, "kind": kind, "value": v, "unit": u, "call_ms": call_ms,
                "kernel_ms": kern_ms, "kernel_value": kv,
                "frac_of_peak": (kv / pk) if kv else None, "peak": pk,
                "peak_source": peak_kind, "work": work}
        line.update(extra or {})
        print(json.dumps(line), flush=True)

    groups = {g for g in args.sweep_only.split(",") if g}
    want = lambda g: not groups or g in groups  # noqa: E731
    D, Hq, Hkv = 128, 32, 8
    # prefill workloads
    if want("tiny"):
        st = wl.cfg1_tiny(dev)
        c = wl.whole_prefill(st)
        cm, km = time_calls([prefill_fn(st, c)])
        emit("cfg1 tiny prefill (256 tok, 4q/1kv, d64, page 16)", "prefill",
             prefill_flops(c, 64, 4), cm, km)
    if want("cfg2") or want("append"):
        st = wl.cfg2_prefill(dev)
        c = wl.whole_prefill(st)
        if want("cfg2"):
            cm, km = time_calls([prefill_fn(st, c)])
            emit("cfg2 batched prefill (8 req, U[512,8192])", "prefill", prefill_flops(c, D, Hq),
                 cm, km)
        if want("append"):
            k_new, v_new = wl.new_kv_rows(c)
            cm, km = time_calls([append_fn(st, c, k_new, v_new)])
            # read the new rows once, write them once
            emit("paged-KV append of the cfg2 prompts (8 req, U[512,8192], page 1)", "append",
                 4 * k_new.numel() * k_new.element_size(), cm, km)
            del k_new, v_new
        del st, c
    if want("cfg3"):
        st = wl.cfg3_prefix(dev)
        whole = wl.whole_prefill(st)
        cm, km = time_calls([prefill_fn(st, whole)])
        fl = prefill_flops(whole, D, Hq)
        emit("cfg3 prefix extend, unchunked (4 x 16384 new)", "prefill", fl, cm, km)
        fns = [prefill_fn(st, cc) for cc in wl.chunked_calls(st, 256)]
        cm, _ = time_calls(fns)
        emit("cfg3 prefix extend, 64 chunks of 256", "prefill", fl, cm, None)
        del st, whole, fns
    if want("cfg5"):
        sweep_cfg5(wl, dev, D, Hq, Hkv, time_calls, prefill_fn, decode_fn, emit, prefill_flops,
                   kv_bytes)
    if want("d256"):
        sweep_d256(wl, dev, time_calls, prefill_fn, decode_fn, emit, prefill_flops, kv_bytes)
    if want("mla"):
        sweep_mla(wl, bia, dev, stream, time_calls, emit)
    if want("cfg4"):
        for B in (1, 8, 64, 256):
            st = wl.cfg4_decode(dev, B)
            c = wl.whole_prefill(st)
            cm, km = time_calls([decode_fn(st, c)])
            emit(f"cfg4 decode B={B} (ctx U[1024,32768], page 1)", "decode", kv_bytes(c, Hkv, D),
                 cm, km)
            del st, c
            torch.cuda.empty_cache()


def sweep_cfg5(wl, dev, D, Hq, Hkv, time_calls, prefill_fn, decode_fn, emit, prefill_flops,
               kv_bytes):
    pst, dst = wl.cfg5_mixed(dev)
    pc = wl.whole_prefill(pst)
    cm, km = time_calls([prefill_fn(pst, pc)])
    emit("cfg5 mixed prefill call (4096-tok chunk + 64 one-token extends, page 16)", "prefill",
         prefill_flops(pc, D, Hq), cm, km, {"kv_bytes": kv_bytes(pc, Hkv, D)})
    # its two parts on their own: the chunk (tensor bound) and the one-token
    # extends (their single-token q tiles streamed by the decode kernel)
    chunk = wl.make_call(pst, [(0, 0, pst.seqs[0].new)])
    cm, km = time_calls([prefill_fn(pst, chunk)])
    emit("cfg5 chunk alone (4096 new tokens after a 4096-token prefix, page 16)", "prefill",
         prefill_flops(chunk, D, Hq), cm, km)
    ext = wl.make_call(pst, [(i, 0, 1) for i in range(1, len(pst.seqs))])
    cm, km = time_calls([prefill_fn(pst, ext)])
    emit("cfg5 one-token extends alone (64, ctx U[1024,32768], page 16)", "kv-stream",
         kv_bytes(ext, Hkv, D), cm, km)
    dc = wl.whole_prefill(dst)
    cm, km = time_calls([decode_fn(dst, dc)])
    emit("cfg5 decodes (32 x 131072 ctx, page 16)", "decode", kv_bytes(dc, Hkv, D), cm, km)
    del pst, dst, pc, dc
    torch.cuda.empty_cache()


def sweep_d256(wl, dev, time_calls, prefill_fn, decode_fn, emit, prefill_flops, kv_bytes):
    # head_dim 256 (16 q / 8 kv heads): the wide prefill kernel and decode
    st = wl.wide_prefill(dev)
    c = wl.whole_prefill(st)
    cm, km = time_calls([prefill_fn(st, c)])
    emit("head_dim 256 prefill (cfg2 lengths, 16q/8kv, page 1)", "prefill",
         prefill_flops(c, 256, 16), cm, km)
    del st, c
    st = wl.wide_prefill(dev, page_size=16)
    c = wl.whole_prefill(st)
    cm, km = time_calls([prefill_fn(st, c)])
    emit("head_dim 256 prefill (cfg2 lengths, 16q/8kv, page 16)", "prefill",
         prefill_flops(c, 256, 16), cm, km)
    del st, c
    st = wl.wide_decode(dev, 64)
    c = wl.whole_prefill(st)
    cm, km = time_calls([decode_fn(st, c)])
    emit("head_dim 256 decode B=64 (ctx U[1024,32768], 16q/8kv, page 1)", "decode",
         kv_bytes(c, 8, 256), cm, km)
    del st, c
    torch.cuda.empty_cache()


def sweep_mla(wl, bia, dev, stream, time_calls, emit):
    # multi-head latent attention decode: 16 heads over one 512 + 64 latent cache
    ctx = wl.uniform_lengths(64, 1024, 32768, 4000)
    mst = wl.MLAStore([wl.Sequence(7700 + i, c - 1, 1) for i, c in enumerate(ctx)], 16, 512, 64,
                      1, dev, layout_seed=7997)
    mc = wl.mla_call(mst, [(i, 0, 1) for i in range(len(mst.seqs))])
    mdesc = bia.make_mla_desc(16, 1, 1.0 / 192 ** 0.5)
    mws = torch.empty(bia.bia_mla_decode_workspace_size(mdesc, mc.kv_indptr,
                                                        mc.kv_last_page_len),
                      dtype=torch.uint8, device=dev)
    mout = torch.empty((64, 16, 512), dtype=torch.bfloat16, device=dev)
    margs = [mc.kv_indptr.to(dev), mc.kv_indices.to(dev), mc.kv_last_page_len.to(dev)]

    def mla_f(evs):
        if evs:
            bia.bia_set_profile_events(*evs)
        bia.bia_mla_decode_paged(mdesc, mc.q_nope, mc.q_pe, mst.ckv_cache, mst.kpe_cache, *margs,
                                 mc.kv_indptr, mc.kv_last_page_len, mws, mout, stream=stream)
        if evs:
            bia.bia_set_profile_events(None, None)
    cm, km = time_calls([mla_f])
    emit("MLA decode B=64, 16 heads, latent 512+64 (ctx U[1024,32768], page 1)", "decode",
         sum(mc.kv_lens) * (512 + 64) * 2, cm, km)
    del mst, mc, mws, mout
    torch.cuda.empty_cache()

    # MLA extend: 64 requests each verifying 4 speculative tokens, same lengths
    est = wl.MLAStore([wl.Sequence(7800 + i, c - 4, 4) for i, c in enumerate(ctx)], 16, 512,
                      64, 1, dev, layout_seed=7998)
    ec = wl.mla_call(est, [(i, 0, 4) for i in range(len(est.seqs))])
    ews = torch.empty(bia.bia_mla_prefill_workspace_size(mdesc, ec.qo_indptr, ec.kv_indptr,
                                                         ec.kv_last_page_len),
                      dtype=torch.uint8, device=dev)
    eout = torch.empty((int(ec.qo_indptr[-1]), 16, 512), dtype=torch.bfloat16, device=dev)
    eargs = [ec.qo_indptr.to(dev), ec.kv_indptr.to(dev), ec.kv_indices.to(dev),
             ec.kv_last_page_len.to(dev)]

    def mla_ext_f(evs):
        if evs:
            bia.bia_set_profile_events(*evs)
        bia.bia_mla_prefill_paged(mdesc, ec.q_nope, ec.q_pe, est.ckv_cache, est.kpe_cache,
                                  *eargs, ec.qo_indptr, ec.kv_indptr, ec.kv_last_page_len, ews,
                                  eout, stream=stream)
        if evs:
            bia.bia_set_profile_events(None, None)
    cm, km = time_calls([mla_ext_f])
    # token t of a request sees kv_len - 3 + t keys; 2 flops per multiply-add
    # over 576 score columns and 512 value columns, 16 heads
    visible = sum(4 * kv - 6 for kv in ec.kv_lens)
    emit("MLA extend B=64 x 4 tokens, 16 heads, latent 512+64 (ctx U[1024,32768], page 1)",
         "prefill", visible * 16 * 2 * (576 + 512), cm, km,
         {"latent_bytes_per_token_pass": visible * (512 + 64) * 2,
          "note": "16 heads: two tokens per CTA, so the rows are read once per pair"})
    del est, ec, ews, eout
    torch.cuda.empty_cache()


class Leg:
    """One call timed on its own: warm-up calls, then `steps` calls each
    preceded by an untimed L2 flush (a 256 MiB write, more than the 129 MB
    L2) and bracketed by CUDA events on the launching stream; the attention
    kernel alone is timed by the events the library records around it.  The
    timed calls are enqueued back to back (one synchronize at the end), so the
    host prepares the next call while the GPU flushes L2 and the events time
    the GPU's execution of each call, not the binding's argument checks."""

    def __init__(self, bia, stream, flush):
        self.bia, self.stream, self.flush = bia, stream, flush

    def run(self, fns, steps, warmup):
        ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
        for _ in range(warmup):
            for f in fns:
                f()
        torch.cuda.synchronize()
        launches0 = self.bia.bia_launch_count()
        evs = []
        for _ in range(steps):
            self.flush.zero_()
            a0, a1, k0, k1 = ev(), ev(), ev(), ev()
            if len(fns) == 1:
                self.bia.bia_set_profile_events(k0, k1)
            a0.record(self.stream)
            for f in fns:
                f()
            a1.record(self.stream)
            self.bia.bia_set_profile_events(None, None)
            evs.append((a0, a1, k0, k1))
        torch.cuda.synchronize()
        call_ms = [a0.elapsed_time(a1) for a0, a1, _, _ in evs]
        kern_ms = [k0.elapsed_time(k1) for _, _, k0, k1 in evs] if len(fns) == 1 else []
        launches = (self.bia.bia_launch_count() - launches0) // max(steps, 1)
        return (statistics.median(call_ms), statistics.median(kern_ms) if kern_ms else None,
                int(launches))


def roofline_of(kind, work, kern_ms, peaks, peak_kind, kernel, traffic=None):
    if kind == "tensor":
        achieved = work / kern_ms / 1e9
        return {"bound": "tensor", "kernel": kernel, "achieved": achieved,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"],
                "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                "peak_source": f"bf16 dense burst, of {peak_kind}",
                "algorithmic_flops_per_launch": work, "kernel_ms": kern_ms, "traffic": traffic}
    achieved = work / kern_ms / 1e6
    return {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
            "peak_source": f"HBM copy, of {peak_kind}", "kv_bytes_per_launch": work,
            "kernel_ms": kern_ms, "traffic": traffic}


def refuse_multi_gpu(args, world, rank):
    """The library runs on one GPU per process, and its prefill kernels
    multicast K/V gathers inside thread-block clusters, which it does for one
    GPU's own memory only: there is no multi-GPU bench.  Rank 0 says so in one
    JSON line; every rank exits without touching a GPU."""
    if rank == 0:
        print(json.dumps({"metric": METRIC, "n_gpus": max(world, args.gpus),
                          "unavailable": "one GPU only: the attention shards into independent "
                                         "requests with no exchange step, and this library "
                                         "runs on the GPU of the calling process alone"}),
              flush=True)


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args)
        return
    if world > 1 or args.gpus != 1:
        refuse_multi_gpu(args, world, rank)
        return
    if args.sweep:
        run_sweep(args)
        return

    import invariant_paged_attention_gb300 as bia
    from invariant_paged_attention_gb300 import build as bia_build

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(0)
    dev = "cuda:0"
    bia_build.build()
    bia.load()

    # ---- inputs resident in HBM
    do_p, do_d = args.only in ("both", "prefill"), args.only in ("both", "decode")
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    stream = torch.cuda.current_stream()

    def dev_idx(call):
        return [call.qo_indptr.to(dev), call.kv_indptr.to(dev), call.kv_indices.to(dev),
                call.kv_last_page_len.to(dev)]

    def prefill_call(store, call):
        desc = bia.make_desc(store.num_qo_heads, store.num_kv_heads, store.head_dim,
                             store.page_size)
        qo, kvp, idx, last = dev_idx(call)
        ws = torch.empty(bia.bia_prefill_workspace_size(desc, call.qo_indptr, call.kv_indptr,
                                                        call.kv_last_page_len),
                         dtype=torch.uint8, device=dev)
        out = torch.empty_like(call.q)
        lse = torch.empty(call.total_q, store.num_qo_heads, dtype=torch.float32, device=dev)

        def f(q=None, k=None, v=None, idx4=None, o=None, lo=None):
            bia.bia_prefill_paged(desc, call.q if q is None else q,
                                  store.k_cache if k is None else k,
                                  store.v_cache if v is None else v,
                                  *(idx4 or (qo, kvp, idx, last)), call.qo_indptr,
                                  call.kv_indptr, call.kv_last_page_len, ws,
                                  out if o is None else o, lse if lo is None else lo,
                                  stream=stream)
        f.out, f.lse = out, lse
        return f

    def decode_call(store, call):
        desc = bia.make_desc(store.num_qo_heads, store.num_kv_heads, store.head_dim,
                             store.page_size)
        _, kvp, idx, last = dev_idx(call)
        ws = torch.empty(bia.bia_decode_workspace_size(desc, call.kv_indptr,
                                                       call.kv_last_page_len),
                         dtype=torch.uint8, device=dev)
        out = torch.empty_like(call.q)
        lse = torch.empty(call.total_q, store.num_qo_heads, dtype=torch.float32, device=dev)

        def f(q=None, k=None, v=None, idx3=None, o=None, lo=None):
            bia.bia_decode_paged(desc, call.q if q is None else q,
                                 store.k_cache if k is None else k,
                                 store.v_cache if v is None else v,
                                 *(idx3 or (kvp, idx, last)), call.kv_indptr,
                                 call.kv_last_page_len, ws, out if o is None else o,
                                 lse if lo is None else lo, stream=stream)
        f.out, f.lse = out, lse
        return f

    flops = dbytes = 0
    prefill = decode = None
    if do_p:
        pstore = wl.cfg2_prefill(dev)
        pcall = wl.whole_prefill(pstore)
        Hq, Hkv, D = pstore.num_qo_heads, pstore.num_kv_heads, pstore.head_dim
        prefill = prefill_call(pstore, pcall)
        flops = prefill_flops(pcall, D, Hq)
    if do_d:
        dstore = wl.cfg4_decode(dev, args.decode_batch)
        dcall = wl.whole_prefill(dstore)
        Hq, Hkv, D = dstore.num_qo_heads, dstore.num_kv_heads, dstore.head_dim
        decode = decode_call(dstore, dcall)
        dbytes = kv_bytes(dcall, Hkv, D)

    # ---- device-timed loop: a step = the prefill call then the decode call
    n = args.warmup + args.steps
    e_step = [(ev(), ev(), ev()) for _ in range(n)]
    e_pk = [(ev(), ev()) for _ in range(n)]
    e_dk = [(ev(), ev()) for _ in range(n)]

    def step(i):
        s0, s1, s2 = e_step[i]
        s0.record(stream)
        if prefill:
            bia.bia_set_profile_events(*e_pk[i])
            prefill()
        s1.record(stream)
        if decode:
            bia.bia_set_profile_events(*e_dk[i])
            decode()
        s2.record(stream)

    for i in range(args.warmup):
        step(i)
    bia.bia_set_profile_events(None, None)
    torch.cuda.synchronize()
    launches0 = bia.bia_launch_count()
    with ClockSampler(0) as clocks:
        torch.cuda.synchronize()
        t_wall0 = time.perf_counter()
        for i in range(args.warmup, n):
            step(i)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
    bia.bia_set_profile_events(None, None)
    launches = bia.bia_launch_count() - launches0
    timed = range(args.warmup, n)
    K = args.steps
    pre_s = sum(e_step[i][0].elapsed_time(e_step[i][1]) for i in timed) / 1000.0
    dec_s = sum(e_step[i][1].elapsed_time(e_step[i][2]) for i in timed) / 1000.0
    pk_s = sum(e_pk[i][0].elapsed_time(e_pk[i][1]) for i in timed) / 1000.0 if prefill else 0.0
    dk_s = sum(e_dk[i][0].elapsed_time(e_dk[i][1]) for i in timed) / 1000.0 if decode else 0.0
    value = flops * K / pre_s / 1e12 if prefill else None
    dec_gbs = dbytes * K / dec_s / 1e9 if decode else None
    pk_avg, dk_avg = pk_s / K, dk_s / K

    # ---- the timed outputs are finite (parity is the test suite's job)
    if prefill:
        assert torch.isfinite(prefill.out.float()).all()
    if decode:
        assert torch.isfinite(decode.out.float()).all()

    peaks, peak_kind = load_peaks()
    # counters are keyed by the kernel's own translation unit
    pre_src = ["invariant_paged_attention_gb300/csrc/prefill.cu",
               "invariant_paged_attention_gb300/csrc/softmax_rows.cuh",
               "invariant_paged_attention_gb300/csrc/ptx.cuh"]
    dec_src = ["invariant_paged_attention_gb300/csrc/decode_tc.cu",
               "invariant_paged_attention_gb300/csrc/ptx.cuh"]
    roofline = roofline_of("tensor", flops, pk_avg * 1e3, peaks, peak_kind, "prefill_kernel<128>",
                           traffic_from_profiles("prefill_kernel<128>", pre_src, flops)) \
        if prefill else None
    dec_roof = roofline_of("hbm", dbytes, dk_avg * 1e3, peaks, peak_kind,
                           "decode_tc_kernel<4,false>",
                           traffic_from_profiles("decode_tc_kernel<4,false>", dec_src, dbytes)) \
        if decode else None

    # ---- end to end through host buffers: each step copies its inputs from
    # pinned host memory (q, the K/V caches, the index arrays), makes the
    # call, and copies out + lse back
    def pin(t):
        h = torch.empty(tuple(t.shape), dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        return h

    def host_available_bytes():
        try:
            with open("/proc/meminfo") as fh:
                for ln in fh:
                    if ln.startswith("MemAvailable:"):
                        return int(ln.split()[1]) * 1024
        except OSError:
            pass
        return 0

    def e2e_leg(fn, store, call, is_decode, work, unit_scale, steps):
        """Steps of one call through the C ABI with host buffers: each step
        copies its inputs (q, the K/V caches, the index arrays) from pinned
        host memory, makes the call and copies out + lse back.  Two sets of
        device buffers and separate copy streams let step i+1's uploads and
        step i-1's downloads run while step i computes, as a serving loop
        would; every step still moves all its bytes inside the timed region."""
        cache_bytes = 2 * store.k_cache.numel() * store.k_cache.element_size()
        if host_available_bytes() < 4 * cache_bytes:
            return {"value": None, "skipped": "pinned host copies of the caches would take "
                                              "more than a quarter of the free host memory"}
        hq, hk, hv = pin(call.q), pin(store.k_cache), pin(store.v_cache)
        names = (call.kv_indptr, call.kv_indices, call.kv_last_page_len) if is_decode else \
            (call.qo_indptr, call.kv_indptr, call.kv_indices, call.kv_last_page_len)
        h_idx = [pin(t) for t in names]
        h_out = torch.empty(tuple(hq.shape), dtype=hq.dtype, pin_memory=True)
        h_lse = torch.empty(tuple(fn.lse.shape), dtype=torch.float32, pin_memory=True)
        bufs = [dict(q=torch.empty_like(call.q), k=torch.empty_like(store.k_cache),
                     v=torch.empty_like(store.v_cache),
                     idx=[torch.empty_like(t, device=dev) for t in h_idx],
                     out=torch.empty_like(fn.out), lse=torch.empty_like(fn.lse))
                for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in [hq, hk, hv] + h_idx)
        d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

        def run(n):
            done_in, done_comp, done_out = [], [], []
            start = ev()
            start.record(s_in)
            for i in range(n):
                bf = bufs[i % 2]
                with torch.cuda.stream(s_in):
                    if i >= 2:  # the inputs of step i-2 have been consumed
                        s_in.wait_event(done_comp[i - 2])
                    bf["q"].copy_(hq, non_blocking=True)
                    bf["k"].copy_(hk, non_blocking=True)
                    bf["v"].copy_(hv, non_blocking=True)
                    for dst, src in zip(bf["idx"], h_idx):
                        dst.copy_(src, non_blocking=True)
                    e = ev()
                    e.record(s_in)
                    done_in.append(e)
                stream.wait_event(done_in[i])
                if i >= 2:  # the outputs of step i-2 have been copied out
                    stream.wait_event(done_out[i - 2])
                fn(bf["q"], bf["k"], bf["v"], bf["idx"], bf["out"], bf["lse"])
                e = ev()
                e.record(stream)
                done_comp.append(e)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(done_comp[i])
                    h_out.copy_(bf["out"], non_blocking=True)
                    h_lse.copy_(bf["lse"], non_blocking=True)
                    e = ev()
                    e.record(s_out)
                    done_out.append(e)
            return start, done_out[-1]
        run(3)
        torch.cuda.synchronize()
        a, b = run(steps)
        torch.cuda.synchronize()
        secs = a.elapsed_time(b) / 1000.0
        del bufs, hk, hv
        return {"value": work * steps / secs / unit_scale, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "steps": steps,
                "pipelining": "2 device buffer sets; uploads, compute and downloads on "
                              "separate streams"}

    e2e = dec_e2e = None
    if not args.no_e2e:
        if prefill:
            e2e = e2e_leg(prefill, pstore, pcall, False, flops, 1e12, min(K, 20))
            e2e.update(unit="TFLOP/s", scope="prefill call incl. H2D of q/K/V/index arrays "
                                              "from pinned host memory and D2H of out+lse")
        if decode:
            dec_e2e = e2e_leg(decode, dstore, dcall, True, dbytes, 1e9, min(K, 8))
            dec_e2e.update(unit="GB/s", scope="decode call incl. H2D of q/K/V/index arrays "
                                               "from pinned host memory and D2H of out+lse")

    # ---- every other workload, each call timed alone (L2 flushed before each)
    configs = {}
    if args.only == "both" and not args.no_configs:
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        leg = Leg(bia, stream, flush)
        cs, cw = max(3, min(args.steps, 10)), 3

        def put(name, kind, work, cm, km, launches, kernel, desc_txt, extra=None):
            unit, scale = ("TFLOP/s", 1e9) if kind == "tensor" else ("GB/s", 1e6)
            rec = {"workload": desc_txt, "value": work / cm / scale, "unit": unit,
                   "call_ms": cm, "gpu_launches_per_call": launches,
                   "roofline": roofline_of(kind, work, km, peaks, peak_kind, kernel) if km else None}
            rec.update(extra or {})
            configs[name] = rec

        st = wl.cfg3_prefix(dev)
        whole = wl.whole_prefill(st)
        fl = prefill_flops(whole, 128, 32)
        f = prefill_call(st, whole)
        cm, km, nl = leg.run([f], cs, cw)
        put("cfg3_unchunked", "tensor", fl, cm, km, nl, "prefill_kernel<128>",
            "prefixes 1/511/2048/4097 + 16384 new tokens, one extend call, page 1")
        fns = [prefill_call(st, c) for c in wl.chunked_calls(st, 256)]
        cm, _, nl = leg.run(fns, cs, cw)
        put("cfg3_chunks256", "tensor", fl, cm, None, nl, "prefill_kernel<128>",
            "the same extend as 64 calls of 256-token chunks (on the 32-token grid)",
            {"note": "call_ms covers all 64 chunk calls"})
        del st, whole, f, fns
        pst, dst = wl.cfg5_mixed(dev)
        pc, dc = wl.whole_prefill(pst), wl.whole_prefill(dst)
        f = prefill_call(pst, pc)
        cm, km, nl = leg.run([f], cs, cw)
        fl5, kb5 = prefill_flops(pc, 128, 32), kv_bytes(pc, 8, 128)
        put("cfg5_prefill_call", "tensor", fl5, cm, km, nl,
            "prefill_kernel<128> + streamed tiles",
            "one 4096-token chunk (prefix 4096) + 64 one-token extends (ctx U[1024,32768]), "
            "page 16", {"kv_bytes": kb5})
        if km:
            # the chunk's tiles are tensor-bound, the 64 extends stream their
            # keys: the call's floor is both kernels at their own roofline,
            # one after the other
            floor = fl5 / (peaks["bf16_tflops"] * 1e9) + kb5 / (peaks["hbm_gbs"] * 1e6)
            configs["cfg5_prefill_call"]["roofline_mixed"] = {
                "bound": "tensor + hbm", "floor_ms": floor, "kernel_ms": km,
                "frac": floor / km,
                "note": "floor = flops / bf16 peak + kv bytes / HBM peak (of "
                        f"{peak_kind}); frac = floor / the kernels' time"}
        f = decode_call(dst, dc)
        cm, km, nl = leg.run([f], cs, cw)
        put("cfg5_decodes", "hbm", kv_bytes(dc, 8, 128), cm, km, nl,
            "decode_tc_kernel<4,false>", "32 decodes at 131072 context, page 16")
        del pst, dst, pc, dc, f
        for B in (1, 8, 64):
            st = wl.cfg4_decode(dev, B)
            c = wl.whole_prefill(st)
            f = decode_call(st, c)
            cm, km, nl = leg.run([f], cs, cw)
            put(f"cfg4_b{B}", "hbm", kv_bytes(c, 8, 128), cm, km, nl,
                "decode_tc_kernel<4,false>", f"{B} decodes, ctx U[1024,32768], page 1")
            del st, c, f
        del flush
        torch.cuda.empty_cache()

    cpu = None
    if prefill and not args.no_cpu_baseline:
        v, cores, desc, _ = oracle_sample_rate(pcall, args.cpu_seconds)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc}

    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": K, "warmup": args.warmup,
            "ms_per_step": (pre_s + dec_s) * 1000.0 / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16, random page tables)",
            "config": {"workload": WORKLOAD if args.only == "both" and args.decode_batch == 256
                       else f"{args.only} only (decode batch {args.decode_batch})",
                       "prefill_tokens": pcall.total_q if prefill else 0,
                       "prefill_algorithmic_flops": flops,
                       "decode_requests": dcall.batch if decode else 0,
                       "decode_kv_bytes": dbytes, "parallelism": "one GPU",
                       "l2": "main step: inputs larger than L2 (prefill q+K+V ~0.43 GB, decode "
                             "K+V ~17.2 GB streamed between prefill steps); configs: L2 flushed "
                             "(256 MiB write) before every timed call"},
            "decode": {"value": dec_gbs, "unit": "GB/s",
                       "ms_per_call": dec_s * 1000.0 / K, "roofline": dec_roof, "e2e": dec_e2e},
            "prefill_ms_per_call": pre_s * 1000.0 / K,
            "roofline": roofline if prefill else dec_roof, "e2e": e2e, "cpu_baseline": cpu,
            "configs": configs, "clocks": clocks.summary(), "gpu_launches": int(launches),
            "wall_s_timed": t_wall}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
