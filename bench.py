#!/usr/bin/env python3
"""Benchmark of the batch-invariant paged attention path on GB300.

A step is one pass of the whole path over one synthetic batch: a causal
prefill call on the Qwen3-8B-shaped batch (8 requests, lengths uniform in
[512, 8192], 32 q / 8 kv heads, head_dim 128, page size 1, split-KV 4096)
followed by a decode call on the decode sweep's largest batch (256 requests,
contexts uniform in [1024, 32768], page size 1, split-KV 2048).  Each call
runs the device planner, the attention kernel and the split merge.

Printed (rank 0, one JSON line): prefill algorithmic TFLOP/s as `value`
(causal-exact flops 4*D*sum(visible keys) over the prefill call time),
decode K+V GB/s under `decode`, the attention kernels' rooflines against
the measured peaks, an end-to-end number through host buffers, clocks
sampled during the timed region, the number of kernel launches, and the CPU
oracle timed on a bounded sample as a baseline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
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
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer e2e leg")
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


def aggregate_over_ranks(local_seconds, units_per_rank, steps, dist=None, device="cpu"):
    """Whole-job throughput of N replicas: every rank contributes its summed
    times, the slowest rank's time is the job's time (max over ranks), and the
    job's work is the sum over ranks.  Returns (units per second, max seconds
    per item of local_seconds)."""
    t = torch.tensor(list(local_seconds), dtype=torch.float64, device=device)
    w = torch.tensor([float(units_per_rank)], dtype=torch.float64, device=device)
    if dist is not None and dist.is_initialized():
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(w, op=dist.ReduceOp.SUM)
    tmax = t.tolist()
    return (w.item() * steps / tmax[0] if tmax[0] > 0 else 0.0), tmax


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
    stream (median of --steps after --warmup), kernel time from the library's
    profile events.  For tables; not the driver's single-line contract."""
    import invariant_paged_attention_gb300 as bia
    from invariant_paged_attention_gb300 import build as bia_build
    bia_build.build()
    bia.load()
    dev = "cuda:0"
    stream = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    peaks, peak_kind = load_peaks()

    def dev_idx(call):
        return [call.qo_indptr.to(dev), call.kv_indptr.to(dev), call.kv_indices.to(dev),
                call.kv_last_page_len.to(dev)]

    def time_calls(fns):
        for _ in range(args.warmup):
            for f in fns:
                f(None)
        call_ms, kern_ms = [], []
        for _ in range(args.steps):
            a0, a1, k0, k1 = ev(), ev(), ev(), ev()
            a0.record(stream)
            for f in fns:
                f((k0, k1) if len(fns) == 1 else None)
            a1.record(stream)
            torch.cuda.synchronize()
            call_ms.append(a0.elapsed_time(a1))
            if len(fns) == 1:
                kern_ms.append(k0.elapsed_time(k1))
        bia.bia_set_profile_events(None, None)
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
         {"latent_bytes_per_token_pass": visible * (512 + 64) * 2})
    del est, ec, ews, eout
    torch.cuda.empty_cache()


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
        return
    if args.sweep:
        run_sweep(args)
        return

    import invariant_paged_attention_gb300 as bia
    from invariant_paged_attention_gb300 import build as bia_build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(dev))
    if rank == 0 or world == 1:
        bia_build.build()
    if dist:
        dist.barrier()
    bia.load()

    # ---- inputs resident in HBM
    do_p, do_d = args.only in ("both", "prefill"), args.only in ("both", "decode")
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    stream = torch.cuda.current_stream()

    def dev_idx(call):
        return [call.qo_indptr.to(dev), call.kv_indptr.to(dev), call.kv_indices.to(dev),
                call.kv_last_page_len.to(dev)]

    flops = dbytes = 0
    prefill = decode = None
    if do_p:
        pstore = wl.cfg2_prefill(dev)
        pcall = wl.whole_prefill(pstore)
        Hq, Hkv, D = pstore.num_qo_heads, pstore.num_kv_heads, pstore.head_dim
        pdesc = bia.make_desc(Hq, Hkv, D, pstore.page_size)
        p_qo, p_kvp, p_idx, p_last = dev_idx(pcall)
        p_ws = torch.empty(bia.bia_prefill_workspace_size(pdesc, pcall.qo_indptr,
                                                          pcall.kv_indptr,
                                                          pcall.kv_last_page_len),
                           dtype=torch.uint8, device=dev)
        p_out = torch.empty_like(pcall.q)
        p_lse = torch.empty(pcall.total_q, Hq, dtype=torch.float32, device=dev)
        flops = prefill_flops(pcall, D, Hq)

        def prefill():
            bia.bia_prefill_paged(pdesc, pcall.q, pstore.k_cache, pstore.v_cache, p_qo, p_kvp,
                                  p_idx, p_last, pcall.qo_indptr, pcall.kv_indptr,
                                  pcall.kv_last_page_len, p_ws, p_out, p_lse, stream=stream)
    if do_d:
        dstore = wl.cfg4_decode(dev, args.decode_batch)
        dcall = wl.whole_prefill(dstore)
        Hq, Hkv, D = dstore.num_qo_heads, dstore.num_kv_heads, dstore.head_dim
        ddesc = bia.make_desc(Hq, Hkv, D, dstore.page_size)
        _, d_kvp, d_idx, d_last = dev_idx(dcall)
        d_ws = torch.empty(bia.bia_decode_workspace_size(ddesc, dcall.kv_indptr,
                                                         dcall.kv_last_page_len),
                           dtype=torch.uint8, device=dev)
        d_out = torch.empty_like(dcall.q)
        d_lse = torch.empty(dcall.total_q, Hq, dtype=torch.float32, device=dev)
        dbytes = kv_bytes(dcall, Hkv, D)

        def decode():
            bia.bia_decode_paged(ddesc, dcall.q, dstore.k_cache, dstore.v_cache, d_kvp, d_idx,
                                 d_last, dcall.kv_indptr, dcall.kv_last_page_len, d_ws, d_out,
                                 d_lse, stream=stream)

    # ---- device-timed loop
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
    if dist:
        dist.barrier()
    launches0 = bia.bia_launch_count()
    with ClockSampler(local) as clocks:
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        t_wall0 = time.perf_counter()
        for i in range(args.warmup, n):
            step(i)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
        if dist:
            dist.barrier()
    bia.bia_set_profile_events(None, None)
    launches = bia.bia_launch_count() - launches0
    timed = range(args.warmup, n)
    pre_ms = [e_step[i][0].elapsed_time(e_step[i][1]) for i in timed]
    dec_ms = [e_step[i][1].elapsed_time(e_step[i][2]) for i in timed]
    pk_ms = [e_pk[i][0].elapsed_time(e_pk[i][1]) if prefill else 0.0 for i in timed]
    dk_ms = [e_dk[i][0].elapsed_time(e_dk[i][1]) if decode else 0.0 for i in timed]
    K = args.steps
    local = [sum(pre_ms) / 1000.0, sum(dec_ms) / 1000.0, sum(pk_ms) / 1000.0,
             sum(dk_ms) / 1000.0]
    flops_rate, (pre_s, dec_s, pk_s, dk_s) = aggregate_over_ranks(local, flops, K, dist, dev)
    value = flops_rate / 1e12 if prefill else None
    dec_gbs = world * dbytes * K / dec_s / 1e9 if decode else None
    pk_avg, dk_avg = pk_s / K, dk_s / K

    # ---- the timed outputs are finite (parity is the test suite's job)
    if prefill:
        assert torch.isfinite(p_out.float()).all()
    if decode:
        assert torch.isfinite(d_out.float()).all()

    # ---- end to end through host buffers (prefill call, the headline metric)
    e2e = None
    if prefill and not args.no_e2e:
        pin = lambda t: t.cpu().pin_memory()  # noqa: E731
        hq, hk, hv = pin(pcall.q), pin(pstore.k_cache), pin(pstore.v_cache)
        h_idx = [pin(t) for t in (pcall.qo_indptr, pcall.kv_indptr, pcall.kv_indices,
                                  pcall.kv_last_page_len)]
        h_out, h_lse = torch.empty_like(hq).pin_memory(), torch.empty_like(p_lse.cpu()).pin_memory()
        dq, dk, dv = torch.empty_like(pcall.q), torch.empty_like(pstore.k_cache), \
            torch.empty_like(pstore.v_cache)
        d_idx4 = [torch.empty_like(t, device=dev) for t in h_idx]
        h2d = sum(t.numel() * t.element_size() for t in [hq, hk, hv] + h_idx)
        d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()

        def e2e_step():
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            for dst, src in zip(d_idx4, h_idx):
                dst.copy_(src, non_blocking=True)
            bia.bia_prefill_paged(pdesc, dq, dk, dv, *d_idx4, pcall.qo_indptr, pcall.kv_indptr,
                                  pcall.kv_last_page_len, p_ws, p_out, p_lse, stream=stream)
            h_out.copy_(p_out, non_blocking=True)
            h_lse.copy_(p_lse, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        ke = min(K, 20)
        a, b = ev(), ev()
        a.record(stream)
        for _ in range(ke):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        e2e_s = torch.tensor([a.elapsed_time(b) / 1000.0], dtype=torch.float64, device=dev)
        if dist:
            dist.all_reduce(e2e_s, op=dist.ReduceOp.MAX)
        e2e = {"value": world * flops * ke / e2e_s.item() / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "steps": ke, "scope": "prefill call incl. H2D of q/K/V/index arrays from pinned "
                                     "host memory and D2H of out+lse"}

    peaks, peak_kind = load_peaks()
    pk_achieved = flops / pk_avg / 1e12 if prefill else 0.0
    dk_achieved = dbytes / dk_avg / 1e9 if decode else 0.0
    # counters are keyed by the kernel's own translation unit
    pre_src = ["invariant_paged_attention_gb300/csrc/prefill.cu"]
    dec_src = ["invariant_paged_attention_gb300/csrc/decode.cu"]
    roofline = {"bound": "tensor", "kernel": "prefill_kernel<128>", "achieved": pk_achieved,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": pk_achieved / peaks["bf16_tflops"],
                "frac_of_sustained": pk_achieved / peaks["bf16_tflops_sustained"],
                "peak_source": f"bf16 dense burst, of {peak_kind}",
                "algorithmic_flops_per_launch": flops, "kernel_ms": pk_avg * 1e3,
                "traffic": traffic_from_profiles("prefill_kernel<128>", pre_src, flops)}
    dec_roof = {"bound": "hbm", "kernel": "decode_kernel<128,4,false>", "achieved": dk_achieved,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": dk_achieved / peaks["hbm_gbs"],
                "peak_source": f"HBM copy, of {peak_kind}", "kv_bytes_per_launch": dbytes,
                "kernel_ms": dk_avg * 1e3,
                "traffic": traffic_from_profiles("decode_kernel<128,4,false>", dec_src, dbytes)
                if decode else None}

    cpu = None
    if rank == 0 and prefill and not args.no_cpu_baseline:
        v, cores, desc, _ = oracle_sample_rate(pcall, args.cpu_seconds)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
                "steps": K, "warmup": args.warmup,
                "ms_per_step": (pre_s + dec_s) * 1000.0 / K, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic (seeded N(0,1) bf16, random page tables)",
                "config": {"workload": WORKLOAD if args.only == "both" and args.decode_batch == 256
                           else f"{args.only} only (decode batch {args.decode_batch})",
                           "prefill_tokens": pcall.total_q if prefill else 0,
                           "prefill_algorithmic_flops": flops,
                           "decode_requests": dcall.batch if decode else 0,
                           "decode_kv_bytes": dbytes, "parallelism": f"replicas x{world}",
                           "l2": "inputs larger than L2 (prefill q+K+V ~0.43 GB, decode K+V "
                                 "~17.7 GB streamed between prefill steps)"},
                "decode": {"value": dec_gbs, "unit": "GB/s",
                           "ms_per_call": dec_s * 1000.0 / K, "roofline": dec_roof},
                "prefill_ms_per_call": pre_s * 1000.0 / K,
                "roofline": roofline if prefill else dec_roof, "e2e": e2e, "cpu_baseline": cpu,
                "clocks": clocks.summary(), "gpu_launches": int(launches) * world,
                "wall_s_timed": t_wall}
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
