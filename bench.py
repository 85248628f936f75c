"""Benchmark of the paged quantized KV-cache hot path on GB300.

One step = the long-context mix: an NVFP4 paged store of 131072 tokens
(256 requests x 512, 4 KV heads, head_size 256, block_size 32, bf16 N(0,1))
followed by an indexer-K gather of 256 sequences x 512 tokens (block_size
64, head_dim 128, 8192-block cache).  Inputs are seeded synthetic arrays
copied to HBM before timing; steps run back to back with inputs larger than
L2 (the store streams 689 MB per step; the gather rotates over 8 buffer
sets).  The JSON line also carries, per kernel, the median and spread of
repeated back-to-back spans, and for every named configuration (tiny,
decode store, prefill store, prefill gather, long mix) single launches on a
clean L2 and back-to-back spans, beside the oracle timed on the host cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the host cores on a bounded sample of the same workload.  Under torchrun
each rank runs its own replica (different seeds, no data exchange): weak
scaling, the slowest rank's time counts.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("HBM GB/s (% of GB300 peak) and tokens/s for NVFP4 KV store and "
          "indexer-K gather")
WORKLOAD = ("long-context mix: NVFP4 store 131072 tokens (256 req x 512), "
            "4 KV heads, head_size 256, block_size 32, 4096-block cache + "
            "indexer-K gather 256 seqs x 512 tokens, block_size 64, "
            "head_dim 128, 8192-block cache")
FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 256 << 20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--cpu-sample-tokens", type=int, default=65536)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clock-window-s", type=float, default=1.5)
    ap.add_argument("--kernel-only",
                    choices=["store", "gather", "load", "istore", "attn"],
                    help="launch only this kernel (each launch after an L2 "
                         "flush) and print its mean time; used for ncu")
    ap.add_argument("--gather-bulk", action="store_true",
                    help="with --kernel-only gather: build and use the "
                         "library with the bulk-copy gather "
                         "(KVQ_GATHER_BULK=1) instead of the default one")
    return ap.parse_args()


# --- distributed plumbing (host side only) ------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def rank_seed(base: int, rank: int) -> int:
    """Each replica draws its own requests."""
    return base + 1000 * rank


# --- workload -------------------------------------------------------------------

def make_workload(rank: int):
    from paged_quantized_kv_gb300 import workloads as W
    st = W.store_workload(4, seed=rank_seed(4, rank))
    ga = W.gather_workload(4, seed=rank_seed(4, rank))
    return st, ga


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_sha(fname: str) -> str:
    path = os.path.join(ROOT, "paged_quantized_kv_gb300", "csrc", fname)
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(profile_md: str, src_file: str):
    """DRAM bytes per launch from a committed ncu summary, or None if the
    summary is absent or was taken on a different kernel source."""
    path = os.path.join(ROOT, "profiles", profile_md)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_sha = re.search(r"source_sha256_16:\s*([0-9a-f]+)", text)
    m_b = re.search(r"dram_bytes_per_full_launch:\s*([0-9]+)", text)
    if not (m_sha and m_b) or m_sha.group(1) != kernel_sha(src_file):
        return None
    return int(m_b.group(1))


# --- clocks ---------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,"
             "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv",
                                               delete=False)
        self.proc = None
        self.dev = device_index

    def start(self):
        import torch
        sel = []
        try:
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            sel = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50", *sel],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        rows = [r.split(",") for r in self.out.read().splitlines()
                if r.strip()]
        os.unlink(self.out.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, flag in zip(names, r[5:9]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


# --- our arm ----------------------------------------------------------------------

QUEUE_S_PER_CALL = 40e-6  # GPU sleep per queued call (host enqueue time)
GATHER_SETS = 8  # gather buffer sets rotated so no launch finds its data in
# L2 (8 x 35 MB > the 129 MB L2, even in the gather-only loop)
SPANS = 11  # timed spans per kernel leg, after one untimed warm-up span
COLD_REPS = 100  # single launches per cold (clean-L2) median


class Timer:
    """CUDA-event timing on one stream.

    ``span_ms``: mean GPU time per call of `count` back-to-back calls
    between two events.  The calls are queued behind a GPU sleep long enough
    for the host to enqueue all of them (the binding spends ~10 us of host
    time per call, more than a short kernel's GPU time, and would otherwise
    pace the GPU); the sleep runs before the first event.

    ``stats``: one untimed span (the first calls on freshly allocated
    buffers measure up to 15 % slower), then SPANS timed spans of `calls`
    calls each; median, min and max of the per-call times.

    ``cold``: single launches, each after the L2 is emptied of anything the
    call uses and left clean (a 256 MiB write, then a 256 MiB read, so the
    write's dirty lines are written back before the launch), an event on
    each side of the launch; the mean of the middle 80 % of `reps`."""

    def __init__(self, dev, stream):
        import torch
        self.torch = torch
        self.dev = dev
        self.stream = stream
        self._flush_w = None
        self._flush_r = None

    def span_ms(self, fn, count):
        torch = self.torch
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(int(2e9 * max(0.005, count * QUEUE_S_PER_CALL)))
        e0.record(self.stream)
        for i in range(count):
            fn(i)
        e1.record(self.stream)
        torch.cuda.synchronize(self.dev)
        return e0.elapsed_time(e1) / count

    def stats(self, fn, calls, spans=SPANS):
        self.span_ms(fn, calls)  # warm-up span
        ms = sorted(self.span_ms(fn, calls) for _ in range(spans))
        return {"ms": round(statistics.median(ms), 5),
                "ms_min": round(ms[0], 5), "ms_max": round(ms[-1], 5),
                "spans": spans, "calls_per_span": calls}

    def clean_l2(self, i):
        torch = self.torch
        if self._flush_w is None:
            self._flush_w = torch.empty(FLUSH_BYTES // 8, dtype=torch.int64,
                                        device=self.dev)
            self._flush_r = torch.zeros(FLUSH_BYTES // 8, dtype=torch.int64,
                                        device=self.dev)
        self._flush_w.fill_(i)
        self._flush_r.max()

    def cold(self, fn, reps=COLD_REPS):
        torch = self.torch
        ms = []
        for i in range(reps + 2):
            self.clean_l2(i)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            fn(i)
            e1.record(self.stream)
            torch.cuda.synchronize(self.dev)
            if i >= 2:
                ms.append(e0.elapsed_time(e1))
        ms.sort()
        # single-launch event times cluster about 2 us apart on this GPU, so
        # the median jumps between clusters from run to run; the mean of
        # the middle 80 % is the figure used
        k = reps // 10
        mid = ms[k:len(ms) - k]
        return {"us": round(statistics.fmean(mid) * 1e3, 2),
                "us_median": round(statistics.median(ms) * 1e3, 2),
                "us_min": round(ms[0] * 1e3, 2),
                "us_max": round(ms[-1] * 1e3, 2), "launches": reps}

    def free(self):
        self._flush_w = self._flush_r = None


def gbs(byts, ms):
    return round(byts / (ms / 1e3) / 1e9, 1)


def leg(st, byts, peak, tokens=None, tokens_key="tokens_per_s"):
    """A per-kernel record: the median time with its spread, GB/s and
    fraction of the HBM peak of the median."""
    out = dict(st)
    out["GB_s"] = gbs(byts, st["ms"])
    out["frac_of_peak"] = round(byts / (st["ms"] / 1e3) / 1e9 / peak, 4)
    if tokens is not None:
        out[tokens_key] = round(tokens / (st["ms"] / 1e3), 1)
    out["algorithmic_bytes"] = int(byts)
    return out


def store_tensors(st, kvq, dev, fill=0xAA, sets=1):
    """Device copies of a store workload: `sets` copies of the K/V source
    (and of the cache, each pre-filled with `fill`) at different addresses,
    the slots and the scales."""
    import torch
    T, H, D = st.num_tokens, st.num_heads, st.head_size
    out = []
    slots = torch.from_numpy(st.slot_mapping).to(dev)
    ks = torch.tensor([float(st.k_scale)], dtype=torch.float32, device=dev)
    vs = torch.tensor([float(st.v_scale)], dtype=torch.float32, device=dev)
    for _ in range(sets):
        src = torch.from_numpy(st.src.view(np.int16)).to(dev).view(
            torch.bfloat16)
        key = src.as_strided((T, H, D), (st.key_stride0, D, 1),
                             st.key_offset)
        value = src.as_strided((T, H, D), (st.value_stride0, D, 1),
                               st.value_offset)
        kv, kc, vc = kvq.alloc_nvfp4_cache(st.num_blocks, st.block_size, H,
                                           D, device=dev, fill=fill)
        out.append(dict(key=key, value=value, kv=kv, kc=kc, vc=vc,
                        slots=slots, ks=ks, vs=vs))
    return out


def gather_tensors(ga, dev, sets=1):
    import torch
    n = ga.total_tokens
    return [dict(cache=torch.from_numpy(ga.cache).to(dev).view(
                     ga.num_blocks, -1),
                 bt=torch.from_numpy(ga.block_table).to(dev),
                 cu=torch.from_numpy(ga.cu_seq_lens).to(dev),
                 k=torch.empty((n, ga.head_dim), dtype=torch.uint8,
                               device=dev),
                 s=torch.empty((n, 4), dtype=torch.uint8, device=dev))
            for _ in range(sets)]


def run_store(kvq, t, flags, dev_err, sh):
    kvq.kvq_store_nvfp4(t["key"], t["value"], t["kc"], t["vc"], t["slots"],
                        t["ks"], t["vs"], flags=flags, dev_error=dev_err,
                        stream=sh)


def run_gather(kvq, g, block_size, flags, dev_err, sh):
    kvq.kvq_gather_indexer_k(g["cache"], g["k"], g["s"], g["bt"], g["cu"],
                             block_size=block_size, flags=flags,
                             dev_error=dev_err, stream=sh)


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    import __graft_entry__
    __graft_entry__.build()
    from paged_quantized_kv_gb300 import kvq
    from paged_quantized_kv_gb300 import workloads as wlmod

    st, ga = make_workload(rank)
    T, H, D = st.num_tokens, st.num_heads, st.head_size

    # ---- device-resident inputs and outputs -------------------------------
    (s4,) = store_tensors(st, kvq, dev)
    n = ga.total_tokens
    gsets = gather_tensors(ga, dev, GATHER_SETS)  # same bytes, other addresses
    dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    tm = Timer(dev, stream)
    EARLY = kvq.KVQ_F_PDL_EARLY_READ
    PDL = kvq.KVQ_F_PDL

    def store(flags):
        run_store(kvq, s4, flags, dev_err, sh)

    def gather(i, flags):
        run_gather(kvq, gsets[i % GATHER_SETS], ga.block_size, flags,
                   dev_err, sh)

    def step(i, flags):
        store(EARLY if flags else 0)
        gather(i, EARLY if flags else 0)

    W = max(args.warmup, 3)
    for i in range(W):
        step(i, PDL)
        step(i, 0)
    torch.cuda.synchronize(dev)

    # ---- timed region: K steps back to back -------------------------------
    K = args.steps
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.2)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    step_ms = tm.span_ms(lambda i: step(i, PDL), K)
    if world > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - t0
    # the same K-step span repeated, for its spread
    step_rep = sorted(tm.span_ms(lambda i: step(i, PDL), K) for _ in range(5))
    peak, peak_kind = measured_hbm_peak()
    st_bytes = st.algorithmic_bytes()
    ga_bytes = ga.algorithmic_bytes()

    # ---- per-kernel legs: SPANS spans each, median and spread -------------
    # (inputs larger than L2: the store streams 689 MB per call; the gather
    # rotates over GATHER_SETS buffer sets)
    store_st = tm.stats(lambda i: store(EARLY), 20)
    store_pdl = tm.stats(lambda i: store(PDL), 20)
    gather_st = tm.stats(lambda i: gather(i, EARLY), 200)
    gather_meta = tm.stats(lambda i: gather(i, kvq.KVQ_F_PDL_EARLY_META), 200)
    plain = {"step": tm.stats(lambda i: step(i, 0), 20),
             "store": tm.stats(lambda i: store(0), 20),
             "gather": tm.stats(lambda i: gather(i, 0), 200)}
    # the store's other input type and cache layout, same shape
    key16 = s4["key"].to(torch.float16)
    value16 = s4["value"].to(torch.float16)
    kv_n, kc_n, vc_n = kvq.alloc_nvfp4_cache(
        st.num_blocks, st.block_size, H, D, layout=kvq.KVQ_LAYOUT_NHD,
        device=dev, fill=0xAA)
    variants = {
        "store_fp16_hnd": tm.stats(lambda i: kvq.kvq_store_nvfp4(
            key16, value16, s4["kc"], s4["vc"], s4["slots"], s4["ks"],
            s4["vs"], flags=PDL, dev_error=dev_err, stream=sh), 20),
        "store_bf16_nhd": tm.stats(lambda i: kvq.kvq_store_nvfp4(
            s4["key"], s4["value"], kc_n, vc_n, s4["slots"], s4["ks"],
            s4["vs"], flags=PDL, dev_error=dev_err, stream=sh), 20),
    }
    del key16, value16, kv_n, kc_n, vc_n
    # the read side: the long-context pages read back to bf16 rows
    lbt, lcu = wlmod.sequences_of_store(st, 512)
    lbt_d = torch.from_numpy(lbt).to(dev)
    lcu_d = torch.from_numpy(lcu).to(dev)
    k_out = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
    v_out = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
    load_st = tm.stats(lambda i: kvq.kvq_load_nvfp4(
        s4["kc"], s4["vc"], lbt_d, lcu_d, s4["ks"], s4["vs"], k_out, v_out,
        flags=kvq.KVQ_F_PDL_EARLY_META, dev_error=dev_err, stream=sh), 20)
    load_bytes = wlmod.load_algorithmic_bytes(st, lbt, lcu)
    del k_out, v_out
    # the indexer cache's write side on the gather's shape (K rows rotated
    # over GATHER_SETS copies: 33.5 MB each, none L2-resident at launch)
    iw = wlmod.make_indexer_store("long_indexer_store", rank_seed(4, rank),
                                  [512] * 256, 64, 128, 8192)
    ik = [torch.from_numpy(iw.k.view(np.int16)).to(dev).view(torch.bfloat16)
          for _ in range(GATHER_SETS)]
    islots = torch.from_numpy(iw.slot_mapping).to(dev)
    icache = torch.empty((iw.num_blocks, iw.block_size, iw.head_dim + 4),
                         dtype=torch.uint8, device=dev)
    istore_st = tm.stats(lambda i: kvq.kvq_store_indexer_k(
        ik[i % GATHER_SETS], icache, islots, flags=EARLY, dev_error=dev_err,
        stream=sh), 200)
    istore_pdl = tm.stats(lambda i: kvq.kvq_store_indexer_k(
        ik[i % GATHER_SETS], icache, islots, flags=PDL, dev_error=dev_err,
        stream=sh), 200)
    istore_bytes = iw.algorithmic_bytes()
    del ik, icache
    # decode attention over NVFP4 pages: one step of Llama-3.1-70B-shaped
    # attention (200 sequences, 64 query / 8 KV heads, contexts 512..2560;
    # 359 MB of pages per call, larger than L2)
    aw = wlmod.attention_workload(rank_seed(5, rank))
    attn = attention_inputs(aw, kvq, dev)
    # back to back with early metadata reads: the kernel before each call
    # is the previous call's partition merge, which writes only the output
    early = kvq.KVQ_F_PDL_EARLY_META
    attn_st = tm.stats(
        lambda i: run_attention(attn, kvq, early, dev_err, sh), 25)
    attn_bytes = aw.algorithmic_bytes()
    attn_ctx = int(aw.context_lens.astype(np.int64).sum())
    del attn
    # the same step on NHD pages (the same bytes read in that layout)
    attn = attention_inputs(
        dataclasses.replace(aw, layout=wlmod.LAYOUT_NHD), kvq, dev)
    attn_nhd_st = tm.stats(
        lambda i: run_attention(attn, kvq, early, dev_err, sh), 25)
    del attn
    # keep the same steps running so the clock sampler sees the load
    t1 = time.perf_counter()
    j = 0
    while time.perf_counter() - t1 < args.clock_window_s:
        step(j, PDL)
        j += 1
        if j % 50 == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    assert int(dev_err.item()) == 0, "device error flag raised"

    # ---- each named configuration on its own ------------------------------
    configs = config_legs(kvq, wlmod, tm, dev, dev_err, sh, peak, rank,
                          long_step=dict(store=(lambda i: store(0), st_bytes),
                                         gather=(lambda i: gather(i, 0),
                                                 ga_bytes)))
    tm.free()
    assert int(dev_err.item()) == 0, "device error flag raised"

    step_s = max_over_ranks(step_ms / 1e3, world, dev)
    total_bytes = sum_over_ranks(float(st_bytes + ga_bytes), world, dev)
    total_tokens = sum_over_ranks(float(T + n), world, dev)
    store_gbs = st_bytes / (store_st["ms"] / 1e3) / 1e9
    traffic = profiled_traffic("store_nvfp4_long.md", "store_nvfp4.cu")

    e2e = run_e2e(args, st, ga, dev, kvq)

    line = {
        "metric": METRIC,
        "value": round(total_bytes / step_s / 1e9, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(step_s * 1e3, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": WORKLOAD,
            "store": {"tokens": T, "num_heads": H, "head_size": D,
                      "block_size": st.block_size,
                      "num_blocks": st.num_blocks, "layout": "HND",
                      "io": "bf16 in, e2m1 data + e4m3 scales out"},
            "gather": {"seqs": ga.num_seqs, "tokens": n,
                       "block_size": ga.block_size,
                       "head_dim": ga.head_dim,
                       "num_blocks": ga.num_blocks, "io": "u8 copy"},
            "l2": "inputs larger than L2: each step streams the store's "
                  "537 MB of bf16 K/V and 151 MB of pages; the gather "
                  f"rotates over {GATHER_SETS} buffer sets (35 MB each, "
                  f"{GATHER_SETS * 35} MB in all), so no launch finds its "
                  "data in L2",
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
            "timing": "K steps (store and gather both with "
                      "KVQ_F_PDL_EARLY_READ: the gather writes none of the "
                      "store's inputs, the store none of the gather's) back "
                      "to back on one stream "
                      "between two CUDA events, all K queued behind a GPU "
                      "sleep before the first event (so the binding's host "
                      "time per call does not pace the GPU); ms_per_step = "
                      "span / K, max over ranks.  Per-kernel legs: one "
                      f"untimed span, then {SPANS} spans of back-to-back "
                      "calls of that kernel alone, queued the same way; "
                      "ms = the median span's time per call, with the min "
                      "and max",
        },
        "ms_per_step_spans": {
            "ms": round(statistics.median(step_rep), 5),
            "ms_min": round(step_rep[0], 5), "ms_max": round(step_rep[-1], 5),
            "spans": len(step_rep), "calls_per_span": K},
        "tokens_per_s": round(total_tokens / step_s, 1),
        "kernels": {
            "store_nvfp4": dict(
                leg(store_st, st_bytes, peak, T),
                pdl_only=leg(store_pdl, st_bytes, peak)),
            "gather_indexer_k": dict(
                leg(gather_st, ga_bytes, peak, n),
                early_meta_only=leg(gather_meta, ga_bytes, peak)),
        },
        "without_pdl": {k: leg(v, st_bytes + ga_bytes if k == "step" else
                               st_bytes if k == "store" else ga_bytes, peak)
                        for k, v in plain.items()},
        "load_nvfp4": dict(
            leg(load_st, load_bytes, peak, T),
            note="read side: the long-context pages read back to bf16 "
                 "rows through the block table (not part of the step)"),
        "store_variants": {k: leg(v, st_bytes, peak)
                           for k, v in variants.items()},
        "store_indexer_k": dict(
            leg(istore_st, istore_bytes, peak, iw.num_tokens),
            pdl_only=leg(istore_pdl, istore_bytes, peak),
            note="write side of the indexer cache on the gather's shape "
                 "(131072 tokens, head_dim 128, block_size 64), not part "
                 "of the step; back to back with KVQ_F_PDL_EARLY_READ (K "
                 "rotated over the buffer sets, the kernel before writes "
                 "only the cache)"),
        "paged_attention_nvfp4": dict(
            leg(attn_st, attn_bytes, peak, aw.num_seqs,
                "decode_tokens_per_s"),
            context_tokens_per_s=round(attn_ctx / (attn_st["ms"] / 1e3), 1),
            note="decode attention over the NVFP4 pages, one step of "
                 "Llama-3.1-70B-shaped attention: 200 sequences, 64 query / "
                 "8 KV heads, head_size 128, block_size 16, contexts 512 + "
                 "U[0, 2048]; partition_size 512 (on these contiguous "
                 "pages a context splits into ceil(L / 1792) stretches in "
                 "the proportions 4 : ... : 4 : 1, one CTA each, launched "
                 "stretch-major, then the partition merge); back to back "
                 "with KVQ_F_PDL_EARLY_META (the kernel before each call is "
                 "the previous call's partition merge, which writes only "
                 "the output); not part of the step"),
        "paged_attention_nvfp4_nhd": dict(
            leg(attn_nhd_st, attn_bytes, peak, aw.num_seqs,
                "decode_tokens_per_s"),
            note="the same attention step on NHD pages (block_size 16: a "
                 "head's token rows 8 rows apart, copied row by row); not "
                 "part of the step"),
        "configs": configs,
        "roofline": {
            "bound": "hbm",
            "kernel": "store_nvfp4",
            "achieved": round(store_gbs, 1),
            "peak": peak,
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                           if peak_kind == "measured" else "fallback 6.8 TB/s",
            "unit": "GB/s",
            "frac": round(store_gbs / peak, 4),
            "traffic": traffic,
        },
        "wall_s_timed_region": round(wall, 4),
        "e2e": e2e,
        "gpu_launches": 2 * K,
        "gpu_launches_note": "in the timed step region (store + gather per "
                             "step); the legs after it launch their own",
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(st, ga, args.cpu_sample_tokens)
        line["paged_attention_nvfp4"]["cpu_oracle"] = cpu_attention_baseline(
            aw)
        cpu_config_legs(configs, rank)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def config_legs(kvq, wlmod, tm, dev, dev_err, sh, peak, rank, long_step):
    """Every named configuration timed alone: single launches after a clean
    L2 flush (COLD_REPS of them) and back-to-back spans (median of SPANS),
    beside the floor of an empty launch measured the same way."""
    import torch
    EARLY = kvq.KVQ_F_PDL_EARLY_READ
    out = {}
    floor = tm.cold(lambda i: torch.cuda._sleep(0))
    floor_b2b = tm.stats(lambda i: torch.cuda._sleep(0), 200)
    out["empty_launch_floor"] = {
        "cold_single_launch": floor,
        "back_to_back_us": round(floor_b2b["ms"] * 1e3, 3),
        "note": "a zero-length kernel timed the same two ways: what any "
                "single launch measured with events costs at least"}

    def store_cfg(idx, name, sets, calls, note):
        st = wlmod.store_workload(idx, seed=rank_seed(idx, rank))
        ts = store_tensors(st, kvq, dev, sets=sets)
        byts = st.algorithmic_bytes()
        cold = tm.cold(lambda i: run_store(kvq, ts[i % sets], 0, dev_err, sh))
        b2b = tm.stats(lambda i: run_store(kvq, ts[i % sets], EARLY, dev_err,
                                           sh), calls)
        rec = {"kernel": "store_nvfp4", "tokens": st.num_tokens,
               "stored_tokens": st.stored_tokens,
               "algorithmic_bytes": int(byts),
               "cold_single_launch": dict(
                   cold, GB_s=gbs(byts, cold["us"] / 1e3),
                   frac_of_peak=round(byts / cold["us"] / 1e3 / peak, 4)),
               "back_to_back": leg(b2b, byts, peak, st.stored_tokens),
               "note": note}
        out[name] = rec
        del ts

    def gather_cfg(idx, name, sets, calls, note):
        ga = wlmod.gather_workload(idx, seed=rank_seed(idx, rank))
        gs = gather_tensors(ga, dev, sets)
        byts = ga.algorithmic_bytes()
        cold = tm.cold(lambda i: run_gather(kvq, gs[i % sets], ga.block_size,
                                            0, dev_err, sh))
        b2b = tm.stats(lambda i: run_gather(kvq, gs[i % sets], ga.block_size,
                                            EARLY, dev_err, sh), calls)
        out[name] = {"kernel": "gather_indexer_k", "seqs": ga.num_seqs,
                     "tokens": ga.total_tokens,
                     "algorithmic_bytes": int(byts),
                     "cold_single_launch": dict(
                         cold, GB_s=gbs(byts, cold["us"] / 1e3),
                         frac_of_peak=round(byts / cold["us"] / 1e3 / peak,
                                            4)),
                     "back_to_back": leg(b2b, byts, peak, ga.total_tokens),
                     "note": note}
        del gs

    store_cfg(0, "0_tiny_store", 1, 200,
              "24 tokens (3 skipped), 2 heads, head_size 64: launch-bound; "
              "back to back the inputs stay in L2")
    gather_cfg(0, "0_tiny_gather", 1, 200,
               "sequences of 5 and 37 tokens: launch-bound; back to back "
               "the inputs stay in L2")
    store_cfg(1, "1_decode_store", 1, 200,
              "256 single-token requests, 8 KV heads, head_size 128, "
              "random slots over a 65536-block cache: launch-bound (1.35 "
              "MB); back to back the 1 MB of K/V and the written lines stay "
              "in L2 (warm), the cold single launch reads from HBM")
    store_cfg(2, "2_prefill_store", 3, 40,
              "16 requests x 1024 tokens, 8 KV heads, head_size 128, rows "
              "2x strided; back to back over 3 input/cache sets (201 MB of "
              "K/V, none L2-resident at launch)")
    gather_cfg(3, "3_prefill_gather", GATHER_SETS, 200,
               "16 sequences of U[1000, 8192] tokens, block_size 64, "
               "head_dim 128; back to back over 8 buffer sets (a 35 MB "
               "cache and 10 MB of outputs each)")
    # the long-context mix's two kernels, cold (launch, algorithmic bytes)
    for key, (fn, byts) in (("4_long_store", long_step["store"]),
                            ("4_long_gather", long_step["gather"])):
        cold = tm.cold(fn)
        out[key] = {"algorithmic_bytes": int(byts),
                    "cold_single_launch": dict(
                        cold, GB_s=gbs(byts, cold["us"] / 1e3),
                        frac_of_peak=round(byts / cold["us"] / 1e3 / peak,
                                           4)),
                    "back_to_back": "kernels.store_nvfp4 / "
                                    "kernels.gather_indexer_k"}
    return out


def cpu_config_legs(configs, rank):
    """The oracle on each named configuration's full inputs, one thread and
    every host core (store split by tokens, gather by sequences)."""
    import oracle
    from paged_quantized_kv_gb300 import workloads as wlmod
    o = oracle.get()
    threads = max(1, os.cpu_count() or 1)
    for name, idx, kind in (("0_tiny_store", 0, "store"),
                            ("0_tiny_gather", 0, "gather"),
                            ("1_decode_store", 1, "store"),
                            ("2_prefill_store", 2, "store"),
                            ("3_prefill_gather", 3, "gather")):
        rec = configs.get(name)
        if rec is None:
            continue
        if kind == "store":
            st = wlmod.store_workload(idx, seed=rank_seed(idx, rank))
            ga = oracle_empty_gather(wlmod.gather_workload(0))
        else:
            ga = wlmod.gather_workload(idx, seed=rank_seed(idx, rank))
            st = oracle_empty_store(wlmod.store_workload(0))
        res = {"kind": "oracle"}
        for label, nt in (("one_thread", 1), ("all_cores", threads)):
            cache = np.full(st.cache_bytes, 0xAA, dtype=np.uint8)
            k = np.empty(max(ga.total_tokens, 1) * ga.head_dim, np.uint8)
            s = np.empty(max(ga.total_tokens, 1) * 4, np.uint8)
            t = time.perf_counter()
            oracle_step_threaded(o, st, ga, cache, k, s, nt)
            dt = time.perf_counter() - t
            res[label] = {"seconds": round(dt, 5), "cores": nt,
                          "GB_s": round(rec["algorithmic_bytes"] / dt / 1e9,
                                        4)}
            del cache
        rec["cpu_oracle"] = res


def oracle_empty_store(st):
    """A store workload with no tokens (the other half of a one-kernel
    oracle leg)."""
    from paged_quantized_kv_gb300 import workloads as W
    return W.StoreWorkload(
        name="none", num_tokens=0, num_heads=st.num_heads,
        head_size=st.head_size, block_size=st.block_size, num_blocks=1,
        src=st.src, key_offset=0, key_stride0=st.key_stride0, value_offset=0,
        value_stride0=st.value_stride0,
        slot_mapping=np.zeros(0, np.int64), k_scale=st.k_scale,
        v_scale=st.v_scale)


def oracle_empty_gather(ga):
    from paged_quantized_kv_gb300 import workloads as W
    return W.GatherWorkload(
        name="none", block_size=ga.block_size, head_dim=ga.head_dim,
        num_blocks=ga.num_blocks, cache=ga.cache,
        block_table=ga.block_table[:0], cu_seq_lens=np.zeros(1, np.int32),
        block_stride=ga.block_stride)


def attention_inputs(aw, kvq, dev):
    """Device copies of an attention workload's inputs, output and
    scratch."""
    import torch
    kv, kc, vc = kvq.alloc_nvfp4_cache(aw.num_blocks, aw.block_size,
                                       aw.num_kv_heads, aw.head_size,
                                       aw.layout, device=dev)
    kv.view(-1).copy_(torch.from_numpy(aw.cache))
    q = torch.from_numpy(aw.query.view(np.int16)).to(dev).view(torch.bfloat16)
    mcl = int(aw.context_lens.max())
    return dict(kv=kv, kc=kc, vc=vc, q=q, out=torch.empty_like(q),
                bt=torch.from_numpy(aw.block_table).to(dev),
                lens=torch.from_numpy(aw.context_lens).to(dev),
                ks=torch.tensor([float(aw.k_scale)], device=dev),
                vs=torch.tensor([float(aw.v_scale)], device=dev),
                scale=float(aw.scale), mcl=mcl,
                scratch=kvq.attention_scratch(aw.num_seqs, aw.num_q_heads,
                                              mcl, 512, aw.head_size, dev))


def run_attention(a, kvq, flags, dev_err, stream):
    es, ml, tmp = a["scratch"]
    kvq.kvq_paged_attention_nvfp4(
        a["q"], a["kc"], a["vc"], a["bt"], a["lens"], a["ks"], a["vs"],
        a["scale"], a["out"], a["mcl"], 512, es, ml, tmp, flags=flags,
        dev_error=dev_err, stream=stream)


def run_e2e(args, st, ga, dev, kvq):
    """Same step through the public binding with pinned HOST buffers: every
    step copies its inputs host->device, runs both calls, and reads the
    gathered rows and the written cache pages back to the host.  Steps are
    pipelined on three streams -- copy-in (double-buffered inputs),
    compute, copy-out -- with events, so step i's copy-out overlaps step
    i+1's copy-in; a store waits for the previous step's page copy-out, a
    gather for its row copy-out."""
    import torch
    T, H, D = st.num_tokens, st.num_heads, st.head_size
    h_src = torch.from_numpy(st.src.view(np.int16)).pin_memory()
    h_slots = torch.from_numpy(st.slot_mapping).pin_memory()
    h_scales = torch.tensor([float(st.k_scale), float(st.v_scale)],
                            dtype=torch.float32).pin_memory()
    h_bt = torch.from_numpy(ga.block_table).pin_memory()
    h_cu = torch.from_numpy(ga.cu_seq_lens).pin_memory()
    n = ga.total_tokens
    h_k = torch.empty((n, ga.head_dim), dtype=torch.uint8).pin_memory()
    h_s = torch.empty((n, 4), dtype=torch.uint8).pin_memory()
    kv, kc, vc = kvq.alloc_nvfp4_cache(st.num_blocks, st.block_size, H, D,
                                       device=dev, fill=0xAA)
    h_cache = torch.empty(kv.shape, dtype=torch.uint8).pin_memory()
    ins = [dict(src=torch.empty(h_src.shape, dtype=torch.int16, device=dev),
                slots=torch.empty_like(h_slots, device=dev),
                scales=torch.empty(2, dtype=torch.float32, device=dev),
                bt=torch.empty_like(h_bt, device=dev),
                cu=torch.empty_like(h_cu, device=dev)) for _ in range(2)]
    gcache = torch.from_numpy(ga.cache).to(dev).view(ga.num_blocks, -1)
    k_fp8 = torch.empty((n, ga.head_dim), dtype=torch.uint8, device=dev)
    k_scale = torch.empty((n, 4), dtype=torch.uint8, device=dev)
    s_in, s_cp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = lambda: torch.cuda.Event(enable_timing=False)
    state = {"out_done": None, "comp_done": [None, None]}

    def step(i):
        b = ins[i % 2]
        with torch.cuda.stream(s_in):
            if state["comp_done"][i % 2] is not None:  # buffer reuse
                s_in.wait_event(state["comp_done"][i % 2])
            b["src"].copy_(h_src, non_blocking=True)
            b["slots"].copy_(h_slots, non_blocking=True)
            b["scales"].copy_(h_scales, non_blocking=True)
            b["bt"].copy_(h_bt, non_blocking=True)
            b["cu"].copy_(h_cu, non_blocking=True)
            in_done = ev()
            in_done.record(s_in)
        with torch.cuda.stream(s_cp):
            s_cp.wait_event(in_done)
            if state["out_done"] is not None:  # pages / rows read back
                s_cp.wait_event(state["out_done"])
            src = b["src"].view(torch.bfloat16)
            key = src.as_strided((T, H, D), (st.key_stride0, D, 1),
                                 st.key_offset)
            value = src.as_strided((T, H, D), (st.value_stride0, D, 1),
                                   st.value_offset)
            kvq.kvq_store_nvfp4(key, value, kc, vc, b["slots"],
                                b["scales"][0:1], b["scales"][1:2],
                                stream=s_cp.cuda_stream)
            kvq.kvq_gather_indexer_k(gcache, k_fp8, k_scale, b["bt"],
                                     b["cu"], block_size=ga.block_size,
                                     stream=s_cp.cuda_stream)
            comp = ev()
            comp.record(s_cp)
            state["comp_done"][i % 2] = comp
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp)
            h_k.copy_(k_fp8, non_blocking=True)
            h_s.copy_(k_scale, non_blocking=True)
            h_cache.copy_(kv, non_blocking=True)
            out = ev()
            out.record(s_out)
            state["out_done"] = out

    for i in range(2):
        step(i)
    torch.cuda.synchronize(dev)
    E = max(args.e2e_steps, 1)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(E):
        step(i)
    s_in.wait_stream(s_out)
    e1.record(s_in)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / E
    h2d = (h_src.numel() * 2 + h_slots.numel() * 8 + 8 + h_bt.numel() * 4
           + h_cu.numel() * 4)
    d2h = h_k.numel() + h_s.numel() + h_cache.numel()
    byts = st.algorithmic_bytes() + ga.algorithmic_bytes()
    return {"value": round(byts / (ms / 1e3) / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": E,
            "note": "pinned host buffers; copy-in, compute and copy-out "
                    "pipelined across steps on three streams; the host link "
                    "measures ~210 GB/s host->device and ~193 GB/s "
                    "device->host per direction on this system"}


# --- CPU oracle legs ----------------------------------------------------------------

def oracle_sample(st, ga, sample_tokens):
    """A bounded slice of the workload: the first requests of the store and
    the first sequences of the gather, same shapes and distributions."""
    from paged_quantized_kv_gb300 import workloads as W
    T = min(sample_tokens, st.num_tokens)
    sub = W.StoreWorkload(
        name="sample", num_tokens=T, num_heads=st.num_heads,
        head_size=st.head_size, block_size=st.block_size,
        num_blocks=st.num_blocks, src=st.src, key_offset=st.key_offset,
        key_stride0=st.key_stride0, value_offset=st.value_offset,
        value_stride0=st.value_stride0, slot_mapping=st.slot_mapping[:T],
        k_scale=st.k_scale, v_scale=st.v_scale, layout=st.layout,
        flags=st.flags)
    n_seq = max(1, (ga.num_seqs * T) // st.num_tokens)
    cu = ga.cu_seq_lens[: n_seq + 1].copy()
    gsub = W.GatherWorkload(
        name="sample", block_size=ga.block_size, head_dim=ga.head_dim,
        num_blocks=ga.num_blocks, cache=ga.cache,
        block_table=ga.block_table[:n_seq], cu_seq_lens=cu,
        block_stride=ga.block_stride)
    return sub, gsub


def oracle_step(o, sub, gsub, cache, k, s):
    o.store_nvfp4(sub.src, sub.key_stride0, sub.src, sub.value_stride0,
                  sub.num_tokens, sub.num_heads, sub.head_size, cache, 0,
                  sub.value_side_offset, sub.page_stride, sub.block_size,
                  sub.num_blocks, sub.layout, sub.slot_mapping, sub.k_scale,
                  sub.v_scale, sub.flags, key_base=sub.key_offset,
                  value_base=sub.value_offset)
    o.gather_indexer_k(gsub.cache, gsub.block_stride, gsub.num_blocks,
                       gsub.block_size, gsub.head_dim, gsub.block_table,
                       gsub.cu_seq_lens, gsub.total_tokens, k, s)


def cpu_baseline(st, ga, sample_tokens):
    import oracle
    o = oracle.get()
    sub, gsub = oracle_sample(st, ga, sample_tokens)
    cache = np.full(sub.cache_bytes, 0xAA, dtype=np.uint8)
    k = np.empty(gsub.total_tokens * gsub.head_dim, dtype=np.uint8)
    s = np.empty(gsub.total_tokens * 4, dtype=np.uint8)
    t = time.perf_counter()
    oracle_step(o, sub, gsub, cache, k, s)
    dt = time.perf_counter() - t
    byts = sub.algorithmic_bytes() + gsub.algorithmic_bytes()
    return {"value": round(byts / dt / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle",
            "seconds": round(dt, 3),
            "sample": f"first {sub.num_tokens} store tokens "
                      f"({sub.num_tokens // 512} requests) and first "
                      f"{gsub.num_seqs} gather sequences of the same "
                      f"workload, single-threaded plain C oracle",
            "all_cores": cpu_baseline_all_cores(o, sub, gsub, byts)}


def oracle_step_threaded(o, sub, gsub, cache, k, s, threads):
    """`oracle_step` with the oracle's calls split over `threads` host
    threads: the store by tokens (slots are distinct, so the pieces write
    disjoint bytes), the gather by sequences (each piece writes its own rows).
    The oracle is unchanged; each thread calls it on its own piece (ctypes
    releases the GIL during the call)."""
    import concurrent.futures as cf
    D = gsub.head_dim
    cu = gsub.cu_seq_lens.astype(np.int64)

    def store_piece(c):
        t0 = sub.num_tokens * c // threads
        t1 = sub.num_tokens * (c + 1) // threads
        if t1 > t0:
            o.store_nvfp4(sub.src, sub.key_stride0, sub.src, sub.value_stride0,
                          t1 - t0, sub.num_heads, sub.head_size, cache, 0,
                          sub.value_side_offset, sub.page_stride,
                          sub.block_size, sub.num_blocks, sub.layout,
                          sub.slot_mapping[t0:t1], sub.k_scale, sub.v_scale,
                          sub.flags,
                          key_base=sub.key_offset + t0 * sub.key_stride0,
                          value_base=sub.value_offset + t0 * sub.value_stride0)

    def gather_piece(c):
        b0 = gsub.num_seqs * c // threads
        b1 = gsub.num_seqs * (c + 1) // threads
        if b1 > b0:
            r0, r1 = int(cu[b0]), int(cu[b1])
            o.gather_indexer_k(gsub.cache, gsub.block_stride, gsub.num_blocks,
                               gsub.block_size, D,
                               np.ascontiguousarray(gsub.block_table[b0:b1]),
                               (cu[b0:b1 + 1] - r0).astype(np.int32),
                               r1 - r0, k[r0 * D:r1 * D], s[r0 * 4:r1 * 4])

    with cf.ThreadPoolExecutor(threads) as ex:
        list(ex.map(store_piece, range(threads)))
        list(ex.map(gather_piece, range(threads)))


def cpu_baseline_all_cores(o, sub, gsub, byts):
    """The single-thread sample again, split over every host core."""
    threads = max(1, os.cpu_count() or 1)
    cache = np.full(sub.cache_bytes, 0xAA, dtype=np.uint8)
    k = np.empty(gsub.total_tokens * gsub.head_dim, dtype=np.uint8)
    s = np.empty(gsub.total_tokens * 4, dtype=np.uint8)
    t = time.perf_counter()
    oracle_step_threaded(o, sub, gsub, cache, k, s, threads)
    dt = time.perf_counter() - t
    return {"value": round(byts / dt / 1e9, 4), "unit": "GB/s",
            "cores": threads, "seconds": round(dt, 3),
            "sample": "the same sample, store tokens and gather sequences "
                      f"split evenly over {threads} threads"}


def cpu_attention_baseline(aw, nseq=4):
    """The attention oracle (plain C, double, one thread) on the first
    `nseq` sequences of the attention workload: algorithmic GB/s and
    context tokens/s of that sample."""
    import oracle
    from paged_quantized_kv_gb300 import workloads as wlmod
    o = oracle.get()
    sub = wlmod.AttentionWorkload(
        name="sample", query=aw.query[:nseq], num_kv_heads=aw.num_kv_heads,
        block_size=aw.block_size, num_blocks=aw.num_blocks, cache=aw.cache,
        block_table=aw.block_table[:nseq],
        context_lens=aw.context_lens[:nseq], k_scale=aw.k_scale,
        v_scale=aw.v_scale, scale=aw.scale)
    t = time.perf_counter()
    o.paged_attention_nvfp4(sub.query, sub.cache, 0, sub.side_bytes,
                            sub.page_stride, sub.block_size, sub.num_blocks,
                            sub.layout, sub.num_kv_heads, sub.block_table,
                            sub.context_lens, sub.k_scale, sub.v_scale,
                            sub.scale, 0, sub.dtype)
    dt = time.perf_counter() - t
    ctx = int(sub.context_lens.astype(np.int64).sum())
    return {"value": round(sub.algorithmic_bytes() / dt / 1e9, 4),
            "unit": "GB/s", "cores": 1, "kind": "oracle",
            "seconds": round(dt, 3),
            "context_tokens_per_s": round(ctx / dt, 1),
            "sample": f"first {nseq} sequences ({ctx} context tokens, all "
                      f"{aw.num_q_heads} query heads) of the same step, "
                      "single-threaded plain C oracle in double"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return  # the reference arm runs on rank 0 only
    import oracle
    st, ga = make_workload(0)
    o = oracle.get()
    sub, gsub = oracle_sample(st, ga, 4096)
    cache = np.full(sub.cache_bytes, 0xAA, dtype=np.uint8)
    k = np.empty(gsub.total_tokens * gsub.head_dim, dtype=np.uint8)
    s = np.empty(gsub.total_tokens * 4, dtype=np.uint8)
    for _ in range(max(args.warmup, 3)):
        oracle_step(o, sub, gsub, cache, k, s)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(o, sub, gsub, cache, k, s)
    dt = (time.perf_counter() - t) / max(args.steps, 1)
    byts = sub.algorithmic_bytes() + gsub.algorithmic_bytes()
    val = round(byts / dt / 1e9, 4)
    sample = (f"per step: first {sub.num_tokens} store tokens and first "
              f"{gsub.num_seqs} gather sequences of the workload")
    print(json.dumps({
        "impl": "reference",
        "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": val, "unit": "GB/s", "cores": 1,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def run_kernel_only(args):
    """One kernel of the long-context mix, warmup + steps launches, each
    after a 256 MiB L2 flush; prints the mean CUDA-event time."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from paged_quantized_kv_gb300 import kvq
    if args.gather_bulk:
        from paged_quantized_kv_gb300 import build as kbuild
        kvq.LIB_PATH = kbuild.build(
            defines={"KVQ_GATHER_BULK": 1},
            out=os.path.join(tempfile.gettempdir(), "libkvq_gather_bulk.so"))
        kvq._lib = None
    dev = torch.device("cuda", 0)
    st, ga = make_workload(0)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    if args.kernel_only in ("store", "load"):
        T, H, D = st.num_tokens, st.num_heads, st.head_size
        src = torch.from_numpy(st.src.view(np.int16)).to(dev).view(
            torch.bfloat16)
        key = src.as_strided((T, H, D), (st.key_stride0, D, 1),
                             st.key_offset)
        value = src.as_strided((T, H, D), (st.value_stride0, D, 1),
                               st.value_offset)
        slots = torch.from_numpy(st.slot_mapping).to(dev)
        ks = torch.tensor([float(st.k_scale)], device=dev)
        vs = torch.tensor([float(st.v_scale)], device=dev)
        kv, kc, vc = kvq.alloc_nvfp4_cache(st.num_blocks, st.block_size, H,
                                           D, device=dev, fill=0xAA)

        def launch():
            kvq.kvq_store_nvfp4(key, value, kc, vc, slots, ks, vs)
        byts = st.algorithmic_bytes()
        if args.kernel_only == "load":
            from paged_quantized_kv_gb300 import workloads as wlmod
            launch()  # pages to read back
            lbt, lcu = wlmod.sequences_of_store(st, 512)
            lbt_d = torch.from_numpy(lbt).to(dev)
            lcu_d = torch.from_numpy(lcu).to(dev)
            k_out = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
            v_out = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
            del key, value, src

            def launch():
                kvq.kvq_load_nvfp4(kc, vc, lbt_d, lcu_d, ks, vs, k_out,
                                   v_out)
            byts = wlmod.load_algorithmic_bytes(st, lbt, lcu)
    elif args.kernel_only == "istore":
        from paged_quantized_kv_gb300 import workloads as wlmod
        iw = wlmod.make_indexer_store("long_indexer_store", 4, [512] * 256,
                                      64, 128, 8192)
        ik = torch.from_numpy(iw.k.view(np.int16)).to(dev).view(
            torch.bfloat16)
        islots = torch.from_numpy(iw.slot_mapping).to(dev)
        icache = torch.empty((iw.num_blocks, iw.block_size, iw.head_dim + 4),
                             dtype=torch.uint8, device=dev)

        def launch():
            kvq.kvq_store_indexer_k(ik, icache, islots)
        byts = iw.algorithmic_bytes()
    elif args.kernel_only == "attn":
        from paged_quantized_kv_gb300 import workloads as wlmod
        aw = wlmod.attention_workload(5)
        attn = attention_inputs(aw, kvq, dev)

        def launch():
            run_attention(attn, kvq, 0, None, None)
        byts = aw.algorithmic_bytes()
    else:
        gcache = torch.from_numpy(ga.cache).to(dev).view(ga.num_blocks, -1)
        bt = torch.from_numpy(ga.block_table).to(dev)
        cu = torch.from_numpy(ga.cu_seq_lens).to(dev)
        n = ga.total_tokens
        k_fp8 = torch.empty((n, ga.head_dim), dtype=torch.uint8, device=dev)
        k_scale = torch.empty((n, 4), dtype=torch.uint8, device=dev)

        def launch():
            kvq.kvq_gather_indexer_k(gcache, k_fp8, k_scale, bt, cu,
                                     block_size=ga.block_size)
        byts = ga.algorithmic_bytes()
    for i in range(args.warmup):
        flush.fill_(i & 0xFF)
        launch()
    ms = []
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        launch()
        e1.record()
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    mean = statistics.fmean(ms)
    print(json.dumps({"kernel": args.kernel_only, "ms": round(mean, 5),
                      "GB_s": round(byts / (mean / 1e3) / 1e9, 1),
                      "launches": args.warmup + args.steps}), flush=True)


def main():
    args = parse_args()
    if args.kernel_only:
        run_kernel_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
