"""Benchmark of the paged quantized KV-cache hot path on GB300.

One step = the long-context mix: an NVFP4 paged store of 131072 tokens
(256 requests x 512, 4 KV heads, head_size 256, block_size 32, bf16 N(0,1))
followed by an indexer-K gather of 256 sequences x 512 tokens (block_size
64, head_dim 128, 8192-block cache).  Inputs are seeded synthetic arrays
copied to HBM before timing; steps run back to back with inputs larger than
L2 (the store streams 689 MB per step; the gather rotates over 4 buffer
sets).  The JSON line also carries single-launch times after an L2 flush.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the host cores on a bounded sample of the same workload.  Under torchrun
each rank runs its own replica (different seeds, no data exchange): weak
scaling, the slowest rank's time counts.
"""
from __future__ import annotations

import argparse
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

    st, ga = make_workload(rank)
    T, H, D = st.num_tokens, st.num_heads, st.head_size

    # ---- device-resident inputs and outputs -------------------------------
    src = torch.from_numpy(st.src.view(np.int16)).to(dev).view(torch.bfloat16)
    key = src.as_strided((T, H, D), (st.key_stride0, D, 1), st.key_offset)
    value = src.as_strided((T, H, D), (st.value_stride0, D, 1),
                           st.value_offset)
    slots = torch.from_numpy(st.slot_mapping).to(dev)
    ks = torch.tensor([float(st.k_scale)], dtype=torch.float32, device=dev)
    vs = torch.tensor([float(st.v_scale)], dtype=torch.float32, device=dev)
    kv, kc, vc = kvq.alloc_nvfp4_cache(st.num_blocks, st.block_size, H, D,
                                       device=dev, fill=0xAA)
    n = ga.total_tokens
    gsets = []
    for _ in range(GATHER_SETS):  # same bytes at different addresses
        gsets.append(dict(
            cache=torch.from_numpy(ga.cache).to(dev).view(ga.num_blocks, -1),
            bt=torch.from_numpy(ga.block_table).to(dev),
            cu=torch.from_numpy(ga.cu_seq_lens).to(dev),
            k=torch.empty((n, ga.head_dim), dtype=torch.uint8, device=dev),
            s=torch.empty((n, 4), dtype=torch.uint8, device=dev)))
    dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    def store(flags):
        kvq.kvq_store_nvfp4(key, value, kc, vc, slots, ks, vs, flags=flags,
                            dev_error=dev_err, stream=sh)

    def gather(i, flags):
        g = gsets[i % GATHER_SETS]
        kvq.kvq_gather_indexer_k(g["cache"], g["k"], g["s"], g["bt"], g["cu"],
                                 block_size=ga.block_size, flags=flags,
                                 dev_error=dev_err, stream=sh)

    def step(i, flags):
        store(kvq.KVQ_F_PDL_EARLY_READ if flags else 0)
        gather(i, kvq.KVQ_F_PDL_EARLY_READ if flags else 0)

    def span_ms(fn, count):
        """Mean GPU time per call of `count` back-to-back calls between two
        events.  The calls are queued behind a GPU sleep long enough for the
        host to enqueue all of them: the binding spends ~10 us of host time
        per call, more than a short kernel's GPU time, and would otherwise
        pace the GPU.  The sleep runs before the first event."""
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(int(2e9 * max(0.005, count * QUEUE_S_PER_CALL)))
        e0.record(stream)
        for i in range(count):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / count

    W = max(args.warmup, 3)
    PDL = kvq.KVQ_F_PDL
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
    step_ms = span_ms(lambda i: step(i, PDL), K)
    if world > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - t0
    # per-kernel averages: each kernel alone, back to back (inputs larger
    # than L2: the store streams 689 MB per call; the gather rotates over
    # GATHER_SETS buffer sets)
    store_ms = span_ms(lambda i: store(kvq.KVQ_F_PDL_EARLY_READ), K)
    store_pdl_ms = span_ms(lambda i: store(PDL), K)
    gather_ms = span_ms(lambda i: gather(i, kvq.KVQ_F_PDL_EARLY_READ), K)
    gather_meta_ms = span_ms(lambda i: gather(i, kvq.KVQ_F_PDL_EARLY_META), K)
    plain = {"step_ms": span_ms(lambda i: step(i, 0), K),
             "store_ms": span_ms(lambda i: store(0), K),
             "gather_ms": span_ms(lambda i: gather(i, 0), K)}
    # the store's other input type and cache layout, same shape
    key16 = key.to(torch.float16)
    value16 = value.to(torch.float16)
    kv_n, kc_n, vc_n = kvq.alloc_nvfp4_cache(
        st.num_blocks, st.block_size, H, D, layout=kvq.KVQ_LAYOUT_NHD,
        device=dev, fill=0xAA)
    variants_ms = {
        "store_fp16_hnd": span_ms(lambda i: kvq.kvq_store_nvfp4(
            key16, value16, kc, vc, slots, ks, vs, flags=PDL,
            dev_error=dev_err, stream=sh), K),
        "store_bf16_nhd": span_ms(lambda i: kvq.kvq_store_nvfp4(
            key, value, kc_n, vc_n, slots, ks, vs, flags=PDL,
            dev_error=dev_err, stream=sh), K),
    }
    del key16, value16, kv_n, kc_n, vc_n
    # the read side: the long-context pages read back to bf16 rows
    from paged_quantized_kv_gb300 import workloads as wlmod
    lbt, lcu = wlmod.sequences_of_store(st, 512)
    lbt_d = torch.from_numpy(lbt).to(dev)
    lcu_d = torch.from_numpy(lcu).to(dev)
    k_out = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
    v_out = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
    load_ms = span_ms(lambda i: kvq.kvq_load_nvfp4(
        kc, vc, lbt_d, lcu_d, ks, vs, k_out, v_out,
        flags=kvq.KVQ_F_PDL_EARLY_META, dev_error=dev_err, stream=sh), K)
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
    istore_ms = span_ms(lambda i: kvq.kvq_store_indexer_k(
        ik[i % GATHER_SETS], icache, islots, flags=kvq.KVQ_F_PDL_EARLY_READ,
        dev_error=dev_err, stream=sh), K)
    istore_pdl_ms = span_ms(lambda i: kvq.kvq_store_indexer_k(
        ik[i % GATHER_SETS], icache, islots, flags=PDL, dev_error=dev_err,
        stream=sh), K)
    istore_bytes = iw.algorithmic_bytes()
    del ik, icache
    # decode attention over NVFP4 pages: one step of Llama-3.1-70B-shaped
    # attention (200 sequences, 64 query / 8 KV heads, contexts 512..2560;
    # 359 MB of pages per call, larger than L2)
    aw = wlmod.attention_workload(rank_seed(5, rank))
    attn = attention_inputs(aw, kvq, dev)
    attn_ms = span_ms(lambda i: run_attention(attn, kvq, PDL, dev_err, sh),
                      K)
    attn_pipe_ms = span_ms(lambda i: run_attention(
        attn, kvq, PDL | kvq.KVQ_F_ATTN_PIPELINED, dev_err, sh), K)
    attn_tc_ms = span_ms(lambda i: run_attention(
        attn, kvq, PDL | kvq.KVQ_F_ATTN_TCGEN05, dev_err, sh), K)
    attn_bytes = aw.algorithmic_bytes()
    attn_ctx = int(aw.context_lens.astype(np.int64).sum())
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
    region_ms = step_ms * K
    cold = single_launch_cold(lambda: store(0), lambda: gather(0, 0), dev)

    st_bytes = st.algorithmic_bytes()
    ga_bytes = ga.algorithmic_bytes()
    step_s = max_over_ranks(step_ms / 1e3, world, dev)
    total_bytes = sum_over_ranks(float(st_bytes + ga_bytes), world, dev)
    total_tokens = sum_over_ranks(float(T + n), world, dev)
    peak, peak_kind = measured_hbm_peak()
    store_gbs = st_bytes / (store_ms / 1e3) / 1e9
    gather_gbs = ga_bytes / (gather_ms / 1e3) / 1e9
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
                      "span / K, max over ranks.  Per-kernel times: K "
                      "launches of that kernel alone, back to back, same "
                      "flags, queued the same way",
        },
        "tokens_per_s": round(total_tokens / step_s, 1),
        "kernels": {
            "store_nvfp4": {
                "ms": round(store_ms, 5),
                "pdl_only_ms": round(store_pdl_ms, 5),
                "GB_s": round(store_gbs, 1),
                "frac_of_peak": round(store_gbs / peak, 4),
                "tokens_per_s": round(T / (store_ms / 1e3), 1),
                "algorithmic_bytes": st_bytes},
            "gather_indexer_k": {
                "ms": round(gather_ms, 5),
                "GB_s": round(gather_gbs, 1),
                "frac_of_peak": round(gather_gbs / peak, 4),
                "tokens_per_s": round(n / (gather_ms / 1e3), 1),
                "algorithmic_bytes": ga_bytes,
                "early_meta_only_ms": round(gather_meta_ms, 5)},
        },
        "without_pdl": {k: round(v, 5) for k, v in plain.items()},
        "load_nvfp4": {
            "note": "read side: the long-context pages read back to bf16 "
                    "rows through the block table (not part of the step)",
            "ms": round(load_ms, 5),
            "GB_s": round(load_bytes / load_ms / 1e6, 1),
            "frac_of_peak": round(load_bytes / load_ms / 1e6 / peak, 4),
            "tokens_per_s": round(T / (load_ms / 1e3), 1),
            "algorithmic_bytes": load_bytes},
        "store_variants": {
            k: {"ms": round(v, 5),
                "GB_s": round(st_bytes / v / 1e6, 1),
                "frac_of_peak": round(st_bytes / v / 1e6 / peak, 4)}
            for k, v in variants_ms.items()},
        "store_indexer_k": {
            "note": "write side of the indexer cache on the gather's shape "
                    "(131072 tokens, head_dim 128, block_size 64), not part "
                    "of the step; back to back with KVQ_F_PDL_EARLY_READ "
                    "(K rotated over the buffer sets, the kernel before "
                    "writes only the cache)",
            "ms": round(istore_ms, 5),
            "pdl_only_ms": round(istore_pdl_ms, 5),
            "GB_s": round(istore_bytes / istore_ms / 1e6, 1),
            "frac_of_peak": round(istore_bytes / istore_ms / 1e6 / peak, 4),
            "tokens_per_s": round(iw.num_tokens / (istore_ms / 1e3), 1),
            "algorithmic_bytes": istore_bytes},
        "paged_attention_nvfp4": {
            "note": "decode attention over the NVFP4 pages, one step of "
                    "Llama-3.1-70B-shaped attention: 200 sequences, 64 "
                    "query / 8 KV heads, head_size 128, block_size 16, "
                    "contexts 512 + U[0, 2048]; partition_size 512 (the "
                    "default warp-level-MMA kernel covers up to 1280 tokens "
                    "per CTA, then the partition merge); not part of the "
                    "step",
            "ms": round(attn_ms, 5),
            "GB_s": round(attn_bytes / attn_ms / 1e6, 1),
            "frac_of_peak": round(attn_bytes / attn_ms / 1e6 / peak, 4),
            "decode_tokens_per_s": round(aw.num_seqs / (attn_ms / 1e3), 1),
            "context_tokens_per_s": round(attn_ctx / (attn_ms / 1e3), 1),
            "algorithmic_bytes": attn_bytes,
            "pipelined_kernel_ms": round(attn_pipe_ms, 5),
            "pipelined_kernel_frac_of_peak": round(
                attn_bytes / attn_pipe_ms / 1e6 / peak, 4),
            "tcgen05_kernel_ms": round(attn_tc_ms, 5),
            "tcgen05_kernel_frac_of_peak": round(
                attn_bytes / attn_tc_ms / 1e6 / peak, 4)},
        "single_launch_after_l2_write_flush": {
            "note": "each kernel alone after writing a 256 MiB buffer "
                    "(L2 left dirty), events around the launch; includes "
                    "the ~4 us event/launch floor an empty kernel shows",
            "store_ms": cold[0], "gather_ms": cold[1],
            "store_GB_s": round(st_bytes / cold[0] / 1e6, 1),
            "gather_GB_s": round(ga_bytes / cold[1] / 1e6, 1)},
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
                             "step); the per-kernel loops after it launch "
                             "their own",
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(st, ga, args.cpu_sample_tokens)
        line["paged_attention_nvfp4"]["cpu_oracle"] = cpu_attention_baseline(
            aw)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def attention_inputs(aw, kvq, dev):
    """Device copies of an attention workload's inputs, output and
    scratch."""
    import torch
    kv, kc, vc = kvq.alloc_nvfp4_cache(aw.num_blocks, aw.block_size,
                                       aw.num_kv_heads, aw.head_size,
                                       device=dev)
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


def single_launch_cold(store, gather, dev, reps=20):
    """Median single-launch times (ms) after a 256 MiB write flush."""
    import torch
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    out = []
    for fn in (store, gather):
        ms = []
        for i in range(reps + 2):
            flush.fill_(i & 0xFF)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize(dev)
            if i >= 2:
                ms.append(e0.elapsed_time(e1))
        out.append(round(statistics.median(ms), 5))
    del flush
    return out


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
