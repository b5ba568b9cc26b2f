#!/usr/bin/env python3
"""Benchmark of one paged-attention step (reshape_and_cache + attention) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload gqa_decode] [--seed 0] [--dtype bf16|fp16]
                    [--kv-dtype fp8_e4m3] [--block-size 8|16|32] [--rope]

A step is one pass of the whole path over one batch: pa_reshape_and_cache of
the step's new K/V rows, then pa_attention_varlen (planning, split-KV
attention, prefill tiles when the batch has chunks, log-sum-exp merge); with
--kv-dtype fp8_e4m3 the 8-bit-cache calls, with --rope the rotary scatter. Inputs are seeded synthetic data resident in
HBM before timing starts. The KV working set (1.7 GB for the default
workload) is far larger than the 126 MB L2, so no L2 flush is needed between
steps. Prints one JSON line (rank 0). Its "scatter" record times the cache
scatter alone (the step's first call), back to back after the step's timed
regions.

The default run (gqa_decode, bf16, N=1) adds to its line the same step drawn
from two more seeds ("seed_spread") and one record per other named
configuration ("configs": tiny, MHA, long-context, mixed), each with its
step time, the dominant kernel's roofline and the oracle timed on the host
cores (one thread as well for the tiny, MHA and GQA configurations).

--impl reference times the fp64 CPU oracle on this machine's host cores on a
bounded sample of the same workload.

Multi-GPU (torchrun): each rank runs its own copy of the workload with its own
seed (independent batches, no collective on the data path); the timing is the
max over ranks and the value counts the bytes of all ranks ("weak" scaling).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged-attn KV GB/s & fraction of GB300 HBM peak; decode tokens/s per layer"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

WORKLOAD_TEXT = {
    "tiny_decode": "tiny decode: 4 requests, seq_lens {1,7,16,33}, H=4, Hkv=1, D=64, bs=16",
    "mha_decode": "MHA 7B-like decode layer: batch 64, H=Hkv=32, D=128, bs=16, seq_lens U[128,2048]",
    "gqa_decode": "GQA 8B-like decode layer: batch 256, H=32, Hkv=8, D=128, bs=16, seq_lens lognormal "
                  "(median 1024, sigma 1.0) clipped [16,8192], reshape_and_cache of 256 new rows",
    "long_decode": "long-context decode: batch 8, seq_len 32768, H=64, Hkv=8, D=128, bs=16",
    "mixed_step": "mixed continuous-batching step: 16 prefill chunks x 512 (ctx U[0,4096]) + 240 decode "
                  "(ctx U[256,4096], 64 share a 64-block prefix), H=32, Hkv=8, D=128, bs=16",
    "copy_blocks": "copy-on-write block copy: 4096 (source, destination) pairs per step over a pool of 16384 "
                   "blocks of the GQA cache shape (bs=16, Hkv=8, D=128; 32 KB per block and cache)",
}
COPY_POOL_BLOCKS, COPY_PAIRS = 16384, 4096
COPY_METRIC = "CoW block copy GB/s (read + write) & fraction of GB300 HBM peak"


# --------------------------------------------------------------------------
# Byte and FLOP accounting (algorithmic: what the step must move at minimum)
# --------------------------------------------------------------------------

def step_accounting(w, rope: bool = False) -> dict:
    H, Hkv, D, bs = w.num_heads, w.num_kv_heads, w.head_dim, w.block_size
    cache_elem = 1 if w.kv_fp8 else 2  # 8-bit caches: one byte per element
    kv_tok = 2 * Hkv * D * cache_elem
    uniq = w.kv_tokens_unique()
    logical = w.kv_tokens_logical()
    T = w.total_q
    tables = int(sum(-(-int(L) // bs) for L in w.seq_lens)) * 4
    meta = (2 * w.num_seqs + 1) * 4
    q_out = 2 * T * H * D * 2
    reshape = T * (2 * Hkv * D) * (2 + cache_elem) + T * 8  # read 16-bit rows, write cache rows
    if rope:  # q rotated in place (read + write), positions, one table row per token
        reshape += 2 * T * H * D * 2 + T * 8 + T * D * 4
    kv_bytes = uniq * kv_tok
    flops = tile_flops = 0
    ql = w.query_lens
    rows_per_item = 8 // (H // Hkv)  # longer requests go to the tensor-core tiles
    decode_reqs = []
    for b in range(w.num_seqs):
        L, n = int(w.seq_lens[b]), int(ql[b])
        visible = n * (L - n) + n * (n + 1) // 2
        flops += 4 * H * D * visible
        if n > rows_per_item:
            tile_flops += 4 * H * D * visible
        elif n > 0:
            decode_reqs.append(b)
    # bytes the split-KV decode kernel must move: unique KV of its requests, their q and out
    seen = {}
    for b in decode_reqs:
        L = int(w.seq_lens[b])
        for i in range(-(-L // bs)):
            blk = int(w.block_tables[b, i])
            seen[blk] = max(seen.get(blk, 0), min(bs, L - i * bs))
    dec_q = int(sum(int(ql[b]) for b in decode_reqs))
    decode_bytes = (sum(seen.values()) * kv_tok + 2 * dec_q * H * D * 2 + tables + meta)
    return {
        "tile_flops": tile_flops,
        "decode_bytes": decode_bytes,
        "kv_bytes": kv_bytes,
        "kv_bytes_logical": logical * kv_tok,
        "attention_bytes": kv_bytes + q_out + tables + meta,
        "step_bytes": kv_bytes + q_out + tables + meta + reshape,
        "scatter_bytes": reshape,
        "flops": flops,
        "query_tokens": T,
    }


# --------------------------------------------------------------------------
# Multi-rank helpers (also exercised by the gloo tests)
# --------------------------------------------------------------------------

def rank_seed(seed: int, rank: int) -> int:
    """Each rank draws an independent batch of the same shape."""
    return seed + 7919 * rank


def reduce_max(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def aggregate_rate(total_units: float, max_seconds: float) -> float:
    return total_units / max_seconds if max_seconds > 0 else float("nan")


# --------------------------------------------------------------------------
# Clocks sampled during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", self.gpu_id], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------------------
# CPU oracle on a bounded sample (the CPU baseline and the reference arm)
# --------------------------------------------------------------------------

def sub_workload(w, reqs):
    """The listed requests of `w` as their own batch (arrays sliced, not recomputed)."""
    reqs = np.asarray(sorted(reqs))
    ql = w.query_lens[reqs]
    qsl = np.zeros(reqs.size + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(ql)
    rows = np.concatenate([np.arange(w.query_start_loc[b], w.query_start_loc[b + 1]) for b in reqs])
    return dict(q=w.q[rows], block_tables=w.block_tables[reqs], seq_lens=w.seq_lens[reqs], query_start_loc=qsl)


def oracle_rate(w, kc, vc, target_s: float, rng, threads: int):
    """Time the oracle on random requests until about target_s of CPU work; returns
    (KV GB/s, query tokens/s, seconds, requests, threads)."""
    import oracle as oracle_mod
    orc = oracle_mod.default()
    kv_tok = 2 * w.num_kv_heads * w.head_dim * (1 if w.kv_fp8 else 2)
    order = rng.permutation(w.num_seqs)
    done_bytes = done_tok = 0
    used = 0
    t_total = 0.0
    n = 1
    while t_total < target_s:
        pos = used % w.num_seqs  # wraps around: a small workload is sampled more than once
        take = order[pos:pos + n]
        used += take.size
        s = sub_workload(w, take)
        t0 = time.perf_counter()
        orc.attention(s["q"], kc, vc, s["block_tables"], s["seq_lens"], s["query_start_loc"], w.num_heads,
                      w.scale, num_threads=threads, dtype=w.dtype, k_scale=w.k_scale, v_scale=w.v_scale)
        t_total += time.perf_counter() - t0
        done_bytes += int(s["seq_lens"].astype(np.int64).sum()) * kv_tok
        done_tok += int(s["query_start_loc"][-1])
        n = min(2 * n, 64)
    return done_bytes / t_total / 1e9, done_tok / t_total, t_total, used, threads


def scattered_caches(w):
    """Host copies of the caches after the oracle's scatter of the step's new rows."""
    import oracle as oracle_mod
    orc = oracle_mod.default()
    kc, vc = w.key_cache.copy(), w.value_cache.copy()
    if w.kv_fp8:
        orc.reshape_and_cache_fp8(w.key, w.value, kc, vc, w.slot_mapping, w.block_size, w.k_scale, w.v_scale,
                                  dtype=w.dtype)
    else:
        orc.reshape_and_cache(w.key, w.value, kc, vc, w.slot_mapping, w.block_size)
    return kc, vc


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# --------------------------------------------------------------------------
# The committed ncu traffic of the timed kernel (valid only for unchanged source)
# --------------------------------------------------------------------------

KERNEL_SOURCES = ["paged_kv_cache_55_gb300/csrc/attention_splitkv.cu", "paged_kv_cache_55_gb300/csrc/pa_common.cuh"]


def kernel_source_hash(root: str = ROOT) -> str:
    """Hash of the timed kernel's code: its sources without `//` comments,
    trailing blanks and empty lines, so that a comment edit keeps the committed
    counters while any change to the code drops them. (The sources hold no
    string literal with `//` in it; a CPU test checks that.)"""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(root, rel), encoding="utf-8") as f:
            for line in f:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode("utf-8") + b"\n")
    return h.hexdigest()[:16]


def committed_traffic(workload: str):
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        data = json.load(open(path))
    except ValueError:
        return None
    rec = data.get(workload)
    if not rec or rec.get("source_hash") != kernel_source_hash():
        return None
    return rec.get("dram_bytes_per_launch")


# --------------------------------------------------------------------------

def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS, "source": "fallback"}


def run_reference(args, world, rank) -> None:
    if rank != 0:
        return
    from paged_kv_cache_55_gb300 import workloads as W
    import oracle as oracle_mod
    kw = {"batch": args.batch} if args.batch else {}
    kw["dtype"] = args.dtype
    if args.block_size != 16:
        kw["block_size"] = args.block_size
    if args.kv_dtype:
        kw["kv_dtype"] = args.kv_dtype
    w = W.by_name(args.workload, seed=args.seed, **kw)
    kc, vc = scattered_caches(w)
    threads = host_threads()
    rng = np.random.default_rng(args.seed)
    per_step = max(1.0, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_rate(w, kc, vc, per_step / 4, rng, threads)
    rates, toks, secs, reqs = [], [], [], []
    for _ in range(args.steps):
        r, t, s, n, _ = oracle_rate(w, kc, vc, per_step, rng, threads)
        rates.append(r)
        toks.append(t)
        secs.append(s)
        reqs.append(n)
    value = float(np.mean(rates))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": float(np.mean(secs)) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "decode_tokens_per_s": float(np.mean(toks)),
        "config": {"workload": workload_text(args), "seed": args.seed},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"per step: {np.mean(reqs):.0f} request evaluations drawn in random order "
                                   f"from the workload's {w.num_seqs} requests (wrapping around), about "
                                   f"{per_step:.1f} s of fp64 oracle work"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_text(args) -> str:
    text = WORKLOAD_TEXT[args.workload]
    if args.dtype != "bf16":
        text += f" [{args.dtype} elements]"
    if getattr(args, "block_size", 16) != 16:
        text += f" [block_size {args.block_size}]"
    if getattr(args, "rope", False):
        text += " [rotary embedding fused into the cache scatter]"
    if getattr(args, "kv_dtype", ""):
        text += " [8-bit E4M3 KV cache, one scale per cache]"
    return text + (f" [batch overridden to {args.batch}]" if args.batch else "")


def step_timing(st, acct, steps: int, warmup: int, stream):
    """Device-timed steps of a built DeviceStep: the mean over `steps` back-to-back
    steps (one event pair around all of them), then a second pass with an event
    pair around every step and around its split-KV and prefill-tile kernels
    (per-step median, kernel durations)."""
    import torch
    from paged_kv_cache_55_gb300 import binding as B
    has_tiles = acct["tile_flops"] > 0
    ev = lambda: torch.cuda.Event(enable_timing=True)
    step_ev = [(ev(), ev()) for _ in range(steps)]
    kern_ev = [(ev(), ev()) for _ in range(steps)]
    tile_ev = [(ev(), ev()) for _ in range(steps)]
    for a, b in step_ev + kern_ev + tile_ev:  # create the events before timing
        a.record(stream)
        b.record(stream)
    for _ in range(max(warmup, 1)):
        st.run()
    torch.cuda.synchronize()
    if B.pa_debug_status() != 0:
        raise RuntimeError("device status flags set during warm-up")
    t0, t1 = ev(), ev()
    launches0 = B.pa_launch_count()
    t0.record(stream)
    for _ in range(steps):
        st.run()
    t1.record(stream)
    torch.cuda.synchronize()
    launches = B.pa_launch_count() - launches0
    step_ms = t0.elapsed_time(t1) / steps
    for k in range(steps):
        step_ev[k][0].record(stream)
        B.pa_attention_set_timing_events(*kern_ev[k])
        if has_tiles:
            B.pa_attention_set_tile_timing_events(*tile_ev[k])
        st.run()
        step_ev[k][1].record(stream)
    torch.cuda.synchronize()
    if B.pa_debug_status() != 0:
        raise RuntimeError("device status flags set during timing")
    return {
        "step_ms": step_ms,
        "step_ms_median": statistics.median(a.elapsed_time(b) for a, b in step_ev),
        "kern_ms": statistics.mean(a.elapsed_time(b) for a, b in kern_ev),
        "tile_ms": statistics.mean(a.elapsed_time(b) for a, b in tile_ev) if has_tiles else 0.0,
        "launches": launches,
    }


def rooflines(acct, t, peaks):
    """The split-KV kernel against HBM (bytes of the requests it serves) and, when the
    step has prefill chunks, the tensor-core tile kernel against the bf16 peak
    (algorithmic FLOPs: 4 H D per visible (query, key) pair of the chunks)."""
    has_tiles = acct["tile_flops"] > 0
    dec_bytes = acct["attention_bytes"] if not has_tiles else acct["decode_bytes"]
    kern_achieved = dec_bytes / (t["kern_ms"] * 1e-3) / 1e9
    decode = {"bound": "hbm", "kernel": "splitkv_attention_kernel", "achieved": kern_achieved,
              "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": kern_achieved / peaks["hbm_gbs"],
              "peak_source": peaks["source"], "kernel_ms": t["kern_ms"],
              "algorithmic_bytes_per_launch": dec_bytes, "traffic": None}
    tile = None
    if has_tiles:
        tile_achieved = acct["tile_flops"] / (t["tile_ms"] * 1e-3) / 1e12
        tile = {"bound": "tensor", "kernel": "prefill_tile_kernel", "achieved": tile_achieved,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": tile_achieved / peaks["bf16_tflops"],
                "peak_source": peaks["source"], "kernel_ms": t["tile_ms"],
                "algorithmic_flops_per_launch": acct["tile_flops"], "traffic": None}
    return decode, tile


EXTRA_CONFIGS = ["tiny_decode", "mha_decode", "long_decode", "mixed_step"]
SINGLE_THREAD_ORACLE = {"tiny_decode", "mha_decode", "gqa_decode"}


def config_record(name, seed, steps, warmup, device, stream, peaks, cpu_seconds):
    """One named configuration on one GPU: device-timed steps, the dominant kernel's
    roofline, and the oracle on the host cores (all of them, and one thread for the
    small and decode configurations) on a bounded sample of the same workload."""
    import torch
    from paged_kv_cache_55_gb300 import workloads as W
    from paged_kv_cache_55_gb300.runner import DeviceStep
    w = W.by_name(name, seed=seed)
    acct = step_accounting(w)
    st = DeviceStep(w, device=str(device))
    t = step_timing(st, acct, steps, warmup, stream)
    del st
    torch.cuda.empty_cache()
    peaks_d, tile = rooflines(acct, t, peaks)
    value = acct["step_bytes"] / (t["step_ms"] * 1e-3) / 1e9
    rec = {"workload": WORKLOAD_TEXT[name], "seed": seed, "steps": steps, "warmup": warmup,
           "ms_per_step": t["step_ms"], "ms_per_step_median": t["step_ms_median"], "value": value, "unit": UNIT,
           "hbm_frac": value / peaks["hbm_gbs"], "query_tokens_per_s": acct["query_tokens"] / (t["step_ms"] * 1e-3),
           "step_bytes": acct["step_bytes"], "flops": acct["flops"], "gpu_launches_per_step": t["launches"] / steps,
           "roofline": tile if tile is not None else peaks_d,
           "roofline_decode_kernel": peaks_d if tile is not None else None}
    if name == "tiny_decode":
        rec["roofline"]["bound"] = "launch latency (15 KB of work: the bytes are not the limit)"
    kc, vc = scattered_caches(w)
    rng = np.random.default_rng(1)
    r, _, secs, n, threads = oracle_rate(w, kc, vc, cpu_seconds, rng, host_threads())
    rec["cpu_baseline"] = {"value": r, "unit": UNIT, "cores": threads, "kind": "oracle",
                           "sample": f"{n} request evaluations drawn in random order from the workload's "
                                     f"{w.num_seqs} requests, {secs:.1f} s of fp64 oracle attention"}
    if name in SINGLE_THREAD_ORACLE:
        r1, _, secs1, n1, _ = oracle_rate(w, kc, vc, cpu_seconds / 2, np.random.default_rng(2), 1)
        rec["cpu_baseline_single_thread"] = {"value": r1, "unit": UNIT, "cores": 1, "kind": "oracle",
                                             "sample": f"{n1} request evaluations, {secs1:.1f} s on one thread"}
    return rec


def run_ours(args, world, rank, local_rank) -> None:
    import torch
    import torch.distributed as dist

    from paged_kv_cache_55_gb300 import binding as B
    from paged_kv_cache_55_gb300 import build as build_mod
    from paged_kv_cache_55_gb300 import workloads as W
    from paged_kv_cache_55_gb300.runner import DeviceStep

    build_mod.build()
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    kw = {"batch": args.batch} if args.batch else {}
    kw["dtype"] = args.dtype
    if args.block_size != 16:
        kw["block_size"] = args.block_size
    if args.kv_dtype:
        kw["kv_dtype"] = args.kv_dtype
    w = W.by_name(args.workload, seed=rank_seed(args.seed, rank), **kw)
    acct = step_accounting(w, rope=args.rope)
    rope = None
    if args.rope:
        pos = np.concatenate([int(w.seq_lens[b]) - int(w.query_lens[b]) + np.arange(int(w.query_lens[b]))
                              for b in range(w.num_seqs)]).astype(np.int64)
        rope = (W.rope_cos_sin_cache(int(w.max_seq_len) + 1, w.head_dim), pos, True)
    st = DeviceStep(w, device=str(device), rope=rope)
    stream = torch.cuda.current_stream()

    # warm-up (the first call also creates the timing events)
    ev_pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)]
    tile_pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
    for a, b in ev_pairs + tile_pairs:
        a.record(stream)
        b.record(stream)
    has_tiles = acct["tile_flops"] > 0
    for _ in range(max(args.warmup, 1)):
        st.run()
    torch.cuda.synchronize()
    if B.pa_debug_status() != 0:
        raise RuntimeError("device status flags set during warm-up")

    gpu_id = str(torch.cuda.get_device_properties(device).uuid)
    gpu_id = gpu_id if gpu_id.startswith("GPU-") else f"GPU-{gpu_id}"
    sampler = ClockSampler(gpu_id)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    launches0 = B.pa_launch_count()
    t0.record(stream)
    for k in range(args.steps):
        st.run()
    t1.record(stream)
    torch.cuda.synchronize()
    launches = B.pa_launch_count() - launches0
    if world > 1:
        dist.barrier()
    step_ms = t0.elapsed_time(t1) / args.steps
    # Second pass of the same steps, with events around the split-KV kernel
    # and the prefill-tile kernel alone (they serialise the kernels against
    # their neighbours, so the step time above is taken without them).
    step_pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
    for k in range(args.steps):
        step_pairs[k][0].record(stream)
        B.pa_attention_set_timing_events(*ev_pairs[k])
        if has_tiles:
            B.pa_attention_set_tile_timing_events(*tile_pairs[k])
        st.run()
        step_pairs[k][1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    step_ms_median = statistics.median(a.elapsed_time(b) for a, b in step_pairs)
    kern_ms = statistics.mean(a.elapsed_time(b) for a, b in ev_pairs)
    tile_ms = statistics.mean(a.elapsed_time(b) for a, b in tile_pairs) if has_tiles else 0.0

    max_ms = reduce_max(step_ms, device)
    total_bytes = reduce_sum(float(acct["step_bytes"]), device)
    total_tok = reduce_sum(float(acct["query_tokens"]), device)
    value = aggregate_rate(total_bytes, max_ms * 1e-3) / 1e9

    # End to end through the C ABI with host buffers: every step uploads its
    # inputs from pinned host memory and reads its output back. Two sets of
    # device buffers alternate so that, as a serving loop would, step k+1's
    # upload (one copy stream) and step k-1's download (another) overlap step
    # k's kernels; every copy of every step is inside the timed region.
    pin = lambda t: t.cpu().pin_memory()
    names = ("q", "key", "value", "slot_mapping", "block_tables", "seq_lens", "query_start_loc")

    def inputs_of(s):
        lst = [getattr(s, k) for k in names]
        if s.rope is not None:
            lst.append(s.rope[1])  # this step's positions (the rotary table stays resident, like weights)
        return lst

    sets = [st, DeviceStep(w, device=str(device), rope=rope)]
    host_in = [pin(d) for d in inputs_of(st)]
    host_out = [torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(h.numel() * h.element_size() for h in host_in)
    d2h = host_out[0].numel() * host_out[0].element_size()
    up, down = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_steps(n, start_event=None):
        for k in range(n):
            i = k % 2
            s = sets[i]
            if k == 0 and start_event is not None:
                up.wait_event(start_event)
            if k >= 2:
                up.wait_event(ev_done[i])  # the set's previous step has read its inputs
            with torch.cuda.stream(up):
                for d, h in zip(inputs_of(s), host_in):
                    d.copy_(h, non_blocking=True)
                ev_in[i].record(up)
            stream.wait_event(ev_in[i])
            if k >= 2:
                stream.wait_event(ev_out[i])  # the set's previous output has been read back
            s.run(stream)
            ev_done[i].record(stream)
            down.wait_event(ev_done[i])
            with torch.cuda.stream(down):
                host_out[i].copy_(s.out, non_blocking=True)
                ev_out[i].record(down)
        for i in range(min(n, 2)):
            stream.wait_event(ev_out[i])

    e2e_steps(4)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_steps(args.steps, start_event=e0)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1) / args.steps, device)
    e2e_value = aggregate_rate(total_bytes, e2e_ms * 1e-3) / 1e9

    # the cache scatter (a1) alone, timed on its own after the step's timed regions
    for _ in range(3):
        st.reshape_and_cache(stream)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(args.steps):
        st.reshape_and_cache(stream)
    a1.record(stream)
    torch.cuda.synchronize()
    scatter_ms = reduce_max(a0.elapsed_time(a1) / args.steps, device)

    peaks = load_peaks()
    # the split-KV kernel against HBM: the bytes of the requests it serves
    dec_bytes = acct["attention_bytes"] if not has_tiles else acct["decode_bytes"]
    kern_achieved = dec_bytes / (kern_ms * 1e-3) / 1e9
    # committed counters exist for the default bf16 line and its 8-bit-cache variant
    traffic = (committed_traffic(args.workload + ("+" + args.kv_dtype if args.kv_dtype else ""))
               if args.dtype == "bf16" and args.block_size == 16 and not args.rope and not args.batch else None)
    roof_decode = {"bound": "hbm", "kernel": "splitkv_attention_kernel", "achieved": kern_achieved,
                   "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": kern_achieved / peaks["hbm_gbs"],
                   "peak_source": peaks["source"], "kernel_ms": kern_ms,
                   "algorithmic_bytes_per_launch": dec_bytes, "traffic": traffic}
    roof = roof_decode
    if has_tiles:
        # a step with prefill chunks: the dominant kernel is the tensor-core tile kernel
        # (algorithmic FLOPs: 4 H D per visible (query, key) pair of the chunks; the bf16
        # burst peak, the fp16 rate being the same)
        tile_achieved = acct["tile_flops"] / (tile_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": "prefill_tile_kernel", "achieved": tile_achieved,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": tile_achieved / peaks["bf16_tflops"],
                "peak_source": peaks["source"], "kernel_ms": tile_ms,
                "algorithmic_flops_per_launch": acct["tile_flops"], "traffic": None}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": max_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": args.dtype, "data": "synthetic",
        "ms_per_step_median": step_ms_median,
        "hbm_frac": value / peaks["hbm_gbs"],
        "decode_tokens_per_s": total_tok / (max_ms * 1e-3),
        "config": {"workload": workload_text(args), "seed": args.seed,
                   "parallelism": f"replicas{world}" if world > 1 else "single",
                   "l2": "no flush: KV working set per step is larger than L2",
                   "step": ("pa_rope_reshape_and_cache" if args.rope else "pa_reshape_and_cache")
                           + ("_fp8 + pa_attention_varlen_fp8" if args.kv_dtype else " + pa_attention_varlen")
                           + " (plan, split-KV, merge)",
                   "kv_cache": args.kv_dtype or args.dtype,
                   "step_bytes": acct["step_bytes"], "kv_bytes": acct["kv_bytes"],
                   "kv_bytes_logical": acct["kv_bytes_logical"], "flops": acct["flops"]},
        "roofline": roof,
        "roofline_decode_kernel": roof_decode if has_tiles else None,
        "e2e": {"value": e2e_value, "unit": UNIT, "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "copies": "pinned host buffers; two device buffer sets, uploads and downloads on their own "
                          "streams overlapping the neighbouring steps' kernels"},
        "gpu_launches": launches,
        "clocks": clocks,
        "scatter": {"call": ("pa_rope_reshape_and_cache" if args.rope else "pa_reshape_and_cache")
                            + ("_fp8" if args.kv_dtype else ""),
                    "ms": scatter_ms, "bytes": acct["scatter_bytes"],
                    "GB/s": acct["scatter_bytes"] / (scatter_ms * 1e-3) / 1e9,
                    "note": "timed alone, back to back, after the step's timed regions: launch-bound at small T, "
                            "and its inputs stay in L2 between repeats, so the rate can exceed HBM's"},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        kc, vc = scattered_caches(w)
        r, _, secs, n, threads = oracle_rate(w, kc, vc, args.cpu_seconds, np.random.default_rng(1), host_threads())
        line["cpu_baseline"] = {"value": r, "unit": UNIT, "cores": threads, "kind": "oracle",
                                "sample": f"{n} request evaluations drawn in random order from the workload's "
                                          f"{w.num_seqs} requests, {secs:.1f} s of fp64 oracle attention "
                                          f"(KV bytes of the evaluated requests / time)"}
        if args.workload in SINGLE_THREAD_ORACLE:
            r1, _, secs1, n1, _ = oracle_rate(w, kc, vc, args.cpu_seconds / 3, np.random.default_rng(2), 1)
            line["cpu_baseline_single_thread"] = {"value": r1, "unit": UNIT, "cores": 1, "kind": "oracle",
                                                  "sample": f"{n1} request evaluations, {secs1:.1f} s on one thread"}
        del kc, vc
    default_line = (args.workload == "gqa_decode" and args.dtype == "bf16" and not args.kv_dtype and
                    args.block_size == 16 and not args.rope and not args.batch)
    if rank == 0 and world == 1 and default_line and not args.no_extra_configs:
        # the other named configurations and two more seeds of this one, each timed
        # on its own (outside the headline's timed region)
        del sets
        torch.cuda.empty_cache()
        n_extra = max(3, min(args.steps, 20))
        spread = {"seeds": [args.seed], "value": [value], "kernel_frac": [roof_decode["frac"]],
                  "ms_per_step": [max_ms]}
        for sd in (args.seed + 1, args.seed + 2):
            w2 = W.by_name(args.workload, seed=sd)
            a2 = step_accounting(w2)
            st2 = DeviceStep(w2, device=str(device))
            t2 = step_timing(st2, a2, n_extra, max(args.warmup, 3), stream)
            del st2
            torch.cuda.empty_cache()
            d2, _ = rooflines(a2, t2, peaks)
            spread["seeds"].append(sd)
            spread["value"].append(a2["step_bytes"] / (t2["step_ms"] * 1e-3) / 1e9)
            spread["kernel_frac"].append(d2["frac"])
            spread["ms_per_step"].append(t2["step_ms"])
        line["seed_spread"] = spread
        line["configs"] = {}
        for name in EXTRA_CONFIGS:
            line["configs"][name] = config_record(name, args.seed, n_extra, max(args.warmup, 3), device, stream,
                                                  peaks, args.extra_cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# Copy-on-write block copy (a separate workload: pa_copy_blocks alone)
# --------------------------------------------------------------------------

def copy_mapping(seed: int) -> np.ndarray:
    """COPY_PAIRS distinct sources and distinct destinations, no destination a source."""
    ids = np.random.default_rng(seed + 4000).permutation(COPY_POOL_BLOCKS)
    return np.stack([ids[:COPY_PAIRS], ids[COPY_PAIRS:2 * COPY_PAIRS]], axis=1).astype(np.int64)


def copy_oracle_rate(target_s: float, seed: int):
    """The oracle's block copy on a host pool (512 blocks, 128 pairs per call) until
    about target_s; returns (GB/s read + write, seconds, pairs)."""
    import oracle as oracle_mod
    orc = oracle_mod.default()
    rng = np.random.default_rng(seed)
    shape = (512, 16, 8, 128)
    kc = rng.integers(0, 65535, size=shape, dtype=np.uint16)
    vc = rng.integers(0, 65535, size=shape, dtype=np.uint16)
    per_pair = 2 * 2 * int(np.prod(shape[1:])) * 2  # K and V, read and write
    t_total, pairs = 0.0, 0
    while t_total < target_s:
        ids = rng.permutation(shape[0])
        m = np.stack([ids[:128], ids[128:256]], axis=1)
        t0 = time.perf_counter()
        orc.copy_blocks(kc, vc, m)
        t_total += time.perf_counter() - t0
        pairs += 128
    return pairs * per_pair / t_total / 1e9, t_total, pairs


def run_copy_reference(args, world, rank) -> None:
    if rank != 0:
        return
    per_step = max(0.5, min(5.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        copy_oracle_rate(per_step / 4, args.seed)
    rates, secs, pairs = [], 0.0, 0
    for k in range(args.steps):
        r, t, n = copy_oracle_rate(per_step, args.seed + k)
        rates.append(r)
        secs += t
        pairs += n
    value = statistics.median(rates)
    line = {
        "metric": COPY_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": secs * 1e3 / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "raw 16-bit", "data": "synthetic", "impl": "reference",
        "config": {"workload": "copy-on-write block copy on the host: bounded sample (128 pairs per call over a "
                               "512-block pool of the GQA block shape)", "seed": args.seed},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{pairs} block pairs, {secs:.1f} s of memcpy-based oracle copy"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_copy_blocks(args, world, rank, local_rank) -> None:
    import torch
    import torch.distributed as dist

    from paged_kv_cache_55_gb300 import binding as B
    from paged_kv_cache_55_gb300 import build as build_mod

    build_mod.build()
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    tdt = torch.float16 if args.dtype == "fp16" else torch.bfloat16
    gen = torch.Generator(device=device)
    gen.manual_seed(rank_seed(args.seed, rank))
    shape = (COPY_POOL_BLOCKS, 16, 8, 128)
    # seeded random 16-bit patterns (the copy moves raw bits; NaN patterns included)
    kc = torch.randint(-32768, 32767, shape, dtype=torch.int16, device=device, generator=gen).view(tdt)
    vc = torch.randint(-32768, 32767, shape, dtype=torch.int16, device=device, generator=gen).view(tdt)
    m_host = torch.from_numpy(copy_mapping(rank_seed(args.seed, rank))).pin_memory()
    m = m_host.to(device)
    block_bytes = 16 * 8 * 128 * 2
    step_bytes = COPY_PAIRS * 2 * 2 * block_bytes  # K and V blocks, read once and written once
    stream = torch.cuda.current_stream()

    for _ in range(max(args.warmup, 1)):
        B.pa_copy_blocks(kc, vc, m)
    torch.cuda.synchronize()
    if B.pa_debug_status() != 0:
        raise RuntimeError("device status flags set during warm-up")
    gpu_id = str(torch.cuda.get_device_properties(device).uuid)
    gpu_id = gpu_id if gpu_id.startswith("GPU-") else f"GPU-{gpu_id}"
    sampler = ClockSampler(gpu_id)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    launches0 = B.pa_launch_count()
    t0.record(stream)
    for _ in range(args.steps):
        B.pa_copy_blocks(kc, vc, m)
    t1.record(stream)
    torch.cuda.synchronize()
    launches = B.pa_launch_count() - launches0
    clocks = sampler.stop()
    if world > 1:
        dist.barrier()
    step_ms = t0.elapsed_time(t1) / args.steps
    max_ms = reduce_max(step_ms, device)
    total_bytes = reduce_sum(float(step_bytes), device)
    value = aggregate_rate(total_bytes, max_ms * 1e-3) / 1e9

    # end to end: the mapping from pinned host memory, the copy, one destination block's first row back
    host_out = torch.empty((8, 128), dtype=tdt).pin_memory()
    probe_block = int(m_host[-1, 1])

    def e2e_step():
        m.copy_(m_host, non_blocking=True)
        B.pa_copy_blocks(kc, vc, m)
        host_out.copy_(vc[probe_block, 0], non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1) / args.steps, device)
    assert B.pa_debug_status() == 0
    peaks = load_peaks()
    line = {
        "metric": COPY_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": max_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": args.dtype, "data": "synthetic (seeded random 16-bit patterns)",
        "hbm_frac": value / peaks["hbm_gbs"],
        "config": {"workload": workload_text(args), "seed": args.seed,
                   "parallelism": f"replicas{world}" if world > 1 else "single",
                   "l2": "no flush: 512 MB moved per step, larger than L2", "step_bytes": step_bytes},
        "roofline": {"bound": "hbm", "kernel": "copy_blocks_kernel", "achieved": value, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": value / peaks["hbm_gbs"], "peak_source": peaks["source"],
                     "kernel_ms": step_ms, "algorithmic_bytes_per_launch": step_bytes, "traffic": None},
        "e2e": {"value": aggregate_rate(total_bytes, e2e_ms * 1e-3) / 1e9, "unit": UNIT,
                "h2d_bytes_per_step": int(m_host.numel() * 8),
                "d2h_bytes_per_step": int(host_out.numel() * host_out.element_size())},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r, secs, pairs = copy_oracle_rate(min(args.cpu_seconds, 5.0), args.seed)
        line["cpu_baseline"] = {"value": r, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": f"{pairs} block pairs over a 512-block host pool, {secs:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOAD_TEXT), default="gqa_decode")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--dtype", choices=["bf16", "fp16"], default="bf16",
                    help="element type of q, K/V and out (the metric's workload is bf16)")
    ap.add_argument("--kv-dtype", choices=["", "fp8_e4m3"], default="",
                    help="cache element type: empty = the element type of q (16-bit), fp8_e4m3 = 8-bit codes")
    ap.add_argument("--block-size", type=int, choices=[8, 16, 32], default=16,
                    help="tokens per cache block (the configurations are quoted at 16)")
    ap.add_argument("--rope", action="store_true",
                    help="the step rotates q and K (pa_rope_reshape_and_cache, neox pairing, rotary_dim = D) "
                         "instead of pa_reshape_and_cache")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's number of requests (small profiling cases only)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-configs", action="store_true",
                    help="skip the records of the other named configurations and seeds")
    ap.add_argument("--extra-cpu-seconds", type=float, default=4.0,
                    help="oracle seconds per extra configuration record")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if args.workload == "copy_blocks":
            run_copy_reference(args, world, rank)
        else:
            run_reference(args, world, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        if args.workload == "copy_blocks":
            run_copy_blocks(args, world, rank, local_rank)
        else:
            run_ours(args, world, rank, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
