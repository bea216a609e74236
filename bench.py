"""Decode-step benchmark: paged decode attention HBM GB/s and decode tokens/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pkv|reference]

Workload (one step = the whole hot path over one batch): the GQA decode
batch -- 64 sequences with context lengths uniform on 512..4096, block size
16, 32 query heads over 8 KV heads, head dim 128, bf16, blocks shuffled over
a pool of 1.2x the blocks needed.  Each step writes one new token per
sequence into its slot (kv_write, preceded by copy_blocks when the block
manager reports copy-on-write pairs: none for this batch) and runs paged
decode attention over context + 1 tokens (split into 512-token partitions
with the log-sum-exp merge).  The KV pools (~0.7 GB) are larger than L2, so
no flush is needed between steps.

``value`` is algorithmic bytes per step (K + V of every attended token, q,
out, the block-table entries and sequence lengths read, and kv_write's
reads and writes) over the device time of a step.  ``roofline`` reports the
paged_decode_attention call alone against the measured HBM peak.

With N > 1 (torchrun), every rank runs its own replica of the batch (weak
scaling, no collective on the data path); the time is the max over ranks.

``--impl reference`` times the CPU oracle (fp64, OpenMP) on a bounded sample
of the same batch and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "paged decode attention achieved HBM GB/s (% of GB300 peak) and decode tokens/s"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
SINGLE_WORKLOADS = ("tiny", "opt13b_like", "long_context", "long_context_fp8", "prefix_sharing",
                    "prefix_sharing_cow", "swap", "writes", "beam_search", "decode_shapes",
                    "prefill_shapes")


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["pkv", "reference"], default="pkv")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end measurement")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-extra", action="store_true", help="skip the long-context line")
    ap.add_argument("--all-configs", action="store_true",
                    help="also measure the tiny, OPT-13B-like and prefix-sharing workloads")
    ap.add_argument("--partition-size", type=int, default=0)
    ap.add_argument("--only", choices=["prefill"] + sorted(SINGLE_WORKLOADS), default=None,
                    help="time one workload alone and print one JSON line: the causal paged "
                         "prefill of the prefill batch, or the decode attention of one of the "
                         "other workloads (used for per-workload profiles)")
    ap.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                    help="pool format of the timed step: 16-bit pools, or 8-bit E4M3 pools "
                         "(quantised from the same values) with the 8-bit write and attention")
    ap.add_argument("--seed", type=int, default=244)
    return ap.parse_args()


# ----------------------------------------------------------------------------
# accounting
# ----------------------------------------------------------------------------
def attention_bytes(step, kv_scalar_bytes: int = 2) -> int:
    """Algorithmic bytes of one paged_decode_attention call (1-byte scalars: 8-bit pools)."""
    lens = step.seq_lens.to(torch.int64)
    b = 2  # bytes per scalar of q and out
    kv = int(lens.sum()) * step.num_kv_heads * step.head_dim * kv_scalar_bytes * 2
    qo = 2 * step.num_seqs * step.num_q_heads * step.head_dim * b
    tables = int(((lens + step.block_size - 1) // step.block_size).sum()) * 4 + 4 * step.num_seqs
    return kv + qo + tables


def kv_write_bytes(step, kv_scalar_bytes: int = 2) -> int:
    """New 16-bit keys / values read, pool scalars written, slot mapping read."""
    T = int(step.slot_mapping.numel())
    return 2 * T * step.num_kv_heads * step.head_dim * (2 + kv_scalar_bytes) + 8 * T


def copy_bytes(step) -> int:
    per_block = step.num_kv_heads * step.block_size * step.head_dim * 2 * 2  # K and V
    return int(step.cow_pairs.shape[0]) * per_block * 2  # read + write


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        return float(peaks["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


TRAFFIC_SOURCES = ("decode_stream.cuh", "decode_policy.cuh", "decode_tile.cuh", "decode_stream.cu",
                   "decode_stream_fp8.cu", "pkv_device.cuh", "pkv_internal.h")


def kernel_source_digest() -> str:
    """sha256 over the sources the streaming attention kernel is built from."""
    h = hashlib.sha256()
    for name in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, "paged_kv_cache_242_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def traffic_for(kv: str = "bf16"):
    """DRAM bytes per launch from a committed ncu capture of these exact sources."""
    path = os.path.join(ROOT, "profiles", "decode_stream_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256") != kernel_source_digest():
        return None
    key = "dram_bytes_per_launch_gqa_batch" + ("" if kv == "bf16" else "_fp8")
    return rec.get(key)


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a host float over all ranks (identity at world size 1)."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------
# CPU oracle timing (baseline and reference arm)
# ----------------------------------------------------------------------------
def oracle_sample_rate(step, max_seconds: float, max_seqs=None, min_reps=1, threads=None):
    """Run the oracle (kv_write replay + attention) on the first sequences,
    with `threads` OpenMP threads (default: every host core).

    Returns (bytes per second, seconds, description, threads).
    """
    import numpy as np

    import oracle
    from paged_kv_cache_242_gb300.workloads import bits

    S = step.num_seqs if max_seqs is None else min(max_seqs, step.num_seqs)
    threads = oracle.max_threads() if threads is None else int(threads)
    kc, vc = bits(step.k_cache), bits(step.v_cache)
    q = np.ascontiguousarray(bits(step.q)[:S])
    bt = np.ascontiguousarray(step.block_tables.numpy()[:S])
    sl = np.ascontiguousarray(step.seq_lens.numpy()[:S])
    kn = np.ascontiguousarray(bits(step.k_new)[:S])
    vn = np.ascontiguousarray(bits(step.v_new)[:S])
    slots = np.ascontiguousarray(step.slot_mapping.numpy()[:S])
    per_rep = (int(sl.astype(np.int64).sum()) * step.num_kv_heads * step.head_dim * 4 +
               2 * S * step.num_q_heads * step.head_dim * 2)
    # the 64-token slot write is replayed once, untimed (the wrapper copies
    # the whole pools to keep its inputs immutable, which is not oracle work)
    kc, vc, _ = oracle.kv_write(kn, vn, slots, kc, vc)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.attention(q, kc, vc, bt, sl, step.scale, step.dtype, num_threads=threads)
        reps += 1
        elapsed = time.perf_counter() - t0
        if reps >= min_reps and elapsed >= max_seconds:
            break
    desc = (f"{S} of {step.num_seqs} sequences of the batch: fp64 attention over the "
            f"written caches, {reps} repetition(s), {elapsed:.1f} s, {threads} OpenMP threads")
    return per_rep * reps / elapsed, elapsed / reps, desc, threads


# ----------------------------------------------------------------------------
def run_reference(args, rank, world):
    """Reference arm: the CPU oracle, timed on the host, on rank 0 only."""
    if rank != 0:
        return
    from paged_kv_cache_242_gb300 import workloads as W

    step = W.gqa_batch(seed=args.seed)
    # size the per-step sample so K + W steps end within ~2 minutes
    probe_rate, probe_t, _, _ = oracle_sample_rate(step, 0.0, max_seqs=1)
    budget = 120.0 / max(1, args.steps + args.warmup)
    seqs = max(1, min(step.num_seqs, int(budget / max(probe_t, 1e-6))))
    for _ in range(args.warmup):
        oracle_sample_rate(step, 0.0, max_seqs=seqs)
    t0 = time.perf_counter()
    per_bytes = 0.0
    for _ in range(args.steps):
        rate, t_rep, desc, threads = oracle_sample_rate(step, 0.0, max_seqs=seqs)
        per_bytes += rate * t_rep
    elapsed = time.perf_counter() - t0
    value = per_bytes / elapsed / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * elapsed / max(1, args.steps), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(step),
        "cpu_baseline": {"kind": "oracle", "value": round(value, 4), "unit": UNIT,
                         "cores": threads, "sample": desc},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(step, partition=None):
    cfg = {"workload": "gqa_decode_batch", "num_seqs": step.num_seqs,
           "context_lengths": "uniform 512..4096 (+1 written token)",
           "num_q_heads": step.num_q_heads, "num_kv_heads": step.num_kv_heads,
           "head_dim": step.head_dim, "block_size": step.block_size,
           "num_blocks": int(step.k_cache.shape[0]) if step.k_cache is not None else None,
           "kv_tokens": step.kv_tokens, "max_seq_len": step.max_seq_len,
           "l2": "inputs larger than L2 (no flush)"}
    if partition is not None:
        cfg["partition_size"] = partition
    return cfg


def time_calls(call, reps=200, warmup=10):
    """Average time of one call issued back to back from Python (CUDA events)."""
    for _ in range(warmup):
        call()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


L2_FLUSH_BYTES = 512 << 20  # written between calls whose inputs could stay in the 129 MB L2


def time_calls_graph(call, per_graph=20, replays=10, flush=False, clean_l2=True):
    """Average device time of one call replayed from a CUDA graph of `per_graph`
    calls: no host launch cost, as a serving loop that captures its decode
    step would issue it (median over replays, CUDA events).  With `flush`,
    every call follows a 512 MiB write that evicts L2 and the time of a graph
    of the flushes alone is subtracted.  With `clean_l2` the write is followed
    by a read of the same buffer, which leaves L2 holding clean lines, so a
    call that mostly reads does not pay the write-back of the flush.  Calls
    that mostly write take `clean_l2=False`: their own writes would otherwise
    sit in a clean L2 and be written back during the next (subtracted) flush."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    scratch = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda") if flush else None

    def build(with_call):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(per_graph):
                if scratch is not None:
                    scratch.fill_(1)
                    if clean_l2:
                        scratch.view(torch.int32).amax()
                if with_call:
                    call()
        graph.replay()
        torch.cuda.synchronize()
        return graph

    def median_ms(graph):
        stream = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        times = []
        for _ in range(replays):
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) / per_graph)
        times.sort()
        return times[len(times) // 2]

    ms = median_ms(build(True))
    if scratch is not None:
        ms -= median_ms(build(False))
    return ms


def time_attention_only(pkv, step, dev, part, reps=200, warmup=10, graph=False):
    """Average device time of one paged_decode_attention call (CUDA events)."""
    ws_bytes = pkv.decode_workspace_bytes(step.num_seqs, step.num_q_heads, step.max_seq_len,
                                          step.block_size, part)
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev["q"].device)
    out = torch.empty_like(dev["q"])

    def call():
        pkv.paged_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                                   dev["seq_lens"], step.num_kv_heads, step.scale, out,
                                   max_seq_len=step.max_seq_len, partition_size=part,
                                   workspace=ws)

    eager = time_calls(call, reps, warmup)
    if not graph:
        return eager
    plan = pkv.DecodeAttentionPlan(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                                   dev["seq_lens"], out, max_seq_len=step.max_seq_len,
                                   num_kv_heads=step.num_kv_heads, scale=step.scale,
                                   partition_size=part, workspace=ws)
    eager_plan = time_calls(plan.run, reps, warmup)
    return eager, eager_plan, time_calls_graph(call, flush=attention_bytes(step) < L2_FLUSH_BYTES)


def measure_attention(pkv, step, device, label, workload):
    dev = {"q": step.q.to(device), "k_cache": step.k_cache.to(device),
           "v_cache": step.v_cache.to(device), "block_tables": step.block_tables.to(device),
           "seq_lens": step.seq_lens.to(device)}
    eager, eager_plan, ms = time_attention_only(pkv, step, dev, 0, graph=True)
    hbm, _ = measured_peaks()
    gbs = attention_bytes(step) / (ms * 1e-3) / 1e9
    del dev
    torch.cuda.empty_cache()
    timing = "CUDA graph replay" + (", L2 evicted before every call"
                                    if attention_bytes(step) < L2_FLUSH_BYTES else
                                    ", inputs larger than L2")
    return {"workload": workload, "attention_ms": round(ms, 4), "timing": timing,
            "host_call_ms": round(eager, 4), "host_call_ms_plan": round(eager_plan, 4),
            "achieved_gbs": round(gbs, 1),
            "frac_of_measured_peak": round(gbs / hbm, 4),
            "frac_of_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
            "decode_tokens_per_s": round(step.num_seqs / (ms * 1e-3), 1)}


# Scales of the 8-bit pools: N(0, 1) keys / values map onto about +-4.8 / +-4.0.
FP8_K_SCALE, FP8_V_SCALE = 0.0107, 0.0089


def measure_attention_fp8(pkv, step, device, workload, reps=200, warmup=10):
    """Decode attention over 8-bit (E4M3) pools quantised from the step's 16-bit pools."""
    nb, h, b, d = step.k_cache.shape
    kc8 = torch.empty((nb, h, b, d), dtype=torch.uint8, device=device)
    vc8 = torch.empty_like(kc8)
    slots = torch.arange(nb * b, dtype=torch.int64, device=device)
    rows = [pool.permute(0, 2, 1, 3).reshape(nb * b, h, d).contiguous().to(device)
            for pool in (step.k_cache, step.v_cache)]  # every slot, in slot order
    pkv.kv_write_fp8(rows[0], rows[1], slots, kc8, vc8, FP8_K_SCALE, FP8_V_SCALE)
    del rows
    q = step.q.to(device)
    bt, sl = step.block_tables.to(device), step.seq_lens.to(device)
    ws = torch.zeros(max(pkv.decode_workspace_bytes(step.num_seqs, step.num_q_heads,
                                                     step.max_seq_len, step.block_size, 0), 16),
                     dtype=torch.uint8, device=device)
    out = torch.empty_like(q)

    def call():
        pkv.paged_decode_attention_fp8(q, kc8, vc8, bt, sl, FP8_K_SCALE, FP8_V_SCALE, step.scale,
                                       out, max_seq_len=step.max_seq_len, workspace=ws)

    for _ in range(warmup):
        call()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    hbm, kind = measured_peaks()
    gbs = attention_bytes(step, 1) / (ms * 1e-3) / 1e9
    del kc8, vc8, q, bt, sl, ws, out
    torch.cuda.empty_cache()
    return {"workload": workload, "kv_format": "E4M3 codes, one scale per pool",
            "attention_ms": round(ms, 4), "achieved_gbs": round(gbs, 1),
            "frac_of_measured_peak": round(gbs / hbm, 4), "peak_kind": kind,
            "decode_tokens_per_s": round(step.num_seqs / (ms * 1e-3), 1)}


def scenario_steps(pkv, device, sc, steps, physical_blocks):
    """Full decode steps of a block-sharing scenario (copy-on-write copies +
    kv_write + attention), every step's inputs resident on the device, the
    pools restored between an untimed and the timed pass."""
    k_cache, v_cache = sc.k_cache.to(device), sc.v_cache.to(device)
    plan = []
    logical = unique = copies = 0
    for _ in range(steps):
        st = sc.next_step()
        plan.append({k: getattr(st, k).to(device) for k in
                     ("q", "k_new", "v_new", "slot_mapping", "block_tables", "seq_lens", "cow_pairs")}
                    | {"max_seq_len": st.max_seq_len, "step": st})
        logical += attention_bytes(st)
        unique += physical_blocks() * sc.num_kv_heads * sc.block_size * sc.head_dim * 4
        copies += int(st.cow_pairs.shape[0])
    ws_bytes = max(pkv.decode_workspace_bytes(int(p["q"].shape[0]), sc.num_q_heads,
                                              p["max_seq_len"], sc.block_size) for p in plan)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=device)
    outs = {int(p["q"].shape[0]): None for p in plan}
    for S in outs:
        outs[S] = torch.empty((S, sc.num_q_heads, sc.head_dim), dtype=plan[0]["q"].dtype,
                              device=device)
    tokens = sum(int(p["q"].shape[0]) for p in plan)

    def run_all():
        for p in plan:
            if p["cow_pairs"].numel():
                pkv.copy_blocks(k_cache, v_cache, p["cow_pairs"])
            pkv.kv_write(p["k_new"], p["v_new"], p["slot_mapping"], k_cache, v_cache)
            pkv.paged_decode_attention(p["q"], k_cache, v_cache, p["block_tables"], p["seq_lens"],
                                       sc.num_kv_heads, p["step"].scale,
                                       outs[int(p["q"].shape[0])],
                                       max_seq_len=p["max_seq_len"], workspace=ws)

    def restore():  # the initial pools, so every timed pass replays the same work
        k_cache.copy_(sc.k_cache.to(device))
        v_cache.copy_(sc.v_cache.to(device))
        torch.cuda.synchronize()

    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn):
        restore()
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    run_all()  # warm-up pass (also replays the copies and writes once)
    eager_ms = timed(run_all)
    # the same steps captured once in a CUDA graph: device time without the
    # host's per-call cost, as a serving loop that captures its steps runs them
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run_all()
    graph.replay()  # first replay off the clock
    ms = timed(graph.replay)
    hbm, _ = measured_peaks()
    return {"ms_per_step": round(ms / steps, 4),
            "timing": "one CUDA-graph replay of all steps (the pools restored before it)",
            "ms_per_step_eager": round(eager_ms / steps, 4),
            "decode_tokens_per_s": round(tokens / (ms * 1e-3), 1),
            "cow_copies": copies,
            "logical_gbs": round(logical / (ms * 1e-3) / 1e9, 1),
            "logical_frac_of_measured_peak": round(logical / (ms * 1e-3) / 1e9 / hbm, 4),
            "unique_kv_gbs": round(unique / (ms * 1e-3) / 1e9, 1),
            "note": "logical bytes count shared blocks once per sequence that reads them (L2 "
                    "serves the repeats); unique bytes count each physical block once"}


def prefix_sharing_steps(pkv, W, device, prompt_len, steps=256):
    """Decode steps of the prefix-sharing scenario (16 prompts x 8 samples)."""
    sc = W.PrefixSharingScenario(prompt_len=prompt_len, decode_steps=steps)
    res = scenario_steps(pkv, device, sc, steps, sc.unique_blocks_in_use)
    return {"workload": f"16 prompts x {prompt_len} tokens x 8 samples, {steps} decode steps, "
                        "block 32, 32 q / 8 kv heads, bf16", **res}


def beam_search_steps(pkv, W, device, prompt_len=2048, width=16, steps=128):
    """Decode steps of beam search over one prompt: every step a seeded number
    of beams is dropped and a survivor forked in their place, sharing all of
    its blocks; a beam whose last block is shared copies it before writing."""
    sc = W.BeamSearchScenario(prompt_len=prompt_len, width=width, decode_steps=steps)
    res = scenario_steps(pkv, device, sc, steps,
                         lambda: int((sc.manager.refcount > 0).sum()))
    return {"workload": f"beam search over one {prompt_len}-token prompt, {width} beams, "
                        f"{steps} decode steps, block 16, 32 q / 8 kv heads, bf16",
            **res, "mean_block_saving": round(float(sum(sc.savings) / len(sc.savings)), 4)}


def swap_throughput(pkv, W, device, victims=16, reps=20):
    """Preemption by swap: every block of `victims` sequences of the GQA batch
    to a page-locked host pool and back, one launch per direction."""
    st = W.gqa_batch()
    k_dev, v_dev = st.k_cache.to(device), st.v_cache.to(device)
    lens = st.seq_lens.to(torch.int64)
    ids = torch.cat([st.block_tables[s, :(int(lens[s]) + st.block_size - 1) // st.block_size]
                     for s in range(victims)]).to(torch.int64)
    n = int(ids.numel())
    host_k = torch.empty((n,) + tuple(st.k_cache.shape[1:]), dtype=st.k_cache.dtype).pin_memory()
    host_v = torch.empty_like(host_k).pin_memory()
    out_pairs = torch.stack([ids, torch.arange(n, dtype=torch.int64)], 1).to(device)
    in_pairs = torch.stack([torch.arange(n, dtype=torch.int64), ids], 1).to(device)
    block_bytes = st.num_kv_heads * st.block_size * st.head_dim * 2 * 2
    stream = torch.cuda.current_stream()
    res = {}
    for name, args in (("out_d2h", (k_dev, v_dev, host_k, host_v, out_pairs)),
                       ("in_h2d", (host_k, host_v, k_dev, v_dev, in_pairs))):
        for _ in range(3):
            pkv.swap_blocks(*args)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            pkv.swap_blocks(*args)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        res[name] = {"ms": round(ms, 4), "gbs": round(n * block_bytes / (ms * 1e-3) / 1e9, 1)}
    # the link's bound: one contiguous copy engine transfer of the same bytes each way
    flat_host = torch.empty(n * block_bytes, dtype=torch.uint8).pin_memory()
    flat_dev = torch.empty(n * block_bytes, dtype=torch.uint8, device=device)
    for name, (dst, src) in (("out_d2h", (flat_host, flat_dev)), ("in_h2d", (flat_dev, flat_host))):
        for _ in range(3):
            dst.copy_(src, non_blocking=True)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            dst.copy_(src, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        gbs = n * block_bytes / (ms * 1e-3) / 1e9
        res[name]["contiguous_copy_gbs"] = round(gbs, 1)
        res[name]["frac_of_contiguous_copy"] = round(res[name]["gbs"] / gbs, 4)
    del k_dev, v_dev, flat_dev
    torch.cuda.empty_cache()
    return {"workload": f"all {n} blocks ({n * block_bytes / 1e6:.1f} MB of K+V) of {victims} "
                        "GQA-batch sequences, device <-> page-locked host pool, one launch",
            "bound": "the CPU-GPU link: one contiguous copy of the same bytes (copy engine)",
            **res}


def measured_bf16_tflops():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def time_prefill(pkv, st, device, reps=20):
    """Device ms per causal paged prefill call of step `st` (attention alone,
    after its kv_write), CUDA events around `reps` back-to-back calls."""
    dev = {k: getattr(st, k).to(device) for k in
           ("q", "cu_q", "k_new", "v_new", "slot_mapping", "block_tables", "seq_lens",
            "k_cache", "v_cache")}
    pkv.kv_write(dev["k_new"], dev["v_new"], dev["slot_mapping"], dev["k_cache"], dev["v_cache"])
    out = torch.empty_like(dev["q"])

    def call():
        pkv.paged_prefill_attention(dev["q"], dev["cu_q"], dev["k_cache"], dev["v_cache"],
                                    dev["block_tables"], dev["seq_lens"], st.scale, out,
                                    max_q_len=st.max_q_len, max_seq_len=st.max_seq_len)

    for _ in range(3):
        call()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    del dev, out
    torch.cuda.empty_cache()
    return e0.elapsed_time(e1) / reps


def measure_prefill(pkv, W, device, reps=20):
    """Causal paged prefill of the prefill batch (attention alone, after kv_write)."""
    st = W.prefill_batch()
    ms = time_prefill(pkv, st, device, reps)
    flops = st.causal_flops()
    peak, kind = measured_bf16_tflops()
    tflops = flops / (ms * 1e-3) / 1e12
    return {"workload": f"{st.num_seqs} prompts of 512..2048 tokens (total {int(st.q.shape[0])}), "
                        "causal, 32 q / 8 kv heads, bf16, block 16",
            "attention_ms": round(ms, 4), "useful_tflops": round(tflops, 1),
            "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(tflops / peak, 4),
                         "peak_kind": f"{kind} bf16 dense (burst)"},
            "prompt_tokens_per_s": round(int(st.q.shape[0]) / (ms * 1e-3), 1)}


def prefill_shapes(pkv, W, device):
    """Causal paged prefill on other shapes (32 q / 8 kv heads, block 16)."""
    batch = W.prefill_batch()
    q_lens = (batch.cu_q[1:] - batch.cu_q[:-1]).tolist()
    g = torch.Generator().manual_seed(13)
    mixed_ctx = torch.randint(100, 600, (253,), generator=g).tolist()
    mixed_q = [1] * 253
    for i, n in ((7, 1500), (100, 700), (200, 1100)):  # three prompts among one-token steps
        mixed_ctx[i], mixed_q[i] = 0, n
    shapes = {
        "batch_fp16": ("the prefill batch's prompts in fp16", [0] * len(q_lens), q_lens,
                       "float16"),
        "uniform_16x2048": ("16 prompts of 2048 tokens", [0] * 16, [2048] * 16, "bfloat16"),
        "ctx4096_q512x16": ("16 x 512 queries after 4096 cached tokens", [4096] * 16, [512] * 16,
                            "bfloat16"),
        "short_256x128": ("256 prompts of 128 tokens", [0] * 256, [128] * 256, "bfloat16"),
        "mixed_253": ("250 one-token steps (100..599 cached) and prompts of 1500, 700, 1100",
                      mixed_ctx, mixed_q, "bfloat16"),
    }
    peak, kind = measured_bf16_tflops()
    res = {}
    for i, (name, (what, ctx, ql, dtype)) in enumerate(shapes.items()):
        st = W.build_prefill_step(name, ctx, ql, 32, 8, 16, dtype, seed=300 + i)
        ms = time_prefill(pkv, st, device)
        tflops = st.causal_flops() / (ms * 1e-3) / 1e12
        res[name] = {"workload": f"{what}, {dtype}", "attention_ms": round(ms, 4),
                     "useful_tflops": round(tflops, 1),
                     "frac_of_measured_bf16": round(tflops / peak, 4)}
    return res


def other_workloads(pkv, W, device, all_configs):
    extra = {"long_context": measure_attention(
        pkv, W.long_context(), device, "long_context",
        "8 sequences x 32768 tokens, 32 q / 8 kv heads, bf16, block 16"),
        "prefill": measure_prefill(pkv, W, device),
        "gqa_fp8": measure_attention_fp8(
            pkv, W.gqa_batch(), device,
            "GQA decode batch over 8-bit pools: 64 sequences 512..4096, 32 q / 8 kv heads, "
            "bf16 queries, block 16"),
        "long_context_fp8": measure_attention_fp8(
            pkv, W.long_context(), device,
            "8 sequences x 32768 tokens over 8-bit pools, 32 q / 8 kv heads, bf16 queries")}
    if all_configs:
        for bs in (16, 32):
            st = W.tiny(bs)
            extra[f"tiny_B{bs}"] = measure_attention(
                pkv, st, device, "tiny", f"5 sequences 37/91/128/201/511, 8 heads, fp16, block {bs}")
        extra["opt13b_like"] = measure_attention(
            pkv, W.opt13b_like(), device, "opt13b_like",
            "128 sequences, log-normal lengths (cap 2048), 40 heads MHA, fp16, block 16")
        sweep = {}
        for bs in (8, 16, 32, 64, 128):
            st = W.gqa_batch(block_size=bs)
            lens = st.seq_lens.to(torch.int64)
            allocated = int(((lens + bs - 1) // bs).sum()) * bs
            rec = measure_attention(pkv, st, device, "gqa", "GQA batch")
            rec.pop("workload")
            rec["position_utilisation"] = round(int(lens.sum()) / allocated, 5)
            rec["tail_slots"] = allocated - int(lens.sum())
            sweep[str(bs)] = rec
        extra["block_size_sweep_gqa_batch"] = sweep
        extra["swap_gqa_batch"] = swap_throughput(pkv, W, device)
        extra["writes_and_copies"] = writes_throughput(pkv, W, device)
        extra["prefix_sharing"] = prefix_sharing_steps(pkv, W, device, 1024)
        extra["prefix_sharing_cow"] = prefix_sharing_steps(pkv, W, device, 1040)
        extra["beam_search"] = beam_search_steps(pkv, W, device)
        extra["decode_shapes"] = decode_shapes(pkv, W, device)
        extra["prefill_shapes"] = prefill_shapes(pkv, W, device)
    return extra


def writes_throughput(pkv, W, device, n_pairs=2000):
    """kv_write (one decode token per sequence, and a whole prefill batch) and
    copy_blocks (scattered block pairs), each as a CUDA-graph replay."""
    hbm, _ = measured_peaks()
    res = {}
    st = W.gqa_batch()
    kc, vc = st.k_cache.to(device), st.v_cache.to(device)
    pre = W.prefill_batch()
    pk, pv, ps = pre.k_new.to(device), pre.v_new.to(device), pre.slot_mapping.to(device)
    pkc, pvc = pre.k_cache.to(device), pre.v_cache.to(device)
    dk, dv, dsm = st.k_new.to(device), st.v_new.to(device), st.slot_mapping.to(device)
    # distinct sources and destinations drawn from the pool (a seeded permutation)
    g = torch.Generator().manual_seed(11)
    perm = torch.randperm(kc.shape[0], generator=g)[: 2 * n_pairs]
    pairs = torch.stack([perm[:n_pairs], perm[n_pairs:]], 1).to(torch.int64).to(device)
    block_bytes = st.num_kv_heads * st.block_size * st.head_dim * 2 * 2  # K and V
    cases = {
        "kv_write_decode": (lambda: pkv.kv_write(dk, dv, dsm, kc, vc),
                            kv_write_bytes(st), f"{st.num_seqs} tokens, 8 kv heads, bf16"),
        "kv_write_prefill": (lambda: pkv.kv_write(pk, pv, ps, pkc, pvc), kv_write_bytes(pre),
                             f"{int(ps.numel())} prompt tokens, 8 kv heads, bf16"),
        "copy_blocks": (lambda: pkv.copy_blocks(kc, vc, pairs), n_pairs * block_bytes * 2 + 16 * n_pairs,
                        f"{n_pairs} scattered pairs of 16-token blocks, 8 kv heads, bf16 "
                        "(K and V read and written)"),
    }
    for name, (call, nbytes, what) in cases.items():
        ms = time_calls_graph(call, flush=nbytes < L2_FLUSH_BYTES, clean_l2=False)
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[name] = {"workload": what, "us": round(ms * 1e3, 2), "bytes": int(nbytes),
                     "gbs": round(gbs, 1), "frac_of_measured_peak": round(gbs / hbm, 4),
                     "timing": "CUDA graph replay, L2 evicted before every call"}
    del kc, vc, pkc, pvc
    torch.cuda.empty_cache()
    return res


# what the --only lines of the workloads that are not decode attention measure
ONLY_METRICS = {"swap": "block swap GB/s between a device pool and a page-locked host pool",
                "writes": "kv_write / copy_blocks GB/s",
                "prefill_shapes": "causal paged prefill useful TFLOP/s"}

# (sequences, tokens each): from one sequence to a few dozen, 32 q / 8 kv heads
DECODE_SHAPES = ((1, 2048), (4, 4096), (1, 32768), (16, 2048), (32, 1024))


def decode_shapes(pkv, W, device):
    """Equal-length decode batches with few (sequence, KV head) segments, each
    cut over many warps of the streaming grid."""
    res = {}
    for i, (S, n) in enumerate(DECODE_SHAPES):
        st = W.build_decode_step("shape", [n - 1] * S, 32, 8, 16, "bfloat16", seed=90 + i,
                                 pool_factor=1.0)
        res[f"S{S}_n{n}"] = measure_attention(
            pkv, st, device, "shape", f"{S} x {n} tokens, 32 q / 8 kv heads, bf16, block 16")
        del st
    return res


def single_workload(pkv, W, device, name):
    """One workload's decode attention (or full prefix-sharing steps) measured alone."""
    if name == "tiny":
        return {f"B{bs}": measure_attention(
            pkv, W.tiny(bs), device, "tiny",
            f"5 sequences 37/91/128/201/511, 8 heads, fp16, block {bs}") for bs in (16, 32)}
    if name == "opt13b_like":
        return measure_attention(
            pkv, W.opt13b_like(), device, "opt13b_like",
            "128 sequences, log-normal lengths (cap 2048), 40 heads MHA, fp16, block 16")
    if name == "long_context":
        return measure_attention(pkv, W.long_context(), device, "long_context",
                                 "8 sequences x 32768 tokens, 32 q / 8 kv heads, bf16, block 16")
    if name == "long_context_fp8":
        return measure_attention_fp8(
            pkv, W.long_context(), device,
            "8 sequences x 32768 tokens over 8-bit pools, 32 q / 8 kv heads, bf16 queries")
    if name == "swap":
        return swap_throughput(pkv, W, device)
    if name == "writes":
        return writes_throughput(pkv, W, device)
    if name == "beam_search":
        return beam_search_steps(pkv, W, device)
    if name == "decode_shapes":
        return decode_shapes(pkv, W, device)
    if name == "prefill_shapes":
        return prefill_shapes(pkv, W, device)
    return prefix_sharing_steps(pkv, W, device, 1040 if name == "prefix_sharing_cow" else 1024)


def run_pkv(args, rank, world, local_rank):
    import paged_kv_cache_242_gb300 as pkv
    from paged_kv_cache_242_gb300 import workloads as W

    pkv._lib.load()  # fail loudly: no fallback
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    step = W.gqa_batch(seed=args.seed + 7919 * rank)
    dev = {k: v.to(device) for k, v in {
        "q": step.q, "k_new": step.k_new, "v_new": step.v_new, "slot_mapping": step.slot_mapping,
        "block_tables": step.block_tables, "seq_lens": step.seq_lens,
        "cow_pairs": step.cow_pairs, "k_cache": step.k_cache, "v_cache": step.v_cache}.items()}
    fp8 = args.kv == "fp8"
    if fp8:  # 8-bit pools holding the same values, quantised by the 8-bit write
        nb, h, b, d = step.k_cache.shape
        kc8 = torch.empty((nb, h, b, d), dtype=torch.uint8, device=device)
        vc8 = torch.empty_like(kc8)
        rows = [dev[k].permute(0, 2, 1, 3).reshape(nb * b, h, d).contiguous()
                for k in ("k_cache", "v_cache")]
        pkv.kv_write_fp8(rows[0], rows[1], torch.arange(nb * b, dtype=torch.int64, device=device),
                         kc8, vc8, FP8_K_SCALE, FP8_V_SCALE)
        del rows
        dev["k_cache"], dev["v_cache"] = kc8, vc8
        if args.partition_size:
            raise SystemExit("--kv fp8 streams (automatic mode): no --partition-size")
    kvb = 1 if fp8 else 2
    part = pkv.decode_partition_size(step.max_seq_len, step.block_size, args.partition_size)
    split = part < step.max_seq_len
    ws_bytes = pkv.decode_workspace_bytes(step.num_seqs, step.num_q_heads, step.max_seq_len,
                                          step.block_size, args.partition_size)
    workspace = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=device)
    out = torch.empty_like(dev["q"])
    err = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    has_cow = step.cow_pairs.numel() > 0

    def attend(q, block_tables, seq_lens, o=None):
        o = out if o is None else o
        if fp8:
            pkv.paged_decode_attention_fp8(q, dev["k_cache"], dev["v_cache"], block_tables,
                                           seq_lens, FP8_K_SCALE, FP8_V_SCALE, step.scale, o,
                                           max_seq_len=step.max_seq_len, workspace=workspace,
                                           err_flag=err)
        else:
            pkv.paged_decode_attention(q, dev["k_cache"], dev["v_cache"], block_tables, seq_lens,
                                       step.num_kv_heads, step.scale, o,
                                       max_seq_len=step.max_seq_len,
                                       partition_size=args.partition_size, workspace=workspace,
                                       err_flag=err)

    def put(k_new, v_new, slot_mapping):
        if fp8:
            pkv.kv_write_fp8(k_new, v_new, slot_mapping, dev["k_cache"], dev["v_cache"],
                             FP8_K_SCALE, FP8_V_SCALE, err_flag=err)
        else:
            pkv.kv_write(k_new, v_new, slot_mapping, dev["k_cache"], dev["v_cache"], err_flag=err)

    def attention():
        attend(dev["q"], dev["block_tables"], dev["seq_lens"])

    def write():
        if has_cow:
            pkv.copy_blocks(dev["k_cache"], dev["v_cache"], dev["cow_pairs"], err_flag=err)
        put(dev["k_new"], dev["v_new"], dev["slot_mapping"])

    # kv_write, copy_blocks when pairs exist, the attention kernel, and the
    # merge kernel (always in automatic mode; with explicit partitions only
    # when a sequence spans several)
    merges = 1 if (args.partition_size == 0 or split) else 0
    launches_per_step = 1 + (1 if has_cow else 0) + 1 + merges
    for _ in range(max(3, args.warmup)):
        write()
        attention()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()

    K = args.steps
    # Events around the attention call on every 8th step only: an event
    # recorded between two kernels stops them from overlapping their launch
    # (programmatic dependent launch), so the other steps run undisturbed.
    sample_every = 8
    sampled = list(range(0, K, sample_every))
    ev = {i: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for i in sampled}
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(device.index if device.index is not None else 0)
    clocks.start()
    time.sleep(0.3)  # let the sampler take its first reading
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(K):
        write()
        pair = ev.get(i)
        if pair is not None:
            pair[0].record(stream)
        attention()
        if pair is not None:
            pair[1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    clock_info = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    total_ms = start.elapsed_time(end)
    attn_ms = sum(a.elapsed_time(b) for a, b in ev.values()) / len(ev)
    assert int(err.item()) == 0, f"device error flag {int(err.item())}"
    total_ms = max_over_ranks(total_ms, world, device)
    ms_per_step = total_ms / K
    a_bytes = attention_bytes(step, kvb)
    step_bytes = a_bytes + kv_write_bytes(step, kvb) + copy_bytes(step) // (2 // kvb)
    value = world * step_bytes / (ms_per_step * 1e-3) / 1e9
    tokens_per_s = world * step.num_seqs / (ms_per_step * 1e-3)

    # ---------------- end to end through the public API ----------------
    e2e = None
    if not args.no_e2e:
        # A step's host inputs (query, new keys / values, slot mapping, block
        # tables, lengths) staged in one pinned buffer: one host-to-device
        # copy per step, device tensors are views of one device buffer.
        host_inputs = {"q": step.q, "k_new": step.k_new, "v_new": step.v_new,
                       "slot_mapping": step.slot_mapping, "block_tables": step.block_tables,
                       "seq_lens": step.seq_lens}
        layout, off = {}, 0
        for k, t in host_inputs.items():
            layout[k] = (off, t.numel() * t.element_size(), t.dtype, tuple(t.shape))
            off = (off + layout[k][1] + 255) // 256 * 256
        staged = torch.empty(off, dtype=torch.uint8, pin_memory=True)
        for k, t in host_inputs.items():
            o, n, _, _ = layout[k]
            staged[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8))
        h2d = off
        d2h = out.numel() * out.element_size()
        e2e_steps = max(10, min(K, 2000))
        # Two device slots for the inputs and two for the output.  A copy
        # stream moves step i+1's inputs in while step i computes and step
        # i's output out while step i+1 computes; events order each slot's
        # reuse.  Every step still copies its own inputs and reads its output.
        slots_dev = [torch.empty(off, dtype=torch.uint8, device=device) for _ in range(2)]
        slot_inputs = [{k: buf[o:o + n].view(dt).view(shape)
                        for k, (o, n, dt, shape) in layout.items()} for buf in slots_dev]
        slot_out = [torch.empty_like(out) for _ in range(2)]
        out_host = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
        copy_stream = torch.cuda.Stream(device)
        ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of the slot landed
        ev_done = [torch.cuda.Event() for _ in range(2)]  # the slot's step finished
        ev_out = [torch.cuda.Event() for _ in range(2)]   # the slot's output left

        def copy_in(i):
            sl = i % 2
            with torch.cuda.stream(copy_stream):
                if i >= 2:
                    copy_stream.wait_event(ev_done[sl])
                slots_dev[sl].copy_(staged, non_blocking=True)
                ev_in[sl].record(copy_stream)

        # 16-bit pools: each slot's two calls validated and marshalled once (the
        # plans of the public API); 8-bit pools: the plain calls
        plans = None
        if not fp8:
            plans = [(pkv.KVWritePlan(x["k_new"], x["v_new"], x["slot_mapping"], dev["k_cache"],
                                      dev["v_cache"], err_flag=err),
                      pkv.DecodeAttentionPlan(x["q"], dev["k_cache"], dev["v_cache"],
                                              x["block_tables"], x["seq_lens"], slot_out[sl],
                                              max_seq_len=step.max_seq_len,
                                              num_kv_heads=step.num_kv_heads, scale=step.scale,
                                              partition_size=args.partition_size,
                                              workspace=workspace, err_flag=err))
                     for sl, x in enumerate(slot_inputs)]

        def step_calls(sl):
            if plans is not None:
                plans[sl][0].run()
                plans[sl][1].run()
            else:
                x = slot_inputs[sl]
                put(x["k_new"], x["v_new"], x["slot_mapping"])
                attend(x["q"], x["block_tables"], x["seq_lens"], slot_out[sl])

        def compute(i):
            sl = i % 2
            stream.wait_event(ev_in[sl])
            if i >= 2:
                stream.wait_event(ev_out[sl])
            step_calls(sl)
            ev_done[sl].record(stream)

        def copy_out(i):
            sl = i % 2
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(ev_done[sl])
                out_host[sl].copy_(slot_out[sl], non_blocking=True)
                ev_out[sl].record(copy_stream)

        def pipelined(n):
            copy_in(0)
            for i in range(n):
                if i + 1 < n:
                    copy_in(i + 1)
                compute(i)
                copy_out(i)
            torch.cuda.synchronize(device)

        def synchronous_step():
            slots_dev[0].copy_(staged, non_blocking=True)
            step_calls(0)
            out_host[0].copy_(slot_out[0], non_blocking=True)
            stream.synchronize()

        pipelined(4)
        for _ in range(3):
            synchronous_step()
        if world > 1:
            torch.distributed.barrier()
        t0 = time.perf_counter()
        pipelined(e2e_steps)
        e2e_s = (time.perf_counter() - t0) / e2e_steps
        if world > 1:
            torch.distributed.barrier()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            synchronous_step()
        sync_s = (time.perf_counter() - t0) / e2e_steps
        e2e_s = max_over_ranks(e2e_s, world, device)
        sync_s = max_over_ranks(sync_s, world, device)
        # the host copy of the last step's output is that step's device output
        last = (e2e_steps - 1) % 2
        assert torch.equal(out_host[last], slot_out[last].cpu())
        step_b = a_bytes + kv_write_bytes(step, kvb)
        e2e = {"value": round(world * step_b / e2e_s / 1e9, 2),
               "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(e2e_s * 1e3, 4), "steps": e2e_steps,
               "decode_tokens_per_s": round(world * step.num_seqs / e2e_s, 1),
               "mode": "pipelined: step i+1's inputs are copied in and step i's output is "
                       "copied out on a second stream while step i computes; host clock "
                       "around all steps",
               "calls": "KVWritePlan / DecodeAttentionPlan (validated once per input slot)"
                        if plans is not None else "kv_write_fp8 / paged_decode_attention_fp8",
               "synchronous": {"value": round(world * step_b / sync_s / 1e9, 2),
                               "ms_per_step": round(sync_s * 1e3, 4),
                               "mode": "copy in, compute, copy out, synchronise: every step"}}

    # ---------------- other workloads: attention alone ----------------
    extra = {}
    if not args.no_extra and rank == 0:
        del dev, workspace
        torch.cuda.empty_cache()
        extra = other_workloads(pkv, W, device, args.all_configs)

    if rank != 0:
        return
    hbm, kind = measured_peaks()
    achieved = a_bytes / (attn_ms * 1e-3) / 1e9
    roofline = {"kernel": ("paged_decode_attention_fp8" if fp8 else "paged_decode_attention")
                          + " (streaming kernel + merge kernel)",
                "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "peak_kind": f"{kind} (burst copy)",
                "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
                "algorithmic_bytes_per_launch": a_bytes,
                "avg_call_ms": round(attn_ms, 5),
                "traffic": traffic_for(args.kv),
                "traffic_note": "ncu dram__bytes_read.sum + dram__bytes_write.sum of the streaming "
                                "kernel alone (the merge kernel reads its ~4 MB of partials from L2)"}
    cpu = None
    if world == 1 and not args.no_cpu and not fp8:
        rate, _, desc, threads = oracle_sample_rate(step, 10.0)
        cpu = {"kind": "oracle", "value": round(rate / 1e9, 4), "unit": UNIT, "cores": threads,
               "sample": desc}
        # the same oracle on one core, on the first 8 sequences
        rate1, _, desc1, _ = oracle_sample_rate(step, 5.0, max_seqs=8, threads=1)
        cpu["single_core"] = {"value": round(rate1 / 1e9, 4), "unit": UNIT, "cores": 1,
                              "sample": desc1}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": dict(workload_config(step, part),
                                            kv_format="E4M3 codes, one scale per pool" if fp8
                                            else "bf16"),
        "decode_tokens_per_s": round(tokens_per_s, 1),
        "step_bytes": step_bytes, "gpu_launches": launches_per_step * K,
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clock_info,
    }
    if extra:
        line["extra"] = extra
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "gloo" if args.impl == "reference" else "nccl"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        elif args.only in SINGLE_WORKLOADS:
            import paged_kv_cache_242_gb300 as pkv
            from paged_kv_cache_242_gb300 import workloads as W

            pkv._lib.load()
            device = torch.device("cuda", local_rank)
            torch.cuda.set_device(device)
            rec = single_workload(pkv, W, device, args.only)
            if rank == 0:
                print(json.dumps(dict(metric=ONLY_METRICS.get(args.only, METRIC), only=args.only,
                                      **rec)), flush=True)
        elif args.only == "prefill":
            import paged_kv_cache_242_gb300 as pkv
            from paged_kv_cache_242_gb300 import workloads as W

            pkv._lib.load()
            device = torch.device("cuda", local_rank)
            torch.cuda.set_device(device)
            rec = measure_prefill(pkv, W, device)
            if rank == 0:
                print(json.dumps(dict(metric="causal paged prefill useful TFLOP/s",
                                      value=rec["useful_tflops"], unit="TFLOP/s", **rec)),
                      flush=True)
        else:
            run_pkv(args, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
