"""Benchmark: batched decode over the rotated K4/V3 quantised KV cache.

Workload (default): 32 sequences, 16 query heads / 2 kv heads, head_dim 256,
each sequence holding a 32768-token K4/V3 cache (keys with x20 outlier
channels, values ~N(0,1)); one step = append one new token per sequence (K1
append kernel) + attend one bf16 query per sequence (split-KV attention +
combine).  Metric: KV tokens scanned per second (B x tokens attended per step),
whole job.  Inputs are resident in HBM before the timed region; the cache
(537 MB read per step) is larger than the 129 MB L2, so no flush is needed.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs its own replica on its own GPU (the path has
no exchange step); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import seeded_inputs as si  # noqa: E402

METRIC = "quantized-KV decode attention: KV tokens/s and HBM GB/s vs ~8 TB/s roofline"
UNIT = "KV tokens/s"
K_ROW, V_ROW = 144, 112  # algorithmic bytes per token-head: codes + bf16 scales/biases


def row_bytes(bits: int, group_size: int) -> int:
    """Bytes of one packed row: 256 * bits / 8 of codes + a bf16 scale and bias per group."""
    return 256 * bits // 8 + 2 * 2 * (256 // group_size)

# DRAM bytes (read + write) per iq_attend call on the default workload, from one
# ncu capture (dram__bytes_read.sum + dram__bytes_write.sum of attend_kernel and
# combine_kernel).  Reported only while the attention source is the one that
# was measured.
TRAFFIC = {"source": "rotated_bit_quantized_gb300/csrc/iq_attend.cu",
           "sha256": "a338e6b50448f303315622c9ec90818b34a5646a7475357717509774e45c4edd",
           "bytes": ((539.385088 + 2.726912 + 2.936576 + 0.0) + (539.399680 + 0.105728 + 2.934528 + 0.002048)) / 2 * 1e6}


def measured_traffic():
    import hashlib
    if not TRAFFIC["sha256"]:
        return None
    try:
        with open(os.path.join(ROOT, TRAFFIC["source"]), "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()
    except OSError:
        return None
    return TRAFFIC["bytes"] if digest == TRAFFIC["sha256"] else None


# nominal GB300 figures, reported beside the measured peaks: HBM3e "~8 TB/s"
# (the metric's roofline) and dense bf16 tensor throughput
NOMINAL_HBM_GBS = 8000.0
NOMINAL_BF16_TFLOPS = 2250.0


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples (200 ms) while the measured work runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) != 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def physical_gpu(local: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    parts = [x for x in vis.split(",") if x.strip()]
    if local < len(parts) and parts[local].strip().isdigit():
        return int(parts[local])
    return local


def reduce_across_ranks(ms: float, tokens: int, device=None):
    """(max of the ranks' timed milliseconds, sum of their tokens); identity on one rank.

    Replicas share nothing on the data path: this is the only collective, and it
    runs outside the timed region.
    """
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(ms), int(tokens)
    dev = device if device is not None else torch.device("cpu")
    t = torch.tensor([float(ms)], dtype=torch.float64, device=dev)
    n = torch.tensor([float(tokens)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), int(round(n.item()))


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def make_workload(wid: int, steps_total: int, dev, batch: int | None = None, fmt=(4, 3, 64)):
    """Device-resident cache holding the prefill, plus per-step inputs (host and device).

    `batch` replaces the workload's sequence count (smaller cases for profiling)."""
    from rotated_bit_quantized_gb300 import IQCache, Rotation
    w = dict(si.WORKLOADS[wid])
    if batch is not None:
        w["B"] = batch
    B, Hkv, Hq = w["B"], w["Hkv"], w["Hq"]
    rot = Rotation(0, 256, dev)
    cache = IQCache(B, Hkv, device=dev, capacity=256, k_bits=fmt[0], v_bits=fmt[1], group_size=fmt[2])
    cache.reserve(w["prefill"] + w["append"] * steps_total + 256)
    full_k, full_v = si.kv_tokens(w["seed"], B, Hkv, w["prefill"], outliers=w["outliers"])
    chunk = 4096
    for lo in range(0, w["prefill"], chunk):  # upload in slices to bound device temporaries
        hi = min(lo + chunk, w["prefill"])
        cache.append(full_k[:, :, lo:hi].to(dev), full_v[:, :, lo:hi].to(dev), rot)
    del full_k, full_v
    steps = []
    for s in range(steps_total):
        k, v = si.kv_tokens(w["seed"], B, Hkv, w["append"], outliers=w["outliers"], step=s)
        q = si.queries(w["seed"], B, Hq, w["queries"], step=s)
        steps.append((k.pin_memory(), v.pin_memory(), q.pin_memory()))
    torch.cuda.synchronize(dev)
    return w, rot, cache, steps


def preroll(dev, steps: int, per_step_s: float = 250e-6) -> None:
    """Keep the GPU busy (a spin kernel on the current stream) while the host
    queues the timed steps, so the region measures the device, not the host's
    first launches; the spin itself runs before the start event."""
    torch.cuda._sleep(int(2.1e9 * (1e-3 + per_step_s * steps)))


def run_ours(args):
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    from rotated_bit_quantized_gb300 import build as b
    b.build()
    W, K = args.warmup, args.steps
    fmt = tuple(int(x) for x in args.kv_format.split(","))
    w, rot, cache, steps = make_workload(args.workload, W + K, dev, args.batch, fmt)
    k_row, v_row = row_bytes(fmt[0], fmt[2]), row_bytes(fmt[1], fmt[2])
    B, Hkv, Hq, L = w["B"], w["Hkv"], w["Hq"], w["queries"]
    base_len = cache.lens.copy()
    dsteps = [(k.to(dev), v.to(dev), q.to(dev)) for k, v, q in steps]
    out = torch.empty((B, Hq, L, 256), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    accept = (si.accepted_lengths(W + K, B, w["append"], w["accept_seed"])
              if "accept_seed" in w else None)
    # attend_kernel + combine_kernel, plus append_kernel when the step does not fuse
    # (more than 8 query rows per kv head)
    launches_per_step = 2 if Hq // Hkv * L <= 8 and args.mask == "none" else 3
    if fmt != (4, 3, 64):  # the generic path: append, attention over the splits, split merge
        launches_per_step = 3

    mask = None
    if args.mask != "none":  # an explicit mask instead of the causal one: [B, L, S], ~90% of keys kept
        S = cache.capacity
        g = torch.Generator(device="cpu").manual_seed(w["seed"])
        keep = torch.rand((B, L, S), generator=g) < 0.9
        keep[:, :, :] |= torch.arange(S)[None, None, :] >= S - 256  # never a fully masked row
        mask = (keep if args.mask == "bool" else torch.where(keep, 0.0, float("-inf")).float()).to(dev)

    def step(i, ev=None):
        # append the step's new tokens, then attend (one library call: a single
        # attention launch that also encodes the new rows for decode-shaped
        # steps, the append launch then the attention otherwise)
        k, v, q = dsteps[i]
        if ev is not None and mask is None:
            ev[0].record(stream)
        if mask is None:
            cache.append_attend(k, v, q, rot, causal=w["causal"], out=out)
        else:
            cache.append(k, v, rot)
            if ev is not None:
                ev[0].record(stream)
            cache.attend(q, rot, mask=mask, out=out)
        if ev is not None:
            ev[1].record(stream)
        if accept is not None:  # speculative verify: keep the accepted prefix only
            cache.commit_verified_prefix(w["append"], accept[i])

    # ---- device-resident run
    for i in range(W):
        step(i)
    cache.trim(cache.lens - base_len)  # timed steps start from the 32768-token cache
    torch.cuda.synchronize(dev)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    tokens = 0
    gpu_index = physical_gpu(local)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    region_ms = []
    with ClockSampler(gpu_index) as clk:
        time.sleep(0.25)
        # timed region: K whole steps, events only at its ends (an event between
        # the append and the attention would stop the attention grid's launch
        # from overlapping the append); repeated from the same cache state and
        # the median taken
        for r in range(args.repeats):
            cache.trim(cache.lens - base_len)
            torch.cuda.synchronize(dev)
            if ws > 1:
                torch.distributed.barrier()
            torch.cuda.synchronize(dev)
            preroll(dev, K)
            start.record(stream)
            tokens = 0
            for i in range(K):
                tokens += int(cache.lens.sum()) + B * w["append"]
                step(W + i)
            stop.record(stream)
            torch.cuda.synchronize(dev)
            region_ms.append(start.elapsed_time(stop))
        # the same K steps again from the same cache state, with events around
        # every iq_attend call: the attention call's own duration (roofline)
        cache.trim(cache.lens - base_len)
        attn_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for i in range(K):
            step(W + i, attn_ev[i])
        torch.cuda.synchronize(dev)
        # keep sampling a little so short timed regions still get clock samples under load
        extra_t0 = time.time()
        while time.time() - extra_t0 < 0.6:
            cache.attend(dsteps[W + K - 1][2], rot, causal=w["causal"], out=out)
            torch.cuda.synchronize(dev)
    ms = statistics.median(region_ms)
    attn_ms = [a.elapsed_time(bq) for a, bq in attn_ev]
    status = cache.device_status()
    ms_max, tokens_all = reduce_across_ranks(ms, tokens, dev)

    # ---- end to end through the public API with host buffers
    cache.trim(cache.lens - base_len)
    host_out = torch.empty((B, Hq, L, 256), dtype=torch.bfloat16).pin_memory()
    dk = torch.empty_like(dsteps[0][0])
    dv = torch.empty_like(dsteps[0][1])
    dq = torch.empty_like(dsteps[0][2])
    torch.cuda.synchronize(dev)
    if ws > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_tokens = 0
    e0.record(stream)
    for i in range(K):
        k, v, q = steps[W + i]
        dk.copy_(k, non_blocking=True)
        dv.copy_(v, non_blocking=True)
        dq.copy_(q, non_blocking=True)
        if mask is None:
            cache.append_attend(dk, dv, dq, rot, causal=w["causal"], out=out)
        else:
            cache.append(dk, dv, rot)
            cache.attend(dq, rot, mask=mask, out=out)
        host_out.copy_(out, non_blocking=True)
        e_tokens += int(cache.lens.sum())
        if accept is not None:
            cache.commit_verified_prefix(w["append"], accept[W + i])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e_ms = e0.elapsed_time(e1)
    e_ms_max, e_tokens_all = reduce_across_ranks(e_ms, e_tokens, dev)

    if rank == 0:
        hbm, peak_kind = peaks()
        token_heads = tokens * Hkv / K  # per step, per rank
        # the call's duration in the decode loop: the timed region (events at its
        # two ends) over the K calls, each call's grids overlapping the next
        # call's start; the isolated per-call duration is reported beside it
        call_s = ms / K / 1e3
        attn_avg_s = statistics.mean(attn_ms) / 1e3
        # per call: the cache scanned (256 B per token-head) plus the append
        # (1024 B of bf16 K/V read and 256 B written per new token-head)
        call_bytes = token_heads * (k_row + v_row) + B * Hkv * w["append"] * (4 * 256 + k_row + v_row)
        if mask is not None:  # the mask entries of the scanned keys; the append runs outside the bracket
            call_bytes = token_heads * (k_row + v_row) + token_heads / Hkv * L * mask.element_size()
        achieved = call_bytes / call_s / 1e9
        h2d = (dsteps[0][0].numel() + dsteps[0][1].numel() + dsteps[0][2].numel()) * 2
        d2h = out.numel() * 2
        cpu = None if args.no_cpu_baseline else cpu_baseline_sample(args.workload, budget_s=args.cpu_seconds,
                                                                    one_core_s=args.cpu_one_core_seconds)
        append = append_throughput(dev, rot)
        append.append(append_decode_record(dev, rot))
        extra = {}
        if not args.no_sub_records and fmt == (4, 3, 64) and mask is None and args.workload == 4:
            del dsteps, steps, cache  # free the decode cache before the verify workload's
            torch.cuda.empty_cache()
            extra["single_stream"] = single_stream_record(dev, rot)
            extra["verify"] = verify_record(dev, rot, hbm)
            extra["prefill"] = prefill_record(dev, rot)
        rec = {
            "metric": METRIC, "value": tokens_all / (ms_max / 1e3), "unit": UNIT, "n_gpus": ws,
            "steps": K, "warmup": W, "ms_per_step": ms_max / K, "higher_is_better": True,
            "repeats": {"n": len(region_ms), "ms_per_step_min": min(region_ms) / K,
                        "ms_per_step_max": max(region_ms) / K,
                        "how": "the K-step region timed n times from the same cache state; value and "
                               "ms_per_step from the median region"},
            "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16 in/out, fp32 accumulate (fp16/bf16 tensor-core operands)",
            "data": "synthetic (seeded N(0,1); keys with x20 outlier channels)",
            "config": {"workload": f"{w['name']}: B={B} seqs, Hq={Hq}/Hkv={Hkv}, head_dim=256, "
                                   f"{w['prefill']}-token K{fmt[0]}/V{fmt[1]} cache (groups of {fmt[2]}), "
                                   f"append {w['append']} + attend "
                                   f"{L} query per step"
                                   + ("" if mask is None else f", explicit {args.mask} mask [B, L, {mask.shape[2]}]"),
                       "parallelism": f"replicas x{ws}",
                       "l2": f"no flush: the cache read per step ({token_heads * (k_row + v_row) / 1e6:.0f} MB) "
                             f"{'exceeds' if token_heads * (k_row + v_row) > 129e6 else 'is below'} the 129 MB L2"},
            "roofline": {"bound": "hbm",
                         "kernel": ("iq_cache_append_attend (generic format: append_any_kernel, attend_any_kernel, "
                                    "merge_any_kernel)") if fmt != (4, 3, 64) else
                                   "iq_cache_append_attend: attend_kernel (split-KV attention, new rows encoded "
                                   "in-kernel for decode steps) + combine_kernel (split merge)",
                         "achieved": achieved, "peak": hbm, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": achieved / hbm, "nominal_peak": NOMINAL_HBM_GBS,
                         "nominal_frac": achieved / NOMINAL_HBM_GBS,
                         "traffic": measured_traffic() if fmt == (4, 3, 64) else None,
                         "bytes_per_token_head": k_row + v_row, "token_heads_per_launch": token_heads,
                         "bytes_per_call": call_bytes, "avg_launch_us": call_s * 1e6,
                         "timing": "CUDA events at the two ends of the timed region over its K calls (each "
                                   "call's attention grid starts streaming while the previous call's grids "
                                   "finish); a spin kernel ahead of the start event lets the host queue the "
                                   "steps first",
                         "isolated_call_us": attn_avg_s * 1e6,
                         "isolated_frac": call_bytes / attn_avg_s / 1e9 / hbm,
                         "isolated_timing": "CUDA events around every call in a second pass over the same K "
                                            "steps (an event between calls stops their overlap)"},
            "e2e": {"value": e_tokens_all / (e_ms_max / 1e3), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_step * K,
            "clocks": clk.summary(),
            "device_status": status,
            "cpu_baseline": cpu,
            "append": append,
        }
        rec.update(extra)
        print(json.dumps(rec), flush=True)
    if ws > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


def append_throughput(dev, rot, reps: int = 10):
    """Appended tokens/s of the append kernel (rotate + quantise + pack + store)
    on two shapes: the batched-decode prefill chunks (32 sequences x 2 kv heads x
    4096 tokens per call) and one chunked-prefill chunk (1 sequence x 2 kv heads
    x 2048 tokens).  CUDA events around `reps` calls, queued behind a spin
    kernel so the region times the device, not the host's calls; each call is
    undone by a host-side trim, so every call writes the same rows."""
    from rotated_bit_quantized_gb300 import IQCache
    stream = torch.cuda.current_stream(dev)
    res = []
    for wid, B, n in ((4, 32, 4096), (3, 1, 2048)):
        w = si.WORKLOADS[wid]
        cache = IQCache(B, w["Hkv"], device=dev, capacity=n + 256)
        k, v = si.kv_tokens(w["seed"], B, w["Hkv"], n, outliers=w["outliers"])
        k, v = k.to(dev), v.to(dev)
        for _ in range(3):
            cache.append(k, v, rot)
            cache.trim(n)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        preroll(dev, reps, 100e-6)
        e0.record(stream)
        for _ in range(reps):
            cache.append(k, v, rot)
            cache.trim(n)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        sec = e0.elapsed_time(e1) / 1e3 / reps
        th = B * w["Hkv"] * n
        res.append({"workload": f"{w['name']} append: B={B} x {w['Hkv']} kv heads x {n} tokens per call",
                    "appended_tokens_per_s": B * n / sec, "token_heads_per_s": th / sec,
                    "gbs": th * (4 * 256 + K_ROW + V_ROW) / sec / 1e9, "us_per_call": sec * 1e6,
                    "bytes_per_token_head": 4 * 256 + K_ROW + V_ROW})
    return res


def append_decode_record(dev, rot, reps: int = 50):
    """The append kernel alone at n = 1 (the decode step's append when it does
    not fuse): 32 sequences x 2 kv heads, one token each, CUDA events around
    `reps` back-to-back calls, each undone by a host trim."""
    from rotated_bit_quantized_gb300 import IQCache
    w = si.WORKLOADS[4]
    B, H = w["B"], w["Hkv"]
    cache = IQCache(B, H, device=dev, capacity=512)
    k, v = si.kv_tokens(w["seed"], B, H, 1, outliers=True, step=0)
    k, v = k.to(dev), v.to(dev)
    for _ in range(5):
        cache.append(k, v, rot)
        cache.trim(1)
    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    preroll(dev, reps, 60e-6)
    e0.record(stream)
    for _ in range(reps):
        cache.append(k, v, rot)
        cache.trim(1)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    sec = e0.elapsed_time(e1) / 1e3 / reps
    th = B * H
    return {"workload": f"batched_decode append: B={B} x {H} kv heads x 1 token per call",
            "appended_tokens_per_s": B / sec, "token_heads_per_s": th / sec,
            "gbs": th * (4 * 256 + K_ROW + V_ROW) / sec / 1e9, "us_per_call": sec * 1e6,
            "bytes_per_token_head": 4 * 256 + K_ROW + V_ROW}


def single_stream_record(dev, rot, reps: int = 200):
    """Single-stream decode (1 sequence, 16/2 heads, 4096-token cache, one
    query): microseconds per attention call, back to back (events at the ends
    of `reps` calls) and isolated (events around each call)."""
    from rotated_bit_quantized_gb300 import IQCache
    w = si.WORKLOADS[2]
    B, H, Hq = w["B"], w["Hkv"], w["Hq"]
    cache = IQCache(B, H, device=dev, capacity=w["prefill"] + 256)
    k, v = si.kv_tokens(w["seed"], B, H, w["prefill"], outliers=True)
    cache.append(k.to(dev), v.to(dev), rot)
    q = si.queries(w["seed"], B, Hq, 1).to(dev)
    out = torch.empty((B, Hq, 1, 256), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(10):
        cache.attend(q, rot, out=out)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    preroll(dev, reps, 60e-6)
    e0.record(stream)
    for _ in range(reps):
        cache.attend(q, rot, out=out)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    us = e0.elapsed_time(e1) * 1e3 / reps
    iso = []
    for _ in range(50):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        cache.attend(q, rot, out=out)
        b.record(stream)
        iso.append((a, b))
    torch.cuda.synchronize(dev)
    iso_us = statistics.median(a.elapsed_time(b) * 1e3 for a, b in iso)
    th = B * H * w["prefill"]
    return {"workload": f"single_stream_decode: B={B}, Hq={Hq}/Hkv={H}, {w['prefill']}-token cache, one query",
            "us_per_call": us, "isolated_us_per_call": iso_us, "kv_tokens_per_s": B * w["prefill"] / (us / 1e6),
            "bytes_per_call": th * (K_ROW + V_ROW), "gbs": th * (K_ROW + V_ROW) / (us / 1e6) / 1e9,
            "bound": "launch latency (2.1 MB per call)", "device_status": cache.device_status()}


def verify_record(dev, rot, hbm: float, steps: int = 16, warmup: int = 3):
    """Speculative verify (8 sequences, 131072-token caches, 16/2 heads): per
    step append 4 draft tokens, attend 4 causal queries, trim the rejected
    suffix (accepted lengths from the seeded draw).  Events at the two ends of
    the timed steps; KV tokens scanned per second and the HBM fraction of the
    scanned bytes (256 B per token-head) plus the append."""
    w = si.WORKLOADS[5]
    _, _, cache, steps_in = make_workload(5, warmup + steps, dev)
    B, H, Hq, L = w["B"], w["Hkv"], w["Hq"], w["queries"]
    base = cache.lens.copy()
    dsteps = [(k.to(dev), v.to(dev), q.to(dev)) for k, v, q in steps_in]
    acc = si.accepted_lengths(warmup + steps, B, w["append"], w["accept_seed"])
    out = torch.empty((B, Hq, L, 256), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    for i in range(warmup):
        cache.append_attend(*dsteps[i], rot, causal=True, out=out)
        cache.commit_verified_prefix(w["append"], acc[i])
    cache.trim(cache.lens - base)
    torch.cuda.synchronize(dev)
    tokens, scanned = 0, 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    preroll(dev, steps, 600e-6)
    e0.record(stream)
    for i in range(warmup, warmup + steps):
        tokens += int(cache.lens.sum()) + B * w["append"]
        cache.append_attend(*dsteps[i], rot, causal=True, out=out)
        cache.commit_verified_prefix(w["append"], acc[i])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    sec = e0.elapsed_time(e1) / 1e3 / steps
    step_bytes = tokens / steps * H * (K_ROW + V_ROW) + B * H * w["append"] * (4 * 256 + K_ROW + V_ROW)
    return {"workload": f"spec_verify: B={B}, Hq={Hq}/Hkv={H}, {w['prefill']}-token caches, append {w['append']} + "
                        f"attend {L} causal queries + trim the rejected suffix per step",
            "us_per_step": sec * 1e6, "kv_tokens_per_s": tokens / steps / sec, "bytes_per_step": step_bytes,
            "gbs": step_bytes / sec / 1e9, "hbm_frac": step_bytes / sec / 1e9 / hbm,
            "nominal_frac": step_bytes / sec / 1e9 / NOMINAL_HBM_GBS, "steps": steps,
            "launches_per_step": 3, "device_status": cache.device_status()}


def prefill_record(dev, rot, chunks: int | None = None, warmup: int = 2):
    """Chunked prefill (1 sequence, 16/2 heads): 16 chunks of 2048 tokens, each
    appended and then attended by its own 2048 causal queries over the cache so
    far; attention TFLOP/s (2 * 256 flop for q.k and 2 * 256 for p.v per
    visible query-key pair and query head) against the sustained bf16 peak."""
    from rotated_bit_quantized_gb300 import IQCache
    w = si.WORKLOADS[3]
    B, Hkv, Hq, n = w["B"], w["Hkv"], w["Hq"], w["append"]
    K = w["steps"] if chunks is None else min(chunks, w["steps"])
    cache = IQCache(B, Hkv, device=dev, capacity=256)
    cache.reserve(n * w["steps"] + 256)
    ch = []
    for s_ in range(w["steps"]):
        k, v = si.kv_tokens(w["seed"], B, Hkv, n, outliers=w["outliers"], step=s_)
        q = si.queries(w["seed"], B, Hq, n, step=s_)
        ch.append((k.to(dev), v.to(dev), q.to(dev)))
    out = torch.empty((B, Hq, n, 256), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    for i in range(warmup):
        cache.append_attend(*ch[i % len(ch)], rot, causal=True, out=out)
    torch.cuda.synchronize(dev)
    cache.trim(cache.lens)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    preroll(dev, K, 100e-6)
    e0.record(stream)
    for i in range(K):
        cache.append_attend(*ch[i], rot, causal=True, out=out)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1)
    flops = prefill_flops(n, K, Hq)
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, kind = float(json.load(f)["bf16_tflops_sustained"]), "measured (sustained)"
    except Exception:
        peak, kind = 1700.0, "fallback (sustained)"
    tflops = flops / (ms / 1e3) / 1e12
    return {"workload": f"chunked_prefill: B={B}, Hq={Hq}/Hkv={Hkv}, {K} chunks of {n} tokens, each appended "
                        f"then attended by its {n} causal queries",
            "ms_per_chunk": ms / K, "tflops": tflops, "peak_tflops": peak, "peak_kind": kind,
            "frac": tflops / peak, "nominal_frac": tflops / NOMINAL_BF16_TFLOPS, "flops": flops,
            "appended_tokens_per_s": B * n * K / (ms / 1e3), "device_status": cache.device_status()}


def _oracle_sequence(wid: int, b: int):
    """Oracle cache of sequence b holding the workload's prefill (setup, untimed),
    and that sequence's step-0 inputs."""
    from oracle import rotation as orot
    from oracle.cache import OracleCache
    w = si.WORKLOADS[wid]
    Hkv, Hq = w["Hkv"], w["Hq"]
    mb = orot.blocks_bf16(orot.build_blocks(si.rotation_draws(0, 256)))
    oc = OracleCache(1, Hkv)
    pre = [si.kv_slice(w["seed"], b, h, w["prefill"], outliers=w["outliers"]) for h in range(Hkv)]
    oc.append(np.stack([x[0].float().numpy() for x in pre])[None], np.stack([x[1].float().numpy() for x in pre])[None], mb)
    new = [si.kv_slice(w["seed"], b, h, w["append"], outliers=w["outliers"], step=0) for h in range(Hkv)]
    ks = np.stack([x[0].float().numpy() for x in new])[None]
    vs = np.stack([x[1].float().numpy() for x in new])[None]
    q = si.queries(w["seed"], w["B"], Hq, w["queries"], step=0)[b:b + 1].float().numpy()
    return w, mb, oc, ks, vs, q


def _time_oracle_steps(prep, budget_s: float, max_steps: int):
    """Time whole oracle steps (append the new tokens + attend) on fresh copies
    of the prefilled cache until the budget is spent; returns (tokens, seconds, steps)."""
    import copy
    from oracle import attention
    w, mb, oc, ks, vs, q = prep
    tokens, spent, n = 0, 0.0, 0
    while n < max_steps and (n == 0 or spent < budget_s):
        c = copy.deepcopy(oc)  # untimed: each step starts from the prefilled cache
        t0 = time.perf_counter()
        c.append(ks, vs, mb)
        attention.attend(q, c, mb, causal=w["causal"])
        spent += time.perf_counter() - t0
        tokens += int(c.lens[0])
        n += 1
    return tokens, spent, n


def one_core_sample(wid: int, budget_s: float):
    """The same oracle sample on one core: a fresh interpreter (spawned, no
    CUDA) pinned to one CPU with one BLAS thread.  None if it fails."""
    code = ("import json, os, sys; os.sched_setaffinity(0, {min(os.sched_getaffinity(0))}); "
            f"sys.path.insert(0, {ROOT!r}); import bench; "
            f"t, s, n = bench._time_oracle_steps(bench._oracle_sequence({int(wid)}, 0), {float(budget_s)!r}, 10 ** 6); "
            "print(json.dumps([t, s, n]))")
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                           timeout=10 * budget_s + 300)
        tokens, spent, n = json.loads(r.stdout.strip().splitlines()[-1])
    except Exception:
        return None
    return {"value": tokens / spent, "unit": UNIT, "cores": 1, "seconds": spent, "steps": n}


def cpu_baseline_sample(wid: int, budget_s: float = 15.0, one_core_s: float = 6.0):
    """The oracle as it stands on a bounded sample of the workload's step: one
    sequence (its prefill encoded once, untimed), whole steps (append + attend)
    repeated on copies until about `budget_s` seconds of timed work, on every
    core the process may use; then the same on one core (`one_core`)."""
    prep = _oracle_sequence(wid, 0)
    w = prep[0]
    tokens, spent, n = _time_oracle_steps(prep, budget_s, 10 ** 6)
    cores = len(os.sched_getaffinity(0))
    return {"value": tokens / spent, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} repetitions of one sequence's step (append {w['append']} + attend over "
                      f"{w['prefill'] + w['append']} tokens x {w['Hkv']} kv heads, {w['Hq']} query heads); "
                      f"NumPy oracle, BLAS threads up to {cores}; prefill encode untimed",
            "seconds": spent,
            "one_core": one_core_sample(wid, one_core_s) if one_core_s > 0 else None}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    W, K = args.warmup, args.steps
    prep = _oracle_sequence(args.workload, 0)
    w = prep[0]
    _time_oracle_steps(prep, 0.0, W)  # warm-up steps, untimed
    tokens, sec, _ = _time_oracle_steps(prep, float("inf"), K)
    value = tokens / sec
    cores = len(os.sched_getaffinity(0))
    rec = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K,
           "warmup": W, "ms_per_step": 1e3 * sec / K, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64 (NumPy oracle)", "data": "synthetic",
           "config": {"workload": f"{w['name']}: one sequence of the B={w['B']} batch per step (append "
                                  f"{w['append']} + attend over {w['prefill'] + w['append']} tokens)"},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                            "sample": "one sequence per step, prefill encode untimed"},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(rec), flush=True)


def prefill_flops(chunk: int, chunks: int, q_heads: int, head_dim: int = 256) -> float:
    """Attention FLOPs of a causal chunked prefill: per query head and visible
    (query, key) pair, 2 * D for q.k and 2 * D for p.v."""
    pairs = 0
    for c in range(chunks):
        pairs += chunk * chunk * c + chunk * (chunk + 1) // 2
    return float(pairs) * q_heads * 4 * head_dim


def run_prefill(args):
    """Chunked prefill (workload 3) as its own bench line: the `prefill`
    sub-record of the default run, reported against the bf16 tensor peak."""
    ws, rank, local = dist_env()
    if rank != 0:
        return
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    from rotated_bit_quantized_gb300 import build as b
    b.build()
    from rotated_bit_quantized_gb300 import Rotation
    rot = Rotation(0, 256, dev)
    with ClockSampler(physical_gpu(local)) as clk:
        time.sleep(0.25)
        r = prefill_record(dev, rot, chunks=args.steps, warmup=args.warmup)
    rec = {"metric": "chunked prefill: attention TFLOP/s", "value": r["tflops"], "unit": "TFLOP/s", "n_gpus": 1,
           "steps": min(args.steps, 16),
           "warmup": args.warmup, "ms_per_step": r["ms_per_chunk"], "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16 in/out, fp32 accumulate (fp16 tensor-core operands)",
           "data": "synthetic", "config": {"workload": r["workload"]},
           "roofline": {"bound": "tensor", "achieved": r["tflops"], "peak": r["peak_tflops"], "peak_kind": r["peak_kind"],
                        "unit": "TFLOP/s", "frac": r["frac"], "nominal_peak": NOMINAL_BF16_TFLOPS,
                        "nominal_frac": r["nominal_frac"], "flops": r["flops"],
                        "tokens_per_s": r["appended_tokens_per_s"]},
           "clocks": clk.summary(), "device_status": r["device_status"]}
    print(json.dumps(rec), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", type=int, default=4, choices=[2, 3, 4, 5])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--cpu-one-core-seconds", type=float, default=6.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--mask", default="none", choices=["none", "bool", "add"],
                    help="attend with an explicit bool / additive mask [B, L, S] instead of the causal one")
    ap.add_argument("--kv-format", default="4,3,64",
                    help="k_bits,v_bits,group_size of the cache (4,3,64 runs the tuned kernels)")
    ap.add_argument("--batch", type=int, default=None,
                    help="sequences per step instead of the workload's own count (smaller profiling cases)")
    ap.add_argument("--repeats", type=int, default=5, help="times the K-step region is timed (median reported)")
    ap.add_argument("--no-sub-records", action="store_true",
                    help="skip the single-stream, verify and prefill sub-records")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == 3:
        run_prefill(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
