#!/usr/bin/env python3
"""Benchmark of the int8 (C8) paged KV-cache store + dequant-gather on GB300.

One step = one store of a batch's new K/V tokens into the paged cache plus one
dequant-gather of every sequence's full context (metadata plan + gather), i.e.
the whole hot path, through the C ABI of libkvc8.

Default workload: "decode" -- batch 256, one new token per sequence appended
after U{1..8192} cached tokens, 8 kv heads x head_dim 128, block 128,
18000-block pool, dynamic per-token scales: the store of 256 tokens plus the
gather of 1.13 M positions (7 GB of algorithmic traffic per step), the largest
configuration that runs both ops.  Other workloads: --workload
tiny|prefill|mixed|longctx|...  --path bf16 runs the same step on the bf16
cache without quantisation (kvc8_store_bf16 + kvc8_gather_bf16) instead of the
int8 one.  On one GPU the int8 path also times the prefill, decode, mixed and
long-context batches after the headline region and reports each op of each in
"ops"["by_workload"] (skip with --no-workload-sweep).

Timing: W untimed warm-up steps, then exactly K steps.  L2 is flushed (a
256 MiB write, then a 256 MiB read) before each timed kernel; each op is bracketed by CUDA events on
the launching stream; the step time is the sum of its ops' event times.
Barrier + synchronize on both sides; max over ranks.  SM clocks are sampled
with nvidia-smi during the timed region.

Printed: one JSON line (rank 0).  value = algorithmic HBM bytes of store +
gather per step / step time, in GB/s; tokens/s and GB/s of each op are in
"ops".  e2e = the same metric through the public API with the new tokens and
metadata copied host->device and the gathered K/V copied device->host (pinned
buffers) inside the timed region; consecutive steps overlap their uploads,
kernels and downloads on three streams, as a serving loop would.  --impl reference times the CPU oracle
instead (the reference arm: a plain single-threaded restatement of the method).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from dequant_kvc8_store_gb300 import workloads as W  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 256 << 20
DEFAULT_WORKLOAD = "decode"
# the full-size batches whose ops the int8 path also reports, one by one
SWEEP_WORKLOADS = ["prefill", "decode", "mixed", "longctx"]
L2_TEXT = "flushed before each timed op (256 MiB write, then 256 MiB read)"
METRIC = "achieved HBM GB/s (% of ~8 TB/s) and K+V tokens/s for store and dequant"
KERNEL_SOURCES = ["dequant_kvc8_store_gb300/csrc/kvc8_store.cu",
                  "dequant_kvc8_store_gb300/csrc/kvc8_gather.cu",
                  "dequant_kvc8_store_gb300/csrc/kvc8_bf16.cu",
                  "dequant_kvc8_store_gb300/csrc/kvc8_attention.cu",
                  "dequant_kvc8_store_gb300/csrc/kvc8_internal.cuh"]
PATH_TEXT = {"c8": "int8 cache", "bf16": "bf16 cache, no quantisation",
             "fused": "int8 cache, store and gather fused into one append + gather launch",
             "attention": "int8 cache, decode attention with the dequantisation fused in "
                          "(one query per sequence, 4 query heads per kv head)"}
WORKLOAD_TEXT = {
    "tiny": "tiny round trip: batch 2, q {5,19} after {3,0} cached, 2 kv heads x 64, block 16, "
            "8 blocks, dynamic scales",
    "prefill": "prefill store+gather: batch 16, prompts U[512,4096] into an empty cache, 8 kv "
               "heads x 128, block 128, 1024-block pool, dynamic per-token scales, N(0,1) with "
               "4 outlier channels/head x20",
    "decode": "decode append + full-context gather: batch 256, 1 new token, cached U[1,8192], "
              "8 x 128, block 128, 18000-block pool, dynamic scales",
    "mixed": "chunked-prefill mix: 64 seqs (32 decode, 32 chunks U[256,2048]), cached "
             "U[0,16384], 8 x 128, block 64, 20480-block pool, static scales U[0.005,0.05]",
    "longctx": "long-context gather: 8 x 131072 cached tokens, 8 x 128, block 128, 8192 "
               "blocks, dynamic scales U[0.01,0.1]",
    "prefill_block": "prefill store+gather with per-block scales: the prefill batch shapes, "
                     "one static scale per (block, kv head) U[0.01,0.1]",
    "decode_small": "decode batch cut to 64 sequences (profiling size): 1 new token, cached "
                    "U[1,8192], 8 x 128, block 128, 4160-block pool, dynamic scales",
    "mixed_small": "chunked-prefill mix with short contexts (profiling size): 64 seqs (32 "
                   "decode, 32 chunks U[256,2048]), cached U[0,1024], 8 x 128, block 64, "
                   "3328-block pool, static scales U[0.005,0.05]",
}


# the sources each timed kernel is built from (its traffic figure stays valid
# while they are unchanged)
KERNEL_FILES = {
    "store_kernel": ["kvc8_store.cu", "kvc8_internal.cuh"],
    "gather_kernel": ["kvc8_gather.cu", "kvc8_internal.cuh"],
    "append_gather_kernel": ["kvc8_gather.cu", "kvc8_internal.cuh"],
    "store_bf16_kernel": ["kvc8_bf16.cu", "kvc8_internal.cuh"],
    "gather_bf16_kernel": ["kvc8_bf16.cu", "kvc8_internal.cuh"],
    "attention_kernel": ["kvc8_attention.cu", "kvc8_internal.cuh"],
}


def _hash_files(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def source_hash() -> str:
    """Hash of all kernel sources."""
    return _hash_files(KERNEL_SOURCES)


def kernel_hash(kernel: str) -> str:
    """Hash of the sources one kernel is built from."""
    return _hash_files("dequant_kvc8_store_gb300/csrc/" + f for f in KERNEL_FILES[kernel])


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def ncu_entry(workload: str, kernel: str):
    """The committed ncu figures of one kernel on one workload, or None unless
    they were taken on the kernel's current sources.  An entry holds `bytes`
    (dram__bytes_read.sum + dram__bytes_write.sum of one full launch; scaled by
    the units processed when the capture ran on a smaller batch, named in
    `captured_on`), and, when known, `captured_bytes` and `captured_ns`
    (gpu__time_duration.sum) of the captured launch itself."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            e = json.load(f)["workloads"][workload][kernel]
        if kernel in KERNEL_FILES and e["source_hash"] == kernel_hash(kernel):
            return e
    except Exception:
        pass
    return None


def ncu_traffic(workload: str, kernel: str):
    """Per-launch DRAM bytes of one kernel on one workload (see ncu_entry)."""
    e = ncu_entry(workload, kernel)
    return None if e is None else int(e["bytes"])


def ncu_dram_frac(workload: str, kernel: str, peak: float):
    """The captured launch's DRAM bytes / its ncu duration / peak: the DRAM
    rate ncu saw, beside the algorithmic-byte fraction (writes still in L2 when
    a short kernel ends count in the algorithmic figure, not in this one)."""
    e = ncu_entry(workload, kernel)
    if e is None or not e.get("captured_ns"):
        return None
    return round(int(e["captured_bytes"]) / (float(e["captured_ns"]) * 1e-9) / 1e9 / peak, 4)


# ---------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock/throttle sampling in a background process."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None, period_ms: int = 50):
        self.uuid = uuid
        self.period_ms = period_ms
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.reader.join(timeout=2)

    def summary(self):
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            if self.uuid and parts[0] != self.uuid:
                continue
            rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------- ranks
# One process per GPU.  The path has no exchange step: every rank stores and
# gathers its own batch (its own seed), so the job scales weakly and the only
# cross-rank traffic is the barrier and the max of the timings.

def rank_seed(workload: str, rank: int) -> int:
    """Seed of a rank's batch: the workload's own seed, shifted per rank."""
    return 1000 + list(W.NAMED).index(workload) + 7919 * rank


def reduce_max(values, device=None):
    """Element-wise max of a list of floats over all ranks (no-op on one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_throughput(bytes_per_rank_step: int, world: int, step_ms_max: float) -> float:
    """Whole-job GB/s: the bytes all ranks moved in one step / the slowest rank's step."""
    return world * bytes_per_rank_step / (step_ms_max * 1e-3) / 1e9


# ---------------------------------------------------------------------------- GPU arm

class Timer:
    """L2 flush, barrier and per-op CUDA-event timing of one batch's steps."""

    def __init__(self, dev, world):
        import torch
        self.torch = torch
        self.world = world
        self.stream = torch.cuda.current_stream()
        self.flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.clean = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def flush_l2(self, v):
        # write more than L2 holds, then read another buffer that size, so L2
        # ends up holding clean lines (no write-back competes with the next op)
        self.flush.fill_(v)
        self.torch.sum(self.clean, dim=0, out=self.sink)

    def barrier(self):
        if self.world > 1:
            self.torch.distributed.barrier()
        self.torch.cuda.synchronize()

    def run(self, d, attn, path, has_store, steps, warmup, clocks=None):
        """W untimed steps, then exactly `steps` timed ones; returns the mean
        store / gather / step milliseconds (each op between its own events on
        the launching stream) and the wall time of the timed region."""
        torch, stream = self.torch, self.stream
        one_op = path in ("fused", "attention")  # no separate store op
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]

        def step(e=None):
            if not one_op:
                self.flush_l2(1)
            if e: e[0].record(stream)
            if has_store and not one_op:
                d.store(stream)
            if e: e[1].record(stream)
            self.flush_l2(2)
            if e: e[2].record(stream)
            if attn is not None:
                attn(stream)  # split plan + attention kernel + merge kernel
            elif path == "fused":
                d.append_gather(stream)  # plan kernel + fused append/gather kernel
            else:
                d.gather(stream)  # plan kernel + gather kernel (programmatic dependent launch)
            if e: e[3].record(stream)

        for _ in range(warmup):
            step()
        if d.error_code() != 0:
            raise RuntimeError("device error during warm-up")
        self.barrier()
        t0 = time.perf_counter()
        for i in range(steps):
            step(ev[i])
        self.barrier()
        wall = time.perf_counter() - t0
        st_ms = [0.0 if one_op else e[0].elapsed_time(e[1]) for e in ev]
        ga_ms = [e[2].elapsed_time(e[3]) for e in ev]
        if d.error_code() != 0:
            raise RuntimeError("device error during the timed steps")
        return {"step_ms": float(np.mean([a + b for a, b in zip(st_ms, ga_ms)])),
                "store_ms": float(np.mean(st_ms)), "gather_ms": float(np.mean(ga_ms)),
                "wall_s": wall}


def gpu_uuid(dev):
    import torch
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        return None


def run_gpu(args, rank, world):
    import torch
    import dequant_kvc8_store_gb300 as kv
    from dequant_kvc8_store_gb300.device import Bf16Batch, DecodeAttention, DeviceBatch

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    kv.load()
    w = W.NAMED[args.workload](seed=rank_seed(args.workload, rank))
    nbytes = path_bytes(w, args.path)
    if args.path == "bf16":
        d = Bf16Batch(w, device=dev, seed=rank_seed(args.workload, rank))
    else:
        d = DeviceBatch(w, device=dev)
    attn = (DecodeAttention(d, ATTN_GROUP, seed=rank_seed(args.workload, rank))
            if args.path == "attention" else None)
    has_store = w.has_store and w.num_tokens > 0 and attn is None
    timer = Timer(dev, world)
    with ClockSampler(gpu_uuid(dev)) as clocks:
        local = timer.run(d, attn, args.path, has_store, args.steps, args.warmup)
    local["step_ms"], local["store_ms"], local["gather_ms"] = reduce_max(
        [local["step_ms"], local["store_ms"], local["gather_ms"]], device=dev)

    def make_twin():
        # a second device copy of the batch for the overlapped end-to-end loop
        if args.path == "bf16":
            d2 = Bf16Batch(w, device=dev, seed=rank_seed(args.workload, rank))
        else:
            d2 = DeviceBatch(w, device=dev)
        a2 = (DecodeAttention(d2, ATTN_GROUP, seed=rank_seed(args.workload, rank))
              if attn is not None else None)
        return d2, a2
    e2e = run_e2e(args, w, d, dev, nbytes, attn, make_twin) if rank == 0 else None
    del d, attn
    sweep = None
    if args.path == "c8" and world == 1 and not args.no_workload_sweep:
        sweep = run_sweep(args, w, local, timer, dev)
    return w, nbytes, local, clocks.summary(), e2e, has_store, sweep


def op_figures(w, nbytes, t, peak):
    """Per-op time, GB/s (algorithmic bytes / time), fraction of peak and
    tokens/s of one batch's store and gather."""
    out = {}
    if w.has_store and w.num_tokens > 0 and t["store_ms"] > 0:
        gbs = nbytes["store"] / (t["store_ms"] * 1e-3) / 1e9
        out["store"] = {"ms": round(t["store_ms"], 5), "GB_s": round(gbs, 1),
                        "frac": round(gbs / peak, 4),
                        "tokens_per_s": round(w.num_tokens / (t["store_ms"] * 1e-3), 1),
                        "bytes": nbytes["store"]}
    gbs = nbytes["gather"] / (t["gather_ms"] * 1e-3) / 1e9
    out["dequant_gather"] = {"ms": round(t["gather_ms"], 5), "GB_s": round(gbs, 1),
                             "frac": round(gbs / peak, 4),
                             "tokens_per_s": round(w.total_context / (t["gather_ms"] * 1e-3), 1),
                             "bytes": nbytes["gather"]}
    return out


def run_sweep(args, w_head, t_head, timer, dev):
    """Store and gather of each full-size batch, timed like the headline (its
    own warm-up, the same L2 flush and events), one batch on the device at a
    time.  The headline batch reuses its own timing."""
    from dequant_kvc8_store_gb300.device import DeviceBatch
    peak, _ = measured_peak()
    steps, warm = max(3, min(args.steps, 100)), max(3, min(args.warmup, 10))
    out = {"steps": steps, "warmup": warm}
    with ClockSampler(gpu_uuid(dev)) as clocks:
        for name in SWEEP_WORKLOADS:
            if name == args.workload:
                out[name] = op_figures(w_head, W.algorithmic_bytes(w_head), t_head, peak)
                continue
            w = W.NAMED[name](seed=rank_seed(name, 0))
            d = DeviceBatch(w, device=dev)
            t = timer.run(d, None, "c8", w.has_store and w.num_tokens > 0, steps, warm)
            out[name] = op_figures(w, W.algorithmic_bytes(w), t, peak)
            del d
    out["clocks"] = clocks.summary()
    return out


def run_e2e(args, w, d, dev, nbytes, attn, make_twin):
    """Same step through the public API with host buffers: H2D of the new K/V
    and the batch metadata from pinned memory, store, plan, gather, D2H of the
    gathered K/V into pinned memory -- all of every step inside the timed
    region.  As a serving loop would, consecutive steps overlap on three
    streams: step i+1's inputs go up while step i computes and step i-1's
    results come down (two device buffer sets, used alternately)."""
    import torch
    from dequant_kvc8_store_gb300.device import _bf16

    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    host = {}
    if d.k_states is not None:
        host["k_states"] = _bf16(w.k_states).pin_memory()
        host["v_states"] = _bf16(w.v_states).pin_memory()
    host["block_table"] = torch.from_numpy(w.block_table).pin_memory()
    if w.cu_q_lens is not None:
        host["cu_q_lens"] = torch.from_numpy(w.cu_q_lens).pin_memory()
    host["context_kv_lens"] = torch.from_numpy(w.context_kv_lens).pin_memory()
    host["context_lengths"] = torch.from_numpy(w.context_lengths).pin_memory()
    pair = [(d, attn), make_twin()]
    if attn is not None:  # the decode step: queries and metadata in, attention out
        host = {"block_table": host["block_table"],
                "context_lengths": host["context_lengths"]}
        q_host = _bf16(attn.q_bits).pin_memory()
        outs = [(torch.empty(attn.out.shape, dtype=torch.bfloat16).pin_memory(), None)
                for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in host.values()) + q_host.numel() * 2
        d2h = outs[0][0].numel() * 2
    else:
        outs = [(torch.empty(d.k_out.shape, dtype=torch.bfloat16).pin_memory(),
                 torch.empty(d.v_out.shape, dtype=torch.bfloat16).pin_memory()) for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = outs[0][0].numel() * 2 * 2
    # bounded: at most ~32 GB of host<->device traffic, at least 3 steps
    steps = max(3, min(args.steps, 50, int(32e9 // max(1, h2d + d2h))))
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        j = i & 1
        dj, aj = pair[j]
        ok, ov = outs[j]
        if i >= 2:
            s_in.wait_event(ev_comp[j])  # step i-2 has consumed this buffer's inputs
        with torch.cuda.stream(s_in):
            for name, t in host.items():
                getattr(dj, name).copy_(t, non_blocking=True)
            if aj is not None:
                aj.query.copy_(q_host, non_blocking=True)
            ev_in[j].record(s_in)
        comp.wait_event(ev_in[j])
        if i >= 2:
            comp.wait_event(ev_out[j])  # step i-2's results are down
        if aj is not None:
            aj(comp)
        elif args.path == "fused":
            dj.append_gather(comp)
        else:
            dj.store(comp)
            dj.gather(comp)
        ev_comp[j].record(comp)
        s_out.wait_event(ev_comp[j])
        with torch.cuda.stream(s_out):
            if aj is not None:
                ok.copy_(aj.out, non_blocking=True)
            else:
                ok.copy_(dj.k_out, non_blocking=True)
                ov.copy_(dj.v_out, non_blocking=True)
            ev_out[j].record(s_out)

    for i in range(4):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(steps):
        step(i)
    comp.wait_event(ev_out[(steps - 1) & 1])
    e1.record(comp)
    torch.cuda.synchronize()
    for (dj, aj), (ok, ov) in zip(pair, outs):
        if dj.error_code() != 0:
            raise RuntimeError("device error during the end-to-end steps")
        # both buffer sets ran the same step: their downloads match the device
        # results bit for bit (a race between the streams would show here)
        same = (torch.equal(ok.view(torch.int16), aj.out.view(torch.int16).cpu()) if aj is not None
                else torch.equal(ok.view(torch.int16), dj.k_out.view(torch.int16).cpu()) and
                torch.equal(ov.view(torch.int16), dj.v_out.view(torch.int16).cpu()))
        if not same:
            raise RuntimeError("end-to-end downloads differ from the device results")
    ms = e0.elapsed_time(e1) / steps
    total = nbytes["store"] + nbytes["gather"]
    return {"value": round(total / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(ms, 4), "steps": steps,
            "overlap": "step i+1 H2D, step i kernels and step i-1 D2H on three streams, "
                       "two device buffer sets"}


# ---------------------------------------------------------------------------- CPU arm

def sub_workload(w: W.Workload, token_budget: int) -> W.Workload:
    """The first sequences of a workload, the last one cut, holding about
    token_budget stored + gathered positions: a bounded sample of it."""
    import copy
    s = copy.copy(w)
    q = w.q_lens().astype(np.int64)
    ctx0 = w.context_kv_lens.astype(np.int64)
    keep_q, keep_c, used = [], [], 0
    for b in range(w.num_seqs):
        cost = int(q[b]) + int(ctx0[b] + q[b])
        if used + cost > token_budget and keep_q:
            break
        keep_q.append(int(q[b]))
        keep_c.append(int(ctx0[b]))
        used += cost
        if used >= token_budget:
            break
    B = len(keep_q)
    if B == 1 and used > token_budget:  # cut the one sequence
        frac = token_budget / max(used, 1)
        keep_c[0] = int(keep_c[0] * frac)
        keep_q[0] = max(0 if not w.has_store else 1, int(keep_q[0] * frac))
        if not w.has_store:
            keep_q[0] = 0
    s.block_table = w.block_table[:B]
    s.context_kv_lens = np.array(keep_c, np.int32)
    s.context_lengths = (np.array(keep_c) + np.array(keep_q)).astype(np.int32)
    if w.has_store:
        n = int(sum(keep_q))
        if w.cu_q_lens is not None:
            s.cu_q_lens = np.concatenate([[0], np.cumsum(keep_q)]).astype(np.int32)
        s.k_states = w.k_states[:n]
        s.v_states = w.v_states[:n]
    return s


def oracle_pass(w: W.Workload, path: str = "c8"):
    import oracle
    if path == "attention":
        rng = np.random.default_rng(7)
        x = rng.standard_normal((w.num_seqs, w.kv_heads * ATTN_GROUP, w.head_dim)).astype(np.float32)
        qb = (x.view(np.uint32) >> 16).astype(np.uint16)
        t0 = time.perf_counter()
        oracle.paged_decode_attention(w.quant_mode, qb, w.k_cache, w.v_cache, w.k_scale,
                                      w.v_scale, w.block_table, w.context_lengths,
                                      w.head_dim ** -0.5)
        return time.perf_counter() - t0
    if path == "bf16":
        # a zero pool of the workload's shape: its prior bits do not change
        # what the copy costs
        shape = w.k_cache.shape
        kc = np.zeros(shape, np.uint16)
        vc = np.zeros(shape, np.uint16)
        t0 = time.perf_counter()
        if w.has_store:
            cu = w.cu_q_lens if w.cu_q_lens is not None else np.arange(w.num_tokens + 1, dtype=np.int32)
            oracle.store_bf16(w.k_states, w.v_states, kc, vc, w.block_table, cu, w.context_kv_lens)
        oracle.gather_bf16(kc, vc, w.block_table, w.context_lengths)
        return time.perf_counter() - t0
    kc, vc = w.k_cache, w.v_cache
    ks, vs = w.k_scale, w.v_scale
    t0 = time.perf_counter()
    if w.has_store:
        oracle.store(w.quant_mode, w.k_states, w.v_states, kc, vc, ks, vs, w.block_table,
                     w.cu_q_lens, w.context_kv_lens)
    oracle.dequant_gather(w.quant_mode, kc, vc, ks, vs, w.block_table, w.context_lengths)
    return time.perf_counter() - t0


ATTN_GROUP = 4  # 32 query heads on the 8 kv heads of the workloads


def path_bytes(w: W.Workload, path: str) -> dict:
    if path == "attention":
        return W.algorithmic_bytes_attention(w, ATTN_GROUP)
    if path == "bf16":
        return W.algorithmic_bytes_bf16(w)
    if path == "fused":
        return W.algorithmic_bytes_fused(w)
    return W.algorithmic_bytes(w)


def host_cpu() -> str:
    """The host CPU as the cpu_baseline reports it: model, architecture, and
    the cores the OS reports (the oracle itself runs on one)."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key, _, val = line.partition(":")
                key, val = key.strip().lower(), val.strip()
                if key == "model name":
                    model = val
                    break
                if key == "cpu part" and model is None:
                    model = {"0xd4f": "Arm Neoverse-V2"}.get(val, "Arm CPU part " + val)
    except OSError:
        pass
    return f"{model or platform.processor() or 'unknown CPU'}, {platform.machine()}, nproc {os.cpu_count()}"


def cpu_baseline(w: W.Workload, path: str = "c8", seconds: float = 12.0,
                 per_pass_cap: float = 3.0):
    """The oracle as it stands on one host core, on a bounded sample of the
    workload (whole passes when one pass is cheap enough)."""
    full = int(w.q_lens().sum() + w.context_lengths.astype(np.int64).sum())
    budget = full
    s = w
    # shrink the sample until one pass takes at most per_pass_cap seconds
    probe = sub_workload(w, min(full, 20000))
    t = oracle_pass(probe, path)
    rate = (int(probe.q_lens().sum()) + int(probe.context_lengths.astype(np.int64).sum())) / max(t, 1e-9)
    if full / rate > per_pass_cap:
        budget = int(rate * per_pass_cap)
        s = sub_workload(w, budget)
    bytes_pass = sum(path_bytes(s, path).values())
    times, t_end = [], time.perf_counter() + seconds
    while time.perf_counter() < t_end or not times:
        times.append(oracle_pass(s, path))
    gbs = bytes_pass / statistics.median(times) / 1e9
    sample = (f"{len(times)} oracle passes of {'the full workload' if s is w else 'its first %d sequences' % s.num_seqs} "
              f"({int(s.q_lens().sum())} stored + {int(s.context_lengths.astype(np.int64).sum())} "
              f"gathered positions, {bytes_pass / 1e6:.1f} MB algorithmic per pass), median pass")
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": sample, "host": host_cpu()}


def config_of(args) -> dict:
    """The `config` object of both arms' lines (identical for the same flags)."""
    return {"workload": WORKLOAD_TEXT[args.workload], "path": PATH_TEXT[args.path],
            "l2": L2_TEXT}


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = W.NAMED[args.workload](seed=rank_seed(args.workload, 0))
    steps, warm = args.steps, args.warmup
    # each step a bounded sample, sized so the whole run stays within ~2 minutes
    per_step = min(2.0, 100.0 / max(1, steps + warm))
    probe = sub_workload(w, 4000)
    t = oracle_pass(probe, args.path)
    rate = (int(probe.q_lens().sum()) + int(probe.context_lengths.astype(np.int64).sum())) / max(t, 1e-9)
    s = sub_workload(w, max(64, int(rate * per_step)))
    bytes_step = sum(path_bytes(s, args.path).values())
    for _ in range(warm):
        oracle_pass(s, args.path)
    times = [oracle_pass(s, args.path) for _ in range(steps)]
    ms = 1e3 * sum(times) / len(times)
    value = bytes_step / (ms * 1e-3) / 1e9
    positions = int(s.q_lens().sum() + s.context_lengths.astype(np.int64).sum())
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": steps, "warmup": warm, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if args.path == "bf16" else "f32",
        "data": "synthetic", "config": config_of(args),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"each step: oracle store+gather of the first {s.num_seqs} "
                                   f"sequences of the workload ({positions} stored + gathered "
                                   f"positions, {bytes_step / 1e6:.2f} MB algorithmic)",
                         "host": host_cpu()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def result_line(args, world, w, nbytes, t, clocks, e2e, has_store, sweep=None):
    """The JSON line of the GPU arm from the measured op times (t: ms per op)."""
    peak, peak_kind = measured_peak()
    total = nbytes["store"] + nbytes["gather"]
    value = job_throughput(total, world, t["step_ms"])
    fused = args.path == "fused"
    attention = args.path == "attention"
    timed_store = has_store and not fused and not attention and t["store_ms"] > 0
    ops = {
        "store": {"ms": round(t["store_ms"], 5),
                  "GB_s": round(nbytes["store"] / (t["store_ms"] * 1e-3) / 1e9, 1) if timed_store else None,
                  "tokens_per_s": round(w.num_tokens / (t["store_ms"] * 1e-3), 1) if timed_store else None,
                  "bytes": nbytes["store"]},
        "dequant_gather": {"ms": round(t["gather_ms"], 5),
                           "kernels": "plan + fused append/gather" if fused else "plan + gather",
                           "GB_s": round(nbytes["gather"] / (t["gather_ms"] * 1e-3) / 1e9, 1),
                           "tokens_per_s": round(w.total_context / (t["gather_ms"] * 1e-3), 1),
                           "bytes": nbytes["gather"]},
    }
    if attention:  # one op: decode attention straight from the int8 cache
        ops = {"decode_attention": {"ms": round(t["gather_ms"], 5),
                                    "kernels": "split plan + attention + merge",
                                    "GB_s": ops["dequant_gather"]["GB_s"],
                                    "positions_per_s": ops["dequant_gather"]["tokens_per_s"],
                                    "bytes": nbytes["gather"], "query_heads": ATTN_GROUP * w.kv_heads}}
    if fused:  # one op: the store is inside the fused launch
        ops["store"] = {"ms": 0.0, "GB_s": None, "tokens_per_s": None, "bytes": 0,
                        "note": "done inside the fused append + gather launch"}
        ops["dequant_gather"]["appended_tokens_per_s"] = round(
            w.num_tokens / (t["gather_ms"] * 1e-3), 1) if has_store else None
    if sweep is not None:
        ops["by_workload"] = sweep
    # the dominant kernel: the op with the larger device time
    dom = "dequant_gather" if (t["gather_ms"] >= t["store_ms"] or not timed_store) else "store"
    dom_bytes = nbytes["gather"] if dom == "dequant_gather" else nbytes["store"]
    dom_ms = t["gather_ms"] if dom == "dequant_gather" else t["store_ms"]
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    if attention:
        dom = "decode_attention"
    kname = "gather" if dom == "dequant_gather" else "store"
    if args.path == "bf16":
        kname += "_bf16"
    if fused:
        kname = "append_gather"
    if attention:
        kname = "attention"
    traffic = ncu_traffic(args.workload, kname + "_kernel")
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t["step_ms"], 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if args.path == "bf16" else "f32",
        "data": "synthetic",
        "config": config_of(args),
        "hbm_frac_of_step": round(total / (t["step_ms"] * 1e-3) / 1e9 / peak, 4),
        "tokens_per_s": ({"decode_attention": ops["decode_attention"]["positions_per_s"]}
                         if attention else
                         {"store": ops["store"]["tokens_per_s"],
                          "dequant_gather": ops["dequant_gather"]["tokens_per_s"]}),
        "ops": ops,
        "roofline": {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_kind": peak_kind, "traffic": traffic,
                     "dram_frac": ncu_dram_frac(args.workload, kname + "_kernel", peak),
                     "algorithmic_bytes": dom_bytes},
        # fused: plan + fused kernel, or store + plan + gather for a long append
        "gpu_launches": args.steps * (3 if (has_store and not fused) or attention or
                                      (fused and w.num_tokens * 2 * w.kv_heads > 16384) else 2),
        "clocks": clocks,
        "e2e": e2e,
        "wall_s": round(t["wall_s"], 3),
    }
    return line


# ---------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["kvc8", "reference"], default="kvc8")
    ap.add_argument("--workload", choices=list(W.NAMED), default=DEFAULT_WORKLOAD)
    ap.add_argument("--path", choices=["c8", "bf16", "fused", "attention"], default="c8",
                    help="c8: the int8 cache (default); bf16: the cache without quantisation; "
                         "fused: the int8 store and gather as one append + gather pass; "
                         "attention: decode attention (4 query heads per kv head) read "
                         "straight from the int8 cache")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workload-sweep", action="store_true",
                    help="int8 path on one GPU: do not also time the prefill, decode, mixed "
                         "and long-context batches")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    w, nbytes, t, clocks, e2e, has_store, sweep = run_gpu(args, rank, world)
    if rank == 0:
        line = result_line(args, world, w, nbytes, t, clocks, e2e, has_store, sweep)
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w, args.path)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
