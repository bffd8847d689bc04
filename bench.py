"""Benchmark: microseconds per decode step and effective KV GB/s of Quest-style
sparse decode attention on one GB300, at long context.

A step is one whole pass of the decode hot path for one new token per
sequence, through the C ABI (kvd_decode_step): append the token's K/V
(quantizing and updating the block envelope), score every block's bound,
select top-K + sink + recent blocks, and attend over the selected blocks.
Before each step the cache length is reset to the workload's L, so every
step sees the same context (L is a multiple of 64, so the token opens a
fresh block and its bounds are exact again).

Timing: W untimed warm-up steps, then K timed steps bracketed by a barrier
and a device synchronize; each step is timed with CUDA events on the stream
it runs on; L2 is flushed between steps, outside the events: a 256 MiB
write (larger than the 129 MB L2) evicts every input, then a 256 MiB read of
another buffer replaces the dirty lines that write leaves with clean ones, so
the timed kernels do not pay for the flush's own write-backs.  Under torchrun
every rank runs the same per-GPU workload (independent sequences: weak
scaling) and rank 0 prints the max over ranks.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                       [--impl reference]
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
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import long_context_decode_kv_gb300 as kvd  # noqa: E402
from long_context_decode_kv_gb300 import synth  # noqa: E402

DEFAULT_WORKLOAD = synth.CTX1M.name
FLUSH_BYTES = 256 << 20


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kv_bytes_per_token(dtype, D=128):
    # K row + V row, plus one f32 scale each (int8) or D / 32 f16 group scales
    # each (q8_0, q4_0; a q4_0 row is D / 2 bytes)
    if dtype == kvd.INT8:
        return 2 * D + 2 * 4
    if dtype == kvd.Q8_0:
        return 2 * D + 2 * (D // 32) * 2
    if dtype == kvd.Q4_0:
        return 2 * (D // 2) + 2 * (D // 32) * 2
    return 2 * 2 * D


def dtype_name(dtype):
    return {kvd.F16: "f16", kvd.INT8: "int8", kvd.Q8_0: "q8_0", kvd.Q4_0: "q4_0"}[dtype]


def attended_tokens(sel_idx, sel_cnt, L):
    idx = sel_idx.cpu().numpy()
    cnt = sel_cnt.cpu().numpy()
    tot = 0
    for b in range(cnt.shape[0]):
        for g in range(cnt.shape[1]):
            blks = idx[b, g, :cnt[b, g]].astype(np.int64)
            tot += int(np.minimum(64, L - blks * 64).sum())
    return tot


def decode_kernel_bytes(w, tokens, n_sel_total):
    # selected rows (+ scales), the block lists, q in, out
    return (tokens * kv_bytes_per_token(w.dtype, w.D) + n_sel_total * 4 +
            w.B * w.H * w.D * 4 * 2)


def step_bytes(w, tokens, n_sel_total, L1):
    """Algorithmic bytes of one whole step: the decode kernel's, plus the
    bounds of every scored (non-forced) block, the selection keys written and
    read once, and the one-token append (inputs read, row and bounds written)."""
    nb = (L1 + 63) // 64
    forced = kvd.selected_count(L1, 0, w.sink_tokens, w.recent_tokens)
    n_cand = nb - forced
    P = w.B * w.Hkv
    scored = P * n_cand * 2 * w.D * 2
    keys = P * n_cand * 4 * 2
    row_out = kv_bytes_per_token(w.dtype, w.D)
    append = P * (2 * w.D * 2 + row_out + 2 * w.D * 2)
    return decode_kernel_bytes(w, tokens, n_sel_total) + scored + keys + append


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
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
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def max_over_ranks(x, world):
    """Max of a host number over all ranks (NCCL: through the GPU; gloo: CPU)."""
    if world == 1:
        return x
    import torch.distributed as dist
    device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# The files the decode kernel's translation unit is compiled from.
DECODE_SOURCES = ("long_context_decode_kv_gb300/csrc/decode.cu",
                  "long_context_decode_kv_gb300/csrc/decode_dev.cuh",
                  "long_context_decode_kv_gb300/csrc/common.cuh",
                  "long_context_decode_kv_gb300/csrc/internal.h",
                  "include/kvdecode.h")


def source_digest():
    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def measured_traffic(workload, tokens):
    """DRAM bytes (read + write) of one decode-kernel launch, from the committed
    ncu summary: bytes per attended token measured on a capture of this
    workload's recipe (at the context the summary names), times the tokens this
    launch attends.  Valid only while the kernel sources are unchanged since the
    capture (the summary line carries their digest); None otherwise."""
    path = os.path.join(ROOT, "profiles", "decode_kernel_traffic.txt")
    if not os.path.exists(path):
        return None
    digest = source_digest()
    for line in open(path):
        parts = line.split()
        if len(parts) == 5 and parts[0] == workload and parts[2] == digest:
            return float(parts[3]) / float(parts[4]) * tokens
    return None


def launches_per_step(w, L1):
    """Kernels one sparse step (kvd_decode_step) launches on a cache of L1
    tokens after its append.  When there is a top-K to rank and the token's
    block is forced (a recent window), the token is appended inside the
    selection kernel: selection + decode.  Otherwise: append, then the
    selection (or the fill kernel when nothing has to be ranked), then decode."""
    nb = (L1 + 63) // 64
    se = min((w.sink_tokens + 63) // 64, nb)
    rb = nb if w.recent_tokens <= 0 else max(se, max(0, L1 - w.recent_tokens) // 64)
    n_cand = rb - se
    keff = min(w.k_sel, n_cand)
    fused = 0 < keff < n_cand and w.recent_tokens > 0
    return 2 if fused else 3


# --------------------------------------------------------------------------
# CPU oracle leg (the only place bench.py runs the oracle)
# --------------------------------------------------------------------------
def oracle_leg(w, q, k, v, steps, problem=(0, 0)):
    """Time the fp64 CPU oracle doing the same decode step on one (sequence,
    KV head) problem; scale to the workload's B*Hkv independent problems."""
    import oracle
    b, g = problem
    G = w.G
    oc = oracle.OracleCache(w.dtype, 1, 1, w.D, w.L + 64, 64)
    oc.append(k[b:b + 1, :, g:g + 1].contiguous().cpu().numpy(),
              v[b:b + 1, :, g:g + 1].contiguous().cpu().numpy())
    qg = q[b:b + 1, g * G:(g + 1) * G].cpu().numpy()
    times = []
    for s in range(steps):
        kn, vn = synth.make_step_token(w, s, device="cpu")
        t0 = time.perf_counter()
        oc.len = w.L
        oc.append(kn[b:b + 1, :, g:g + 1].numpy(), vn[b:b + 1, :, g:g + 1].numpy())
        oc.decode(qg, w.scale, k_sel=w.k_sel, sink_tokens=w.sink_tokens,
                  recent_tokens=w.recent_tokens, n_threads=1)
        times.append(time.perf_counter() - t0)
    per_problem_us = statistics.median(times) * 1e6
    n_prob = w.B * w.Hkv
    return per_problem_us * n_prob, {
        "kind": "oracle", "cores": 1,
        "sample": (f"1 of {n_prob} (sequence, KV head) problems of {w.name}, {steps} steps "
                   f"(append + select + attend, fp64, 1 thread), median per-problem time "
                   f"x {n_prob} problems")}


def oracle_leg_all_cores(w, q, k, v, steps):
    """The same oracle step on all host cores: every KV-head problem of
    sequence 0 at once, their selections and then their (problem, query head)
    attentions spread over the OpenMP threads (the arithmetic of each head is
    the same on any thread count); the step time is scaled by the workload's
    B sequences."""
    import oracle
    threads = max(1, len(os.sched_getaffinity(0)))
    hk = w.Hkv
    G = w.G
    oc = oracle.OracleCache(w.dtype, 1, hk, w.D, w.L + 64, 64)
    oc.append(k[0:1, :, :hk].contiguous().cpu().numpy(), v[0:1, :, :hk].contiguous().cpu().numpy())
    qg = q[0:1, :hk * G].cpu().numpy()
    times = []
    for s in range(steps):
        kn, vn = synth.make_step_token(w, s, device="cpu")
        t0 = time.perf_counter()
        oc.len = w.L
        oc.append(kn[0:1, :, :hk].numpy(), vn[0:1, :, :hk].numpy())
        oc.decode(qg, w.scale, k_sel=w.k_sel, sink_tokens=w.sink_tokens,
                  recent_tokens=w.recent_tokens, n_threads=threads)
        times.append(time.perf_counter() - t0)
    n_prob = w.B * w.Hkv
    batches = w.B
    used = min(threads, hk * G)
    return statistics.median(times) * 1e6 * batches, {
        "kind": "oracle", "cores": used, "threads_available": threads,
        "sample": (f"the {hk} KV-head problems of sequence 0 of {w.name} ({hk * G} query "
                   f"heads) at once on {used} threads, {steps} steps (append + select + "
                   f"attend, fp64), median step time x {batches} sequence(s) = {n_prob} "
                   f"problems")}


def run_reference(args, w):
    # the oracle, as cpu_baseline runs it (every host core it may use), on rank
    # 0 only; other ranks exit without work
    if int(os.environ.get("RANK", "0")) != 0:
        return
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    q, k, v, _ = synth.make_workload(w, device="cuda")
    steps = max(1, args.steps)
    for _ in range(max(0, min(args.warmup, 1))):
        oracle_leg_all_cores(w, q, k, v, 1)
    value, base = oracle_leg_all_cores(w, q, k, v, steps)
    base["value"] = value
    base["unit"] = "us/step"
    line = {"impl": "reference", "metric": "us_per_decode_step", "value": value,
            "unit": "us/step", "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup,
            "higher_is_better": False, "dtype": "f64", "data": "synthetic",
            "config": config_of(w), "cpu_baseline": base,
            "e2e": {"value": value, "unit": "us/step", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_of(w):
    return {"workload": w.name, "batch": w.B, "n_heads": w.H, "n_kv_heads": w.Hkv,
            "head_dim": w.D, "context": w.L, "kv_dtype": dtype_name(w.dtype),
            "block": 64, "k_sel": w.k_sel, "sink_tokens": w.sink_tokens,
            "recent_tokens": w.recent_tokens, "keys": w.keys, "n_needles": w.n_needles,
            "step": "append 1 token + select + sparse attend (kvd_decode_step)",
            "l2": ("flushed between timed steps, outside the events: 256 MiB write, then "
                   "256 MiB read of another buffer (drains the write-backs)"),
            "parallelism": "replicas"}


def run_sweep(args):
    """Sparse and dense decode steps (append + select + attend, as in the bench
    line) over a sweep of workloads; one JSON line per point."""
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    drain = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    points = {"context": synth.context_sweep, "coverage": synth.coverage_sweep,
              "head_dim": synth.head_dim_sweep}[args.sweep]()
    steps, warm = max(1, args.steps), max(3, args.warmup)
    for w in points:
        q, k, v, _ = synth.make_workload(w, device=dev)
        cache = kvd.KVCache(w.dtype, w.B, w.Hkv, w.L + 64, head_dim=w.D, device=dev)
        kvd.kv_append(cache, k, v)
        del k, v
        ws = kvd.make_workspace(cache, w.H)
        nbmax = cache.max_seq // 64
        sel_idx = torch.zeros((w.B, w.Hkv, nbmax), dtype=torch.int32, device=dev)
        sel_cnt = torch.zeros((w.B, w.Hkv), dtype=torch.int32, device=dev)
        out = torch.empty(w.B, w.H, w.D, device=dev)
        toks = [synth.make_step_token(w, s, device=dev) for s in range(8)]

        def step(i, dense):
            cache.len = w.L
            kn, vn = toks[i % len(toks)]
            kvd.decode_step(cache, q, kn, vn, w.scale, -1 if dense else w.k_sel,
                            w.sink_tokens, w.recent_tokens, out, ws, sel_idx=sel_idx,
                            sel_cnt=sel_cnt)

        res = {}
        for dense in (False, True):
            ms = []
            for i in range(warm + steps):
                flush.fill_(i & 0xFF)
                drain.sum()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                step(i, dense)
                e1.record(stream)
                if i >= warm:
                    ms.append((e0, e1))
            torch.cuda.synchronize()
            res[dense] = statistics.mean(a.elapsed_time(b) for a, b in ms) * 1e3
        L1 = w.L + 1
        n_sel = int(sel_cnt.sum().item())
        tokens = attended_tokens(sel_idx, sel_cnt, L1) if n_sel else 0
        # the step's selection and sparse decode timed apart (same flush)
        cache.len = L1
        max_sel = kvd.selected_count(L1, w.k_sel, w.sink_tokens, w.recent_tokens)
        calls = {"select": lambda: kvd.select_blocks(cache, q, w.k_sel, w.sink_tokens,
                                                     w.recent_tokens, sel_idx, sel_cnt, ws),
                 "decode": lambda: kvd.decode_attn(cache, q, w.scale, sel_idx, sel_cnt, max_sel,
                                                   out, ws)}
        part = {}
        for name, fn in calls.items():
            ms = []
            for i in range(warm + steps):
                flush.fill_(i & 0xFF)
                drain.sum()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                if i >= warm:
                    ms.append((e0, e1))
            torch.cuda.synchronize()
            part[name] = statistics.mean(a.elapsed_time(b) for a, b in ms) * 1e3
        assert cache.device_status() == 0, "device-side fault reported"
        print(json.dumps({
            "sweep": args.sweep, "workload": w.name, "context": w.L, "batch": w.B,
            "kv_dtype": dtype_name(w.dtype), "head_dim": w.D, "k_sel": w.k_sel,
            "kernels": "tuned (head dim 128)" if w.D == 128 else "general head dim",
            "coverage": n_sel / (w.B * w.Hkv) / ((L1 + 63) // 64),
            "sparse_step_us": res[False], "dense_step_us": res[True],
            "dense_over_sparse": res[True] / res[False],
            "select_us": part["select"], "decode_us": part["decode"],
            "decode_kv_gbs": decode_kernel_bytes(w, tokens, n_sel) / (part["decode"] * 1e-6) / 1e9,
            "effective_kv_gbs": step_bytes(w, tokens, n_sel, L1) / (res[False] * 1e-6) / 1e9,
            "dense_kv_gbs": (w.B * w.Hkv * L1 * kv_bytes_per_token(w.dtype, w.D) /
                             (res[True] * 1e-6) / 1e9),
            "steps": steps, "l2": "write + read flush between steps"}), flush=True)
        del cache, ws
        torch.cuda.empty_cache()


SPARSE_V_EPS = (0.0, 0.05, 0.5, 2.0)


def run_sparse_v_sweep(args):
    """Decode attention alone with sparse-V (eps mode) at several eps, on the
    selection of the workloads' decode step; one JSON line per point."""
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    drain = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    steps, warm = max(1, args.steps), max(3, args.warmup)
    for name in ("ctx1m_int8", "qwen3_4b_gqa_32k_f16"):
        w = synth.WORKLOADS[name]
        q, k, v, _ = synth.make_workload(w, device=dev)
        cache = kvd.KVCache(w.dtype, w.B, w.Hkv, w.L + 64, device=dev)
        kvd.kv_append(cache, k, v)
        del k, v
        ws = kvd.make_workspace(cache, w.H)
        nbmax = cache.max_seq // 64
        sel_idx = torch.zeros((w.B, w.Hkv, nbmax), dtype=torch.int32, device=dev)
        sel_cnt = torch.zeros((w.B, w.Hkv), dtype=torch.int32, device=dev)
        kvd.select_blocks(cache, q, w.k_sel, w.sink_tokens, w.recent_tokens, sel_idx, sel_cnt, ws)
        max_sel = kvd.selected_count(w.L, w.k_sel, w.sink_tokens, w.recent_tokens)
        out = torch.empty(w.B, w.H, w.D, device=dev)
        base = None
        for eps in SPARSE_V_EPS:
            ms = []
            for i in range(warm + steps):
                flush.fill_(i & 0xFF)
                drain.sum()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                kvd.decode_attn_sv(cache, q, w.scale, sel_idx, sel_cnt, max_sel, eps, out, ws)
                e1.record(stream)
                if i >= warm:
                    ms.append((e0, e1))
            torch.cuda.synchronize()
            us = statistics.mean(a.elapsed_time(b) for a, b in ms) * 1e3
            base = us if base is None else base
            print(json.dumps({
                "sweep": "sparse_v", "workload": w.name, "context": w.L,
                "kv_dtype": dtype_name(w.dtype), "eps": eps,
                "decode_us": us, "vs_eps0": us / base, "steps": steps,
                "l2": "write + read flush between steps"}), flush=True)
        del cache, ws
        torch.cuda.empty_cache()


def run_tail_sweep(args):
    """Decode attention over the step's selection, without and with the moment
    tail of the blocks it leaves out, at the workload's K_SEL and a quarter of
    it: device time (write + read L2 flush between calls) and the relative L2
    error of each output against dense attention; one JSON line per point."""
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    drain = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    steps, warm = max(1, args.steps), max(3, args.warmup)

    def timed_us(fn):
        ms = []
        for i in range(warm + steps):
            flush.fill_(i & 0xFF)
            drain.sum()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            if i >= warm:
                ms.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ms) * 1e3

    def rel_err(x, ref):
        e = ((x - ref).norm(dim=-1) / ref.norm(dim=-1)).flatten()
        return float(e.median()), float(e.max())

    for name in ("ctx1m_int8", "qwen3_4b_gqa_32k_f16"):
        w = synth.WORKLOADS[name]
        q, k, v, _ = synth.make_workload(w, device=dev)
        cache = kvd.KVCache(w.dtype, w.B, w.Hkv, w.L + 64, device=dev, moments=True)
        kvd.kv_append(cache, k, v)
        del k, v
        ws = kvd.make_workspace(cache, w.H)
        nbmax = cache.max_seq // 64
        dense = torch.empty(w.B, w.H, w.D, device=dev)
        kvd.decode_attn_dense(cache, q, w.scale, dense, ws)
        for k_sel in (w.k_sel, w.k_sel // 4):
            sel_idx = torch.zeros((w.B, w.Hkv, nbmax), dtype=torch.int32, device=dev)
            sel_cnt = torch.zeros((w.B, w.Hkv), dtype=torch.int32, device=dev)
            kvd.select_blocks(cache, q, k_sel, w.sink_tokens, w.recent_tokens, sel_idx, sel_cnt,
                              ws)
            max_sel = kvd.selected_count(w.L, k_sel, w.sink_tokens, w.recent_tokens)
            plain = torch.empty_like(dense)
            tail = torch.empty_like(dense)
            us_plain = timed_us(lambda: kvd.decode_attn(cache, q, w.scale, sel_idx, sel_cnt,
                                                        max_sel, plain, ws))
            us_tail = timed_us(lambda: kvd.decode_attn_tail(cache, q, w.scale, sel_idx, sel_cnt,
                                                            max_sel, tail, ws))
            assert cache.device_status() == 0, "device-side fault reported"
            nb = (w.L + 63) // 64
            print(json.dumps({
                "sweep": "tail", "workload": w.name, "context": w.L,
                "kv_dtype": dtype_name(w.dtype), "k_sel": k_sel,
                "coverage": max_sel / nb, "decode_us": us_plain, "decode_tail_us": us_tail,
                "tail_moment_bytes": w.B * w.Hkv * nb * 512,
                "err_vs_dense_median": rel_err(plain, dense)[0],
                "err_vs_dense_max": rel_err(plain, dense)[1],
                "tail_err_vs_dense_median": rel_err(tail, dense)[0],
                "tail_err_vs_dense_max": rel_err(tail, dense)[1], "steps": steps,
                "l2": "write + read flush between calls"}), flush=True)
        del cache, ws
        torch.cuda.empty_cache()


def run_gqa_sweep(args):
    """The GQA-shared selection against one selection per query head, at the
    workload's K_SEL: device time of select and decode (write + read L2 flush
    before each call), the K/V bytes each decode reads, the distinct blocks
    the heads of a group pick, and each output's relative L2 error against
    dense attention; one JSON line per workload."""
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    drain = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    steps, warm = max(1, args.steps), max(3, args.warmup)

    def timed_us(fn):
        ms = []
        for i in range(warm + steps):
            flush.fill_(i & 0xFF)
            drain.sum()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            if i >= warm:
                ms.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ms) * 1e3

    def rel_err(x, ref):
        e = ((x - ref).norm(dim=-1) / ref.norm(dim=-1)).flatten()
        return float(e.median()), float(e.max())

    for name in ("qwen3_4b_gqa_32k_f16", "ctx1m_int8"):
        w = synth.WORKLOADS[name]
        q, k, v, _ = synth.make_workload(w, device=dev)
        cache = kvd.KVCache(w.dtype, w.B, w.Hkv, w.L + 64, device=dev)
        kvd.kv_append(cache, k, v)
        del k, v
        ws = kvd.make_workspace(cache, w.H)
        nbmax = cache.max_seq // 64
        dense = torch.empty(w.B, w.H, w.D, device=dev)
        kvd.decode_attn_dense(cache, q, w.scale, dense, ws)
        s_idx = torch.zeros((w.B, w.Hkv, nbmax), dtype=torch.int32, device=dev)
        s_cnt = torch.zeros((w.B, w.Hkv), dtype=torch.int32, device=dev)
        h_idx = torch.zeros((w.B, w.H, nbmax), dtype=torch.int32, device=dev)
        h_cnt = torch.zeros((w.B, w.H), dtype=torch.int32, device=dev)
        args_sel = (w.k_sel, w.sink_tokens, w.recent_tokens)
        us_sel_s = timed_us(lambda: kvd.select_blocks(cache, q, *args_sel, s_idx, s_cnt, ws))
        us_sel_h = timed_us(lambda: kvd.select_blocks_per_head(cache, q, *args_sel, h_idx,
                                                                h_cnt, ws))
        max_sel = kvd.selected_count(w.L, *args_sel)
        shared, per_head = torch.empty_like(dense), torch.empty_like(dense)
        us_dec_s = timed_us(lambda: kvd.decode_attn(cache, q, w.scale, s_idx, s_cnt, max_sel,
                                                    shared, ws))
        us_dec_h = timed_us(lambda: kvd.decode_attn_per_head(cache, q, w.scale, h_idx, h_cnt,
                                                             max_sel, per_head, ws))
        assert cache.device_status() == 0, "device-side fault reported"
        blk_bytes = 64 * kv_bytes_per_token(w.dtype)
        si, sc = s_idx.cpu().numpy(), s_cnt.cpu().numpy()
        hi, hc = h_idx.cpu().numpy(), h_cnt.cpu().numpy()
        shared_blocks = int(sc.sum())
        head_blocks = int(hc.sum())
        union = sum(len(set().union(*[set(hi[b, g * w.G + j, :hc[b, g * w.G + j]].tolist())
                                      for j in range(w.G)]))
                    for b in range(w.B) for g in range(w.Hkv))
        print(json.dumps({
            "sweep": "gqa", "workload": w.name, "context": w.L, "group": w.G,
            "kv_dtype": dtype_name(w.dtype), "k_sel": w.k_sel,
            "shared": {"select_us": us_sel_s, "decode_us": us_dec_s,
                       "kv_bytes": shared_blocks * blk_bytes,
                       "err_vs_dense_median": rel_err(shared, dense)[0],
                       "err_vs_dense_max": rel_err(shared, dense)[1]},
            "per_head": {"select_us": us_sel_h, "decode_us": us_dec_h,
                         "kv_bytes": head_blocks * blk_bytes,
                         "distinct_blocks_per_group_vs_shared": union / shared_blocks,
                         "err_vs_dense_median": rel_err(per_head, dense)[0],
                         "err_vs_dense_max": rel_err(per_head, dense)[1]},
            "bytes_per_head_over_shared": head_blocks / shared_blocks, "steps": steps,
            "l2": "write + read flush between calls"}), flush=True)
        del cache, ws
        torch.cuda.empty_cache()


SELECT_MARKS = {0: "entry", 1: "first bounds in", 2: "warp 0 scored", 3: "all warps scored",
                4: "ticket taken", 6: "keys in shared memory", 7: "first digit",
                8: "above-bitmap + bin collected", 9: "threshold found", 5: "list written",
                10: "exit", 11: "first-digit keys counted (thread 0)",
                12: "list offsets scanned", 13: "list written (last warp)"}
DECODE_MARKS = {0: "entry", 1: "dependency wait over", 8: "first copy issued",
                2: "first stage in", 3: "all stages consumed", 4: "partial written",
                5: "arrival counted", 6: "splits merged"}


def run_stage_marks(args, w):
    """Per-stage timings of one decode step from the kernels' %globaltimer marks
    (a library built with KVD_MARKS=1 only).  Each of K steps runs after the
    L2 flush; the marks of every CTA are read back after each step.  Printed:
    per kernel and mark, the median over steps of the min / median / max over
    CTAs, in microseconds from the step's first mark."""
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    marks = torch.zeros(kvd.MARK_KINDS * kvd.MARK_CTAS * kvd.MARK_SLOTS, dtype=torch.int64,
                        device=dev)
    kvd.debug_stage_marks(marks)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    drain = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    q, k, v, _ = synth.make_workload(w, device=dev)
    cache = kvd.KVCache(w.dtype, w.B, w.Hkv, w.L + 64, head_dim=w.D, device=dev)
    kvd.kv_append(cache, k, v)
    del k, v
    ws = kvd.make_workspace(cache, w.H)
    nbmax = cache.max_seq // 64
    sel_idx = torch.zeros((w.B, w.Hkv, nbmax), dtype=torch.int32, device=dev)
    sel_cnt = torch.zeros((w.B, w.Hkv), dtype=torch.int32, device=dev)
    out = torch.empty(w.B, w.H, w.D, device=dev)
    toks = [synth.make_step_token(w, s, device=dev) for s in range(8)]
    per = {0: {}, 1: {}}
    steps = max(1, args.steps)
    for i in range(max(3, args.warmup) + steps):
        flush.fill_(i & 0xFF)
        drain.sum()
        marks.zero_()
        cache.len = w.L
        kn, vn = toks[i % len(toks)]
        kvd.decode_step(cache, q, kn, vn, w.scale, w.k_sel, w.sink_tokens, w.recent_tokens,
                        out, ws, sel_idx=sel_idx, sel_cnt=sel_cnt)
        torch.cuda.synchronize()
        if i < max(3, args.warmup):
            continue
        m = marks.view(kvd.MARK_KINDS, kvd.MARK_CTAS, kvd.MARK_SLOTS).cpu().numpy()
        live = m[:, :, 0] > 0
        t0 = min(int(m[kind, live[kind], 0].min()) for kind in (0, 1) if live[kind].any())
        for kind in (0, 1):
            for slot in range(kvd.MARK_SLOTS):
                vals = m[kind, :, slot]
                vals = vals[vals > 0]
                if vals.size:
                    d = (vals - t0) / 1e3
                    per[kind].setdefault(slot, []).append(
                        (float(d.min()), float(np.median(d)), float(d.max()), int(vals.size)))
    assert cache.device_status() == 0, "device-side fault reported"
    kvd.debug_stage_marks(None)
    for kind, names in ((0, SELECT_MARKS), (1, DECODE_MARKS)):
        rows = []
        for slot, vals in sorted(per[kind].items(), key=lambda kv: statistics.median(
                x[1] for x in kv[1])):
            med = [statistics.median(x[j] for x in vals) for j in range(4)]
            rows.append({"mark": names.get(slot, str(slot)), "slot": slot,
                         "us_min": round(med[0], 2), "us_median": round(med[1], 2),
                         "us_max": round(med[2], 2), "ctas": int(med[3])})
        print(json.dumps({"stage_marks": "select" if kind == 0 else "decode",
                          "workload": w.name, "context": w.L, "steps": steps, "rows": rows}),
              flush=True)


# The metric's other contexts, reported beside the 1M headline.
CONTEXT_WORKLOADS = ("qwen3_4b_gqa_32k_f16", "ctx128k_b8_int8")


def measure(w, dev, steps, warmup, flush_l2, world, local, headline):
    """The bench protocol on one workload: K timed decode steps (value), then
    the decode kernel, the selection and the append alone, the dense step, and
    (headline) the end-to-end step through host buffers.  Returns a dict."""
    stream = torch.cuda.current_stream(dev)
    q, k, v, needles = synth.make_workload(w, device=dev)
    cache = kvd.KVCache(w.dtype, w.B, w.Hkv, w.L + 64, head_dim=w.D, device=dev)
    kvd.kv_append(cache, k, v)
    if not headline:
        del k, v
        k = v = None
    ws = kvd.make_workspace(cache, w.H)
    nbmax = cache.max_seq // 64
    sel_idx = torch.zeros((w.B, w.Hkv, nbmax), dtype=torch.int32, device=dev)
    sel_cnt = torch.zeros((w.B, w.Hkv), dtype=torch.int32, device=dev)
    out = torch.empty(w.B, w.H, w.D, device=dev)
    toks = [synth.make_step_token(w, s, device=dev) for s in range(8)]
    L1 = w.L + 1
    max_sel = kvd.selected_count(L1, w.k_sel, w.sink_tokens, w.recent_tokens)

    def step(i, dense=False):
        cache.len = w.L
        kn, vn = toks[i % len(toks)]
        kvd.decode_step(cache, q, kn, vn, w.scale, -1 if dense else w.k_sel, w.sink_tokens,
                        w.recent_tokens, out, ws, sel_idx=sel_idx, sel_cnt=sel_cnt)

    def timed(fn, n, warm):
        for i in range(warm):
            flush_l2(i)
            fn(i)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        barrier(world)
        t0 = time.perf_counter()
        for i in range(n):
            flush_l2(i)
            ev[i][0].record(stream)
            fn(i)
            ev[i][1].record(stream)
        barrier(world)
        wall = time.perf_counter() - t0
        ms = [a.elapsed_time(b) for a, b in ev]
        return ms, wall

    # ---- the timed decode steps (value).  Clocks are sampled from a short
    # stretch of the same steps just before the timed region through its end
    # (the sampler's period is 200 ms, longer than K steps take).
    with Clocks(local) as clk:
        t_end = time.perf_counter() + 0.8
        i = 0
        while time.perf_counter() < t_end:
            flush_l2(i)
            step(i)
            i += 1
            if i % 64 == 0:
                torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("kvd_timed" if headline else "kvd_context")
        step_ms, wall = timed(lambda i: step(i), steps, warmup)
        torch.cuda.nvtx.range_pop()
    clocks = clk.summary()
    assert cache.device_status() == 0, "device-side fault reported"
    us_step = max_over_ranks(statistics.mean(step_ms) * 1e3, world)

    # ---- selection statistics of the timed configuration
    tokens = attended_tokens(sel_idx, sel_cnt, L1)
    n_sel_total = int(sel_cnt.sum().item())
    needle_ok = all(int(p) // 64 in set(sel_idx[b, g, :sel_cnt[b, g]].tolist())
                    for b in range(w.B) for g in range(w.Hkv) for p in needles[b, g].tolist())

    # ---- the decode kernel alone (roofline of the dominant kernel)
    cache.len = L1

    def dec(i):
        kvd.decode_attn(cache, q, w.scale, sel_idx, sel_cnt, max_sel, out, ws)
    dec_ms, _ = timed(dec, steps, 3)
    dec_us = statistics.mean(dec_ms) * 1e3

    def sel(i):
        kvd.select_blocks(cache, q, w.k_sel, w.sink_tokens, w.recent_tokens, sel_idx, sel_cnt,
                          ws)
    sel_ms, _ = timed(sel, steps, 3)

    def app(i):
        cache.len = w.L
        kn, vn = toks[i % len(toks)]
        kvd.kv_append(cache, kn, vn)
    app_ms, _ = timed(app, steps, 3)

    # ---- dense arm at the same context (append + dense attend)
    dense_ms, _ = timed(lambda i: step(i, dense=True), max(5, steps // 5), 2)

    e2e = None
    if headline:
        # ---- e2e: host buffers through the C ABI, copies inside the timed region
        qh = q.cpu().pin_memory()
        kh = [(a.cpu().pin_memory(), b.cpu().pin_memory()) for a, b in toks]
        oh = torch.empty(w.B, w.H, w.D).pin_memory()

        def host_step(i):
            cache.len = w.L
            a, b = kh[i % len(kh)]
            kvd.decode_step_host(cache, qh, a, b, w.scale, w.k_sel, w.sink_tokens,
                                 w.recent_tokens, oh, ws)
        e2e_ms, _ = timed(host_step, steps, 3)
        e2e_us = max_over_ranks(statistics.mean(e2e_ms) * 1e3, world)
        e2e = {"value": e2e_us, "unit": "us/step",
               "h2d_bytes_per_step": qh.numel() * 4 + 2 * kh[0][0].numel() * 2,
               "d2h_bytes_per_step": oh.numel() * 4,
               "host_buffers": "pinned; the kernels read q, k, v and write out in place "
                               "over the host link (no staging copies)"}
    assert cache.device_status() == 0, "device-side fault reported"

    peak, peak_kind = peaks()
    dbytes = decode_kernel_bytes(w, tokens, n_sel_total)
    sbytes = step_bytes(w, tokens, n_sel_total, L1)
    achieved = dbytes / (dec_us * 1e-6) / 1e9
    eff_step = sbytes / (us_step * 1e-6) / 1e9
    kernel = ("decode_kernel" if w.D == 128 else "gd_decode_kernel") + " (kvd_decode_attn)"
    res = {
        "step_us": us_step, "effective_kv_gbs": eff_step, "effective_kv_frac": eff_step / peak,
        "step_bytes": sbytes,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind, "kernel": kernel,
                     "bytes": dbytes, "us": dec_us,
                     "traffic": measured_traffic(w.name, tokens) if w.D == 128 else None,
                     "tokens_attended": tokens},
        "breakdown_us": {"append": statistics.mean(app_ms) * 1e3,
                         "select": statistics.mean(sel_ms) * 1e3, "decode": dec_us,
                         "step": us_step, "dense_step": statistics.mean(dense_ms) * 1e3},
        "selected_blocks_per_problem": n_sel_total / (w.B * w.Hkv),
        "coverage": n_sel_total / (w.B * w.Hkv) / ((L1 + 63) // 64),
        "needles_selected": needle_ok, "e2e": e2e, "clocks": clocks,
        "wall_s_timed_region": wall, "launches_per_step": launches_per_step(w, L1),
        "_inputs": (q, k, v),
    }
    del cache, ws
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--stage-marks", action="store_true",
                    help="print per-stage timings of the step from the kernels' timer marks "
                         "(needs the library built with KVD_MARKS=1)")
    ap.add_argument("--no-contexts", action="store_true",
                    help="leave out the 32K and 128K x 8 sub-records of the default line")
    ap.add_argument("--context", type=int, default=None,
                    help="run the workload's recipe at this context instead (a multiple "
                         "of 64; a smaller case for profiling)")
    ap.add_argument("--head-dim", type=int, default=None,
                    help="run the workload's recipe with this head dim instead (a multiple "
                         "of 16 up to 1024; 128 runs the tuned kernels, others the general "
                         "ones)")
    ap.add_argument("--sweep", choices=["context", "coverage", "sparse_v", "tail", "gqa",
                                        "head_dim"],
                    default=None,
                    help="instead of the bench line: sparse vs dense decode steps over the "
                         "context sweep (16K..1M, 25%% coverage) or the 128K x 8 coverage "
                         "sweep, decode attention with sparse-V at several eps, or decode "
                         "attention with the moment tail, or the GQA-shared selection "
                         "against one per query head; one JSON line per point")
    args = ap.parse_args()
    if args.sweep == "sparse_v":
        return run_sparse_v_sweep(args)
    if args.sweep == "tail":
        return run_tail_sweep(args)
    if args.sweep == "gqa":
        return run_gqa_sweep(args)
    if args.sweep:
        return run_sweep(args)
    w = synth.WORKLOADS[args.workload]
    if args.context is not None:
        if args.context < 64 or args.context % 64:
            ap.error("--context must be a positive multiple of 64")
        w = w.with_(L=args.context)
    if args.head_dim is not None:
        if not (16 <= args.head_dim <= 1024 and args.head_dim % 16 == 0):
            ap.error("--head-dim must be a multiple of 16 in [16, 1024]")
        w = w.with_(D=args.head_dim)
    if args.impl == "reference":
        return run_reference(args, w)
    if args.stage_marks:
        return run_stage_marks(args, w)

    world, rank, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    warmup = max(3, args.warmup)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    drain = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2(i):
        flush.fill_(i & 0xFF)
        return drain.sum()

    m = measure(w, dev, args.steps, warmup, flush_l2, world, local, headline=True)
    q, k, v = m.pop("_inputs")

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        try:
            v_all, cpu = oracle_leg_all_cores(w, q, k, v, 3)
            v_one, one = oracle_leg(w, q, k, v, 3)
            cpu["value"] = v_all
            cpu["unit"] = "us/step"
            cpu["value_1_thread"] = v_one
            cpu["sample_1_thread"] = one["sample"]
        except Exception as e:  # the baseline must not hide the GPU number
            cpu = {"kind": "oracle", "value": None, "error": str(e)[:200]}
    del q, k, v
    torch.cuda.empty_cache()

    # ---- the metric's other contexts (32K f16 GQA, 128K x 8 int8), measured
    # in the same run with the same protocol; the headline stays the workload's
    contexts = {}
    if args.workload == DEFAULT_WORKLOAD and args.context is None and args.head_dim is None \
            and not args.no_contexts:
        for name in CONTEXT_WORKLOADS:
            cm = measure(synth.WORKLOADS[name], dev, args.steps, warmup, flush_l2, world, local,
                         headline=False)
            cm.pop("_inputs")
            contexts[name] = cm
            torch.cuda.empty_cache()

    if rank != 0:
        return
    line = {
        "metric": "us_per_decode_step", "value": m["step_us"], "unit": "us/step",
        "n_gpus": world, "steps": args.steps, "warmup": warmup,
        "ms_per_step": m["step_us"] / 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": dtype_name(w.dtype), "data": "synthetic",
        "config": config_of(w),
        "effective_kv_gbs": m["effective_kv_gbs"],
        "effective_kv_frac": m["effective_kv_frac"],
        "step_bytes": m["step_bytes"],
        "roofline": m["roofline"],
        "breakdown_us": m["breakdown_us"],
        "sparse_over_dense": m["breakdown_us"]["dense_step"] / m["step_us"],
        "selected_blocks_per_problem": m["selected_blocks_per_problem"],
        "coverage": m["coverage"],
        "needles_selected": m["needles_selected"],
        "e2e": m["e2e"],
        "gpu_launches": m["launches_per_step"] * args.steps,
        "clocks": m["clocks"],
        "wall_s_timed_region": m["wall_s_timed_region"],
        "cpu_baseline": cpu,
    }
    if contexts:
        line["contexts"] = {
            name: {"config": config_of(synth.WORKLOADS[name]), "step_us": cm["step_us"],
                   "select_us": cm["breakdown_us"]["select"],
                   "decode_us": cm["breakdown_us"]["decode"],
                   "dense_step_us": cm["breakdown_us"]["dense_step"],
                   "sparse_over_dense": cm["breakdown_us"]["dense_step"] / cm["step_us"],
                   "effective_kv_gbs": cm["effective_kv_gbs"],
                   "effective_kv_frac": cm["effective_kv_frac"],
                   "roofline": cm["roofline"], "coverage": cm["coverage"],
                   "needles_selected": cm["needles_selected"], "clocks": cm["clocks"]}
            for name, cm in contexts.items()}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
