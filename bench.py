"""Benchmark of the exact blocked attention path on GB300.

Default (N=1): the batched GQA decode workload (batch 32, 32 query / 8 KV
heads, d=128, T_q=1, cache lengths uniform in [512, 8192], bf16).  One step is
one blkattn_fwd call over the whole batch (for this shape one launch of the
tcgen05 decode kernel, which also folds the units it splits across CTAs).
``value`` is KV-cache GB/s: the algorithmic K+V bytes of the visible cache
rows (each (sequence, KV head) row read once) over the device time.

Under torchrun (N > 1) every rank runs its own batch (weak scaling, seed
offset by rank); the only collectives are a barrier and the max of the step
time over the ranks.

The other workloads (tiny fp32, long-context decode, speculative verify,
causal prefill) are measured in the same run and reported under
``workloads`` with their own roofline figures.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import shutil
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from exact_blocked_attention_gb300 import workloads  # noqa: E402

HEADLINE = "decode_gqa"
METRIC = "decode attn KV-cache GB/s (batched GQA decode, bf16)"
L2_BYTES = 129 * 1024 * 1024


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return {"hbm_gbs": float(j["hbm_gbs"]), "bf16_tflops": float(j["bf16_tflops"]),
                "bf16_tflops_sustained": float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def code_digest(sources):
    """sha256 (first 16 hex digits) over the given C/CUDA sources with their
    comments and blank space removed: a comment-only edit keeps the digest."""
    import hashlib
    import re
    m = hashlib.sha256()
    for src in sources:
        with open(os.path.join(ROOT, src)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        m.update(" ".join(text.split()).encode())
    return m.hexdigest()[:16]


def measured_traffic(workload):
    """DRAM bytes per launch of the workload's main kernel from the committed
    ncu capture (profiles/traffic.json), or None when the kernel's code
    changed since that capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            entry = json.load(f)["workloads"][workload]
        if code_digest(entry["sources"]) != entry["code_sha256_16"]:
            return None
        return entry["dram_bytes_per_launch"]
    except (OSError, KeyError, ValueError):
        return None


def describe(s):
    return (f"{s.name}: B={s.B} Hq={s.Hq} Hkv={s.Hkv} d={s.d} Tq={s.Tq} Tmax={s.Tmax} "
            f"lens={s.lens} pos={s.pos} {s.dtype}" + (f" bias={s.bias}" if s.bias != "none" else ""))


def algorithmic_bytes(s, inp):
    """K+V of the visible cache rows (once per KV head) + Q + O (+ lse), and
    the token-tree masks of a tree workload."""
    kv = workloads.kv_bytes(s, inp["seqlens"].numpy())
    elt = 2 if s.dtype == "bf16" else 4
    q = s.B * s.Hq * s.Tq * s.d * elt
    o = s.B * s.Hq * s.Tq * (s.d * 4 + 4)  # fp32 out + lse
    tr = 0 if inp.get("tree") is None else inp["tree"].numel() * 8  # token-tree node masks
    return kv, kv + q + o + tr


def causal_flops(s, inp):
    """4 * d per (row, visible key): QK^T and PV, 2 flops per multiply-add
    (a sliding window keeps the keys pos - W < j <= pos)."""
    lens = inp["seqlens"].numpy().astype(np.int64)
    pos = inp["qpos"].numpy().astype(np.int64)
    end = np.clip(np.minimum(lens[:, None], pos + 1), 0, None)  # [B, Tq]
    start = np.maximum(pos - s.window + 1, 0) if s.window else np.zeros_like(pos)
    vis = np.clip(end - start, 0, None)
    return float(vis.sum()) * s.Hq * 4 * s.d


def tensor_bound(s):
    """Workloads measured in FLOP/s (many query rows per head on tcgen05)."""
    return s.name in ("prefill", "window_prefill")


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def __enter__(self):
        if shutil.which("nvidia-smi") is None:
            return self
        self.file = tempfile.TemporaryFile(mode="w+")
        self.proc = subprocess.Popen(
            ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
             "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.file is None:
            return None
        self.file.seek(0)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.file.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, flag in zip(names, parts[4:8]):
                if flag.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return rank, local, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def flush_l2(buf):
    """Evict L2 by reading a buffer of twice its size (a written buffer would
    leave dirty lines whose write-back lands in the timed step)."""
    buf.sum()


def queue_ahead(ms: float = 5.0):
    """Keep the device busy (a timed sleep) while the host enqueues the timed
    steps, so that host launch gaps never land inside the device-timed
    region; the sleep itself precedes the first step's start event."""
    if hasattr(torch.cuda, "_sleep"):
        torch.cuda._sleep(int(ms * 1e-3 * 2.0e9))


def device_times(call, steps: int, warmup: int, before=None):
    """Device time (ms) of each of `steps` calls, CUDA events around each on
    the current stream, after `warmup` untimed calls.  All steps are enqueued
    behind a device sleep (queue_ahead) with one synchronize at the end, so
    the host's marshalling of a call never lands between its events.
    `before` (an L2 eviction) runs ahead of every call, outside its events."""
    for _ in range(warmup):
        if before is not None:
            before()
        call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    queue_ahead()
    for e0, e1 in ev:
        if before is not None:
            before()
        e0.record()
        call()
        e1.record()
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) for e0, e1 in ev]


class Runner:
    """Inputs resident on the device plus the call the user makes."""

    def __init__(self, name, seed_offset=0):
        from exact_blocked_attention_gb300 import blkattn
        self.blkattn = blkattn
        s = workloads.spec(name)
        if seed_offset:
            s = workloads.replace(s, seed=s.seed + 1000 * seed_offset)
        self.s = s
        self.cpu = workloads.generate(s)
        self.dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in self.cpu.items()}
        self.out = torch.empty(s.B, s.Hq, s.Tq, s.d, device="cuda")
        self.lse = torch.empty(s.B, s.Hq, s.Tq, device="cuda")
        self.plan = blkattn.debug_plan(s.B, s.Hq, s.Hkv, s.Tq, s.Tmax, s.d,
                                       torch.bfloat16 if s.dtype == "bf16" else torch.float32,
                                       torch.cuda.get_device_properties(0).multi_processor_count)

    def launches_per_call(self):
        # the tcgen05 decode kernel (kernel 3) folds its split units itself;
        # the split-KV kernels are followed by the merge kernel when split
        if self.plan["kernel"] == 3:
            return 1
        return 1 + (1 if self.plan["n_splits"] > 1 else 0)

    def call(self):
        g = self.dev
        self.blkattn.fwd(g["q"], g["k"], g["v"], g["seqlens"], g["qpos"], g["bias"], g["scale"],
                         self.out, self.lse, tree=g.get("tree"), window=g.get("window", 0))

    def free(self):
        del self.dev, self.out, self.lse


def time_steps(r: Runner, steps: int, warmup: int, world: int, flush: bool):
    """Device times (ms) per step: the whole call (the timed region, K steps
    between barrier + synchronize), then, in a second pass, the main kernel
    alone (an event recorded by the library between its two kernels; kept out
    of the first pass because it serialises the programmatic-dependent merge
    launch)."""
    blk = r.blkattn
    flush_buf = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda") if flush else None
    for _ in range(warmup):
        r.call()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    queue_ahead()
    for i in range(steps):
        if flush_buf is not None:
            flush_l2(flush_buf)
        starts[i].record()
        r.call()
        ends[i].record()
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    total = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    # second pass: main kernel only
    queue_ahead()
    for i in range(steps):
        if flush_buf is not None:
            flush_l2(flush_buf)
        blk.set_split_event(mids[i])
        starts[i].record()
        r.call()
    blk.set_split_event(None)
    torch.cuda.synchronize()
    main = [s.elapsed_time(m) for s, m in zip(starts, mids)]
    return total, main, wall


def _cudart():
    """The CUDA runtime library (for pitched host-to-device copies), or None."""
    import ctypes
    import glob
    names = ["libcudart.so", "libcudart.so.13"]
    names += glob.glob(os.path.join(os.path.dirname(torch.__file__), "lib", "libcudart*.so*"))
    names += glob.glob("/usr/local/cuda/lib64/libcudart.so*")
    for n in names:
        try:
            lib = ctypes.CDLL(n)
            lib.cudaMemcpy2DAsync.restype = ctypes.c_int
            lib.cudaMemcpy2DAsync.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_size_t,
                                              ctypes.c_size_t, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
            return lib
        except (OSError, AttributeError):
            continue
    return None


def time_e2e(r: Runner, steps: int, warmup: int):
    """The user's call end to end: pinned host inputs -> device, fwd, result
    -> pinned host, every step (device-timed with events).  Of the K/V cache
    only the valid rows of each sequence move (one pitched copy per sequence
    and tensor: H_kv runs of len_b rows); the rows past len_b are never read."""
    g = r.dev
    host = {k: r.cpu[k].pin_memory() for k in ("q", "k", "v", "seqlens", "qpos")}
    for opt in ("bias", "tree"):
        if r.cpu.get(opt) is not None:
            host[opt] = r.cpu[opt].pin_memory()
    out_h = torch.empty(r.out.shape, dtype=r.out.dtype).pin_memory()
    lse_h = torch.empty(r.lse.shape, dtype=r.lse.dtype).pin_memory()
    r.call()
    ref_out, ref_lse = r.out.cpu(), r.lse.cpu()  # the device-resident result
    rt = _cudart()
    if rt is not None and (g["k"].stride() != host["k"].stride() or g["v"].stride() != host["v"].stride()):
        rt = None
    lens = [min(max(int(x), 0), r.s.Tmax) for x in r.cpu["seqlens"].tolist()]
    whole = [k_ for k_ in host if rt is None or k_ not in ("k", "v")]
    h2d = sum(host[k_].numel() * host[k_].element_size() for k_ in whole)
    if rt is not None:
        row = r.s.d * host["k"].element_size()
        h2d += 2 * sum(r.s.Hkv * ln * row for ln in lens)
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()

    def step():
        for k_ in whole:
            g[k_].copy_(host[k_], non_blocking=True)
        if rt is not None:
            stream = torch.cuda.current_stream().cuda_stream
            for k_ in ("k", "v"):
                dt, ht = g[k_], host[k_]
                pitch = ht.stride(1) * ht.element_size()
                for b, ln in enumerate(lens):
                    if ln == 0:
                        continue
                    st = rt.cudaMemcpy2DAsync(dt[b].data_ptr(), pitch, ht[b].data_ptr(), pitch,
                                              ln * r.s.d * ht.element_size(), r.s.Hkv, 1, stream)
                    if st != 0:
                        raise RuntimeError(f"cudaMemcpy2DAsync failed: {st}")
        r.call()
        out_h.copy_(r.out, non_blocking=True)
        lse_h.copy_(r.lse, non_blocking=True)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        step()
    t1.record()
    torch.cuda.synchronize()
    # the copies moved what the call reads: the result is the device-resident run's
    if not (torch.equal(out_h, ref_out) and torch.equal(lse_h, ref_lse)):
        raise RuntimeError("end-to-end result differs from the device-resident call")
    return t0.elapsed_time(t1) / steps, h2d, d2h


def roofline_entry(r: Runner, main_ms, peaks, flops=None):
    s = r.s
    kv, total_bytes = algorithmic_bytes(s, r.cpu)
    if tensor_bound(s):
        achieved = flops / (main_ms * 1e-3) / 1e12
        return {"bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(achieved / peaks["bf16_tflops"], 4), "traffic": measured_traffic(s.name),
                "algorithmic_flops": flops, "algorithmic_bytes": total_bytes,
                "peak_note": f"dense bf16 burst, {peaks['source']}"}
    achieved = total_bytes / (main_ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": measured_traffic(s.name),
            "algorithmic_bytes": total_bytes, "peak_note": f"HBM copy bandwidth, {peaks['source']}"}


def oracle_rate(s, inp, budget_s: float, threads: int = 0):
    """Time the fp64 oracle on a bounded row sample; return (seconds per full
    workload, rows sampled, cores used)."""
    import oracle
    total_rows = s.B * s.Hq * s.Tq
    rng = np.random.default_rng(0)
    cores = oracle.max_threads() if threads <= 0 else threads
    n = min(total_rows, 64)
    spent, done = 0.0, 0
    while True:
        rows = rng.choice(total_rows, size=n, replace=False)
        t0 = time.perf_counter()
        oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"], inp["qpos"], inp["scale"],
                         bias=inp["bias"], rows=rows, nthreads=threads, tree=inp.get("tree"),
                         window=inp.get("window", 0))
        spent += time.perf_counter() - t0
        done += n
        if spent >= budget_s or done >= total_rows:
            break
        n = min(total_rows, n * 2)
    return spent / done * total_rows, done, cores


def line_config(s, inp, world):
    """The `config` of the JSON line: the workload, its per-step work and how
    L2 is kept out of the timing (the same dict on both arms)."""
    kv, total_bytes = algorithmic_bytes(s, inp)
    in_bytes = sum(t.numel() * t.element_size() for t in inp.values() if torch.is_tensor(t))
    return {"workload": describe(s), "kv_bytes_per_step": kv, "algorithmic_bytes_per_step": total_bytes,
            "l2": "evicted between steps (a read of 2x L2)" if in_bytes < 2 * L2_BYTES else f"inputs ({in_bytes / 1e6:.0f} MB) larger than L2",
            "parallelism": f"weak: {world} rank(s), own batch each"}


def run_reference(args, rank, world):
    """--impl reference: the fp64 CPU oracle on the host cores (rank 0 only)."""
    if rank != 0:
        return
    s = workloads.spec(args.workload)
    inp = workloads.generate(s)
    kv, _ = algorithmic_bytes(s, inp)
    budget = max(0.25, args.ref_budget_s / max(1, args.steps + args.warmup))
    import oracle
    for _ in range(args.warmup):
        oracle_rate(s, inp, budget / 4)
    per_step = []
    rows_total = 0
    cores = 1
    for _ in range(args.steps):
        sec, rows, cores = oracle_rate(s, inp, budget)
        per_step.append(sec)
        rows_total += rows
    sec = statistics.mean(per_step)
    value = kv / sec / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": line_config(s, inp, world),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows_total} random query rows over {args.steps} steps, "
                                   f"scaled to all {s.B * s.Hq * s.Tq} rows"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def measure_other(name, peaks):
    ro = Runner(name)
    fl = tensor_bound(ro.s)
    steps_o = 10 if not fl else 5
    # inputs larger than L2 need no flush (writing a flush buffer between
    # steps would leave dirty lines whose write-back lands in the timed step)
    in_bytes = sum(t.numel() * t.element_size() for t in ro.dev.values() if torch.is_tensor(t))
    tot, mn, _ = time_steps(ro, steps_o, 3, 1, flush=in_bytes < 2 * L2_BYTES)
    t_ms = sum(tot) / len(tot)
    m_ms = sum(mn) / len(mn)
    roof = roofline_entry(ro, m_ms, peaks, causal_flops(ro.s, ro.cpu) if fl else None)
    ro.free()
    # whole call (us) against the roofline; the main kernel's own figures are in `roofline`
    work = roof.get("algorithmic_flops", roof.get("algorithmic_bytes"))
    per_s = work / (t_ms * 1e-3) / (1e12 if fl else 1e9)
    return compact(name, t_ms * 1e3, per_s, roof, m_ms * 1e3)


# workloads that are BASELINE configurations (the others are "next" rows)
CONFIG_OF = {"tiny_fp32": 1, "decode_gqa": 2, "long_decode": 3, "spec_verify": 4, "prefill": 5}


def compact(name, us, achieved, roof, main_us=None):
    """One short entry per workload: whole-call time and throughput, its
    fraction of the roofline's peak, and DRAM traffic over algorithmic bytes
    (from the committed ncu record; null when the kernel changed since)."""
    e = {}
    if name in CONFIG_OF:
        e["config"] = CONFIG_OF[name]
    e.update({"us": round(us, 2), "achieved": round(achieved, 1), "unit": roof["unit"],
              "frac": round(achieved / roof["peak"], 4), "bound": roof["bound"]})
    if main_us is not None:
        e["main_us"] = round(main_us, 2)
    t, ab = roof.get("traffic"), roof.get("algorithmic_bytes")
    e["traffic_ratio"] = round(t / ab, 3) if (t and ab) else None
    return e


def measure_spec_sample(peaks, steps=10, warmup=3, full=False):
    """The speculative-sampling step (blkattn_spec_sample) on its full-size
    workload: device time per call with L2 cleared by a read of twice its size
    before each call (the rows a call reads fit in L2), and the bytes of the
    rows each sequence draws from (p_i and q_i of the first rejected position,
    or p_{k+1})."""
    from exact_blocked_attention_gb300 import blkattn
    s = workloads.sample_spec("spec_sample")
    cpu = workloads.generate_sampling(s)
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in cpu.items()}
    n_acc = torch.empty(s.B, dtype=torch.int32, device="cuda")
    tok = torch.empty(s.B, dtype=torch.int32, device="cuda")
    call = lambda: blkattn.spec_sample(dev["p"], dev["q"], dev["draft"], dev["u_accept"], dev["u_sample"],
                                       n_acc, tok)
    call()
    torch.cuda.synchronize()
    n = n_acc.cpu().numpy()
    row = s.V * 4
    drawn = int(sum(2 * row if int(x) < s.k else row for x in n))
    small = int(sum((int(x) + 1) * 12 for x in n)) + s.B * 12  # candidate p, q, u; s; outputs
    total = drawn + small
    # evict the rows by READING a buffer twice the L2 size: a written flush
    # buffer would leave dirty lines whose write-back lands in the timed call
    flush = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
    times = device_times(call, steps, warmup, before=lambda: flush.sum())
    t_ms = sum(times) / len(times)
    achieved = total / (t_ms * 1e-3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "traffic": measured_traffic("spec_sample"),
            "algorithmic_bytes": total}
    if full:
        return {"workload": f"spec_sample: B={s.B} k={s.k} V={s.V} f32 probabilities",
                "us_per_call": t_ms * 1e3, "l2": "evicted between steps by reading 2x its size",
                "kept_candidates_histogram": np.bincount(n, minlength=s.k + 1).tolist(), "roofline": roof}
    return compact("spec_sample", t_ms * 1e3, achieved, roof)


def measure_backward(peaks, steps=5, warmup=3, name="prefill", full=False):
    """The backward pass (blkattn_bwd: row facts, dQ, dK/dV) on the causal
    prefill workload with an upstream gradient; inputs come from the
    library's own forward.  Algorithmic work: the five products of eqs.
    33.6-33.8, 10 * d flops per (row, visible key) (2.5x the forward's 4 * d);
    the kernels form S and G_P twice, 7 products in all."""
    from exact_blocked_attention_gb300 import blkattn
    s = workloads.spec(name)
    cpu = workloads.generate_backward(s)
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in cpu.items()}
    W = cpu.get("window", 0)
    out, lse = blkattn.attention(dev["q"], dev["k"], dev["v"], dev["seqlens"], dev["qpos"], None, cpu["scale"],
                                 window=W)
    dq = torch.empty(dev["q"].shape, dtype=torch.float32, device="cuda")
    dk = torch.empty(dev["k"].shape, dtype=torch.float32, device="cuda")
    dv = torch.empty(dev["v"].shape, dtype=torch.float32, device="cuda")
    call = lambda: blkattn.bwd(dev["q"], dev["k"], dev["v"], dev["seqlens"], dev["qpos"], None, cpu["scale"],
                               out, lse, dev["go"], dq, dk, dv, window=W)
    in_bytes = sum(t.numel() * t.element_size() for t in (dev["q"], dev["k"], dev["v"], dev["go"], out, lse))
    times = device_times(call, steps, warmup)
    assert blkattn.check_device_error() == 0
    t_ms = sum(times) / len(times)
    flops = causal_flops(s, cpu) * 2.5
    achieved = flops / (t_ms * 1e-3) / 1e12
    # bytes every call must move at least once: q, k, v, g_o, o, lse in; dq, dk, dv out
    moved = sum(t.numel() * t.element_size() for t in (dev["q"], dev["k"], dev["v"], dev["go"], out, lse, dq, dk, dv))
    roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": achieved / peaks["bf16_tflops"], "traffic": measured_traffic(f"{name}_backward"),
            "algorithmic_flops": flops, "algorithmic_bytes": moved}
    if full:
        return {"workload": f"{name}_backward: {describe(s)}" + (f" window={W}" if W else "") +
                            " + g_o bf16; dq, dk, dv f32",
                "us_per_call": t_ms * 1e3, "l2": f"inputs ({in_bytes / 1e6:.0f} MB) larger than L2",
                "kernels": "row facts, dQ (3 products per tile pair), dK/dV (4 products per tile pair)",
                "roofline": roof, "frac_of_bf16_sustained": achieved / peaks["bf16_tflops_sustained"]}
    return compact(f"{name}_backward", t_ms * 1e3, achieved, roof)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE, choices=list(workloads.SPECS))
    ap.add_argument("--no-others", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only-sampling", action="store_true",
                    help="time only the speculative-sampling step and print its entry")
    ap.add_argument("--only-backward", action="store_true",
                    help="time only the backward pass and print its entry")
    ap.add_argument("--ref-budget-s", type=float, default=60.0,
                    help="--impl reference: seconds of oracle work over all steps")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    rank, local, world = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    torch.cuda.set_device(local)
    from exact_blocked_attention_gb300 import build as libbuild
    if rank == 0:
        libbuild.build()
    barrier(world)
    peaks = measured_peaks()
    if args.only_sampling:
        from exact_blocked_attention_gb300 import blkattn
        blkattn.load()
        if rank == 0:
            print(json.dumps(measure_spec_sample(peaks, steps=args.steps, warmup=args.warmup, full=True)), flush=True)
        return
    if args.only_backward:
        from exact_blocked_attention_gb300 import blkattn
        blkattn.load()
        if rank == 0:
            print(json.dumps(measure_backward(peaks, steps=args.steps, warmup=args.warmup, full=True)), flush=True)
            print(json.dumps(measure_backward(peaks, steps=args.steps, warmup=args.warmup, name="window_prefill",
                                              full=True)), flush=True)
        return

    # ---- headline workload: every rank runs its own batch (weak scaling) ----
    r = Runner(args.workload, seed_offset=rank)
    s = r.s
    kv, total_bytes = algorithmic_bytes(s, r.cpu)
    in_bytes = sum(t.numel() * t.element_size() for k, t in r.dev.items() if torch.is_tensor(t))
    flush = in_bytes < 2 * L2_BYTES
    with ClockSampler(local) as clk:
        total, main_ms, wall = time_steps(r, args.steps, args.warmup, world, flush)
    clocks = clk.summary()
    step_ms = max_over_ranks(sum(total) / len(total), world)
    main_avg = max_over_ranks(sum(main_ms) / len(main_ms), world)
    spread = {"min": min(total), "median": sorted(total)[len(total) // 2], "max": max(total)}
    value = kv * world / (step_ms * 1e-3) / 1e9
    if tensor_bound(s):
        value = causal_flops(s, r.cpu) * world / (step_ms * 1e-3) / 1e12
    e2e_ms, h2d, d2h = time_e2e(r, max(3, args.steps // 4), 2)
    e2e_ms = max_over_ranks(e2e_ms, world)
    e2e_value = kv * world / (e2e_ms * 1e-3) / 1e9
    roof = roofline_entry(r, main_avg, peaks, causal_flops(s, r.cpu))
    launches = r.launches_per_call() * args.steps
    plan = r.plan
    cpu_inp = r.cpu
    r.free()
    torch.cuda.empty_cache()

    line = {
        "metric": METRIC if s.name == HEADLINE else f"{s.name} throughput",
        "value": value,
        "unit": "GB/s" if not tensor_bound(s) else "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": s.dtype,
        "data": "synthetic",
        "config": line_config(s, cpu_inp, world),
        "plan": {k: plan[k] for k in ("kernel", "rows_per_cta", "n_splits", "ctas", "workspace_bytes")},
        "us_per_call": round(step_ms * 1e3, 2),
        "step_us_spread": [round(min(total) * 1e3, 2), round(spread["median"] * 1e3, 2), round(max(total) * 1e3, 2)],
        "main_kernel_us": round(main_avg * 1e3, 2),
        "frac_of_hbm_peak": round((total_bytes / (step_ms * 1e-3) / 1e9) / peaks["hbm_gbs"], 4),
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": clocks,
    }

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N=1 only) ----
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sec, rows, cores = oracle_rate(s, cpu_inp, 15.0)
        line["cpu_baseline"] = {"value": kv / sec / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
                                "sample": f"{rows} random query rows of the same batch, fp64, "
                                          f"scaled to all {s.B * s.Hq * s.Tq} rows"}
    # ---- the other workloads (rank 0 only), each with its own roofline ----
    if rank == 0 and not args.no_others:
        # (the configurations last: the end of the line is what a short log tail shows)
        order = ["tree_verify", "window_decode", "window_prefill", "prefill_backward", "window_prefill_backward",
                 "spec_sample", "tiny_fp32", "long_decode", "spec_verify", "prefill", "decode_gqa"]
        others = {}
        for name in order:
            if name == s.name:
                continue
            try:
                if name.endswith("_backward"):
                    others[name] = measure_backward(peaks, name=name[: -len("_backward")])
                elif name == "spec_sample":
                    others[name] = measure_spec_sample(peaks)
                else:
                    others[name] = measure_other(name, peaks)
            except Exception as exc:  # report, keep the headline line
                others[name] = {"error": f"{type(exc).__name__}: {exc}"}
            torch.cuda.empty_cache()
        line["workloads"] = others

    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
