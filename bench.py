#!/usr/bin/env python3
"""Benchmark of one paged GQA decode step on GB300.

A step is the whole decode path over one batch: the host block manager's
slot mapping (a1), copy-on-write copies when a block is shared (a2, none in
these workloads), the KV append (a3) and paged attention with its split merge
(a4-a8).  Default workload: the Llama-3.1-70B-shaped GQA decode layer (B=64,
Hq=64, Hkv=8, D=128, bf16, every context 8192 tokens).  Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload 1..5] [--num-splits P]

--impl reference times the CPU oracle (double precision, all host cores) on a
bounded sample of the same workload.  Under torchrun (N > 1) every rank runs
an independent replica; only rank 0 prints.
"""
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged GQA decode attention: achieved HBM GB/s (% of GB300 peak); decode tok/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=3)
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch size (smaller profiling cases)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU time budget of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--q-len", type=int, default=1,
                    help="new tokens per sequence per step (multi-query decode, causal)")
    ap.add_argument("--window", type=int, default=0,
                    help="sliding window: each row attends its W most recent positions")
    ap.add_argument("--calibrated", action="store_true",
                    help="fp8 caches: append with calibrated (running-max, power-of-two) block scales")
    ap.add_argument("--prefill", default="",
                    help="time paged prefill (tensor cores) on a prefill workload: page, llama70b, chunked")
    ap.add_argument("--mq-route", default="auto", choices=["auto", "transposed", "prefill", "units"],
                    help="force the library's kernel route for q_len >= 2 (pkv_set_route)")
    ap.add_argument("--prefill-route", default="auto", choices=["auto", "persistent", "tiles"],
                    help="force the prefill kernel's schedule (pkv_set_route)")
    return ap.parse_args()


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# --- replica aggregation (one process per GPU; no data-path collective) -----
def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    """The slowest rank's time: every rank's number, MAX-reduced."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_rank, world, ms):
    """Whole-job throughput: all ranks' bytes over the slowest rank's time."""
    return world * bytes_per_rank / (ms * 1e-3) / 1e9


def peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured (MEASURED_PEAKS.json hbm_gbs, copy read+write)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""

    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id):
        self.bus_id = (bus_id or "").lower()
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                rows.append(parts)
        os.unlink(self.path)
        if self.bus_id:
            mine = [r for r in rows if r[1].lower().endswith(self.bus_id[-12:])]
            rows = mine or rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


TRAFFIC_RECORDS = {"bf16": ("decode_traffic.json",), "f16": ("decode_traffic_f16.json",),
                   "fp8_e4m3": ("decode_traffic_fp8.json", "decode_traffic_fp8_qlen4.json")}


def kernel_traffic(w, kernel="", profiles_dir=None):
    """DRAM bytes per launch of the dominant kernel, from the committed ncu
    capture of that kernel (the decode kernel for the cache's dtype, or the
    transposed multi-query kernel) on a smaller case of the same kernel:
    reads scale with the K/V bytes a launch attends, writes (partials and
    outputs) are kept as captured.  None when the kernel's sources changed
    since the capture, the record covers another q_len, or the workload's
    sequences share blocks (L2 then serves most of the logical bytes)."""
    if w.window or w.prefix_blocks:
        return None
    mq = kernel.startswith("mq_decode_kernel")
    for name in ("mq_traffic.json",) if mq else TRAFFIC_RECORDS.get(w.dtype, ()):
        try:
            with open(os.path.join(profiles_dir or os.path.join(ROOT, "profiles"), name)) as f:
                rec = json.load(f)
        except Exception:
            continue
        if rec.get("q_len", 1) != w.q_len or "kv_bytes" not in rec:
            continue
        h = hashlib.sha256()
        for src in rec.get("sources", ("common.cuh", "decode.cuh", "internal.h")):
            with open(os.path.join(ROOT, "paged_kv_gqa_03_gb300", "csrc", src), "rb") as f:
                h.update(f.read())
        if rec.get("source_sha256") != h.hexdigest():
            continue
        return int(rec["dram_bytes_read"] / rec["kv_bytes"] * w.kv_bytes() + rec["dram_bytes_write"])
    return None


def oracle_sample_rate(w, seconds, threads=0):
    """Times the oracle's append + decode on the first sequences of w until
    about `seconds` of work; returns (GB/s of KV processed, description, cores)."""
    import numpy as np
    import oracle
    from oracle.block_table import BlockTable

    bt = BlockTable(w.num_blocks)
    for b in range(w.B):
        bt.adopt(b, w.tables[b], w.cached[b])
    L = w.q_len
    slots, _ = bt.append_slots([b for b in range(w.B) for _ in range(L)])
    k_new = w.k_new.reshape(w.B, L, w.Hkv, w.D)
    v_new = w.v_new.reshape(w.B, L, w.Hkv, w.D)
    mb = w.max_blocks
    table = np.full((w.B, mb), -1, dtype=np.int32)
    for b in range(w.B):
        table[b, :len(bt.seq_tables[b])] = bt.seq_tables[b]
    lens = np.array([bt.seq_tokens[b] for b in range(w.B)], dtype=np.int32)
    per_seq = [w.attended(int(lens[b])) * 2 * w.Hkv * w.D
               * {"f32": 4, "f16": 2, "bf16": 2, "fp8_e4m3": 1}[w.dtype] for b in range(w.B)]
    ks = None if w.k_scale is None else w.k_scale.numpy()   # views: the append writes through
    vs = None if w.v_scale is None else w.v_scale.numpy()
    done_bytes, elapsed, n = 0, 0.0, 1
    b0 = 0
    while elapsed < seconds:
        rows = [(b0 + i) % w.B for i in range(n)]
        t0 = time.perf_counter()
        oracle.append(w.k_cache, w.v_cache, w.dtype, k_new[rows].reshape(-1, w.Hkv, w.D),
                      v_new[rows].reshape(-1, w.Hkv, w.D), w.new_dtype,
                      [slots[r * L + t] for r in rows for t in range(L)], ks, vs, inplace=True)
        oracle.decode(w.q[rows], w.q_dtype, w.k_cache, w.v_cache, w.dtype, table[rows], lens[rows],
                      scale=w.scale, k_scale=ks, v_scale=vs, nthreads=threads, window=w.window)
        dt = time.perf_counter() - t0
        elapsed += dt
        done_bytes += sum(per_seq[r] for r in rows)
        b0 = (b0 + n) % w.B
        if dt < seconds / 8:
            n = min(w.B, n * 2)
    cores = oracle.num_threads() if threads <= 0 else threads
    desc = (f"oracle decode (fp64, OpenMP over sequence x kv-head) of {done_bytes / 1e9:.2f} GB of "
            f"KV from the same workload's sequences, {elapsed:.1f} s")
    return done_bytes / elapsed / 1e9, desc, cores


def spot_check(w, out, step):
    """Max-abs error of the timed run's output against the oracle on the first
    and last sequence (the oracle applies the same append on the host copy)."""
    import numpy as np
    import oracle
    rows = sorted({0, w.B - 1})
    L = w.q_len
    slots = step.h_slots.numpy().reshape(w.B, L)
    ks = None if w.k_scale is None else w.k_scale.numpy()
    vs = None if w.v_scale is None else w.v_scale.numpy()
    oracle.append(w.k_cache, w.v_cache, w.dtype, w.k_new[rows].reshape(-1, w.Hkv, w.D),
                  w.v_new[rows].reshape(-1, w.Hkv, w.D), w.new_dtype,
                  slots[rows].reshape(-1), ks, vs, inplace=True)
    table = step.h_table.numpy()[rows]
    lens = step.h_lens.numpy()[rows]
    ref = oracle.decode(w.q[rows], w.q_dtype, w.k_cache, w.v_cache, w.dtype, table, lens,
                        scale=w.scale, k_scale=ks, v_scale=vs, window=w.window)
    got = out[rows].double().cpu().numpy()
    return {"rows": rows, "max_abs_err": float(np.abs(got - ref).max())}


def run_reference(args, world, rank):
    if rank != 0:
        return
    import workloads
    w = _workload(args)
    budget = min(3.0, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample_rate(w, budget / 4)
    rates, times = [], []
    t_start = time.perf_counter()
    for _ in range(args.steps):
        t0 = time.perf_counter()
        r, desc, cores = oracle_sample_rate(w, budget)
        times.append(time.perf_counter() - t0)
        rates.append(r)
    total = time.perf_counter() - t_start
    value = statistics.median(rates)
    kv = w.kv_bytes()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(kv / (value * 1e9) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(w),
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": desc + f"; {args.steps} steps of ~{budget:.1f} s"},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "wall_s": round(total, 1),
    }
    print(json.dumps(line), flush=True)


def _workload(args):
    import workloads
    over = {}
    if args.batch:
        over["B"] = args.batch
    if args.q_len > 1:
        over["q_len"] = args.q_len
    if args.window:
        over["window"] = args.window
    return workloads.config(args.workload, **over)


def _config(w):
    extra = {} if w.q_len == 1 else {"q_len": w.q_len}
    if getattr(w, "calibrated", False):
        extra["fp8_append"] = "calibrated"
    if w.window:
        extra["window"] = w.window
    return extra | {"workload": w.name, "index": w.seed - 1000, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv,
            "D": w.D, "kv_dtype": w.dtype, "q_dtype": w.q_dtype, "block_size": 16,
            "context_lens": (w.context_lens[0] if len(set(w.context_lens)) == 1
                             else f"{min(w.context_lens)}..{max(w.context_lens)}"),
            "num_blocks": w.num_blocks,
            "pool_extra_blocks": getattr(w, "extra_blocks", 0),
            "l2": (f"KV read per step {w.kv_bytes() / 1e9:.2f} GB > 129 MB L2; no flush needed"
                   if w.kv_bytes() > 129e6 else
                   f"KV read per step {w.kv_bytes() / 1e6:.2f} MB < 129 MB L2: L2-resident across steps, "
                   "not flushed (a small case: launch latency, not HBM, bounds it)")}


def grow_pool(w, extra):
    """Appends `extra` free physical blocks (zeros; fp8 scales 1) to the
    workload's pool, so that the end-to-end loop can advance every context
    by one token per step; the block tables and every value already in the
    pool stay as drawn."""
    import torch
    if extra <= 0:
        return
    def grow(t, fill):
        pad = torch.full((extra,) + tuple(t.shape[1:]), fill, dtype=torch.uint8 if t.element_size() == 1 else t.dtype)
        base = t.view(torch.uint8) if t.element_size() == 1 else t
        out = torch.cat([base, pad])
        return out.view(t.dtype) if t.element_size() == 1 else out
    w.k_cache, w.v_cache = grow(w.k_cache, 0), grow(w.v_cache, 0)
    if w.k_scale is not None:
        w.k_scale, w.v_scale = grow(w.k_scale, 1.0), grow(w.v_scale, 1.0)
    w.num_blocks += extra


def run_ours(args, world, rank, local):
    import numpy as np
    import torch

    import workloads
    import paged_kv_gqa_03_gb300 as pkv
    from paged_kv_gqa_03_gb300.step import DecodeStep

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16,
           "fp8_e4m3": torch.float8_e4m3fn}
    w = _workload(args)
    w.calibrated = args.calibrated
    # room for the end-to-end loop's advancing contexts
    e2e_steps = args.steps + 4
    grow_blocks = -(-(e2e_steps + 1) * w.q_len // 16) + 1      # per sequence
    extra = w.B * grow_blocks
    grow_pool(w, extra)
    w.extra_blocks = extra
    pkv.pkv_set_route("multi_query", args.mq_route)
    pkv.pkv_set_route("prefill", args.prefill_route)
    stream = torch.cuda.Stream(dev)
    ks = None if w.k_scale is None else w.k_scale.to(dev)
    vs = None if w.v_scale is None else w.v_scale.to(dev)
    # block tables with room for the end-to-end loop's growth
    step = DecodeStep(w.k_cache.to(dev), w.v_cache.to(dev), w.Hq, tdt[w.q_dtype], w.max_blocks + grow_blocks,
                      ks, vs, num_splits=args.num_splits, stream=stream, scale=w.scale,
                      q_len=w.q_len, window=w.window, calibrated=args.calibrated)
    for b in range(w.B):
        step.adopt(b, w.tables[b], w.cached[b])
    step.prepare()
    step.upload()
    q, kn, vn = w.q.to(dev), w.k_new.to(dev), w.v_new.to(dev)
    out = torch.empty_like(q)
    kv = w.kv_bytes()

    kname = attention_kernel_name(w, args.num_splits, torch.cuda.get_device_properties(dev).multi_processor_count,
                                  args.mq_route)

    # warm-up
    for _ in range(args.warmup):
        step.launch(q, kn, vn, out)
    stream.synchronize()

    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
    except Exception:
        pass
    sampler = ClockSampler(bus)
    sampler.start()

    # (1) device-timed steps: append + attention (+ merge), inputs resident in HBM
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    timed_launches = 0
    for _ in range(args.steps):
        step.launch(q, kn, vn, out)
        timed_launches += launches_per_step(w, kname, step.ncow)
    e1.record(stream)
    e1.synchronize()
    barrier(world)
    ms_step = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)

    # (2) the attention call alone, same stream, for the roofline of the dominant kernel
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a0.record(stream)
    for _ in range(args.steps):
        step.attend(q, out)
    a1.record(stream)
    a1.synchronize()
    ms_attn = max_over_ranks(a0.elapsed_time(a1) / args.steps, world, dev)
    clocks = sampler.stop()

    # host cost of one attention call (argument marshalling, the C ABI's
    # checks and launches), issued back to back without waiting
    torch.cuda.synchronize()
    nh = 100
    th0 = time.perf_counter()
    for _ in range(nh):
        step.attend(q, out)
    host_us = (time.perf_counter() - th0) / nh * 1e6
    stream.synchronize()

    # a spot check of the device-timed step's outputs against the oracle on
    # two sequences, before the serving loop below advances the bookkeeping
    # (the calibrated append re-quantises blocks, so its cache is the
    # oracle's only after the same sequence of appends: no spot check there)
    check = spot_check(w, out, step) if rank == 0 and not args.calibrated else None

    # (3) end to end through the public API from pinned host memory, as a
    # serving loop runs it: every step appends q_len new tokens to every
    # sequence (contexts advance; blocks open every 16 tokens); a captured
    # graph per staging buffer copies the step's inputs and bookkeeping in,
    # appends, attends and writes the output into pinned host memory.  The
    # host keeps one step queued ahead: it issues step n, then waits for step
    # n - 1, reads its output (two pinned output buffers alternate) and runs
    # the a1 of step n + 1 (slot mapping, copy-on-write pairs, tables) into the
    # staging buffer step n - 1 read — all while step n runs on the GPU.
    # Timed by the host's clock from the first issue to the last output read.
    hout = [torch.empty(w.q.shape, dtype=w.q.dtype).pin_memory() for _ in range(2)]
    step.stage_inputs(w.q, w.k_new, w.v_new, both=True)
    step.prepare()
    for i in range(4):                  # the first step eager, then a graph per staging buffer
        step.run(hout[i % 2])
        stream.synchronize()
        step.prepare()
    barrier(world)
    torch.cuda.synchronize()
    a1_us, wait_us, step_lens = [], [], []
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    th_start = time.perf_counter()
    x0.record(stream)
    for n in range(args.steps):
        gev[n][0].record(stream)
        step.run(hout[n % 2])
        gev[n][1].record(stream)         # the step's own GPU time (copies in and out included)
        step_lens.append(step.h_lens.numpy().copy())   # this step's context lengths
        if n > 0:
            t1 = time.perf_counter()
            gev[n - 1][1].synchronize()  # step n - 1 is done ...
            wait_us.append((time.perf_counter() - t1) * 1e6)
            _ = float(hout[(n - 1) % 2].view(-1)[0])   # ... and the host reads its result
        t0 = time.perf_counter()
        step.prepare()                  # a1 of step n + 1, overlapping step n
        a1_us.append((time.perf_counter() - t0) * 1e6)
    x1.record(stream)
    x1.synchronize()
    _ = float(hout[(args.steps - 1) % 2].view(-1)[0])
    th_end = time.perf_counter()
    barrier(world)
    ms_e2e = max_over_ranks((th_end - th_start) * 1e3 / args.steps, world, dev)
    ms_gpu_line = x0.elapsed_time(x1) / args.steps
    kv_e2e = sum(w.kv_bytes(lens) for lens in step_lens) / args.steps
    h2d = step.h2d_bytes(with_inputs=True)
    d2h = hout[0].numel() * hout[0].element_size()
    host_a1_us = statistics.median(a1_us)
    graph_ms = statistics.median(a.elapsed_time(b) for a, b in gev)

    if rank != 0:
        torch.distributed.destroy_process_group() if world > 1 else None
        return
    peak, peak_src = peak_hbm()
    value = job_gbs(kv, world, ms_step)
    attn_gbs = kv / (ms_attn * 1e-3) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        r, desc, cores = oracle_sample_rate(w, args.cpu_seconds)
        cpu = {"value": round(r, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded N(0,1), random block permutation)",
        "config": _config(w) | {"parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "tok_per_s": round(world * w.B * w.q_len / (ms_step * 1e-3), 1),
        "attn_tflops": round(4.0 * w.Hq * w.D * sum(
            min(max(0, c - w.q_len + 1 + i), w.window or 1 << 30)
            for c in w.context_lens for i in range(w.q_len)) / (ms_attn * 1e-3) / 1e12, 2),
        "frac_of_nominal_8tbs": round(value / world / NOMINAL_HBM_GBS, 4),
        "roofline": {"bound": "hbm", "kernel": kname,
                     "achieved": round(attn_gbs, 2), "peak": peak, "peak_source": peak_src,
                     "unit": "GB/s", "frac": round(attn_gbs / peak, 4),
                     "traffic": kernel_traffic(w, kname),
                     "algorithmic_bytes_per_launch": kv,
                     "ms_per_launch": round(ms_attn, 4)},
        "unique_kv": unique_kv_line(w, ms_step, ms_attn, peak),
        "cpu_baseline": cpu,
        "e2e": {"value": round(job_gbs(kv_e2e, world, ms_e2e), 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(ms_e2e, 4),
                "loop": "serving loop, host clock from the first issue to the last output read: contexts "
                        "advance q_len tokens per sequence per step; one step queued ahead (issue step n, "
                        "wait for step n-1 and read its output, a1 of step n+1) while step n runs; a graph "
                        "per staging buffer; two pinned output buffers",
                "a1_us_median": round(host_a1_us, 1),
                "host_wait_for_previous_step_us_median": round(statistics.median(wait_us), 1)
                if wait_us else None,
                "gpu_timeline_ms_per_step": round(ms_gpu_line, 4),
                "gap_vs_device_step_ms": round(ms_e2e - ms_step, 4),
                "graph_gpu_ms_median": round(graph_ms, 4),
                "gap_split": "graph_gpu_ms - ms_per_step of the device loop: the step's copies in and out; "
                             "e2e ms_per_step - graph_gpu_ms: GPU idle between steps (graph launch latency) "
                             "and the last step's output read"},
        "host_a1_us": round(host_a1_us, 1),
        "host_us_per_attention_call": round(host_us, 1),
        "clocks": clocks,
        "gpu_launches": timed_launches,
        "num_splits": args.num_splits,
        "check": check,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def unique_kv_line(w, ms_step, ms_attn, peak):
    """For a workload whose sequences share prefix blocks: the distinct K/V
    bytes a step reads (each shared block once, whole blocks), per step and
    per attention call, against the HBM peak.  The logical figure counts
    every sequence's read of the shared blocks, most of which L2 serves."""
    if not w.prefix_blocks:
        return None
    u = w.unique_kv_bytes()
    return {"bytes": u, "logical_bytes": w.kv_bytes(),
            "step_gbs": round(u / (ms_step * 1e-3) / 1e9, 2),
            "attn_gbs": round(u / (ms_attn * 1e-3) / 1e9, 2),
            "attn_frac": round(u / (ms_attn * 1e-3) / 1e9 / peak, 4)}


def peak_bf16():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    except Exception:
        return 1900.0, "fallback"


def launches_per_step(w, kernel_name, ncow):
    """Our kernels launched by one timed step (DecodeStep.launch): the
    copy-on-write block copy when the step has pairs, the append, and the
    attention call's kernels for its route (decode + merge, plus the plan
    kernel from 2048 sequences on; the transposed kernel + its merge; one
    prefill kernel)."""
    if kernel_name.startswith("mq_decode_kernel"):
        attn = 2
    elif kernel_name.startswith("prefill"):
        attn = 1
    else:
        attn = 2 + (1 if w.B >= 2048 else 0)
    return (1 if ncow else 0) + 1 + attn


def attention_kernel_name(w, num_splits, sms, force="auto"):
    """The kernels the library's attention call runs for this decode
    workload (the C ABI's routing rule, with the route forced by
    pkv_set_route("multi_query", force) honoured)."""
    if w.q_len == 1:
        return "paged_decode_attention (plan + decode + merge)"
    G = w.Hq // w.Hkv
    R = w.q_len * G
    sixteen = w.dtype in ("bf16", "f16")
    fp8_ok = w.dtype == "fp8_e4m3" and R <= 32 and force == "transposed"  # widened to f16 there: forced only
    fills = w.B * w.Hkv * ((R + 127) // 128) >= sms and w.B <= 65535
    if num_splits == 0 and (sixteen or fp8_ok) and force not in ("units", "prefill") and w.D == 128 and R <= 64 \
            and w.B <= 2048 and (R <= 32 or not fills or force == "transposed"):
        return "mq_decode_kernel (transposed tcgen05, stream-K) + mq_merge_kernel"
    if num_splits == 0 and sixteen and force != "units" and fills:
        return "prefill tcgen05 kernel (128-row tiles, uniform q_len)"
    rows = 16 if w.dtype == "fp8_e4m3" and R > 8 else 8  # fp8 kv heads past 8 rows: 16-row units
    return f"paged_decode_attention (plan + decode in {rows}-row units + merge)"


def prefill_kernel_name(c, force="auto"):
    """The kernel the library runs for this workload: one CTA per work item
    when the block table admits a cached prefix of 2048+ positions before
    the new tokens, the persistent kernel otherwise (unless forced)."""
    G = c["Hq"] // c["Hkv"]
    tiles = c["table"].shape[1] * 16 - max(c["n"]) >= (1024 if max(c["n"]) * G <= 64 else 2048)
    if force in ("tiles", "persistent"):
        tiles = force == "tiles"
    return ("prefill_tile_kernel (tcgen05, one CTA per work item)" if tiles
            else "prefill_kernel (tcgen05, persistent)")


def run_prefill(args, world, rank, local):
    """Paged prefill on the tensor cores: each launch attends every new token
    of the workload causally; value = useful TFLOP/s (4 * D per query head and
    visible position), L2 flushed before every timed launch."""
    import numpy as np
    import torch

    import workloads
    import paged_kv_gqa_03_gb300 as pkv

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pkv.pkv_set_route("prefill", args.prefill_route)
    spec = dict(workloads.PREFILL_SPECS[args.prefill])
    c = workloads.make_prefill(2000 + list(workloads.PREFILL_SPECS).index(args.prefill), **spec,
                               free=8, window=args.window)
    flops = workloads.prefill_flops(c)
    q, kc, vc = c["q"].to(dev), c["kc"].to(dev), c["vc"].to(dev)
    table = torch.from_numpy(c["table"]).to(dev)
    lens = torch.from_numpy(c["ctx"]).to(dev)
    q_start = torch.from_numpy(c["q_start"]).to(dev)
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)
    scale = 1.0 / math.sqrt(c["D"])
    max_n = max(c["n"])
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # > 129 MB L2

    def launch():
        pkv.paged_prefill_attention(out, q, kc, vc, table, lens, q_start, max_n, scale,
                                    window=args.window, status=status, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            launch()
    stream.synchronize()
    sampler = ClockSampler(torch.cuda.get_device_properties(dev).pci_bus_id)
    sampler.start()
    times = []
    for _ in range(args.steps):
        with torch.cuda.stream(stream):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            launch()
            e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    clocks = sampler.stop()
    ms = max_over_ranks(statistics.median(times), world, dev)
    tflops = flops / (ms * 1e-3) / 1e12
    assert int(status.item()) == 0

    # end to end: q from pinned host memory, the launch, out back to pinned host memory
    hq = c["q"].pin_memory()
    hout = torch.empty_like(hq).pin_memory()
    e2e = []
    for _ in range(args.steps):
        with torch.cuda.stream(stream):
            x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            x0.record(stream)
            pkv.pkv_copy(q, hq, stream=stream)
            launch()
            pkv.pkv_copy(hout, out, stream=stream)
            x1.record(stream)
        x1.synchronize()
        e2e.append(x0.elapsed_time(x1))
    ms_e2e = statistics.median(e2e)

    # context: torch SDPA (a library kernel) on the same prompts stored contiguously, when
    # nothing is cached and no window is set
    sdpa = None
    if not any(c["prefix"]) and not args.window:
        G = c["Hq"] // c["Hkv"]
        qs = [q[c["q_start"][b]:c["q_start"][b + 1]].transpose(0, 1)[None] for b in range(len(c["n"]))]
        qq = torch.cat(qs)                                                   # [B, Hq, n, D]
        kk = torch.randn((qq.shape[0], c["Hkv"], qq.shape[2], c["D"]), device=dev, dtype=q.dtype)
        vv = torch.randn_like(kk)
        F = torch.nn.functional
        kx = kk.repeat_interleave(G, 1) if G > 1 else kk
        vx = vv.repeat_interleave(G, 1) if G > 1 else vv
        for _ in range(3):
            F.scaled_dot_product_attention(qq, kx, vx, is_causal=True)
        st = []
        for _ in range(args.steps):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            F.scaled_dot_product_attention(qq, kx, vx, is_causal=True)
            e1.record()
            e1.synchronize()
            st.append(e0.elapsed_time(e1))
        sdpa = {"tflops": round(flops / (statistics.median(st) * 1e-3) / 1e12, 1),
                "ms": round(statistics.median(st), 4),
                "what": "torch scaled_dot_product_attention, is_causal, contiguous K/V (GQA heads expanded), same shapes"}

    # oracle sample on the host cores: the first 64 rows' worth of one sequence
    cpu = None
    if not args.no_cpu_baseline and rank == 0:
        import oracle
        rows = np.arange(min(64, c["n"][0]))
        lens = np.array([c["ctx"][0] - c["n"][0] + r + 1 for r in rows], dtype=np.int32)
        t0 = time.perf_counter()
        oracle.decode(c["q"][rows], c["dtype"], c["kc"], c["vc"], c["dtype"], c["table"][np.zeros_like(rows)],
                      lens, scale=scale, window=args.window)
        dt = time.perf_counter() - t0
        f = 4.0 * c["D"] * c["Hq"] * sum(min(l, args.window) if args.window else l for l in lens)
        cpu = {"value": round(f / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
               "kind": "oracle", "sample": f"oracle (fp64) on {len(rows)} rows of sequence 0, {dt:.1f} s"}
    if rank != 0:
        return
    peak, src = peak_bf16()
    line = {
        "metric": "paged prefill attention throughput (causal, useful FLOPs)", "value": round(tflops, 1),
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": c["dtype"], "data": "synthetic (seeded N(0,1), random block permutation)",
        "config": {"workload": f"prefill {args.prefill}", "B": len(c["n"]), "new_tokens": c["n"][0],
                   "cached_prefix": c["prefix"][0], "Hq": c["Hq"], "Hkv": c["Hkv"], "D": c["D"],
                   "window": args.window, "block_size": 16, "l2": "flushed (256 MB write) before every timed launch"},
        "roofline": {"bound": "tensor", "kernel": prefill_kernel_name(c, args.prefill_route), "achieved": round(tflops, 1),
                     "peak": peak, "peak_source": src, "unit": "TFLOP/s", "frac": round(tflops / peak, 4),
                     "traffic": None, "algorithmic_flops_per_launch": flops,
                     "note": "bf16 caches: P . V takes P as a bf16 high part plus residual (two MMAs per k-step)"},
        "e2e": {"value": round(flops / (ms_e2e * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
                "h2d_bytes_per_step": q.numel() * q.element_size(),
                "d2h_bytes_per_step": out.numel() * out.element_size(), "ms_per_step": round(ms_e2e, 4)},
        "sdpa_contiguous": sdpa, "cpu_baseline": cpu, "clocks": clocks, "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.prefill:
        run_prefill(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
