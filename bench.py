#!/usr/bin/env python3
"""Benchmark of one continuous-batching attention step over a paged KV cache.

Headline (`value`): query tokens/s of the mixed step -- 8 chunked-prefill
chunks of 512 tokens (cached context uniform in 0..8192), 192 decode rows
(seq_len uniform in 256..8192) and 32 speculative-verify rows of 1+4 tokens;
32 q / 8 kv heads, head_dim 128, block_size 16, bf16.  One step = one
pa_write_kv_attention call: write the 4448 new K/V rows through the slot
mapping + attention for every row (device planner, split-KV kernel,
tensor-core kernel, fused split merge).  Inputs are
resident in HBM and larger than L2 (about 3.9 GB of KV is read per step), so
no L2 flush is needed between steps.

Also reported on the same line:
  roofline      the attention kernel with the larger share of the step:
                algorithmic bytes (or flops) per launch / its CUDA-event
                duration inside the timed region, against the measured HBM
                copy bandwidth (or bf16 tensor throughput);
  kernels       both attention kernels in that form (split-KV in GB/s,
                tcgen05 prefill in TFLOP/s);
  decode_heavy  256 decode rows, seq_len uniform in 512..4096: KV GB/s;
  cascade       64 requests sharing an 8192-token prefix: cascade decode vs
                plain paged attention over the full tables;
  e2e           the same step through the public API with host buffers
                (pinned host -> device copies of every step's inputs and
                device -> host copy of its out/lse inside the timed region,
                on a second stream that overlaps the neighbouring steps);
  cpu_baseline  the fp64 CPU oracle on a 1/8 sample of the step.

`--impl reference` times the CPU oracle itself (the reference arm).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "decode paged-attn KV GB/s (% HBM peak); mixed-step query tokens/s on 1 GB300"
WORKLOAD = ("mixed continuous-batching step: 8 chunked-prefill chunks x 512 tokens "
            "(context U[0,8192]) + 192 decode rows (seq_len U[256,8192]) + 32 spec-verify "
            "rows of 1+4 tokens; 32 q / 8 kv heads, d=128, block_size 16, bf16")


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---------------------------------------------------------------------------
# environment
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(
            p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------------------------
# workloads on the device
# ---------------------------------------------------------------------------

class DeviceStep:
    """One step's inputs on the device; with fp8=True the pool is an e4m3 pool
    of the same shape (codes and per-kv-head scales drawn by the workload
    generator) and every call passes its scales."""

    def __init__(self, pool, step, dev, fp8=False):
        import paged_kv_cache_284_gb300 as pk
        from paged_kv_cache_284_gb300 import workloads
        self.pk = pk
        self.step = step
        self.dev = dev
        self.scales = {}
        if fp8:
            pool8 = workloads.fp8_pool_like(pool, workloads.SEED_BASE + 80)
            self.kc, self.vc = pool8.k_cache.to(dev), pool8.v_cache.to(dev)
            self.scales = {"k_scale": pool8.k_scale.to(dev), "v_scale": pool8.v_scale.to(dev)}
        else:
            self.kc = pool.k_cache.to(dev)
            self.vc = pool.v_cache.to(dev)
        self.q = step.q.to(dev)
        self.k = step.k.to(dev)
        self.v = step.v.to(dev)
        self.slots = step.slot_mapping.to(dev)
        self.bt = step.block_tables.to(dev)
        self.qsl = step.query_start_loc.to(dev)
        self.ctx = step.context_lens.to(dev)
        self.sl = step.seq_lens.to(dev)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty(self.q.shape[:2], dtype=torch.float32, device=dev)
        T, hq, d = self.q.shape
        nbytes = pk.workspace_size(step.num_seqs, T, hq, step.num_kv_heads, d)
        if fp8:
            # room to stage the long requests' blocks for the tensor-core kernel
            nbytes += pk.fp8_staging_bytes(step.num_kv_heads, d, step.block_size,
                                           staging_blocks(step))
        self.ws = pk.alloc_workspace(nbytes, dev)

    def run(self, write=True, fused=True):
        """One step: the cache write and the attention, through the one-call
        entry point (fused=True; the write runs beside the step's planner)
        or as pa_write_kv then pa_attention; write=False attends only."""
        pk = self.pk
        if write and fused:
            pk.pa_write_kv_attention(self.k, self.v, self.slots, self.q, self.kc, self.vc,
                                     self.bt, self.qsl, self.ctx, self.sl, self.step.scale,
                                     self.out, self.lse, workspace=self.ws, **self.scales)
            return
        if write:
            pk.pa_write_kv(self.k, self.v, self.slots, self.kc, self.vc, **self.scales)
        pk.pa_attention(self.q, self.kc, self.vc, self.bt, self.qsl, self.ctx, self.sl,
                        self.step.scale, self.out, self.lse, workspace=self.ws, **self.scales)


def staging_blocks(step, short_max_rows=64):
    """Blocks of the requests that run on the tensor-core kernel (q_len *
    group > short_max_rows): the bf16 staging room an e4m3 pool needs."""
    group = step.num_q_heads // step.num_kv_heads
    bs = step.block_size
    return sum(-(-int(step.seq_lens[b]) // bs) for b, n in enumerate(step.q_lens.tolist())
               if n * group > short_max_rows)


def split_rows(step, short_max_rows=64):
    """Indices of requests the split-KV kernel takes (q_len*group <= 64)."""
    g = step.num_q_heads // step.num_kv_heads
    ql = step.q_lens.tolist()
    return [b for b, n in enumerate(ql) if 0 < n * g <= short_max_rows]


def algorithmic_bytes(step, reqs, kv_elem_bytes=2):
    """HBM bytes a perfect kernel must move for these requests: each visible
    K and V row once per kv head (kv_elem_bytes per element: 2 for bf16, 1
    for e4m3), q read once, out + lse written once, and the block-table
    entries (per kv head)."""
    hkv, hq, d, bs = step.num_kv_heads, step.num_q_heads, step.head_dim, step.block_size
    total = 0
    for b in reqs:
        L = int(step.seq_lens[b])
        n = int(step.query_start_loc[b + 1] - step.query_start_loc[b])
        total += 2 * L * hkv * d * kv_elem_bytes  # K and V
        total += 2 * n * hq * d * 2 + n * hq * 4  # q, out, lse
        total += math.ceil(L / bs) * 4 * hkv     # block table
    return total


def kv_bytes(step, reqs, kv_elem_bytes=2):
    hkv, d = step.num_kv_heads, step.head_dim
    return sum(2 * int(step.seq_lens[b]) * hkv * d * kv_elem_bytes for b in reqs)


def tensor_core_flops(step, reqs):
    """4 * d * Hq flops per visible (query, key) pair (QK^T and PV)."""
    total = 0
    for b in reqs:
        n = int(step.query_start_loc[b + 1] - step.query_start_loc[b])
        c = int(step.context_lens[b])
        pairs = n * c + n * (n + 1) // 2
        total += 4 * step.head_dim * step.num_q_heads * pairs
    return total


def make_events(n):
    """n (start, end) timing events, created now: torch creates the CUDA
    event lazily at the first record, and the library records them by
    handle, so each is recorded once here, outside any timed region."""
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(n)]
    for a, b in pairs:
        a.record()
        b.record()
    torch.cuda.synchronize()
    return pairs


def max_over_ranks(ms: float, device) -> float:
    """Slowest rank's time (replicas run independently; the job is as slow as
    its slowest GPU).  A no-op without torch.distributed."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, units_per_step: int, steps: int, ms: float) -> float:
    """Whole-job units/s: every rank processed units_per_step per step."""
    return world * units_per_step * steps / (ms / 1000.0)


def time_steps(fn, steps, stream):
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end)


def sharded_mixed_step(world: int, rank: int):
    """The job at N > 1 GPUs: N copies of the mixed-step recipe's requests
    (seeds 284003 + 1000 i), routed to the N replicas by the library's
    request router (KV tokens balanced, greedy longest first).  This rank
    builds a pool and a step for its own requests only; no data crosses
    ranks.  Returns (pool, step, global request list)."""
    import paged_kv_cache_284_gb300 as pk
    from paged_kv_cache_284_gb300 import workloads
    reqs = []
    for i in range(world):
        reqs += workloads.mixed_step_requests(seed=workloads.SEED_BASE + 3 + 1000 * i)
    rank_of, _ = pk.partition_requests([c + n for c, n in reqs], world)
    mine = [reqs[b] for b in range(len(reqs)) if rank_of[b] == rank]
    pool, (step,) = workloads.from_requests(mine, seed=workloads.SEED_BASE + 3 + 1000 * rank,
                                            label=f"mixed step shard {rank}/{world}")
    return pool, step, reqs


def headline_config(args, world, step, pool, global_reqs=None):
    """The `config` object of the JSON line, the same on both arms: the
    whole job's requests, query tokens and KV bytes."""
    fp8 = args.kv_dtype == "fp8"
    elem = 1 if fp8 else 2
    hkv, d = step.num_kv_heads, step.head_dim
    if global_reqs is None:
        reqs = [(int(c), int(n)) for c, n in zip(step.context_lens.tolist(),
                                                 step.q_lens.tolist())]
    else:
        reqs = global_reqs
    cfg = {"workload": (WORKLOAD if args.workload == "mixed_step" else step.label)
           + ("; e4m3 KV pool, per-kv-head scales" if fp8 else ""),
           "kv_dtype": args.kv_dtype,
           "requests": len(reqs),
           "query_tokens": sum(n for _, n in reqs),
           "kv_bytes_read_per_step": sum(2 * (c + n) * hkv * d * elem for c, n in reqs),
           "l2": "inputs larger than L2 (no flush needed)",
           "parallelism": (f"{world} request-sharded replicas: the library's router splits "
                           f"{world} copies of the step's requests over the GPUs by KV tokens; "
                           f"no collective on the data path") if world > 1 else "single GPU",
           "seed": 284003}
    if world == 1:
        cfg["pool_blocks"] = pool.num_blocks
    return cfg


def all_ranks_sum(x: int, device) -> int:
    """Sum of an integer over ranks (each replica's query tokens); a no-op
    without torch.distributed."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.int64, device=device)
    dist.all_reduce(t)
    return int(t.item())


# ---------------------------------------------------------------------------
# CPU oracle baseline
# ---------------------------------------------------------------------------

def oracle_sample(pool, step, fraction=8):
    """1/fraction of the mixed step: every fraction-th request of each kind."""
    from paged_kv_cache_284_gb300 import workloads
    ql = step.q_lens.tolist()
    kinds = {}
    for b, n in enumerate(ql):
        kinds.setdefault(n, []).append(b)
    idx = []
    for n, bs in sorted(kinds.items()):
        idx += bs[::fraction]
    return workloads.subset(step, sorted(idx))


def time_oracle(pool, sub):
    import oracle
    t0 = time.perf_counter()
    kb, vb = oracle.write_kv(sub.k, sub.v, sub.slot_mapping, pool.k_cache, pool.v_cache)
    oracle.attention(sub.q, kb, vb, sub.block_tables, sub.query_start_loc, sub.context_lens,
                     sub.seq_lens, sub.scale)
    return time.perf_counter() - t0


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def traffic_for(kernel: str):
    """dram bytes per KV byte from the committed ncu summary, if the kernel
    source is unchanged since it was captured."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel)
    if not rec:
        return None
    src = os.path.join(ROOT, rec["source"])
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if sha != rec["source_sha256_16"]:
        return None
    return rec


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from paged_kv_cache_284_gb300 import workloads
    oracle.build_oracle()
    global_reqs = None
    if world > 1:
        pool, step, global_reqs = sharded_mixed_step(world, 0)
    else:
        pool, (step,) = workloads.mixed_step()
    sub = oracle_sample(pool, step)
    for _ in range(args.warmup):
        time_oracle(pool, sub)
    t = 0.0
    for _ in range(args.steps):
        t += time_oracle(pool, sub)
    tok = sub.num_q_tokens * args.steps
    value = tok / t
    cores = os.cpu_count()
    sample = (f"1/8 of the mixed step{' shard of rank 0' if world > 1 else ''} per timed "
              f"step ({sub.num_seqs} requests, {sub.num_q_tokens} query tokens): oracle "
              f"write_kv + attention, fp64")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "query tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * t / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": headline_config(args, world, step, pool, global_reqs),
        "cpu_baseline": {"value": value, "unit": "query tokens/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "query tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


KERNEL_TIMING = ("CUDA events around every launch of the kernel, on its stream, in a second "
                 "pass of the same K steps right after the timed pass (with the events set, "
                 "the step launches its kernels one after the other; the timed pass runs the "
                 "split-KV and tensor-core kernels side by side)")


def run_ours(args):
    import paged_kv_cache_284_gb300 as pk
    from paged_kv_cache_284_gb300 import workloads
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    hbm_peak, tc_peak, tc_peak_sus, peak_src = peaks()

    # ---- headline: the mixed step ------------------------------------------
    t0 = time.time()
    global_reqs = None
    if args.workload == "mixed_step" and world > 1:
        pool, step, global_reqs = sharded_mixed_step(world, rank)
    elif args.workload == "mixed_step":
        pool, (step,) = workloads.mixed_step()
    elif args.workload == "decode_heavy":
        pool, (step,) = workloads.decode_heavy(seed=workloads.SEED_BASE + 2 + 1000 * rank)
    else:  # the 8 prefill chunks of the mixed step alone
        pool, (step,) = workloads.mixed_step(seed=workloads.SEED_BASE + 3 + 1000 * rank,
                                             num_decode=0, num_spec=0)
    log(f"[bench] mixed step generated in {time.time() - t0:.1f}s: "
        f"{step.num_seqs} requests, {step.num_q_tokens} tokens, {pool.num_blocks} blocks")
    fp8 = args.kv_dtype == "fp8"
    ds = DeviceStep(pool, step, dev, fp8=fp8)
    stream = torch.cuda.current_stream()
    short_reqs = split_rows(step)
    long_reqs = [b for b in range(step.num_seqs) if b not in set(short_reqs)]
    short_bytes = algorithmic_bytes(step, short_reqs, kv_elem_bytes=1 if fp8 else 2)
    long_flops = tensor_core_flops(step, long_reqs)

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    # warm-up: at least W steps, and at least ~0.5 s of load so the clock
    # samples cover a busy GPU
    ds.run()
    torch.cuda.synchronize()
    t_w = time.time()
    n_w = 0
    while n_w < args.warmup or time.time() - t_w < args.min_warmup_s:
        ds.run()
        n_w += 1
        if n_w % 20 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()

    # timed region: exactly K plain steps.  Each kernel is launched as a
    # programmatic dependent of the one before it (its launch and prologue
    # overlap the previous kernel's tail); an event between two kernels would
    # break that overlap, so the per-kernel times come from a second pass.
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = pk.kernel_launches()
    ms = time_steps(ds.run, args.steps, stream)
    torch.cuda.synchronize()
    # the library's own count of the kernels it enqueued in the timed region
    gpu_launches = pk.kernel_launches() - launches0
    ms = max_over_ranks(ms, dev)
    job_tokens = all_ranks_sum(step.num_q_tokens, dev)
    clocks = sampler.stop() if sampler else None

    # kernel pass: the same K steps with CUDA events around each launch of
    # the two attention kernels, recorded on the launching stream
    ev = {w: make_events(args.steps) for w in (pk.PA_KERNEL_SPLIT_KV, pk.PA_KERNEL_TENSOR_CORE)}
    it = [0]

    def profiled_step():
        i = it[0]
        for w, pairs in ev.items():
            pk.set_profile_events(w, *pairs[i])
        ds.run()
        it[0] += 1

    torch.cuda.synchronize()
    ms_profiled = time_steps(profiled_step, args.steps, stream)
    torch.cuda.synchronize()
    for w in ev:
        pk.set_profile_events(w, None, None)
    status = pk.read_device_status(clear=True)
    if status:
        log(f"[bench] WARNING device status {status:#x}")

    ms_step = ms / args.steps
    value = job_tokens * args.steps / (ms / 1000.0)
    short_ms = statistics.mean(a.elapsed_time(b) for a, b in ev[pk.PA_KERNEL_SPLIT_KV])
    long_ms = statistics.mean(a.elapsed_time(b) for a, b in ev[pk.PA_KERNEL_TENSOR_CORE])
    achieved = short_bytes / (short_ms / 1000.0) / 1e9 if short_bytes else 0.0
    # the committed DRAM record is the bf16 variant's
    tr = None if fp8 else traffic_for("split_kv_mixed_step")
    split_kv = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak,
                "traffic": tr["dram_bytes_per_algorithmic_byte"] * short_bytes if tr else None,
                "kernel": "split-KV decode/short-q kernel (pa_short.cu)",
                "kernel_ms": short_ms, "algorithmic_bytes": short_bytes,
                "timing": KERNEL_TIMING,
                "peak_source": f"{peak_src} hbm_gbs (copy)"}
    tflops = long_flops / (long_ms / 1000.0) / 1e12 if long_flops else 0.0
    tr = traffic_for("tensor_core_mixed_step")
    tensor_core = {"bound": "tensor", "achieved": tflops, "peak": tc_peak, "unit": "TFLOP/s",
                   "frac": tflops / tc_peak,
                   "traffic": tr["dram_bytes_per_flop"] * long_flops if tr else None,
                   "kernel": "tcgen05 prefill kernel (pa_long.cu)",
                   "kernel_ms": long_ms, "flops": long_flops,
                   "timing": KERNEL_TIMING,
                   "peak_source": f"{peak_src} bf16_tflops (burst)"}
    # the roofline object describes the kernel with the larger share of the step
    roofline = split_kv if short_ms >= long_ms else tensor_core

    # ---- e2e through the public API with host buffers ----------------------
    # Every step copies its inputs from pinned host memory and its result
    # (out, lse) back, as a serving loop does; the copies run on a second
    # stream, double-buffered, so step i+1's inputs go up and step i's result
    # comes down while step i computes.  The timed region spans all K steps
    # from the first upload to the last download.
    e2e = None
    if not args.no_e2e:
        host = {name: t.cpu().pin_memory() for name, t in
                (("q", step.q), ("k", step.k), ("v", step.v), ("slots", step.slot_mapping),
                 ("bt", step.block_tables), ("qsl", step.query_start_loc),
                 ("ctx", step.context_lens), ("sl", step.seq_lens))}
        out_h = torch.empty(ds.out.shape, dtype=ds.out.dtype).pin_memory()
        lse_h = torch.empty(ds.lse.shape, dtype=ds.lse.dtype).pin_memory()
        dbuf = [{name: torch.empty_like(t, device=dev) for name, t in host.items()}
                for _ in range(2)]
        outs = [(torch.empty_like(ds.out), torch.empty_like(ds.lse)) for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()
        copy_stream = torch.cuda.Stream()
        in_ready = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]

        def upload(b):
            with torch.cuda.stream(copy_stream):
                for name, t in host.items():
                    dbuf[b][name].copy_(t, non_blocking=True)
                in_ready[b].record(copy_stream)

        def e2e_steps(n):
            copy_stream.wait_stream(stream)
            upload(0)
            for i in range(n):
                b = i & 1
                stream.wait_event(in_ready[b])
                d, (o, l) = dbuf[b], outs[b]
                pk.pa_write_kv_attention(d["k"], d["v"], d["slots"], d["q"], ds.kc, ds.vc,
                                         d["bt"], d["qsl"], d["ctx"], d["sl"], step.scale, o,
                                         l, workspace=ds.ws, **ds.scales)
                done[b].record(stream)
                with torch.cuda.stream(copy_stream):
                    if i + 1 < n:
                        # buffer 1-b was last read by step i-1
                        if i >= 1:
                            copy_stream.wait_event(done[1 - b])
                        upload(1 - b)
                    copy_stream.wait_event(done[b])
                    out_h.copy_(o, non_blocking=True)
                    lse_h.copy_(l, non_blocking=True)
            stream.wait_stream(copy_stream)

        e2e_steps(max(3, args.warmup))
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        e2e_steps(args.steps)
        end.record(stream)
        end.synchronize()
        e_ms = max_over_ranks(start.elapsed_time(end), dev)
        e2e = {"value": job_tokens * args.steps / (e_ms / 1000.0),
               "unit": "query tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e_ms / args.steps,
               "copies": "pinned host buffers; uploads and downloads on a second stream, "
                         "double-buffered, overlapping the neighbouring steps' compute"}

    # ---- secondary: decode-heavy KV GB/s and cascade --------------------------
    decode = cascade = graph = fp8_res = None
    del ds
    torch.cuda.empty_cache()
    if not args.no_secondary:
        decode = bench_decode_heavy(args, dev, hbm_peak)
        cascade = bench_cascade(args, dev)
        graph = bench_graph_decode(args, dev)
        fp8_res = bench_fp8(args, dev, hbm_peak)

    # ---- CPU baseline (rank 0 only) -----------------------------------------
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle
        oracle.build_oracle()
        sub = oracle_sample(pool, step)
        t_cpu = time_oracle(pool, sub)
        cpu = {"value": sub.num_q_tokens / t_cpu, "unit": "query tokens/s",
               "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"1/8 of the mixed step ({sub.num_seqs} requests, "
                         f"{sub.num_q_tokens} query tokens: every 8th chunk, decode and spec "
                         f"request), fp64 oracle write_kv + attention, {t_cpu:.2f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "query tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3 KV, f16 MMA" if fp8 else "bf16",
            "data": "synthetic",
            "config": headline_config(args, world, step, pool, global_reqs),
            "roofline": roofline,
            "kernels": {"split_kv": split_kv, "tensor_core": tensor_core},
            "decode_heavy": decode,
            "cascade": cascade,
            "graph_decode": graph,
            "fp8_kv": fp8_res,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "clocks": clocks,
            "gpu_launches": gpu_launches,
            "device_status": status,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def bench_decode_heavy(args, dev, hbm_peak):
    import paged_kv_cache_284_gb300 as pk
    from paged_kv_cache_284_gb300 import workloads
    pool, (step,) = workloads.decode_heavy()
    ds = DeviceStep(pool, step, dev)
    ds.run()
    for _ in range(max(3, args.warmup)):
        ds.run(write=False)
    torch.cuda.synchronize()
    # plain pass for the attention call, then a pass with kernel events
    ms = time_steps(lambda: ds.run(write=False), args.steps,
                    torch.cuda.current_stream()) / args.steps
    s_ev = make_events(args.steps)
    it = [0]

    def one():
        pk.set_profile_events(pk.PA_KERNEL_SPLIT_KV, *s_ev[it[0]])
        ds.run(write=False)
        it[0] += 1

    time_steps(one, args.steps, torch.cuda.current_stream())
    pk.set_profile_events(pk.PA_KERNEL_SPLIT_KV, None, None)
    k_ms = statistics.mean(a.elapsed_time(b) for a, b in s_ev)
    reqs = range(step.num_seqs)
    kvb = kv_bytes(step, reqs)
    alg = algorithmic_bytes(step, reqs)
    res = {"workload": "256 decode rows, seq_len U[512,4096], 32 q / 8 kv heads, d=128, bs=16",
           "kv_bytes": kvb, "attention_ms": ms, "kv_gbs": kvb / (ms / 1000) / 1e9,
           "kv_frac_of_hbm": kvb / (ms / 1000) / 1e9 / hbm_peak,
           "split_kv_kernel_ms": k_ms,
           "split_kv_kernel_gbs": alg / (k_ms / 1000) / 1e9,
           "split_kv_kernel_frac": alg / (k_ms / 1000) / 1e9 / hbm_peak}
    del ds
    torch.cuda.empty_cache()
    return res


def bench_graph_decode(args, dev):
    """Small decode steps (write + attention) launched one by one versus
    replayed from one captured CUDA graph: the launch overhead the on-device
    plan lets a serving loop remove."""
    from paged_kv_cache_284_gb300 import workloads
    res = {"workload": "decode rows, seq_len U[512,4096], 32 q / 8 kv heads, d=128, bs=16; "
                       "one pa_write_kv_attention call (cache write + attention) per step, "
                       "back to back"}
    for b in (8, 64):
        pool, (step,) = workloads.decode_heavy(seed=workloads.SEED_BASE + 50 + b, num_seqs=b)
        ds = DeviceStep(pool, step, dev)
        stream = torch.cuda.current_stream()
        for _ in range(max(3, args.warmup)):
            ds.run()
        torch.cuda.synchronize()
        n = max(args.steps, 50)
        eager = time_steps(ds.run, n, stream) / n
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            ds.run()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            ds.run()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        graph = time_steps(g.replay, n, stream) / n
        res[f"batch_{b}"] = {"eager_ms": eager, "graph_ms": graph, "speedup": eager / graph}
        del g, ds
    torch.cuda.empty_cache()
    return res


def bench_fp8(args, dev, hbm_peak):
    """The decode-heavy and mixed steps on an e4m3 KV pool (same metadata and
    new tokens, codes drawn by the workload generator, per-kv-head scales):
    half the KV bytes of bf16."""
    import paged_kv_cache_284_gb300 as pk
    from paged_kv_cache_284_gb300 import workloads
    res = {"kv_dtype": "e4m3 (per-kv-head fp32 scales)"}
    for name, fn in (("decode_heavy", workloads.decode_heavy),
                     ("mixed_step", workloads.mixed_step)):
        pool, (step,) = fn()
        pool8 = workloads.fp8_pool_like(pool, workloads.SEED_BASE + 80)
        del pool
        kc, vc = pool8.k_cache.to(dev), pool8.v_cache.to(dev)
        ks, vs = pool8.k_scale.to(dev), pool8.v_scale.to(dev)
        del pool8
        q, k, v = step.q.to(dev), step.k.to(dev), step.v.to(dev)
        slots = step.slot_mapping.to(dev)
        meta = dict(block_tables=step.block_tables.to(dev),
                    query_start_loc=step.query_start_loc.to(dev),
                    context_lens=step.context_lens.to(dev), seq_lens=step.seq_lens.to(dev))
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
        T, hq, d = q.shape
        ws = pk.alloc_workspace(pk.workspace_size(step.num_seqs, T, hq, step.num_kv_heads, d)
                                + pk.fp8_staging_bytes(step.num_kv_heads, d, step.block_size,
                                                       staging_blocks(step)), dev)

        def one(write=True):
            if write:
                pk.pa_write_kv_attention(k, v, slots, q, kc, vc, meta["block_tables"],
                                         meta["query_start_loc"], meta["context_lens"],
                                         meta["seq_lens"], step.scale, out, lse, workspace=ws,
                                         k_scale=ks, v_scale=vs)
                return
            pk.pa_attention(q, kc, vc, scale=step.scale, out=out, lse=lse, workspace=ws,
                            k_scale=ks, v_scale=vs, **meta)

        for _ in range(max(3, args.warmup)):
            one()
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream()
        ms = time_steps(one, args.steps, stream) / args.steps
        s_ev = make_events(args.steps)
        it = [0]

        def prof():
            pk.set_profile_events(pk.PA_KERNEL_SPLIT_KV, *s_ev[it[0]])
            one()
            it[0] += 1

        time_steps(prof, args.steps, stream)
        pk.set_profile_events(pk.PA_KERNEL_SPLIT_KV, None, None)
        k_ms = statistics.mean(a.elapsed_time(b) for a, b in s_ev)
        reqs = range(step.num_seqs)
        # long requests run on the tensor-core kernel over their staged copy
        alg = algorithmic_bytes(step, split_rows(step), kv_elem_bytes=1)
        entry = {"step_ms": ms, "query_tokens_per_s": T / (ms / 1000),
                 "kv_bytes": kv_bytes(step, reqs, 1), "split_kv_kernel_ms": k_ms,
                 "split_kv_kernel_gbs": alg / (k_ms / 1000) / 1e9,
                 "split_kv_kernel_frac": alg / (k_ms / 1000) / 1e9 / hbm_peak}
        res[name] = entry
        del kc, vc, ws
        torch.cuda.empty_cache()
    return res


def bench_cascade(args, dev, compare_full=True, parts=False):
    import paged_kv_cache_284_gb300 as pk
    from paged_kv_cache_284_gb300 import workloads
    pool, (step,) = workloads.cascade()
    ds = DeviceStep(pool, step, dev)
    ds.run()
    pb = step.prefix_blocks.to(dev)
    sbt = step.suffix_block_tables.to(dev)
    sctx = step.suffix_context_lens.to(dev)
    ssl = step.suffix_seq_lens.to(dev)
    out = torch.empty_like(ds.q)
    lse = torch.empty_like(ds.lse)
    ws = pk.alloc_workspace(pk.cascade_workspace_size(step.num_seqs, step.num_q_tokens,
                                                      step.num_q_heads, step.num_kv_heads,
                                                      step.head_dim, step.prefix_len), dev)

    def casc():
        pk.pa_cascade_decode(ds.q, ds.kc, ds.vc, pb, step.prefix_len, sbt, ds.qsl, sctx, ssl,
                             step.scale, out, lse, workspace=ws)

    for _ in range(max(3, args.warmup)):
        casc()
    torch.cuda.synchronize()
    ms_c = time_steps(casc, args.steps, torch.cuda.current_stream()) / args.steps
    ms_p = None
    if compare_full:
        for _ in range(max(3, args.warmup)):
            ds.run(write=False)
        torch.cuda.synchronize()
        ms_p = time_steps(lambda: ds.run(write=False), args.steps,
                          torch.cuda.current_stream()) / args.steps
    if parts:
        # the two passes on their own: the shared-prefix pass (bf16 output)
        # and paged attention over the suffix tables alone
        def prefix_only():
            pk.pa_prefix_attention(ds.q, ds.kc, ds.vc, pb, step.prefix_len, step.scale, out,
                                   lse, workspace=ws)

        def suffix_only():
            pk.pa_attention(ds.q, ds.kc, ds.vc, sbt, ds.qsl, sctx, ssl, step.scale, out, lse,
                            workspace=ws)

        part_ms = {}
        for name, fn in (("prefix_pass_ms", prefix_only), ("suffix_pass_ms", suffix_only)):
            for _ in range(max(3, args.warmup)):
                fn()
            torch.cuda.synchronize()
            part_ms[name] = time_steps(fn, args.steps, torch.cuda.current_stream()) / args.steps
    uniq = sum(int(s) for s in step.suffix_seq_lens) * step.num_kv_heads * step.head_dim * 4
    pref = step.prefix_len * step.num_kv_heads * step.head_dim * 4
    res = {"workload": "64 requests sharing an 8192-token prefix, suffix U[128,1024], q_len 1",
           "cascade_ms": ms_c, "paged_attention_ms": ms_p,
           "speedup": ms_p / ms_c if ms_p else None,
           "cascade_algorithmic_kv_bytes": uniq + pref,
           "cascade_kv_gbs": (uniq + pref) / (ms_c / 1000) / 1e9}
    if parts:
        res.update(part_ms)
    del ds
    torch.cuda.empty_cache()
    return res


def run_cascade_only(args):
    """Profiling case: the cascade decode call alone (no write, no full-table
    comparison), W warm-up calls then K timed calls; one JSON line."""
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    res = bench_cascade(args, dev, compare_full=False, parts=True)
    print(json.dumps({"workload": "cascade", **res}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--kv-dtype", choices=["bf16", "fp8"], default="bf16",
                    help="KV pool element type of the headline step (fp8 = e4m3 + scales)")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--workload", choices=["mixed_step", "decode_heavy", "prefill", "cascade"],
                    default="mixed_step",
                    help="headline workload (mixed_step is the benchmark; the others are "
                         "single-kernel cases for profiling)")
    ap.add_argument("--min-warmup-s", type=float, default=0.5,
                    help="keep warming up at least this long (clock samples need a busy GPU)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "cascade":
        run_cascade_only(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
