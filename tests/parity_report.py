"""Parity and timing report for the five workload configurations (run on a GPU
machine: `python tests/parity_report.py`; prints a markdown table).

For each configuration the GPU path (pa_write_kv, then pa_attention -- or
pa_cascade_decode for the shared-prefix step) runs on the seeded inputs, the
fp64 oracle runs on the same inputs over every row, and the report gives the
cache comparison (bit for bit), the output's max / mean absolute error, the
lse's max absolute error, the GPU step time (CUDA events, warm, inputs
resident) and the oracle's wall time on this machine's host cores.
"""
from __future__ import annotations

import os
import statistics
import sys
import time

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

import oracle  # noqa: E402
import paged_kv_cache_284_gb300 as pk  # noqa: E402
from paged_kv_cache_284_gb300 import workloads  # noqa: E402

DEV = torch.device("cuda:0")


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def gpu_time(fn, n=20):
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    for a, b in evs:
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs)


def report(name, pool, steps, cascade=False):
    kc, vc = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    kb, vb = bits(pool.k_cache), bits(pool.v_cache)
    errs, cache_ok, t_gpu, t_cpu, kv_bytes, toks = [], True, 0.0, 0.0, 0, 0
    for step in steps:
        d = {n: getattr(step, n).to(DEV) for n in
             ("q", "k", "v", "slot_mapping", "block_tables", "query_start_loc",
              "context_lens", "seq_lens")}
        out = torch.empty_like(d["q"])
        lse = torch.empty(d["q"].shape[:2], dtype=torch.float32, device=DEV)
        if cascade:
            pb, sbt = step.prefix_blocks.to(DEV), step.suffix_block_tables.to(DEV)
            sctx, ssl = step.suffix_context_lens.to(DEV), step.suffix_seq_lens.to(DEV)

            def attend():
                pk.pa_cascade_decode(d["q"], kc, vc, pb, step.prefix_len, sbt,
                                     d["query_start_loc"], sctx, ssl, step.scale, out, lse)
        else:
            ws = pk.alloc_workspace(pk.workspace_size(step.num_seqs, step.num_q_tokens,
                                                      step.num_q_heads, step.num_kv_heads,
                                                      step.head_dim), DEV)

            def attend():
                pk.pa_attention(d["q"], kc, vc, d["block_tables"], d["query_start_loc"],
                                d["context_lens"], d["seq_lens"], step.scale, out, lse,
                                workspace=ws)

        def one():
            pk.pa_write_kv(d["k"], d["v"], d["slot_mapping"], kc, vc)
            attend()

        t_gpu += gpu_time(one)
        t0 = time.time()
        kb, vb = oracle.write_kv(step.k, step.v, step.slot_mapping, kb, vb)
        ro, rl = oracle.attention(step.q, kb, vb, step.block_tables, step.query_start_loc,
                                  step.context_lens, step.seq_lens, step.scale)
        t_cpu += time.time() - t0
        cache_ok &= np.array_equal(bits(kc), kb) and np.array_equal(bits(vc), vb)
        o = out.float().cpu().numpy().astype(np.float64)
        e = np.abs(o - ro)
        errs.append((e.max(), e.mean(), np.abs(lse.cpu().numpy() - rl).max()))
        kv_bytes += sum(2 * int(L) * step.num_kv_heads * step.head_dim * 2
                        for L in step.seq_lens)
        toks += step.num_q_tokens
    mx = max(x[0] for x in errs)
    mean = max(x[1] for x in errs)
    ml = max(x[2] for x in errs)
    st = pk.read_device_status(clear=True)
    print(f"| {name} | {'bit-exact' if cache_ok else 'DIFFERS'} | {mx:.2e} / {mean:.2e} / "
          f"{ml:.2e} | {t_gpu * 1000:.1f} | {kv_bytes / (t_gpu / 1000) / 1e9:.0f} | "
          f"{toks / (t_gpu / 1000):.3g} | {t_cpu:.2f} | {toks / t_cpu:.3g} | {st:#x} |",
          flush=True)


def main():
    print(f"host cores: {os.cpu_count()}; GPU: {torch.cuda.get_device_name(0)}")
    print("| config | cache | out max / mean abs err, lse max abs err | GPU step (us) | "
          "KV GB/s | GPU query tok/s | oracle (s) | oracle query tok/s | device status |")
    print("|---|---|---|---|---|---|---|---|---|")
    pool, steps = workloads.tiny_prefill()
    report("1 tiny prefill", pool, steps)
    pool, steps = workloads.chunked_prefix_decode()
    report("2 chunked + prefix hit + decode (3 steps)", pool, steps)
    pool, steps = workloads.decode_heavy()
    report("3 decode-heavy", pool, steps)
    pool, steps = workloads.mixed_step()
    report("4 mixed step", pool, steps)
    pool, steps = workloads.cascade()
    report("5 cascade (pa_cascade_decode)", pool, steps, cascade=True)


if __name__ == "__main__":
    main()
