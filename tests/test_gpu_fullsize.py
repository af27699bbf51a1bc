"""Parity at the benchmark sizes, in the launch configuration bench.py times
(pa_write_kv, then pa_attention with default dispatch and automatic split
size; pa_cascade_decode for the shared-prefix step).

The oracle cannot redo a whole full-size step in test time, so it checks
sampled requests one by one (every kind of row: decode, speculative verify,
chunked-prefill chunk), and every row of the batch is checked for properties
that hold at any size: finite, and each output inside the range of the value
vectors it averages.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_284_gb300 as pk
from paged_kv_cache_284_gb300 import workloads
from gpu_helpers import (DEV, assert_attention_close, assert_status_clean, bits, gpu_attend,
                         gpu_write)

pytestmark = pytest.mark.gpu


def run_full(pool, step):
    kc, vc = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    gpu_write(step, kc, vc)
    out, lse = gpu_attend(step, kc, vc)
    torch.cuda.synchronize()
    return kc, vc, out, lse


def sample_requests(step, per_kind, seed):
    """Up to per_kind[n] requests of each q_len n (first, last, then random)."""
    rng = np.random.default_rng(seed)
    kinds = {}
    for b, n in enumerate(step.q_lens.tolist()):
        kinds.setdefault(n, []).append(b)
    picked = []
    for n, reqs in sorted(kinds.items()):
        k = per_kind.get(n, per_kind.get("default", 2))
        chosen = {reqs[0], reqs[-1]}
        rest = [b for b in reqs if b not in chosen]
        chosen.update(rng.choice(rest, size=min(len(rest), max(0, k - 2)), replace=False).tolist()
                      if rest else [])
        picked += sorted(chosen)[:max(k, 1)]
    return sorted(set(picked))


def check_sampled(pool, step, out, lse, idx, what):
    sub = workloads.subset(step, idx)
    kb, vb = oracle.write_kv(step.k, step.v, step.slot_mapping, pool.k_cache, pool.v_cache)
    ref_o, ref_l = oracle.attention(sub.q, kb, vb, sub.block_tables, sub.query_start_loc,
                                    sub.context_lens, sub.seq_lens, sub.scale)
    qsl = step.query_start_loc
    rows = torch.cat([torch.arange(int(qsl[b]), int(qsl[b + 1])) for b in idx])
    assert_attention_close(out[rows.to(DEV)], lse[rows.to(DEV)], ref_o, ref_l, what)


def check_whole_batch(out, lse, vc):
    o = out.float()
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    vmax = vc.float().abs().max()
    assert o.abs().max() <= vmax * (1 + 2 ** -7)


def test_decode_heavy_full_size():
    pool, (step,) = workloads.decode_heavy()
    kc, vc, out, lse = run_full(pool, step)
    check_whole_batch(out, lse, vc)
    idx = sample_requests(step, {1: 12}, seed=1)
    check_sampled(pool, step, out, lse, idx, "decode_heavy")
    assert_status_clean()


def test_mixed_step_full_size():
    pool, (step,) = workloads.mixed_step()
    kc, vc, out, lse = run_full(pool, step)
    check_whole_batch(out, lse, vc)
    # decode rows, speculative-verify rows (q_len 5) and two 512-token chunks
    idx = sample_requests(step, {1: 8, 5: 4, 512: 2}, seed=2)
    check_sampled(pool, step, out, lse, idx, "mixed_step")
    assert_status_clean()


def test_cascade_full_size():
    pool, (step,) = workloads.cascade()
    kc, vc = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    gpu_write(step, kc, vc)
    q = step.q.to(DEV)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=DEV)
    pk.pa_cascade_decode(q, kc, vc, step.prefix_blocks.to(DEV), step.prefix_len,
                         step.suffix_block_tables.to(DEV), step.query_start_loc.to(DEV),
                         step.suffix_context_lens.to(DEV), step.suffix_seq_lens.to(DEV),
                         step.scale, out, lse)
    torch.cuda.synchronize()
    check_whole_batch(out, lse, vc)
    # against the oracle over the full tables (prefix blocks + suffix blocks)
    idx = sample_requests(step, {1: 10}, seed=3)
    check_sampled(pool, step, out, lse, idx, "cascade")
    # and the plain paged attention over the full tables agrees too
    o2, l2 = gpu_attend(step, kc, vc)
    torch.cuda.synchronize()
    err = (o2.float() - out.float()).abs()
    assert err.max().item() <= 2e-2 and err.mean().item() <= 2e-3
    assert (l2 - lse).abs().max().item() <= 1e-3
    assert_status_clean()
