"""Parity at the benchmark sizes, in the launch configuration bench.py times
(pa_write_kv, then pa_attention with default dispatch and automatic split
size; pa_cascade_decode for the shared-prefix step).

Every row of every request is compared with the fp64 oracle element by
element (the oracle covers a whole full-size step in seconds on the host's
cores), the whole K and V caches bit for bit, and every row is also checked
for properties that hold at any size: finite, and each output inside the
range of the value vectors it averages.
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


def check_every_row(pool, step, kc, vc, out, lse, what):
    """The oracle over the whole step (full block tables), every row, and the
    caches after the write, bit for bit."""
    kb, vb = oracle.write_kv(step.k, step.v, step.slot_mapping, pool.k_cache, pool.v_cache)
    assert np.array_equal(bits(kc), kb), f"{what}: K cache differs"
    assert np.array_equal(bits(vc), vb), f"{what}: V cache differs"
    ref_o, ref_l = oracle.attention(step.q, kb, vb, step.block_tables, step.query_start_loc,
                                    step.context_lens, step.seq_lens, step.scale)
    return assert_attention_close(out, lse, ref_o, ref_l, what)


def check_whole_batch(out, lse, vc):
    o = out.float()
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    vmax = vc.float().abs().max()
    assert o.abs().max() <= vmax * (1 + 2 ** -7)


def test_decode_heavy_full_size():
    """256 decode rows: all 256 x 32 rows against the oracle."""
    pool, (step,) = workloads.decode_heavy()
    kc, vc, out, lse = run_full(pool, step)
    check_whole_batch(out, lse, vc)
    check_every_row(pool, step, kc, vc, out, lse, "decode_heavy")
    assert_status_clean()


def test_mixed_step_full_size():
    """The benchmark step: all 4448 query tokens x 32 heads against the
    oracle (decode rows, speculative-verify rows, 512-token chunks)."""
    pool, (step,) = workloads.mixed_step()
    kc, vc, out, lse = run_full(pool, step)
    check_whole_batch(out, lse, vc)
    check_every_row(pool, step, kc, vc, out, lse, "mixed_step")
    assert_status_clean()


def test_cascade_full_size():
    """64 requests sharing an 8192-token prefix: every row of the cascade call
    against the oracle over the full tables (prefix blocks + suffix blocks),
    and the plain paged attention over the full tables agrees too."""
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
    check_every_row(pool, step, kc, vc, out, lse, "cascade")
    o2, l2 = gpu_attend(step, kc, vc)
    torch.cuda.synchronize()
    err = (o2.float() - out.float()).abs()
    assert err.max().item() <= 2e-2 and err.mean().item() <= 2e-3
    assert (l2 - lse).abs().max().item() <= 1e-3
    assert_status_clean()
