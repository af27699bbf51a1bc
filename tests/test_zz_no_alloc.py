"""The allocation-free entry point, pa_attention_no_alloc.

It exists for callers that cannot allocate device memory when they run a
step (a fixed device-memory arena, a shutdown or memory-pressure path, a
plugin that must not create buffers): the library keeps the step's scratch
in one fixed device array of its own.  This file checks, through the C ABI,
that two calls in a row on different batches give the same attention as
pa_attention with a caller-allocated workspace (same tolerance as the
parity tests), that a repeated batch still agrees after another batch has
left its contents in the shared array, and that a step too large for the
array is refused cleanly.  pytest collects it last; it also passes alone.
"""
import ctypes
import os
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import paged_kv_cache_284_gb300 as pk  # noqa: E402
from paged_kv_cache_284_gb300 import workloads  # noqa: E402

pytestmark = pytest.mark.gpu

OUT_MAX_ABS, OUT_MEAN_ABS, LSE_MAX_ABS = 2e-2, 2e-3, 1e-3


def on_device(pool, step, dev):
    t = {name: getattr(step, name).to(dev) for name in
         ("q", "k", "v", "slot_mapping", "block_tables", "query_start_loc", "context_lens",
          "seq_lens")}
    kc, vc = pool.k_cache.to(dev), pool.v_cache.to(dev)
    pk.pa_write_kv(t["k"], t["v"], t["slot_mapping"], kc, vc)
    return t, kc, vc


def with_workspace(t, kc, vc, scale):
    out = torch.empty_like(t["q"])
    lse = torch.empty(t["q"].shape[:2], dtype=torch.float32, device=t["q"].device)
    pk.pa_attention(t["q"], kc, vc, t["block_tables"], t["query_start_loc"], t["context_lens"],
                    t["seq_lens"], scale, out, lse)
    return out, lse


def no_alloc(t, kc, vc, scale):
    """Straight through the C ABI: no workspace argument at all."""
    out = torch.empty_like(t["q"])
    lse = torch.empty(t["q"].shape[:2], dtype=torch.float32, device=t["q"].device)
    kv = pk.kv_desc(kc, vc)
    T, hq, _ = t["q"].shape
    rc = pk.lib().pa_attention_no_alloc(
        ctypes.c_void_p(t["q"].data_ptr()), ctypes.byref(kv),
        ctypes.c_void_p(t["block_tables"].data_ptr()), int(t["block_tables"].shape[1]),
        ctypes.c_void_p(t["query_start_loc"].data_ptr()),
        ctypes.c_void_p(t["context_lens"].data_ptr()), ctypes.c_void_p(t["seq_lens"].data_ptr()),
        int(t["seq_lens"].shape[0]), T, hq, float(scale), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(lse.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == pk.PA_OK, pk.lib().pa_last_error_message()
    return out, lse


def assert_same(a, b, what):
    (oa, la), (ob, lb) = a, b
    err = (oa.float() - ob.float()).abs()
    lerr = (la - lb).abs()
    assert torch.isfinite(ob.float()).all(), what
    assert err.max().item() <= OUT_MAX_ABS, (what, err.max().item())
    assert err.mean().item() <= OUT_MEAN_ABS, (what, err.mean().item())
    assert lerr.max().item() <= LSE_MAX_ABS, (what, lerr.max().item())


def test_no_alloc_matches_pa_attention_on_two_calls_in_a_row():
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    pool_a, (step_a,) = workloads.decode_heavy(seed=41, num_seqs=48, lo=1, hi=3000)
    pool_b, (step_b,) = workloads.mixed_step(seed=42, num_chunks=2, chunk_len=200,
                                             chunk_ctx=(0, 600), num_decode=12,
                                             decode_len=(1, 2000), num_spec=4,
                                             spec_ctx=(0, 900))
    ta, kca, vca = on_device(pool_a, step_a, dev)
    tb, kcb, vcb = on_device(pool_b, step_b, dev)
    ref_a = with_workspace(ta, kca, vca, step_a.scale)
    ref_b = with_workspace(tb, kcb, vcb, step_b.scale)
    got_a = no_alloc(ta, kca, vca, step_a.scale)      # first call
    got_b = no_alloc(tb, kcb, vcb, step_b.scale)      # second call, other batch
    got_a2 = no_alloc(ta, kca, vca, step_a.scale)     # after B's contents in the scratch
    torch.cuda.synchronize()
    assert_same(ref_a, got_a, "decode batch, first call")
    assert_same(ref_b, got_b, "mixed batch, second call")
    assert_same(ref_a, got_a2, "decode batch again")
    assert pk.read_device_status(clear=True) == 0


def test_no_alloc_refuses_a_step_too_large_for_its_scratch():
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    pool, (step,) = workloads.decode_heavy(seed=43, num_seqs=4, lo=20, hi=40)
    t, kc, vc = on_device(pool, step, dev)
    # a batch claiming 1.5 million sequences needs more work-list room than the
    # fixed scratch has; the call must refuse before launching anything
    huge = 1_500_000
    kv = pk.kv_desc(kc, vc)
    out = torch.empty_like(t["q"])
    rc = pk.lib().pa_attention_no_alloc(
        ctypes.c_void_p(t["q"].data_ptr()), ctypes.byref(kv),
        ctypes.c_void_p(t["block_tables"].data_ptr()), int(t["block_tables"].shape[1]),
        ctypes.c_void_p(t["query_start_loc"].data_ptr()),
        ctypes.c_void_p(t["context_lens"].data_ptr()), ctypes.c_void_p(t["seq_lens"].data_ptr()),
        huge, int(t["q"].shape[0]), int(t["q"].shape[1]), float(step.scale),
        ctypes.c_void_p(out.data_ptr()), None, None)
    assert rc == pk.PA_ERR_WORKSPACE
    assert b"fixed scratch" in pk.lib().pa_last_error_message()
