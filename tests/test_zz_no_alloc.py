"""The allocation-free entry point, pa_attention_no_alloc.

It exists for callers that cannot allocate device memory when they run a
step (a fixed device-memory arena, a shutdown or memory-pressure path, a
plugin that must not create buffers): the library keeps the step's scratch
in one fixed device array of its own.  This file checks, through the C ABI,
that two calls in a row on different batches give the same attention as
pa_attention with a caller-allocated workspace (same tolerance as the
parity tests), that a repeated batch still agrees after another batch has
left its contents in the shared array, that an e4m3 pool (whose long
requests run as split-KV pieces here) agrees too, and that a step too large
for the array is refused cleanly.  pytest collects it last; it also passes alone.
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


def on_device(pool, step, dev, scales=None):
    t = {name: getattr(step, name).to(dev) for name in
         ("q", "k", "v", "slot_mapping", "block_tables", "query_start_loc", "context_lens",
          "seq_lens")}
    kc, vc = pool.k_cache.to(dev), pool.v_cache.to(dev)
    pk.pa_write_kv(t["k"], t["v"], t["slot_mapping"], kc, vc, **(scales or {}))
    return t, kc, vc


def with_workspace(t, kc, vc, scale, scales=None, staging_blocks=0):
    """pa_attention with a caller-allocated workspace (on an e4m3 pool with
    room to stage the long requests for the tensor-core kernel)."""
    out = torch.empty_like(t["q"])
    lse = torch.empty(t["q"].shape[:2], dtype=torch.float32, device=t["q"].device)
    T, hq, d = t["q"].shape
    hkv, bs = kc.shape[1], kc.shape[2]
    ws = pk.alloc_workspace(pk.workspace_size(t["seq_lens"].shape[0], T, hq, hkv, d)
                            + (pk.fp8_staging_bytes(hkv, d, bs, staging_blocks)
                               if staging_blocks else 0), t["q"].device)
    pk.pa_attention(t["q"], kc, vc, t["block_tables"], t["query_start_loc"], t["context_lens"],
                    t["seq_lens"], scale, out, lse, workspace=ws, **(scales or {}))
    return out, lse


def no_alloc(t, kc, vc, scale, scales=None):
    """Straight through the C ABI: no workspace argument at all."""
    out = torch.empty_like(t["q"])
    lse = torch.empty(t["q"].shape[:2], dtype=torch.float32, device=t["q"].device)
    kv = pk.kv_desc(kc, vc, **(scales or {}))
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


def test_no_alloc_on_an_e4m3_pool_matches_pa_attention():
    """On an fp8 pool the fixed scratch has no staging room, so the long
    requests run as split-KV pieces; pa_attention with a staging workspace
    runs them on the tensor-core kernel.  Both must agree."""
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    pool, (step,) = workloads.mixed_step(seed=44, num_chunks=2, chunk_len=200,
                                         chunk_ctx=(0, 600), num_decode=12,
                                         decode_len=(1, 2000), num_spec=4, spec_ctx=(0, 900))
    pool8 = workloads.fp8_pool_like(pool, seed=45)
    scales = {"k_scale": pool8.k_scale.to(dev), "v_scale": pool8.v_scale.to(dev)}
    t, kc, vc = on_device(pool8, step, dev, scales)
    group = step.num_q_heads // step.num_kv_heads
    stage = sum(-(-int(L) // step.block_size) for L, n in
                zip(step.seq_lens.tolist(), step.q_lens.tolist()) if n * group > 64)
    ref = with_workspace(t, kc, vc, step.scale, scales, staging_blocks=stage)
    got = no_alloc(t, kc, vc, step.scale, scales)
    got2 = no_alloc(t, kc, vc, step.scale, scales)
    torch.cuda.synchronize()
    assert_same(ref, got, "e4m3 mixed batch, first call")
    assert_same(ref, got2, "e4m3 mixed batch, second call")
    assert pk.read_device_status(clear=True) == 0


def test_no_alloc_refuses_a_step_too_large_for_its_scratch():
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    pool, (step,) = workloads.decode_heavy(seed=43, num_seqs=4, lo=20, hi=40)
    t, kc, vc = on_device(pool, step, dev)
    # 1.5 million requests need more work-list room than the fixed scratch
    # has, so the call must refuse on the host.  The metadata is valid for
    # every one of them (the 4 real decode rows, then empty requests whose
    # table rows name block 0), so even a call that was wrongly let through
    # would read nothing out of bounds.
    huge = 1_500_000
    nb = int(t["block_tables"].shape[1])
    bt = torch.zeros((huge, nb), dtype=torch.int32, device=dev)
    bt[:4] = t["block_tables"]
    qsl = torch.full((huge + 1,), int(t["q"].shape[0]), dtype=torch.int32, device=dev)
    qsl[:5] = t["query_start_loc"]
    ctx = torch.zeros(huge, dtype=torch.int32, device=dev)
    ctx[:4] = t["context_lens"]
    sl = torch.zeros(huge, dtype=torch.int32, device=dev)
    sl[:4] = t["seq_lens"]
    kv = pk.kv_desc(kc, vc)
    out = torch.empty_like(t["q"])
    rc = pk.lib().pa_attention_no_alloc(
        ctypes.c_void_p(t["q"].data_ptr()), ctypes.byref(kv),
        ctypes.c_void_p(bt.data_ptr()), nb, ctypes.c_void_p(qsl.data_ptr()),
        ctypes.c_void_p(ctx.data_ptr()), ctypes.c_void_p(sl.data_ptr()),
        huge, int(t["q"].shape[0]), int(t["q"].shape[1]), float(step.scale),
        ctypes.c_void_p(out.data_ptr()), None, None)
    torch.cuda.synchronize()
    assert rc == pk.PA_ERR_WORKSPACE
    assert b"fixed scratch" in pk.lib().pa_last_error_message()
