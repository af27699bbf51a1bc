"""pa_write_kv_attention: the step's cache write and its attention in one call,
the write running beside the planner.  It must give exactly what
pa_write_kv followed by pa_attention gives (caches, out and lse bit for bit)
and match the oracle, on bf16 and e4m3 pools, on multi-step chains where
each step reads the rows the previous one wrote, and inside one CUDA graph
replayed on padded smaller batches."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_284_gb300 as pk
from paged_kv_cache_284_gb300 import workloads
from gpu_helpers import (DEV, assert_attention_close, assert_status_clean, bits, codes,
                         dev_meta, oracle_attend, oracle_write)
from test_gpu_graph import padded

pytestmark = pytest.mark.gpu


def two_calls(step, kc, vc, **sc):
    pk.pa_write_kv(step.k.to(DEV), step.v.to(DEV), step.slot_mapping.to(DEV), kc, vc, **sc)
    q = step.q.to(DEV)
    out = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    pk.pa_attention(q, kc, vc, scale=step.scale, out=out, lse=lse, **dev_meta(step), **sc)
    return out, lse


def fused(step, kc, vc, **sc):
    q = step.q.to(DEV)
    out = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    m = dev_meta(step)
    pk.pa_write_kv_attention(step.k.to(DEV), step.v.to(DEV), step.slot_mapping.to(DEV), q, kc,
                             vc, m["block_tables"], m["query_start_loc"], m["context_lens"],
                             m["seq_lens"], step.scale, out, lse, **sc)
    return out, lse


def check_chain(pool, steps):
    """Both paths on their own copy of the pool, step after step."""
    ka, va = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    kf, vf = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    kb, vb = bits(pool.k_cache), bits(pool.v_cache)
    for step in steps:
        oa, la = two_calls(step, ka, va)
        of, lf = fused(step, kf, vf)
        torch.cuda.synchronize()
        kb, vb = oracle_write(step, kb, vb)
        assert np.array_equal(bits(kf), kb) and np.array_equal(bits(vf), vb), step.label
        assert np.array_equal(bits(ka), bits(kf)) and np.array_equal(bits(va), bits(vf))
        assert np.array_equal(bits(oa), bits(of)), f"{step.label}: out differs"
        assert torch.equal(la, lf), f"{step.label}: lse differs"
        ref_o, ref_l = oracle_attend(step, kb, vb)
        assert_attention_close(of, lf, ref_o, ref_l, f"fused {step.label}")
    assert_status_clean()


def test_fused_chunked_prefill_chain():
    """48-token prompt in three chunks (each chunk attends the rows the
    previous call wrote), a prefix hit and decode rows."""
    pool, steps = workloads.chunked_prefix_decode()
    check_chain(pool, steps)


def test_fused_small_decode_and_mixed_steps():
    pool, (step,) = workloads.decode_heavy(seed=284101, num_seqs=8, lo=16, hi=2000,
                                           num_q_heads=8, num_kv_heads=2)
    check_chain(pool, [step])
    pool, (step,) = workloads.mixed_step(seed=284102, num_chunks=2, chunk_len=200,
                                         chunk_ctx=(0, 900), num_decode=20,
                                         decode_len=(20, 1500), num_spec=5, spec_ctx=(20, 900),
                                         num_q_heads=8, num_kv_heads=2)
    check_chain(pool, [step])


def test_fused_fp8_pool():
    pool, (step,) = workloads.mixed_step(seed=284103, num_chunks=2, chunk_len=80,
                                         chunk_ctx=(0, 700), num_decode=20,
                                         decode_len=(20, 1200), num_spec=6, spec_ctx=(20, 1200))
    pool8 = workloads.fp8_pool_like(pool, 7101)
    sc = {"k_scale": pool8.k_scale.to(DEV), "v_scale": pool8.v_scale.to(DEV)}
    ka, va = pool8.k_cache.to(DEV), pool8.v_cache.to(DEV)
    kf, vf = pool8.k_cache.to(DEV), pool8.v_cache.to(DEV)
    oa, la = two_calls(step, ka, va, **sc)
    of, lf = fused(step, kf, vf, **sc)
    torch.cuda.synchronize()
    sk, sv = pool8.k_scale.numpy(), pool8.v_scale.numpy()
    kb, vb = oracle.write_kv_fp8(step.k, step.v, step.slot_mapping, codes(pool8.k_cache),
                                 codes(pool8.v_cache), sk, sv)
    assert np.array_equal(codes(kf), kb) and np.array_equal(codes(vf), vb)
    assert np.array_equal(bits(oa), bits(of)) and torch.equal(la, lf)
    ref_o, ref_l = oracle.attention_fp8(step.q, kb, vb, sk, sv, step.block_tables,
                                        step.query_start_loc, step.context_lens, step.seq_lens,
                                        step.scale)
    assert_attention_close(of, lf, ref_o, ref_l, "fused fp8")
    assert_status_clean()


def test_fused_graph_serves_padded_decode_batches():
    """One fused step captured at 32 decode requests replays batches of 1, 9
    and 32 rows (padded with empty requests, padding tokens slot -1)."""
    N = 32
    pool, (full,) = workloads.decode_heavy(seed=284104, num_seqs=N, lo=16, hi=1500,
                                           num_q_heads=8, num_kv_heads=2)
    kc, vc = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    names = ("q", "k", "v", "slot_mapping", "block_tables", "query_start_loc", "context_lens",
             "seq_lens")
    t = {n: getattr(full, n).to(DEV).clone() for n in names}
    out = torch.empty_like(t["q"])
    lse = torch.empty(t["q"].shape[:2], dtype=torch.float32, device=DEV)
    ws = pk.alloc_workspace(pk.workspace_size(N, N, full.num_q_heads, full.num_kv_heads,
                                              full.head_dim), DEV)

    def run():
        pk.pa_write_kv_attention(t["k"], t["v"], t["slot_mapping"], t["q"], kc, vc,
                                 t["block_tables"], t["query_start_loc"], t["context_lens"],
                                 t["seq_lens"], full.scale, out, lse, workspace=ws)

    run()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    torch.cuda.synchronize()
    kb, vb = oracle_write(full, bits(pool.k_cache), bits(pool.v_cache))
    for b in (1, 9, N):
        step = workloads.subset(full, range(b))
        p = padded(step, N, N)
        for n in names:
            t[n].copy_(getattr(p, n))
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        T = step.num_q_tokens
        ref_o, ref_l = oracle_attend(step, kb, vb)
        assert_attention_close(out[:T], lse[:T], ref_o, ref_l, f"fused graph, batch {b}")
        assert torch.isnan(out[T:].float()).all() and torch.isnan(lse[T:]).all()
    assert np.array_equal(bits(kc), kb) and np.array_equal(bits(vc), vb)
    assert_status_clean()


def test_fused_edge_cases():
    """No request: the write alone.  No new row: the attention alone.  A slot
    beyond the pool: skipped and flagged, as pa_write_kv does."""
    pool, (step,) = workloads.decode_heavy(seed=284105, num_seqs=5, lo=16, hi=400,
                                           num_q_heads=8, num_kv_heads=2)
    kc, vc = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    m = dev_meta(step)
    q = step.q.to(DEV)
    out = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    k, v, slots = step.k.to(DEV), step.v.to(DEV), step.slot_mapping.to(DEV)
    # num_seqs == 0: only the write happens
    pk.pa_write_kv_attention(k, v, slots, q, kc, vc, m["block_tables"][:0],
                             m["query_start_loc"][:1], m["context_lens"][:0],
                             m["seq_lens"][:0], step.scale, out, lse)
    torch.cuda.synchronize()
    kb, vb = oracle_write(step, bits(pool.k_cache), bits(pool.v_cache))
    assert np.array_equal(bits(kc), kb) and np.array_equal(bits(vc), vb)
    # zero new rows: the attention alone, over the rows written above
    pk.pa_write_kv_attention(k[:0], v[:0], slots[:0], q, kc, vc, m["block_tables"],
                             m["query_start_loc"], m["context_lens"], m["seq_lens"],
                             step.scale, out, lse)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle_attend(step, kb, vb)
    assert_attention_close(out, lse, ref_o, ref_l, "fused, no new rows")
    assert_status_clean()
    # a slot past the pool is skipped and flagged; the other rows are written
    bad = slots.clone()
    bad[0] = pool.num_blocks * step.block_size + 3
    pk.pa_write_kv_attention(k, v, bad, q, kc, vc, m["block_tables"], m["query_start_loc"],
                             m["context_lens"], m["seq_lens"], step.scale, out, lse)
    torch.cuda.synchronize()
    assert pk.read_device_status(clear=True) & pk.PA_DEV_BAD_SLOT
    assert np.array_equal(bits(kc), kb) and np.array_equal(bits(vc), vb)
    assert_status_clean()
