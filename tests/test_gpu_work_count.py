"""The tensor-core kernel's work, counted on the GPU ("vLLM中如何实现大模型推理加
速技术？", chunked prefill: a chunk's score block only covers the keys up to
its last row -- 48 tokens in 16-token tiles cost 16^2*6 with causal skipping,
not the dense 16^2*9).

With pa_set_tile_counter the kernel adds up the 128-key tiles for which it
issued Q K^T.  The expected count comes from the oracle's per-row visible key
counts: a 128-row query tile (128/group tokens x group heads) needs
ceil(max visible / 128) key tiles, once per kv head.  A kernel that also
visited fully masked tiles would count more; each case below also checks
that the dense count is larger, so the test can tell the two apart.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_284_gb300 as pk
from paged_kv_cache_284_gb300 import workloads
from gpu_helpers import (DEV, assert_attention_close, assert_status_clean, bits, gpu_attend,
                         gpu_write, oracle_write)

pytestmark = pytest.mark.gpu

KEY_TILE = 128


def expected_tiles(step, visible, short_max_rows):
    """(causal, dense) key-tile counts of the step's tensor-core requests."""
    g = step.num_q_heads // step.num_kv_heads
    tq = 128 // g
    qsl = step.query_start_loc.tolist()
    causal = dense = 0
    for b, n in enumerate(step.q_lens.tolist()):
        if n == 0 or n * g <= short_max_rows:
            continue
        L = int(step.seq_lens[b])
        for t0 in range(0, n, tq):
            last = qsl[b] + min(n, t0 + tq) - 1
            causal += math.ceil(int(visible[last]) / KEY_TILE)
            dense += math.ceil(L / KEY_TILE)
    return causal * step.num_kv_heads, dense * step.num_kv_heads


def count_run(pool, steps, short_max_rows):
    kc, vc = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    kb, vb = bits(pool.k_cache), bits(pool.v_cache)
    counter = torch.zeros(1, dtype=torch.int64, device=DEV)
    got = want = dense = 0
    for step in steps:
        gpu_write(step, kc, vc)
        kb, vb = oracle_write(step, kb, vb)
        counter.zero_()
        pk.set_tile_counter(counter)
        try:
            out, lse = gpu_attend(step, kc, vc, short_q_max_rows=short_max_rows)
            torch.cuda.synchronize()
        finally:
            pk.set_tile_counter(None)
        ref_o, ref_l, vis = oracle.attention(step.q, kb, vb, step.block_tables,
                                             step.query_start_loc, step.context_lens,
                                             step.seq_lens, step.scale, return_visible=True)
        assert_attention_close(out, lse, ref_o, ref_l, step.label)
        c, d = expected_tiles(step, vis, short_max_rows)
        assert int(counter.item()) == c, (step.label, int(counter.item()), c)
        got += int(counter.item())
        want += c
        dense += d
    assert_status_clean()
    return got, want, dense


def test_chunked_prefill_prefix_hit_and_decode_all_on_tensor_cores():
    """The 48 = 16+16+16 prompt, the 107-token prompt with 48 cached and the
    decode rows, every request on the tensor-core kernel."""
    pool, steps = workloads.chunked_prefix_decode()
    got, want, dense = count_run(pool, steps, short_max_rows=0)
    assert got == want > 0 and dense >= want


def test_long_chunks_skip_the_masked_tiles():
    """512-token chunks (empty and cached contexts) and a 107-token prompt:
    later query tiles see more keys than earlier ones, so causal skipping
    does less work than the dense square."""
    pool, (step,) = workloads.mixed_step(seed=284090, num_chunks=3, chunk_len=512,
                                         chunk_ctx=(0, 700), num_decode=4,
                                         decode_len=(50, 900), num_spec=2,
                                         spec_ctx=(10, 300), num_q_heads=8, num_kv_heads=2)
    got, want, dense = count_run(pool, [step], short_max_rows=64)
    assert got == want and dense > want


def test_empty_context_chunk_counts_the_page_ratio_at_128():
    """One 512-token chunk with nothing cached, 4 q / 4 kv heads (group 1, so
    4 query tiles of 128 tokens): they need 1, 2, 3 and 4 key tiles -- 10 per
    kv head against the dense 16, the 128-wide form of the page's 6 of 9."""
    gen = torch.Generator().manual_seed(284091)
    reqs = [(0, 512)]
    nb, tables, _ = workloads._assign_tables(reqs, 16, gen)
    pool = workloads.make_pool(nb, 4, 16, 128, gen)
    step = workloads.build_step(reqs, num_q_heads=4, num_kv_heads=4, head_dim=128,
                                block_size=16, gen=gen, tables=tables, label="512 from empty")
    got, want, dense = count_run(pool, [step], short_max_rows=64)
    assert want == 10 * 4 and dense == 16 * 4 and got == want
