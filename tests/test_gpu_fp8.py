"""FP8 (e4m3) KV pool on the GPU against the oracle: the quantising write is
compared byte for byte, attention within the acceptance tolerance of the fp64
oracle over the dequantised codes (values = code x per-kv-head scale)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_284_gb300 as pk
from paged_kv_cache_284_gb300 import workloads
from gpu_helpers import (DEV, assert_attention_close, assert_status_clean, codes, fp8_dev,
                         gpu_attend_fp8, gpu_write_fp8, long_requests, plan_header,
                         run_and_check_fp8, staging_blocks_for)

pytestmark = pytest.mark.gpu


def test_fp8_chunked_prefill_prefix_hit_and_decode():
    """48-token prompt in three chunks, then a 107-token prompt whose first 48
    tokens hit the cache (59 new rows: cut into pieces of 16 tokens), with
    decode rows in the same batch."""
    pool, steps = workloads.chunked_prefix_decode()
    run_and_check_fp8(workloads.fp8_pool_like(pool, 7001), steps)


def test_fp8_decode_with_forced_splits():
    pool, (step,) = workloads.decode_heavy(num_seqs=24, lo=40, hi=1500)
    pool8 = workloads.fp8_pool_like(pool, 7002)
    for split_keys in (0, 256, 1024):
        run_and_check_fp8(pool8, [step], split_keys=split_keys)


def test_fp8_mixed_small():
    pool, (step,) = workloads.mixed_step(num_chunks=2, chunk_len=80, chunk_ctx=(0, 700),
                                         num_decode=20, decode_len=(20, 1200), num_spec=6,
                                         spec_ctx=(20, 1200))
    run_and_check_fp8(workloads.fp8_pool_like(pool, 7003), [step])


@pytest.mark.parametrize("block_size,hq,hkv", [(32, 8, 2), (64, 16, 2), (16, 8, 8)])
def test_fp8_block_sizes_and_groups(block_size, hq, hkv):
    pool, (step,) = workloads.mixed_step(num_chunks=1, chunk_len=40, chunk_ctx=(0, 300),
                                         num_decode=10, decode_len=(20, 900), num_spec=3,
                                         spec_ctx=(20, 900), num_q_heads=hq, num_kv_heads=hkv,
                                         block_size=block_size)
    run_and_check_fp8(workloads.fp8_pool_like(pool, 7004 + block_size), [step])


def test_fp8_nan_codes_past_seq_len_are_ignored():
    """Slots past each request's last key hold NaN codes; no output may see them."""
    pool, (step,) = workloads.decode_heavy(num_seqs=12, lo=20, hi=400)
    pool8 = workloads.fp8_pool_like(pool, 7010)
    bs = step.block_size
    for b in range(step.num_seqs):
        L = int(step.seq_lens[b])
        last = int(step.block_tables[b, (L - 1) // bs])
        if L % bs:
            pool8.k_cache[last, :, L % bs:] = 0x7F
            pool8.v_cache[last, :, L % bs:] = 0xFF
    run_and_check_fp8(pool8, [step])


def test_fp8_write_quantises_out_of_range_values_by_saturation():
    """New tokens far beyond 448 x scale saturate to +-448 (bit-exact with the
    oracle's saturating encoder)."""
    pool, (step,) = workloads.decode_heavy(num_seqs=6, lo=20, hi=100)
    pool8 = workloads.fp8_pool_like(pool, 7011)
    step.k = (step.k.float() * 300.0).to(torch.bfloat16)
    step.v = (step.v.float() * -300.0).to(torch.bfloat16)
    kc, vc, ks, vs = fp8_dev(pool8)
    gpu_write_fp8(step, kc, vc, ks, vs)
    torch.cuda.synchronize()
    kb, vb = oracle.write_kv_fp8(step.k, step.v, step.slot_mapping, pool8.k_cache,
                                 pool8.v_cache, pool8.k_scale, pool8.v_scale)
    assert np.array_equal(codes(kc), kb) and np.array_equal(codes(vc), vb)
    assert (kb == 0x7E).any() and (vb == 0xFE).any()
    assert_status_clean()


def test_fp8_decode_heavy_full_size():
    """The decode-heavy step at full size on an e4m3 pool: every row finite and
    inside the range of the values it averages, and every row against the
    oracle over the dequantised codes."""
    pool, (step,) = workloads.decode_heavy()
    pool8 = workloads.fp8_pool_like(pool, 7012)
    del pool
    kc, vc, ks, vs = fp8_dev(pool8)
    gpu_write_fp8(step, kc, vc, ks, vs)
    out, lse = gpu_attend_fp8(step, kc, vc, ks, vs)
    torch.cuda.synchronize()
    o = out.float()
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    vmax = float(np.abs(oracle.e4m3_decode(np.arange(256, dtype=np.uint8)[:0x7F])).max()) * \
        float(pool8.v_scale.max())
    assert o.abs().max().item() <= vmax * (1 + 2 ** -7)
    kb, vb = oracle.write_kv_fp8(step.k, step.v, step.slot_mapping, pool8.k_cache,
                                 pool8.v_cache, pool8.k_scale, pool8.v_scale)
    ref_o, ref_l = oracle.attention_fp8(step.q, kb, vb, pool8.k_scale, pool8.v_scale,
                                        step.block_tables, step.query_start_loc,
                                        step.context_lens, step.seq_lens, step.scale)
    assert_attention_close(out, lse, ref_o, ref_l, "fp8 decode_heavy")
    assert_status_clean()


def test_fp8_rejected_where_not_built():
    pool, (step,) = workloads.tiny_prefill()   # head_dim 64
    pool8 = workloads.fp8_pool_like(pool, 7013)
    kc, vc, ks, vs = fp8_dev(pool8)
    with pytest.raises(pk.PaError):
        gpu_write_fp8(step, kc, vc, ks, vs)


def test_fp8_long_rows_on_the_tensor_core_path():
    """With room to stage them, the long requests (chunks, the prefix-hit
    prompt) run on the tensor-core kernel over a bf16 copy of their blocks;
    all of them are staged and the results match the oracle."""
    pool, steps = workloads.chunked_prefix_decode()
    big_pool, big_steps = workloads.mixed_step(num_chunks=3, chunk_len=96, chunk_ctx=(0, 900),
                                               num_decode=12, decode_len=(20, 900), num_spec=4,
                                               spec_ctx=(20, 900))
    for pool8, stps in ((workloads.fp8_pool_like(pool, 7020), steps),
                        (workloads.fp8_pool_like(big_pool, 7021), big_steps)):
        room = max(staging_blocks_for(st, long_requests(st)) for st in stps)
        run_and_check_fp8(pool8, stps, staging_blocks=room)
        longs = long_requests(stps[-1])
        hdr = plan_header(gpu_attend_fp8.last_workspace)
        assert longs and hdr["num_staged"] == len(longs) and hdr["long_items"] > 0, hdr


def test_fp8_partial_staging_splits_long_rows_between_the_paths():
    """Staging room for only the first long request: it runs on the
    tensor-core kernel, the later ones as split-KV pieces."""
    pool, (step,) = workloads.mixed_step(num_chunks=3, chunk_len=64, chunk_ctx=(0, 700),
                                         num_decode=8, decode_len=(20, 700), num_spec=3,
                                         spec_ctx=(20, 700))
    longs = long_requests(step)
    assert len(longs) == 3
    first = staging_blocks_for(step, longs[:1])
    pool8 = workloads.fp8_pool_like(pool, 7022)
    run_and_check_fp8(pool8, [step], staging_blocks=first)
    assert plan_header(gpu_attend_fp8.last_workspace)["num_staged"] == 1


@pytest.mark.parametrize("prefix_len,hq,hkv", [(0, 32, 8), (16, 32, 8), (512, 32, 8),
                                               (2048, 32, 8), (512, 32, 2)])
def test_fp8_cascade_decode_equals_full_attention(prefix_len, hq, hkv):
    """Cascade decode on an e4m3 pool (the prefix decoded to bf16 for the
    tensor-core prefix pass, the suffixes on the fp8 split-KV kernel writing
    fp32 states, the fold merging both) equals the oracle's fp8 attention
    over the full tables.  Group 4 takes the operand-swapped suffix path,
    group 16 the general one."""
    pool, (step,) = workloads.cascade(seed=7200 + prefix_len + hkv, num_seqs=9,
                                      prefix_len=prefix_len, suffix=(1, 300), num_q_heads=hq,
                                      num_kv_heads=hkv)
    pool8 = workloads.fp8_pool_like(pool, 7201)
    kc, vc, ks, vs = fp8_dev(pool8)
    gpu_write_fp8(step, kc, vc, ks, vs)
    sk, sv = pool8.k_scale.numpy(), pool8.v_scale.numpy()
    kb, vb = oracle.write_kv_fp8(step.k, step.v, step.slot_mapping, codes(pool8.k_cache),
                                 codes(pool8.v_cache), sk, sv)
    q = step.q.to(DEV)
    out = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    pk.pa_cascade_decode(q, kc, vc, step.prefix_blocks.to(DEV), step.prefix_len,
                         step.suffix_block_tables.to(DEV), step.query_start_loc.to(DEV),
                         step.suffix_context_lens.to(DEV), step.suffix_seq_lens.to(DEV),
                         step.scale, out, lse, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert np.array_equal(codes(kc), kb) and np.array_equal(codes(vc), vb)
    ro, rl = oracle.attention_fp8(step.q, kb, vb, sk, sv, step.block_tables,
                                  step.query_start_loc, step.context_lens, step.seq_lens,
                                  step.scale)
    assert_attention_close(out, lse, ro, rl, f"fp8 cascade, prefix {prefix_len}, group {hq // hkv}")
    assert_status_clean()


def test_fp8_prefix_attention_matches_oracle():
    """Shared-prefix attention on an e4m3 pool: every query row over all
    prefix keys, against the oracle's fp8 attention with each row a request
    whose table is the prefix (context prefix_len - 1, so no key is masked)."""
    pool, (step,) = workloads.cascade(seed=7210, num_seqs=12, prefix_len=704, suffix=(1, 50))
    pool8 = workloads.fp8_pool_like(pool, 7211)
    kc, vc, ks, vs = fp8_dev(pool8)
    q = step.q.to(DEV)
    out = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    pk.pa_prefix_attention(q, kc, vc, step.prefix_blocks.to(DEV), step.prefix_len, step.scale,
                           out, lse, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    T = step.num_q_tokens
    bt = step.prefix_blocks.view(1, -1).repeat(T, 1).contiguous()
    qsl = torch.arange(T + 1, dtype=torch.int32)
    ctx = torch.full((T,), step.prefix_len - 1, dtype=torch.int32)
    sl = torch.full((T,), step.prefix_len, dtype=torch.int32)
    ro, rl = oracle.attention_fp8(step.q, codes(pool8.k_cache), codes(pool8.v_cache),
                                  pool8.k_scale.numpy(), pool8.v_scale.numpy(), bt, qsl, ctx, sl,
                                  step.scale)
    assert_attention_close(out, lse, ro, rl, "fp8 prefix attention")
    assert_status_clean()
