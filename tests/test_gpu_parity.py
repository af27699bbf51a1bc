"""GPU parity: the CUDA path against the fp64 oracle on the same seeded
inputs, through the C ABI.  Cache writes bit-exact; attention within
max-abs 2e-2 / mean-abs 2e-3 (output) and 1e-3 (LSE).

Sizes here are ones the oracle finishes in seconds while still spanning
several KV tiles, several splits and ragged tails; the full-size workloads
are sampled in test_gpu_fullsize.py.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_284_gb300 as pk
from paged_kv_cache_284_gb300 import workloads
from gpu_helpers import (DEV, assert_attention_close, assert_status_clean, bits, gpu_attend,
                         gpu_write, long_requests, oracle_attend, oracle_write, plan_header,
                         run_and_check, OUT_MAX_ABS, OUT_MEAN_ABS, LSE_MAX_ABS)

pytestmark = pytest.mark.gpu

# short_q_max_rows: -1 = default dispatch, 0 = every request on the tensor-core kernel
PATHS = [dict(), dict(short_q_max_rows=0)]
PATH_IDS = ["default", "tensor_core_only"]


@pytest.mark.parametrize("kw", PATHS, ids=PATH_IDS)
def test_tiny_prefill_31_29_30(kw):
    pool, steps = workloads.tiny_prefill()
    run_and_check(pool, steps, **kw)


@pytest.mark.parametrize("kw", PATHS, ids=PATH_IDS)
def test_chunked_prefill_prefix_hit_decode(kw):
    pool, steps = workloads.chunked_prefix_decode()
    run_and_check(pool, steps, **kw)


@pytest.mark.parametrize("kw", PATHS + [dict(split_keys=64), dict(split_keys=256)],
                         ids=PATH_IDS + ["split64", "split256"])
def test_decode_rows(kw):
    pool, steps = workloads.decode_heavy(seed=7, num_seqs=24, lo=1, hi=700)
    run_and_check(pool, steps, **kw)


@pytest.mark.parametrize("kw", PATHS + [dict(split_keys=128)], ids=PATH_IDS + ["split128"])
def test_mixed_step_small(kw):
    pool, steps = workloads.mixed_step(seed=11, num_chunks=2, chunk_len=150,
                                       chunk_ctx=(0, 400), num_decode=10,
                                       decode_len=(1, 500), num_spec=5, spec_ctx=(0, 300))
    run_and_check(pool, steps, **kw)


@pytest.mark.parametrize("bs", [32, 64, 256])
@pytest.mark.parametrize("hq,hkv,d", [(4, 4, 128), (32, 4, 128), (8, 2, 64)])
def test_block_sizes_groups_head_dims(bs, hq, hkv, d):
    pool, steps = workloads.mixed_step(seed=bs + hq + d, num_chunks=1, chunk_len=70,
                                       chunk_ctx=(0, 300), num_decode=5, decode_len=(1, 400),
                                       num_spec=2, spec_ctx=(0, 200), num_q_heads=hq,
                                       num_kv_heads=hkv, head_dim=d, block_size=bs)
    run_and_check(pool, steps)
    run_and_check(pool, steps, short_q_max_rows=0)


def test_write_kv_skips_padding_and_keeps_other_slots():
    gen = torch.Generator().manual_seed(3)
    pool = workloads.make_pool(20, 4, 32, 128, gen)
    T = 50
    k = torch.randn(T, 4, 128, generator=gen).to(torch.bfloat16)
    v = torch.randn(T, 4, 128, generator=gen).to(torch.bfloat16)
    slots = torch.randperm(20 * 32, generator=gen)[:T].to(torch.int64)
    slots[::7] = -1
    kc, vc = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    pk.pa_write_kv(k.to(DEV), v.to(DEV), slots.to(DEV), kc, vc)
    ek, ev = oracle.write_kv(k, v, slots, pool.k_cache, pool.v_cache)
    assert np.array_equal(bits(kc), ek) and np.array_equal(bits(vc), ev)
    assert_status_clean()


def test_write_kv_out_of_pool_slot_is_flagged_not_written():
    gen = torch.Generator().manual_seed(4)
    pool = workloads.make_pool(4, 2, 16, 64, gen)
    k = torch.randn(3, 2, 64, generator=gen).to(torch.bfloat16)
    slots = torch.tensor([1, 4 * 16 + 3, 9], dtype=torch.int64)
    kc, vc = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    pk.pa_write_kv(k.to(DEV), k.to(DEV), slots.to(DEV), kc, vc)
    st = pk.read_device_status(clear=True)
    assert st & pk.PA_DEV_BAD_SLOT
    ek, _ = oracle.write_kv(k[[0, 2]], k[[0, 2]], slots[[0, 2]], pool.k_cache, pool.v_cache)
    assert np.array_equal(bits(kc), ek)


@pytest.mark.parametrize("kw", PATHS, ids=PATH_IDS)
def test_non_finite_cache_tails_are_never_used(kw):
    """Slots past a sequence's end (and unused blocks) hold NaN/Inf: results
    must not change."""
    pool, (step,) = workloads.mixed_step(seed=5, num_chunks=1, chunk_len=77, chunk_ctx=(3, 90),
                                         num_decode=6, decode_len=(1, 200), num_spec=3,
                                         spec_ctx=(1, 150))
    used = torch.zeros(pool.num_blocks, step.block_size, dtype=torch.bool)
    for b in range(step.num_seqs):
        L = int(step.seq_lens[b])
        for j in range(L):
            used[int(step.block_tables[b, j // step.block_size]), j % step.block_size] = True
    for cache, val in ((pool.k_cache, float("nan")), (pool.v_cache, float("inf"))):
        mask = (~used)[:, None, :, None].expand_as(cache)
        cache[mask] = val
    run_and_check(pool, [step], **kw)


@pytest.mark.parametrize("n,h,d", [(37, 6, 128), (1000, 32, 64), (3, 1, 8)])
def test_merge_states_matches_oracle(n, h, d):
    """The merge operator against the fp64 oracle at the attention tolerance
    (max and mean absolute output error, LSE error), including empty states
    (lse = -inf on one side and on both)."""
    gen = torch.Generator().manual_seed(21 + n)
    oa = torch.randn(n, h, d, generator=gen).to(torch.bfloat16)
    ob = torch.randn(n, h, d, generator=gen).to(torch.bfloat16)
    la = (4 * torch.randn(n, h, generator=gen)).float()
    lb = (4 * torch.randn(n, h, generator=gen)).float()
    la[0, 0] = -float("inf")
    if n > 1 and h > 1:
        la[1, 1] = lb[1, 1] = -float("inf")
    if n > 2:
        lb[2, -1] = -float("inf")
    out = torch.empty(n, h, d, dtype=torch.bfloat16, device=DEV)
    lo = torch.empty(n, h, dtype=torch.float32, device=DEV)
    pk.pa_merge_states(oa.to(DEV), la.to(DEV), ob.to(DEV), lb.to(DEV), out, lo)
    ro, rl = oracle.merge_states(oa.double(), la.double(), ob.double(), lb.double())
    o = out.float().cpu().numpy()
    err = np.abs(o - ro)
    assert err.max() <= OUT_MAX_ABS, err.max()
    assert err.mean() <= OUT_MEAN_ABS, err.mean()
    l = lo.cpu().numpy()
    fin = np.isfinite(rl)
    assert np.abs(l[fin] - rl[fin]).max() <= LSE_MAX_ABS
    assert np.array_equal(np.isneginf(l), np.isneginf(rl))


def cascade_small(seed=31):
    return workloads.cascade(seed=seed, num_seqs=6, prefix_len=512, suffix=(20, 150))


def test_prefix_attention_matches_oracle():
    pool, (step,) = cascade_small()
    kc, vc = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    gpu_write(step, kc, vc)
    kb, vb = oracle_write(step, bits(pool.k_cache), bits(pool.v_cache))
    q = step.q.to(DEV)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=DEV)
    pk.pa_prefix_attention(q, kc, vc, step.prefix_blocks.to(DEV), step.prefix_len, step.scale,
                           out, lse)
    ro, rl = oracle.prefix_attention(step.q, kb, vb, step.prefix_blocks, step.prefix_len,
                                     step.scale)
    assert_attention_close(out, lse, ro, rl, "prefix")
    assert_status_clean()


@pytest.mark.parametrize("prefix_len", [0, 16, 512, 2048])
def test_cascade_decode_equals_full_attention(prefix_len):
    """Cascade decode (prefix pass beside the suffix pass, merged by the fold)
    equals paged attention over the full tables, down to an empty prefix."""
    pool, (step,) = workloads.cascade(seed=prefix_len, num_seqs=9, prefix_len=prefix_len,
                                      suffix=(1, 300))
    kc, vc = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    gpu_write(step, kc, vc)
    kb, vb = oracle_write(step, bits(pool.k_cache), bits(pool.v_cache))
    q = step.q.to(DEV)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=DEV)
    pk.pa_cascade_decode(q, kc, vc, step.prefix_blocks.to(DEV), step.prefix_len,
                         step.suffix_block_tables.to(DEV), step.query_start_loc.to(DEV),
                         step.suffix_context_lens.to(DEV), step.suffix_seq_lens.to(DEV),
                         step.scale, out, lse)
    ro, rl = oracle_attend(step, kb, vb)   # full tables: prefix blocks + suffix blocks
    assert_attention_close(out, lse, ro, rl, "cascade")
    # and the merge kernel on the two separate passes gives the same
    assert_status_clean()


def test_empty_batches_are_no_ops():
    pool, (step,) = workloads.decode_heavy(seed=1, num_seqs=2, lo=5, hi=9)
    kc, vc = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    q = torch.empty(0, step.num_q_heads, step.head_dim, dtype=torch.bfloat16, device=DEV)
    out = torch.empty_like(q)
    z = torch.zeros(1, dtype=torch.int32, device=DEV)
    pk.pa_attention(q, kc, vc, step.block_tables[:0].to(DEV), z,
                    torch.zeros(0, dtype=torch.int32, device=DEV),
                    torch.zeros(0, dtype=torch.int32, device=DEV), step.scale, out)
    pk.pa_write_kv(step.k[:0].to(DEV), step.v[:0].to(DEV), step.slot_mapping[:0].to(DEV), kc, vc)
    torch.cuda.synchronize()
    assert_status_clean()


def test_zero_length_request_inside_a_batch():
    """A request with q_len 0 contributes nothing and does not disturb others."""
    pool, (step,) = workloads.decode_heavy(seed=2, num_seqs=5, lo=10, hi=80)
    # make request 2 empty: q_len 0, seq_len = context
    qsl = step.query_start_loc.clone()
    qsl[3:] -= 1
    rows = [i for i in range(step.num_q_tokens) if i != 2]
    step = workloads.dataclasses.replace(
        step, q=step.q[rows].contiguous(), k=step.k[rows].contiguous(),
        v=step.v[rows].contiguous(), slot_mapping=step.slot_mapping[rows].contiguous(),
        query_start_loc=qsl, seq_lens=step.seq_lens.clone())
    step.seq_lens[2] = step.context_lens[2]
    run_and_check(pool, [step])


def test_bad_block_id_is_clamped_and_flagged():
    pool, (step,) = workloads.decode_heavy(seed=3, num_seqs=4, lo=40, hi=60)
    bt = step.block_tables.clone()
    bt[1, 0] = pool.num_blocks + 5
    kc, vc = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    q = step.q.to(DEV)
    out = torch.empty_like(q)
    pk.pa_attention(q, kc, vc, bt.to(DEV), step.query_start_loc.to(DEV),
                    step.context_lens.to(DEV), step.seq_lens.to(DEV), step.scale, out)
    st = pk.read_device_status(clear=True)
    assert st & pk.PA_DEV_BAD_BLOCK
    assert not (st & pk.PA_DEV_WAIT_TIMEOUT)


def test_inconsistent_seq_len_is_flagged_and_skipped():
    pool, (step,) = workloads.decode_heavy(seed=4, num_seqs=3, lo=40, hi=60)
    sl = step.seq_lens.clone()
    sl[0] += 1
    kc, vc = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    q = step.q.to(DEV)
    out = torch.zeros_like(q)
    pk.pa_attention(q, kc, vc, step.block_tables.to(DEV), step.query_start_loc.to(DEV),
                    step.context_lens.to(DEV), sl.to(DEV), step.scale, out)
    st = pk.read_device_status(clear=True)
    assert st & pk.PA_DEV_BAD_METADATA


def test_same_result_on_a_side_stream():
    pool, (step,) = workloads.decode_heavy(seed=9, num_seqs=12, lo=100, hi=900)
    kc, vc = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    gpu_write(step, kc, vc)
    o1, l1 = gpu_attend(step, kc, vc)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        o2, l2 = gpu_attend(step, kc, vc)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert_status_clean()


def test_side_by_side_kernels_match_the_serial_launch_order():
    """The step's default launch order runs the split-KV and tensor-core
    kernels side by side (two tensor-core grids sharing a work counter); with
    per-kernel profiling events set, the same kernels run one after the other
    with a fixed item order.  Every item is computed the same way either
    way, so the outputs agree bit for bit."""
    pool, (step,) = workloads.mixed_step(num_chunks=4, chunk_len=256, chunk_ctx=(0, 3000),
                                         num_decode=64, decode_len=(64, 3000), num_spec=8,
                                         spec_ctx=(64, 3000))
    assert len(long_requests(step)) == 4 and step.num_seqs > 4
    kc, vc = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    gpu_write(step, kc, vc)
    out_a, lse_a = gpu_attend(step, kc, vc)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(2)]
    for a, b in evs:
        a.record()
        b.record()
    torch.cuda.synchronize()
    pk.set_profile_events(pk.PA_KERNEL_SPLIT_KV, *evs[0])
    pk.set_profile_events(pk.PA_KERNEL_TENSOR_CORE, *evs[1])
    try:
        out_b, lse_b = gpu_attend(step, kc, vc)
        torch.cuda.synchronize()
    finally:
        pk.set_profile_events(pk.PA_KERNEL_SPLIT_KV, None, None)
        pk.set_profile_events(pk.PA_KERNEL_TENSOR_CORE, None, None)
    assert np.array_equal(bits(out_a), bits(out_b))
    assert torch.equal(lse_a, lse_b)
    assert_status_clean()


def test_launches_per_step():
    """The library's launch count for one step: write_kv, plan, split-KV and,
    when the step can hold a long request (T >= 64 / group + 1 tokens), the
    tensor-core kernel -- as two grids beside the split-KV grid for a step
    of at least 512 tokens, as one grid after it for a smaller step."""
    pool, (step,) = workloads.mixed_step(num_chunks=2, chunk_len=256, chunk_ctx=(0, 1000),
                                         num_decode=16, decode_len=(64, 1000), num_spec=2,
                                         spec_ctx=(64, 1000))
    assert step.num_q_tokens >= 512
    kc, vc = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    torch.cuda.synchronize()
    n0 = pk.kernel_launches()
    gpu_write(step, kc, vc)
    gpu_attend(step, kc, vc)
    torch.cuda.synchronize()
    assert pk.kernel_launches() - n0 == 5
    spool, (sstep,) = workloads.tiny_prefill()   # 90 tokens: could hold a long request
    skc, svc = spool.k_cache.to(DEV), spool.v_cache.to(DEV)
    n0 = pk.kernel_launches()
    gpu_write(sstep, skc, svc)
    gpu_attend(sstep, skc, svc)
    torch.cuda.synchronize()
    assert pk.kernel_launches() - n0 == 4
    dpool, (dstep,) = workloads.decode_heavy(num_seqs=8, lo=64, hi=600)
    dkc, dvc = dpool.k_cache.to(DEV), dpool.v_cache.to(DEV)
    n0 = pk.kernel_launches()
    gpu_write(dstep, dkc, dvc)
    gpu_attend(dstep, dkc, dvc)
    torch.cuda.synchronize()
    assert pk.kernel_launches() - n0 == 3
    assert_status_clean()


def test_small_decode_batch_is_cut_into_one_round_of_items():
    """A decode batch too small to fill the persistent split-KV grid (8
    requests x 8 kv heads) is cut so that each CTA gets about one item: the
    split size is the smallest that keeps the item count within the grid
    (one round), above the 4-stage floor; results stay at parity."""
    pool, (step,) = workloads.decode_heavy(seed=58, num_seqs=8)
    kc, vc = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    ws = pk.alloc_workspace(pk.workspace_size(step.num_seqs, step.num_q_tokens,
                                              step.num_q_heads, step.num_kv_heads,
                                              step.head_dim), DEV)
    gpu_write(step, kc, vc)
    out, lse = gpu_attend(step, kc, vc, workspace=ws)
    torch.cuda.synchronize()
    h = plan_header(ws)
    ctas = 2 * torch.cuda.get_device_properties(0).multi_processor_count  # 2 per SM here
    assert 0.8 * ctas <= h["short_items"] <= ctas, h
    assert h["split_stages"] > 4, h
    kb, vb = oracle_write(step, bits(pool.k_cache), bits(pool.v_cache))
    ref_o, ref_l = oracle_attend(step, kb, vb)
    assert_attention_close(out, lse, ref_o, ref_l, "one-round split")
    assert_status_clean()


def test_cascade_with_64_prefix_splits():
    """One query tile per kv head (8 requests x 4 heads of 2 kv heads) over an
    8192-token prefix: the prefix pass cuts it into 64 key-range splits, the
    most it makes, so the fold merges states 32-63 too."""
    pool, (step,) = workloads.cascade(seed=64, num_seqs=8, prefix_len=8192, suffix=(1, 200),
                                      num_q_heads=8, num_kv_heads=2)
    kc, vc = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    gpu_write(step, kc, vc)
    kb, vb = oracle_write(step, bits(pool.k_cache), bits(pool.v_cache))
    q = step.q.to(DEV)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=DEV)
    pk.pa_cascade_decode(q, kc, vc, step.prefix_blocks.to(DEV), step.prefix_len,
                         step.suffix_block_tables.to(DEV), step.query_start_loc.to(DEV),
                         step.suffix_context_lens.to(DEV), step.suffix_seq_lens.to(DEV),
                         step.scale, out, lse)
    ro, rl = oracle_attend(step, kb, vb)
    assert_attention_close(out, lse, ro, rl, "cascade, 64 prefix splits")
    assert_status_clean()
