"""Request-sharded replicas on the CPU (no GPU).

The router (pa_partition_requests, host C++ in libpa) hands each request of
one step to one replica, balancing KV tokens greedily longest first
(2048ai.net page on the vLLM V1 engine, data parallelism: a request router
feeds full replicas, and load imbalance between them is the risk).  Checked
here:
  * every request goes to exactly one rank, the per-rank loads add up, and
    the heaviest and lightest rank differ by at most one request's weight
    (the list-scheduling bound);
  * the assignment equals a plain Python greedy model, ties included;
  * two gloo ranks each run the CPU oracle on their shard of one step, and
    rank 0 checks that the gathered rows equal the oracle on the whole step,
    bit for bit (the shards need no exchange on the data path).
"""
import os
import random
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import paged_kv_cache_284_gb300 as pk  # noqa: E402


def greedy_model(weights, ranks):
    """Longest first (stable on request index), least-loaded rank (lowest on
    ties)."""
    order = sorted(range(len(weights)), key=lambda b: (-weights[b], b))
    load = [0] * ranks
    out = [None] * len(weights)
    for b in order:
        r = min(range(ranks), key=lambda i: (load[i], i))
        out[b] = r
        load[r] += weights[b]
    return out, load


@pytest.mark.parametrize("ranks", [1, 2, 3, 8])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_router_balances_kv_tokens_within_one_request(ranks, seed):
    rng = random.Random(seed)
    weights = [rng.randint(0, 8704) for _ in range(rng.randint(1, 500))]
    rank_of, loads = pk.partition_requests(weights, ranks)
    assert all(0 <= r < ranks for r in rank_of)
    per = [0] * ranks
    for b, r in enumerate(rank_of):
        per[r] += weights[b]
    assert per == loads
    assert sum(loads) == sum(weights)
    assert max(loads) - min(loads) <= max(weights)
    assert (rank_of, loads) == greedy_model(weights, ranks)


def test_router_edge_cases():
    assert pk.partition_requests([], 4) == ([], [0, 0, 0, 0])
    # more ranks than requests: one request each, the rest empty
    rank_of, loads = pk.partition_requests([5, 9, 7], 5)
    assert rank_of == [2, 0, 1] and loads == [9, 7, 5, 0, 0]
    # equal weights go round the ranks in request order
    rank_of, _ = pk.partition_requests([3] * 7, 3)
    assert rank_of == [0, 1, 2, 0, 1, 2, 0]
    with pytest.raises(pk.PaError):
        pk.partition_requests([1, -1], 2)
    with pytest.raises(pk.PaError):
        pk.partition_requests([1, 2], 0)


def test_router_on_the_mixed_step_recipe():
    """Eight copies of the mixed-step recipe over eight replicas: each rank's
    KV is within one request (at most 8192 + 512 tokens) of the others'."""
    from paged_kv_cache_284_gb300 import workloads
    reqs = []
    for i in range(8):
        reqs += workloads.mixed_step_requests(seed=workloads.SEED_BASE + 3 + 1000 * i)
    lens = [c + n for c, n in reqs]
    rank_of, loads = pk.partition_requests(lens, 8)
    assert max(loads) - min(loads) <= max(lens)
    assert max(loads) <= sum(lens) / 8 + max(lens)
    assert sorted(set(rank_of)) == list(range(8))


def _small_step():
    from paged_kv_cache_284_gb300 import workloads
    return workloads.mixed_step(seed=284300, num_chunks=3, chunk_len=40, chunk_ctx=(0, 200),
                                num_decode=9, decode_len=(5, 400), num_spec=3,
                                spec_ctx=(0, 300), num_q_heads=8, num_kv_heads=2,
                                head_dim=64)


def _shard_rank(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import oracle
    import paged_kv_cache_284_gb300 as pkr
    from paged_kv_cache_284_gb300 import workloads
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        pool, (step,) = _small_step()
        rank_of, _ = pkr.partition_requests(step.seq_lens.tolist(), world)
        mine = [b for b, r in enumerate(rank_of) if r == rank]
        sub = workloads.subset(step, mine)
        kc, vc = oracle.write_kv(sub.k, sub.v, sub.slot_mapping, pool.k_cache, pool.v_cache)
        o, lse = oracle.attention(sub.q, kc, vc, sub.block_tables, sub.query_start_loc,
                                  sub.context_lens, sub.seq_lens, sub.scale)
        qsl = step.query_start_loc.tolist()
        rows = [t for b in mine for t in range(qsl[b], qsl[b + 1])]
        gathered = [None] * world if rank == 0 else None
        dist.gather_object((rows, o, lse), gathered, dst=0)
        if rank == 0:
            results["gathered"] = gathered
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_on_their_shards_equal_the_whole_step():
    import oracle
    oracle.build_oracle()
    world = 2
    port = 31500 + (os.getpid() % 2000)
    with mp.get_context("spawn").Manager() as m:
        results = m.dict()
        mp.spawn(_shard_rank, args=(world, port, results), nprocs=world, join=True)
        gathered = results["gathered"]
    pool, (step,) = _small_step()
    kc, vc = oracle.write_kv(step.k, step.v, step.slot_mapping, pool.k_cache, pool.v_cache)
    ref_o, ref_l = oracle.attention(step.q, kc, vc, step.block_tables, step.query_start_loc,
                                    step.context_lens, step.seq_lens, step.scale)
    got_o = np.full_like(ref_o, np.nan)
    got_l = np.full_like(ref_l, np.nan)
    seen = []
    for rows, o, lse in gathered:
        assert len(rows) > 0          # both replicas got work
        got_o[rows] = o
        got_l[rows] = lse
        seen += rows
    assert sorted(seen) == list(range(step.num_q_tokens))
    assert np.array_equal(got_o, ref_o)
    assert np.array_equal(got_l, ref_l)
