"""Host block manager (include/pa_blocks.h) with its content-hash prefix cache.

The plain model in oracle/blocks.py is pinned first against what the page
states ("11. 推理加速(一):vLLM 原理", §11.2 and §11.4) and against invariants;
then the C++ manager is compared with the model operation by operation on
random workloads (every return code, emitted array, reference count and
table must be identical)."""
import random

import numpy as np
import pytest

import oracle
from oracle.blocks import BlockManagerModel, INVALID, NO_BLOCKS, OK
from paged_kv_cache_284_gb300 import PA_ERR_INVALID_ARG, PA_ERR_WORKSPACE
from paged_kv_cache_284_gb300.blocks import BlockManager

BS = 16


def run_prompt(m, rid, tokens, max_blocks=64):
    code, cached = m.add_request(rid, tokens)
    assert code == OK
    code, meta = m.schedule([rid], [len(tokens) - cached], max_blocks, 4)
    assert code == OK
    return cached, meta


# ---- pins of the model against the page ----------------------------------------

def test_shared_prefix_blocks_like_the_page_example():
    """§11.2: A = [3,7,11]-style table; B shares A's first two physical blocks
    and gets a new third one; the shared blocks count two references."""
    m = BlockManagerModel(32, BS)
    a = list(range(100, 148))                 # 48 tokens = 3 full blocks
    run_prompt(m, "A", a)
    b = a[:32] + list(range(500, 520))        # same first 32 tokens, then different
    cached, meta = run_prompt(m, "B", b)
    ta, tb = m.reqs["A"].table, m.reqs["B"].table
    assert cached == 32 and tb[:2] == ta[:2] and tb[2] != ta[2]
    assert [m.ref[x] for x in ta] == [2, 2, 1]
    assert meta["context_lens"] == [32] and meta["seq_lens"] == [52]


def test_prefix_hit_prefills_only_the_new_tokens():
    """§11.4 with the 107-token prompt whose first 48 tokens are cached: only
    59 tokens are computed, at positions 48..106, and the table starts with
    the 48-token prompt's three blocks."""
    m = BlockManagerModel(64, BS)
    p48 = list(range(1, 49))
    run_prompt(m, 1, p48)
    p107 = p48 + list(range(1000, 1059))
    cached, meta = run_prompt(m, 2, p107)
    assert cached == 48
    assert meta["query_start_loc"] == [0, 59] and meta["context_lens"] == [48]
    assert m.reqs[2].table[:3] == m.reqs[1].table[:3]
    slots = meta["slot_mapping"]
    assert len(slots) == 59 and all(s // BS not in m.reqs[1].table for s in slots)


def test_fully_cached_prompt_still_computes_its_last_block():
    m = BlockManagerModel(16, BS)
    p = list(range(7, 7 + 32))
    run_prompt(m, 1, p)
    code, cached = m.add_request(2, p)
    assert code == OK and cached == 16


def test_blocks_are_taken_only_when_tokens_reach_them():
    m = BlockManagerModel(16, BS)
    run_prompt(m, 1, list(range(20)))       # 20 tokens -> 2 blocks
    assert len(m.reqs[1].table) == 2
    for step in range(30):
        m.append_tokens(1, [9])
        code, _ = m.schedule([1], [1], 16, 1)
        assert code == OK
        assert len(m.reqs[1].table) == -(-m.reqs[1].computed // BS)


def test_copy_on_write_after_fork():
    m = BlockManagerModel(16, BS)
    run_prompt(m, 1, list(range(20)))       # block 1 holds 4 tokens
    assert m.fork(1, 2) == OK
    shared = m.reqs[1].table[1]
    assert m.ref[shared] == 2
    m.append_tokens(2, [77])
    code, meta = m.schedule([2], [1], 16, 1)
    assert code == OK
    new = m.reqs[2].table[1]
    assert meta["copies"] == [(shared, new)] and new != shared
    assert m.ref[shared] == 1 and m.ref[new] == 1
    assert m.reqs[1].table[1] == shared and m.reqs[2].table[0] == m.reqs[1].table[0]


def test_eviction_takes_the_block_released_longest_ago():
    m = BlockManagerModel(5, 4)
    run_prompt(m, 1, list(range(9)))        # blocks 0, 1 full (cached), 2 holds one token
    run_prompt(m, 2, list(range(50, 54)))   # block 3 full (cached); block 4 free
    assert m.free_request(1) == OK          # releases 2 (free), then 1, then 0 (evictable)
    assert m.free_blocks() == [2, 4] and sorted(m.evictable_blocks()) == [0, 1, 3][:2]
    run_prompt(m, 3, list(range(80, 93)))   # 4 blocks: free 2 and 4, then evict 1, then 0
    assert m.reqs[3].table == [2, 4, 1, 0]
    code, cached = m.add_request(4, list(range(9)))
    assert cached == 0                      # that prefix was evicted
    assert m.reqs[2].table == [3] and m.cache[tuple(range(50, 54))] == 3


def test_out_of_blocks_changes_nothing():
    m = BlockManagerModel(2, 4)
    run_prompt(m, 1, list(range(8)))
    m.add_request(2, list(range(40, 44)))
    before = (list(m.ref), dict(m.cache))
    assert m.schedule([2], [4], 4, 1)[0] == NO_BLOCKS
    assert (list(m.ref), dict(m.cache)) == before


def random_ops(seed, n_ops=400, vocab=3, model=None):
    """A random serving trace: new prompts (short vocabulary and shared
    openings, so prefixes repeat), decode appends, chunked steps, forks and
    frees.  With `model`, step sizes are drawn from each request's pending
    tokens (most steps valid) and requests are freed when the pool runs low;
    yields one operation at a time, so the caller applies it before the next
    is drawn."""
    rng = random.Random(seed)
    live, next_id = [], 0
    for _ in range(n_ops):
        r = rng.random()
        low = model is not None and model.available() < 4
        if (r < 0.25 or not live) and not low:
            n = rng.randint(1, 14)
            base = rng.choice([[], [0, 1, 2, 0], [1, 1, 1, 1, 2, 2, 2, 2]])
            yield ("add", next_id, base + [rng.randrange(vocab) for _ in range(n)])
            live.append(next_id)
            next_id += 1
        elif r < 0.33 and not low:
            yield ("fork", rng.choice(live), next_id)
            live.append(next_id)
            next_id += 1
        elif r < 0.45 or (low and live):
            rid = rng.choice(live)
            yield ("free", rid)
            live.remove(rid)
        elif r < 0.60:
            rid = rng.choice(live)
            yield ("append", rid, [rng.randrange(vocab) for _ in range(rng.randint(1, 3))])
        else:
            k = rng.randint(1, min(4, len(live)))
            rids = rng.sample(live, k)
            news = []
            for rid in rids:
                pend = 0
                if model is not None and rid in model.reqs:
                    q = model.reqs[rid]
                    pend = len(q.tokens) - q.computed
                news.append(rng.randint(1, pend) if pend and rng.random() < 0.9
                            else rng.randint(1, 6))
            yield ("schedule", rids, news, rng.choice([3, 8]))
        if rng.random() < 0.02:
            yield ("bad",)


def apply_model(m, op):
    kind = op[0]
    if kind == "add":
        return m.add_request(op[1], op[2])
    if kind == "fork":
        return m.fork(op[1], op[2])
    if kind == "free":
        return m.free_request(op[1])
    if kind == "append":
        return m.append_tokens(op[1], op[2])
    if kind == "schedule":
        return m.schedule(op[1], op[2], op[3], 4)
    return m.add_request(-5, [])


def model_invariants(m):
    count = [0] * m.n
    for r in m.reqs.values():
        for b in r.table:
            count[b] += 1
        assert len(r.table) == -(-r.computed // m.bs)
    assert count == m.ref
    assert len(m.free_blocks()) + len(m.evictable_blocks()) + sum(c > 0 for c in count) == m.n
    for key, b in m.cache.items():
        assert m.key[b] == key


@pytest.mark.parametrize("seed", range(6))
def test_model_invariants_on_random_traces(seed):
    m = BlockManagerModel(24, 4)
    for op in random_ops(seed, model=m):
        res = apply_model(m, op)
        if op[0] == "schedule" and res[0] == OK:
            slots = res[1]["slot_mapping"]
            assert len(set(slots)) == len(slots)
            for rid, t0, t1 in zip(op[1], res[1]["query_start_loc"], res[1]["query_start_loc"][1:]):
                assert all(s // m.bs in m.reqs[rid].table for s in slots[t0:t1])
        model_invariants(m)


# ---- the metadata drives the attention oracle to dense attention ----------------

def test_manager_metadata_reproduces_dense_attention():
    """K/V of position p of a sequence is a function of its token prefix
    [0..p]; writing each step's new rows through the manager's slot mapping
    (after its copy-on-write copies) and attending through its tables must
    read, for every request, exactly its own positions' K/V in order -- so
    paged attention equals dense causal attention over those arrays."""
    import torch
    hkv, hq, d, bs, nb = 2, 4, 8, 4, 40

    def kv_of(prefix):
        g = torch.Generator().manual_seed(hash(tuple(prefix)) & 0x7FFFFFFF)
        return (torch.randn(2, hkv, d, generator=g).to(torch.bfloat16))

    m = BlockManagerModel(nb, bs)
    kc = torch.zeros(nb, hkv, bs, d, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    seqs = {}
    rng = random.Random(3)
    prompts = {0: [1, 2, 3, 1, 2, 3, 1, 2, 3, 4], 1: [1, 2, 3, 1, 2, 3, 1, 2, 9, 9, 9],
               2: [5] * 13}
    for rid, p in prompts.items():
        m.add_request(rid, p)
        seqs[rid] = list(p)
    m.fork(0, 3)
    seqs[3] = list(seqs[0])
    for step in range(6):
        rids = sorted(seqs)
        new = []
        for rid in rids:
            r = m.reqs[rid]
            if r.computed == len(r.tokens):
                t = rng.randrange(10)
                m.append_tokens(rid, [t])
                seqs[rid].append(t)
            new.append(min(len(r.tokens) - r.computed, rng.randint(1, 5)))
        code, meta = m.schedule(rids, new, 16, 8)
        assert code == OK
        for src, dst in meta["copies"]:
            kc[dst] = kc[src]
            vc[dst] = vc[src]
        T = sum(new)
        k = torch.empty(T, hkv, d, dtype=torch.bfloat16)
        v = torch.empty_like(k)
        q = torch.randn(T, hq, d, generator=torch.Generator().manual_seed(step)).to(torch.bfloat16)
        qsl = meta["query_start_loc"]
        for i, rid in enumerate(rids):
            for j, p in enumerate(range(meta["context_lens"][i], meta["seq_lens"][i])):
                kv = kv_of(seqs[rid][:p + 1])
                k[qsl[i] + j], v[qsl[i] + j] = kv[0], kv[1]
        kb, vb = oracle.write_kv(k, v, np.array(meta["slot_mapping"]), kc, vc)
        kc = torch.from_numpy(kb.view(np.int16)).view(torch.bfloat16)
        vc = torch.from_numpy(vb.view(np.int16)).view(torch.bfloat16)
        bt = np.array(meta["block_tables"], np.int32)
        out, lse = oracle.attention(q, kc, vc, bt, np.array(qsl), np.array(meta["context_lens"]),
                                    np.array(meta["seq_lens"]), 0.3)
        # dense reference: each request's own K/V arrays, contiguous blocks
        for i, rid in enumerate(rids):
            L = meta["seq_lens"][i]
            dk = torch.stack([kv_of(seqs[rid][:p + 1])[0] for p in range(L)])
            dv = torch.stack([kv_of(seqs[rid][:p + 1])[1] for p in range(L)])
            nblk = -(-L // bs)
            pad = nblk * bs - L
            dk = torch.cat([dk, torch.zeros(pad, hkv, d, dtype=torch.bfloat16)])
            dv = torch.cat([dv, torch.zeros(pad, hkv, d, dtype=torch.bfloat16)])
            dkc = dk.view(nblk, bs, hkv, d).transpose(1, 2).contiguous()
            dvc = dv.view(nblk, bs, hkv, d).transpose(1, 2).contiguous()
            rows = slice(qsl[i], qsl[i + 1])
            ro, rl = oracle.attention(q[rows], dkc, dvc, np.arange(nblk, dtype=np.int32)[None],
                                      np.array([0, qsl[i + 1] - qsl[i]]),
                                      np.array([meta["context_lens"][i]]), np.array([L]), 0.3)
            assert np.allclose(out[rows], ro, atol=1e-12) and np.allclose(lse[rows], rl, atol=1e-12)


# ---- the C++ manager against the model -------------------------------------------

def apply_cpp(bm, op):
    kind = op[0]
    try:
        if kind == "add":
            return OK, bm.add_request(op[1], op[2])
        if kind == "fork":
            bm.fork(op[1], op[2])
            return OK
        if kind == "free":
            bm.free_request(op[1])
            return OK
        if kind == "append":
            bm.append_tokens(op[1], op[2])
            return OK
        if kind == "schedule":
            res = bm.try_schedule(op[1], op[2], op[3], max_copies=4)
            if isinstance(res, int):
                return {PA_ERR_INVALID_ARG: INVALID, PA_ERR_WORKSPACE: NO_BLOCKS}[res], None
            return OK, {"block_tables": res["block_tables"].tolist(),
                        "query_start_loc": res["query_start_loc"].tolist(),
                        "context_lens": res["context_lens"].tolist(),
                        "seq_lens": res["seq_lens"].tolist(),
                        "slot_mapping": res["slot_mapping"].tolist(),
                        "copies": [tuple(c) for c in res["copies"].tolist()]}
        bm.add_request(-5, [])
        return OK
    except Exception as e:  # PaError
        code = getattr(e, "code", None)
        code = {PA_ERR_INVALID_ARG: INVALID}.get(code, code)
        return (code, 0) if kind in ("add", "bad") else code


@pytest.mark.parametrize("seed", range(8))
def test_cpp_block_manager_matches_the_model(seed):
    m = BlockManagerModel(24, 4)
    bm = BlockManager(24, 4)
    for i, op in enumerate(random_ops(100 + seed, n_ops=500, model=m)):
        want = apply_model(m, op)
        got = apply_cpp(bm, op)
        assert got == want, (i, op, got, want)
        assert bm.num_free_blocks == m.available(), (i, op)
        assert bm.num_cached_blocks == len(m.cache), (i, op)
        assert [bm.ref_count(b) for b in range(24)] == m.ref, (i, op)
        for rid, r in m.reqs.items():
            assert bm.blocks_of(rid) == r.table and bm.num_computed(rid) == r.computed
    bm.close()
