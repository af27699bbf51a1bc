"""Pins for the CPU oracle (no GPU).

The oracle is trusted only because it agrees with things other than itself:
  * brute force on tiny inputs (independent NumPy loops);
  * torch's scaled_dot_product_attention in float64 on the single-request
    case (a textbook library routine), with torch.logsumexp for the LSE;
  * closed forms (one key, zero query, identical keys);
  * the pages' worked examples (tests/golden/page_examples.json) as
    equivalences: 31/29/30 = 90 batched, 16+16+16 chunks = one-shot 48,
    a 15-token chunk after 16 cached, 107 tokens with 48 cached, shared
    block tables [3,7,11] / [3,7,5], 1+4 speculative rows = 5 decodes,
    cascade merge(prefix, suffix) = full attention;
  * the page's work count for chunked prefill (16^2*9 one-shot dense vs
    16^2*6 chunked), pinned on the oracle's own per-row mask.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_examples.json")))


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def randn_bf16(gen, *shape):
    return torch.randn(*shape, generator=gen).to(torch.bfloat16)


def make_pool(gen, num_blocks, hkv, bs, d):
    return randn_bf16(gen, num_blocks, hkv, bs, d), randn_bf16(gen, num_blocks, hkv, bs, d)


def place(pool_k, pool_v, table, keys, vals):
    """Test-side construction: put dense per-position K/V ([L, Hkv, d]) into
    the pool at the positions the block table names."""
    bs = pool_k.shape[2]
    for j in range(keys.shape[0]):
        pool_k[table[j // bs], :, j % bs] = keys[j]
        pool_v[table[j // bs], :, j % bs] = vals[j]


def meta(reqs):
    """reqs = [(ctx, n)] -> qsl, ctx, seq_lens (int32 tensors)."""
    qsl = [0]
    for _, n in reqs:
        qsl.append(qsl[-1] + n)
    return (torch.tensor(qsl, dtype=torch.int32),
            torch.tensor([c for c, _ in reqs], dtype=torch.int32),
            torch.tensor([c + n for c, n in reqs], dtype=torch.int32))


def tables_tensor(tables, width=None):
    width = width or max(len(t) for t in tables)
    bt = torch.full((len(tables), width), -1, dtype=torch.int32)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = torch.tensor(t, dtype=torch.int32)
    return bt


# ---------------------------------------------------------------------------
# 1. brute force on tiny inputs
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_oracle_matches_brute_force(seed):
    gen = torch.Generator().manual_seed(1000 + seed)
    hq, hkv, d, bs = 4, 2, 8, 4
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 4))
    reqs = []
    for _ in range(B):
        L = int(rng.integers(1, 41))
        n = int(rng.integers(1, L + 1))
        reqs.append((L - n, n))
    nblk = [math.ceil((c + n) / bs) for c, n in reqs]
    num_blocks = sum(nblk) + 3
    perm = torch.randperm(num_blocks, generator=gen).tolist()
    tables, cur = [], 0
    for k in nblk:
        tables.append(perm[cur:cur + k])
        cur += k
    kc, vc = make_pool(gen, num_blocks, hkv, bs, d)
    T = sum(n for _, n in reqs)
    q = randn_bf16(gen, T, hq, d)
    qsl, ctx, sl = meta(reqs)
    bt = tables_tensor(tables)
    scale = 0.37
    o1, l1 = oracle.attention(q, kc, vc, bt, qsl, ctx, sl, scale)
    o2, l2 = brute.attention(bits(q), bits(kc), bits(vc), bt.numpy(), qsl.numpy(), ctx.numpy(),
                             sl.numpy(), scale)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# 2. library special case: torch SDPA (float64) on one request
# ---------------------------------------------------------------------------

def sdpa_reference(q, keys, vals, ctx, scale, group):
    """q [n, Hq, d], keys/vals [L, Hkv, d] (float64) -> out [n, Hq, d], lse [n, Hq]."""
    n, L = q.shape[0], keys.shape[0]
    k = keys.repeat_interleave(group, dim=1).permute(1, 0, 2)   # [Hq, L, d]
    v = vals.repeat_interleave(group, dim=1).permute(1, 0, 2)
    qh = q.permute(1, 0, 2)                                      # [Hq, n, d]
    if ctx == 0:
        out = torch.nn.functional.scaled_dot_product_attention(qh, k, v, is_causal=True,
                                                               scale=scale)
    else:
        allowed = torch.arange(L)[None, :] <= (ctx + torch.arange(n))[:, None]
        out = torch.nn.functional.scaled_dot_product_attention(qh, k, v, attn_mask=allowed,
                                                               scale=scale)
    allowed = torch.arange(L)[None, :] <= (ctx + torch.arange(n))[:, None]
    scores = torch.matmul(qh, k.transpose(1, 2)) * scale
    scores = scores.masked_fill(~allowed, float("-inf"))
    lse = torch.logsumexp(scores, dim=-1)
    return out.permute(1, 0, 2).numpy(), lse.permute(1, 0).numpy()


@pytest.mark.parametrize("hq,hkv,ctx,n", [(2, 2, 0, 37), (8, 2, 0, 33), (6, 3, 21, 12),
                                          (4, 1, 5, 1)])
def test_oracle_matches_torch_sdpa(hq, hkv, ctx, n):
    gen = torch.Generator().manual_seed(77 + hq + ctx)
    d, bs = 16, 8
    L = ctx + n
    nb = math.ceil(L / bs)
    num_blocks = nb + 5
    table = torch.randperm(num_blocks, generator=gen)[:nb].tolist()
    kc, vc = make_pool(gen, num_blocks, hkv, bs, d)
    keys, vals = randn_bf16(gen, L, hkv, d), randn_bf16(gen, L, hkv, d)
    place(kc, vc, table, keys, vals)
    q = randn_bf16(gen, n, hq, d)
    qsl, c, sl = meta([(ctx, n)])
    scale = 1.0 / math.sqrt(d)
    o, l = oracle.attention(q, kc, vc, tables_tensor([table]), qsl, c, sl, scale)
    ro, rl = sdpa_reference(q.double(), keys.double(), vals.double(), ctx, scale, hq // hkv)
    np.testing.assert_allclose(o, ro, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, rl, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# 3. closed forms
# ---------------------------------------------------------------------------

def single_request(gen, L, n, hq=4, hkv=2, d=16, bs=4, q=None, keys=None, vals=None):
    nb = math.ceil(L / bs)
    table = torch.randperm(nb + 2, generator=gen)[:nb].tolist()
    kc, vc = make_pool(gen, nb + 2, hkv, bs, d)
    keys = randn_bf16(gen, L, hkv, d) if keys is None else keys
    vals = randn_bf16(gen, L, hkv, d) if vals is None else vals
    place(kc, vc, table, keys, vals)
    q = randn_bf16(gen, n, hq, d) if q is None else q
    qsl, c, sl = meta([(L - n, n)])
    return q, kc, vc, tables_tensor([table]), qsl, c, sl, keys, vals


def test_closed_form_single_key():
    gen = torch.Generator().manual_seed(5)
    q, kc, vc, bt, qsl, c, sl, keys, vals = single_request(gen, 1, 1)
    o, l = oracle.attention(q, kc, vc, bt, qsl, c, sl, 0.5)
    for h in range(4):
        np.testing.assert_array_equal(o[0, h], vals[0, h // 2].double().numpy())
        s = 0.5 * float((q[0, h].double() * keys[0, h // 2].double()).sum())
        assert abs(l[0, h] - s) < 1e-12


def test_closed_form_zero_query_is_mean_of_visible_values():
    gen = torch.Generator().manual_seed(6)
    L, n = 23, 7
    qz = torch.zeros(n, 4, 16, dtype=torch.bfloat16)
    q, kc, vc, bt, qsl, c, sl, keys, vals = single_request(gen, L, n, q=qz)
    o, l = oracle.attention(q, kc, vc, bt, qsl, c, sl, 0.25)
    for i in range(n):
        nvis = L - n + i + 1
        for h in range(4):
            want = vals[:nvis, h // 2].double().mean(0).numpy()
            np.testing.assert_allclose(o[i, h], want, rtol=0, atol=1e-12)
            assert abs(l[i, h] - math.log(nvis)) < 1e-12


def test_closed_form_identical_keys():
    gen = torch.Generator().manual_seed(7)
    L, n = 19, 4
    one = randn_bf16(gen, 1, 2, 16)
    keys = one.repeat(L, 1, 1)
    q, kc, vc, bt, qsl, c, sl, _, vals = single_request(gen, L, n, keys=keys)
    o, l = oracle.attention(q, kc, vc, bt, qsl, c, sl, 0.3)
    for i in range(n):
        nvis = L - n + i + 1
        for h in range(4):
            s = 0.3 * float((q[i, h].double() * one[0, h // 2].double()).sum())
            np.testing.assert_allclose(o[i, h], vals[:nvis, h // 2].double().mean(0).numpy(),
                                       rtol=0, atol=1e-12)
            assert abs(l[i, h] - (s + math.log(nvis))) < 1e-12


def test_rows_are_probability_weighted_averages():
    """With V = one-hot key index, o[i, h][j] is the softmax weight of key j:
    the weights are non-negative, sum to 1 and vanish on masked keys."""
    gen = torch.Generator().manual_seed(8)
    L, n, d = 16, 5, 16
    vals = torch.zeros(L, 2, d, dtype=torch.bfloat16)
    for j in range(L):
        vals[j, :, j] = 1.0
    q, kc, vc, bt, qsl, c, sl, _, _ = single_request(gen, L, n, vals=vals, d=d)
    o, _ = oracle.attention(q, kc, vc, bt, qsl, c, sl, 0.25)
    for i in range(n):
        nvis = L - n + i + 1
        assert np.all(o[i] >= 0)
        np.testing.assert_allclose(o[i].sum(-1), 1.0, atol=1e-12)
        assert np.all(o[i][:, nvis:] == 0)


# ---------------------------------------------------------------------------
# 4. the pages' worked examples, as equivalences
# ---------------------------------------------------------------------------

def test_concatenated_prefill_equals_separate_prefills():
    g = GOLDEN["concat_prefill"]
    assert sum(g["prompt_lens"]) == g["concatenated_tokens"]
    gen = torch.Generator().manual_seed(9)
    hq, hkv, d, bs = 4, 2, 64, 16
    lens = g["prompt_lens"]
    nbs = [math.ceil(x / bs) for x in lens]
    num_blocks = 32
    perm = torch.randperm(num_blocks, generator=gen).tolist()
    tables, cur = [], 0
    for k in nbs:
        tables.append(perm[cur:cur + k])
        cur += k
    kc, vc = make_pool(gen, num_blocks, hkv, bs, d)
    q = randn_bf16(gen, sum(lens), hq, d)
    qsl, c, sl = meta([(0, x) for x in lens])
    o, l = oracle.attention(q, kc, vc, tables_tensor(tables), qsl, c, sl, 0.125)
    assert o.shape[0] == g["concatenated_tokens"]
    for b, x in enumerate(lens):
        s = int(qsl[b])
        qb, cb, slb = meta([(0, x)])
        ob, lb = oracle.attention(q[s:s + x], kc, vc, tables_tensor([tables[b]]), qb, cb, slb,
                                  0.125)
        np.testing.assert_array_equal(o[s:s + x], ob)
        np.testing.assert_array_equal(l[s:s + x], lb)


def prompt_setup(gen, L, hq=8, hkv=2, d=32, bs=16):
    nb = math.ceil(L / bs)
    table = torch.randperm(nb + 4, generator=gen)[:nb].tolist()
    kc, vc = make_pool(gen, nb + 4, hkv, bs, d)
    q = randn_bf16(gen, L, hq, d)
    return q, kc, vc, table


def test_chunked_prefill_equals_one_shot():
    g = GOLDEN["chunked_prefill"]
    L, C = g["prompt_len"], g["chunk_len"]
    assert L == g["num_chunks"] * C
    gen = torch.Generator().manual_seed(10)
    q, kc, vc, table = prompt_setup(gen, L)
    bt = tables_tensor([table])
    o_all, l_all = oracle.attention(q, kc, vc, bt, *meta([(0, L)]), 0.2)
    for k in range(g["num_chunks"]):
        rows = slice(k * C, (k + 1) * C)
        ok, lk = oracle.attention(q[rows], kc, vc, bt, *meta([(k * C, C)]), 0.2)
        np.testing.assert_array_equal(ok, o_all[rows])
        np.testing.assert_array_equal(lk, l_all[rows])


def test_chunk_of_15_after_16_cached():
    g = GOLDEN["chunk_after_cache"]
    cached, n = g["cached_tokens"], g["chunk_len"]
    gen = torch.Generator().manual_seed(11)
    q, kc, vc, table = prompt_setup(gen, cached + n)
    bt = tables_tensor([table])
    o_all, l_all = oracle.attention(q, kc, vc, bt, *meta([(0, cached + n)]), 0.2)
    o, l = oracle.attention(q[cached:], kc, vc, bt, *meta([(cached, n)]), 0.2)
    np.testing.assert_array_equal(o, o_all[cached:])
    np.testing.assert_array_equal(l, l_all[cached:])


def test_prefix_hit_rows_equal_full_prefill_rows():
    g = GOLDEN["prefix_hit"]
    L, hit = g["prompt_len"], g["cached_tokens"]
    assert g["first_position_id"] == hit
    gen = torch.Generator().manual_seed(12)
    q, kc, vc, table = prompt_setup(gen, L)
    bt = tables_tensor([table])
    o_all, l_all = oracle.attention(q, kc, vc, bt, *meta([(0, L)]), 0.2)
    o, l, vis = oracle.attention(q[hit:], kc, vc, bt, *meta([(hit, L - hit)]), 0.2,
                                 return_visible=True)
    np.testing.assert_array_equal(o, o_all[hit:])
    np.testing.assert_array_equal(l, l_all[hit:])
    # the first new row sits at position 48: it sees 49 keys
    assert vis[0] == hit + 1 and vis[-1] == L


def test_shared_block_tables_read_identical_prefix():
    g = GOLDEN["shared_block_tables"]
    ta, tb = g["request_a"], g["request_b"]
    shared = g["shared_logical_blocks"]
    assert ta[:shared] == tb[:shared] and ta[shared] != tb[shared]
    gen = torch.Generator().manual_seed(13)
    bs, hq, hkv, d = 4, 4, 2, 16
    num_blocks = 12
    kc, vc = make_pool(gen, num_blocks, hkv, bs, d)
    L = len(ta) * bs
    q = randn_bf16(gen, L, hq, d)
    q2 = torch.cat([q, q])
    o, l = oracle.attention(q2, kc, vc, tables_tensor([ta, tb]), *meta([(0, L), (0, L)]), 0.25)
    cut = shared * bs
    np.testing.assert_array_equal(o[:cut], o[L:L + cut])
    np.testing.assert_array_equal(l[:cut], l[L:L + cut])
    assert np.abs(o[cut:L] - o[L + cut:]).max() > 1e-3


def test_spec_verify_rows_equal_sequential_decodes():
    g = GOLDEN["spec_verify"]
    n = g["tokens_in_one_pass"]
    assert n == 1 + g["draft_tokens"]
    gen = torch.Generator().manual_seed(14)
    ctx = 37
    q, kc, vc, table = prompt_setup(gen, ctx + n)
    bt = tables_tensor([table])
    o, l = oracle.attention(q[ctx:], kc, vc, bt, *meta([(ctx, n)]), 0.2)
    for i in range(n):
        oi, li = oracle.attention(q[ctx + i:ctx + i + 1], kc, vc, bt, *meta([(ctx + i, 1)]), 0.2)
        np.testing.assert_array_equal(oi[0], o[i])
        np.testing.assert_array_equal(li[0], l[i])


def test_cascade_merge_equals_full_attention():
    """[AI] §02.1: prefix state ⊕ suffix state = attention over prefix+suffix."""
    gen = torch.Generator().manual_seed(15)
    bs, hq, hkv, d = 4, 8, 2, 16
    P, R = 12, 3
    sfx = [5, 9, 1]
    pblocks = P // bs
    nb_total = pblocks + sum(math.ceil(s / bs) for s in sfx) + 2
    perm = torch.randperm(nb_total, generator=gen).tolist()
    prefix = perm[:pblocks]
    cur, full, own = pblocks, [], []
    for s in sfx:
        k = math.ceil(s / bs)
        own.append(perm[cur:cur + k])
        full.append(prefix + perm[cur:cur + k])
        cur += k
    kc, vc = make_pool(gen, nb_total, hkv, bs, d)
    q = randn_bf16(gen, R, hq, d)
    o_full, l_full = oracle.attention(q, kc, vc, tables_tensor(full),
                                      *meta([(P + s - 1, 1) for s in sfx]), 0.25)
    o_p, l_p = oracle.prefix_attention(q, kc, vc, torch.tensor(prefix, dtype=torch.int32), P,
                                       0.25)
    o_s, l_s = oracle.attention(q, kc, vc, tables_tensor(own), *meta([(s - 1, 1) for s in sfx]),
                                0.25)
    o_m, l_m = oracle.merge_states(o_p, l_p, o_s, l_s)
    np.testing.assert_allclose(o_m, o_full, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l_m, l_full, rtol=0, atol=1e-12)


def random_state(gen, n=6, h=3, d=8):
    o = torch.randn(n, h, d, generator=gen, dtype=torch.float64).numpy()
    l = (3 * torch.randn(n, h, generator=gen, dtype=torch.float64)).numpy()
    return o, l


def test_merge_is_commutative_associative_with_identity():
    gen = torch.Generator().manual_seed(16)
    a, b, c = random_state(gen), random_state(gen), random_state(gen)
    ab = oracle.merge_states(*a, *b)
    ba = oracle.merge_states(*b, *a)
    np.testing.assert_allclose(ab[0], ba[0], rtol=0, atol=1e-14)
    np.testing.assert_allclose(ab[1], ba[1], rtol=0, atol=1e-14)
    ab_c = oracle.merge_states(*ab, *c)
    a_bc = oracle.merge_states(*a, *oracle.merge_states(*b, *c))
    np.testing.assert_allclose(ab_c[0], a_bc[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(ab_c[1], a_bc[1], rtol=0, atol=1e-12)
    ident = (np.zeros_like(a[0]), np.full_like(a[1], -np.inf))
    ai = oracle.merge_states(*a, *ident)
    np.testing.assert_allclose(ai[0], a[0], rtol=0, atol=1e-15)
    np.testing.assert_array_equal(ai[1], a[1])
    ii = oracle.merge_states(*ident, *ident)
    assert np.all(ii[0] == 0) and np.all(np.isneginf(ii[1]))
    # a ⊕ a keeps the output and doubles the mass: lse + ln 2
    aa = oracle.merge_states(*a, *a)
    np.testing.assert_allclose(aa[0], a[0], rtol=0, atol=1e-14)
    np.testing.assert_allclose(aa[1], a[1] + math.log(2), rtol=0, atol=1e-14)


def test_merge_of_disjoint_key_sets_equals_union():
    """Split one request's keys in two halves by hand: the merge of the two
    halves' states (computed with numpy directly) equals the oracle's full
    row -- pins the merge weights against plain softmax algebra."""
    gen = torch.Generator().manual_seed(17)
    s = torch.randn(40, generator=gen, dtype=torch.float64).numpy()
    v = torch.randn(40, 8, generator=gen, dtype=torch.float64).numpy()

    def state(idx):
        w = np.exp(s[idx])
        return (w[:, None] * v[idx]).sum(0) / w.sum(), np.log(w.sum())

    oa, la = state(np.arange(0, 17))
    ob, lb = state(np.arange(17, 40))
    of, lf = state(np.arange(0, 40))
    om, lm = oracle.merge_states(oa[None, None], np.array([[la]]), ob[None, None],
                                 np.array([[lb]]))
    np.testing.assert_allclose(om[0, 0], of, rtol=0, atol=1e-13)
    assert abs(lm[0, 0] - lf) < 1e-13


# ---------------------------------------------------------------------------
# 5. the page's work count for chunked prefill, on the oracle's mask
# ---------------------------------------------------------------------------

def tiles_touched(visible, first_row, tile):
    """Count (q-tile, k-tile) pairs of size tile x tile holding at least one
    visible (row, key) pair, given each row's visible-key count."""
    touched = set()
    for r, nvis in enumerate(visible):
        row = first_row + r
        for kt in range((int(nvis) + tile - 1) // tile):
            touched.add((row // tile, kt))
    return len(touched)


def test_chunked_prefill_work_count():
    g = GOLDEN["chunked_prefill"]
    L, C = g["prompt_len"], g["chunk_len"]
    assert sum(g["chunk_work_terms"]) == C * C * g["chunked_work_in_16x16_units"]
    assert L * L == C * C * g["one_shot_work_in_16x16_units"]
    gen = torch.Generator().manual_seed(18)
    q, kc, vc, table = prompt_setup(gen, L)
    bt = tables_tensor([table])
    _, _, vis_all = oracle.attention(q, kc, vc, bt, *meta([(0, L)]), 0.2, return_visible=True)
    chunk_terms, pairs_chunked, tiles_chunked = [], 0, 0
    for k in range(g["num_chunks"]):
        _, _, vis = oracle.attention(q[k * C:(k + 1) * C], kc, vc, bt, *meta([(k * C, C)]), 0.2,
                                     return_visible=True)
        # the chunk's score block is C rows x (keys up to its last row)
        chunk_terms.append(C * int(vis.max()))
        pairs_chunked += int(vis.sum())
        tiles_chunked += tiles_touched(vis, k * C, C)
    assert chunk_terms == g["chunk_work_terms"]
    assert pairs_chunked == int(vis_all.sum()) == L * (L + 1) // 2
    assert tiles_chunked == tiles_touched(vis_all, 0, C) == g["chunked_work_in_16x16_units"]


# ---------------------------------------------------------------------------
# 6. write path
# ---------------------------------------------------------------------------

def test_write_kv_places_rows_and_skips_padding():
    gen = torch.Generator().manual_seed(19)
    nb, hkv, bs, d = 6, 2, 4, 8
    kc, vc = make_pool(gen, nb, hkv, bs, d)
    T = 7
    k, v = randn_bf16(gen, T, hkv, d), randn_bf16(gen, T, hkv, d)
    slots = torch.tensor([5, 0, -1, 23, 9, 12, -1], dtype=torch.int64)
    nk, nv = oracle.write_kv(k, v, slots, kc, vc)
    kb, vb, kcb, vcb = bits(k), bits(v), bits(kc), bits(vc)
    expect_k, expect_v = kcb.copy(), vcb.copy()
    for t, s in enumerate(slots.tolist()):
        if s >= 0:
            expect_k[s // bs, :, s % bs] = kb[t]
            expect_v[s // bs, :, s % bs] = vb[t]
    np.testing.assert_array_equal(nk, expect_k)
    np.testing.assert_array_equal(nv, expect_v)
    # untouched slots keep their old bits
    untouched = np.ones((nb, bs), bool)
    for s in slots.tolist():
        if s >= 0:
            untouched[s // bs, s % bs] = False
    for blk, off in zip(*np.nonzero(untouched)):
        np.testing.assert_array_equal(nk[blk, :, off], kcb[blk, :, off])


def test_oracle_rejects_inconsistent_metadata():
    gen = torch.Generator().manual_seed(20)
    q, kc, vc, table = prompt_setup(gen, 20)
    qsl, c, sl = meta([(4, 16)])
    sl = sl + 1   # seq_len != context + q_len
    with pytest.raises(ValueError):
        oracle.attention(q[4:], kc, vc, tables_tensor([table]), qsl, c, sl, 0.2)
