"""The host block manager driving the GPU path: a few serving steps of
requests with shared prefixes, a fork, chunked prefill and decode.  Each
step the manager's metadata goes to the device as is: its copy-on-write
copies are applied to the pool, the new K/V are written through its slot
mapping, and attention reads through its block tables; the oracle does the
same on the CPU and the results are compared."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_284_gb300 as pk
from paged_kv_cache_284_gb300.blocks import BlockManager
from gpu_helpers import DEV, assert_attention_close, assert_status_clean, bits

pytestmark = pytest.mark.gpu


def test_block_manager_steps_on_the_gpu():
    hq, hkv, d, bs, nb = 8, 2, 128, 16, 96
    gen = torch.Generator().manual_seed(284900)
    kc = torch.randn(nb, hkv, bs, d, generator=gen).to(torch.bfloat16).to(DEV)
    vc = torch.randn(nb, hkv, bs, d, generator=gen).to(torch.bfloat16).to(DEV)
    kb, vb = bits(kc), bits(vc)
    bm = BlockManager(nb, bs)
    system = list(range(300, 348))                       # a 48-token shared opening
    prompts = {0: system + list(range(10, 30)), 1: system + list(range(40, 71)),
               2: list(range(900, 937))}
    for rid, p in prompts.items():
        bm.add_request(rid, p)
    known = {rid: len(p) for rid, p in prompts.items()}   # tokens in each sequence
    cached_3 = None
    rng = np.random.default_rng(5)
    for step in range(8):
        if step == 2:                                    # hits the 48-token opening
            p3 = system + list(range(60, 75))
            cached_3 = bm.add_request(3, p3)
            known[3] = len(p3)
        if step == 3:                                    # shares 1's blocks, then diverges
            bm.fork(1, 4)
            known[4] = known[1]
        final_ids, final_new = [], []
        for rid in sorted(known):
            comp = bm.num_computed(rid)
            if comp < known[rid]:                        # prefill, 24-token chunks
                n = min(24, known[rid] - comp)
            else:                                        # decode: one new token
                bm.append_tokens(rid, [int(rng.integers(0, 1000))])
                known[rid] += 1
                n = 1
            final_ids.append(rid)
            final_new.append(n)
        meta = bm.schedule(final_ids, final_new, max_blocks_per_seq=12)
        for src, dst in meta["copies"]:
            kc[dst] = kc[src]
            vc[dst] = vc[src]
            kb[dst], vb[dst] = kb[src].copy(), vb[src].copy()
        T = int(sum(final_new))
        k = torch.randn(T, hkv, d, generator=gen).to(torch.bfloat16)
        v = torch.randn(T, hkv, d, generator=gen).to(torch.bfloat16)
        q = torch.randn(T, hq, d, generator=gen).to(torch.bfloat16)
        slots = torch.from_numpy(meta["slot_mapping"])
        pk.pa_write_kv(k.to(DEV), v.to(DEV), slots.to(DEV), kc, vc)
        kb, vb = oracle.write_kv(k, v, slots, kb, vb)
        dm = {n: torch.from_numpy(meta[n]).to(DEV) for n in
              ("block_tables", "query_start_loc", "context_lens", "seq_lens")}
        out = torch.full((T, hq, d), float("nan"), dtype=torch.bfloat16, device=DEV)
        lse = torch.full((T, hq), float("nan"), dtype=torch.float32, device=DEV)
        pk.pa_attention(q.to(DEV), kc, vc, dm["block_tables"], dm["query_start_loc"],
                        dm["context_lens"], dm["seq_lens"], 0.088, out, lse)
        torch.cuda.synchronize()
        assert np.array_equal(bits(kc), kb) and np.array_equal(bits(vc), vb)
        ref_o, ref_l = oracle.attention(q, kb, vb, meta["block_tables"], meta["query_start_loc"],
                                        meta["context_lens"], meta["seq_lens"], 0.088)
        assert_attention_close(out, lse, ref_o, ref_l, f"serving step {step}")
    assert cached_3 == 48
    assert_status_clean()
    bm.close()
