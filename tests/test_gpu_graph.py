"""A whole step (pa_write_kv + pa_attention) captured once in a CUDA graph and
replayed on new metadata.  Planning runs on the device, so nothing the host
passes depends on the metadata's contents: a graph captured for one step of
a given shape serves every later step of that shape, with the inputs copied
into the captured buffers in place."""
import dataclasses

import numpy as np
import pytest
import torch

import paged_kv_cache_284_gb300 as pk
from paged_kv_cache_284_gb300 import workloads
from gpu_helpers import (DEV, assert_attention_close, assert_status_clean, bits, oracle_attend,
                         oracle_write)

pytestmark = pytest.mark.gpu


class StaticStep:
    """Device buffers of one step's shape; the graph reads and writes these."""

    def __init__(self, step, kc, vc):
        self.kc, self.vc = kc, vc
        self.t = {name: getattr(step, name).to(DEV).clone() for name in
                  ("q", "k", "v", "slot_mapping", "block_tables", "query_start_loc",
                   "context_lens", "seq_lens")}
        self.scale = step.scale
        self.out = torch.empty_like(self.t["q"])
        self.lse = torch.empty(self.t["q"].shape[:2], dtype=torch.float32, device=DEV)
        self.ws = pk.alloc_workspace(pk.workspace_size(step.num_seqs, step.num_q_tokens,
                                                       step.num_q_heads, step.num_kv_heads,
                                                       step.head_dim), DEV)

    def load(self, step):
        for name, t in self.t.items():
            t.copy_(getattr(step, name))

    def run(self):
        t = self.t
        pk.pa_write_kv(t["k"], t["v"], t["slot_mapping"], self.kc, self.vc)
        pk.pa_attention(t["q"], self.kc, self.vc, t["block_tables"], t["query_start_loc"],
                        t["context_lens"], t["seq_lens"], self.scale, self.out, self.lse,
                        workspace=self.ws)


def test_graph_replay_on_new_metadata():
    pool, (sa, sb) = workloads.graph_replay_pair()
    kc, vc = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    st = StaticStep(sa, kc, vc)

    # eager reference for step A, then capture (warm-up on a side stream first,
    # as torch's graph capture wants)
    st.run()
    torch.cuda.synchronize()
    eager_out, eager_lse = st.out.clone(), st.lse.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        st.run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st.run()
    torch.cuda.synchronize()

    # replay on A: same result as the eager call, bit for bit
    st.out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(bits(st.out), bits(eager_out))
    assert torch.equal(st.lse, eager_lse)

    # replay on B: new contexts, tables, slots and values through the same graph
    kb, vb = oracle_write(sa, bits(pool.k_cache), bits(pool.v_cache))
    st.load(sb)
    st.out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    kb, vb = oracle_write(sb, kb, vb)
    assert np.array_equal(bits(kc), kb) and np.array_equal(bits(vc), vb)
    ref_o, ref_l = oracle_attend(sb, kb, vb)
    assert_attention_close(st.out, st.lse, ref_o, ref_l, "graph replay on new metadata")

    # and back to A's metadata (its K/V are still in the cache)
    st.load(sa)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(bits(st.out), bits(eager_out))
    assert_status_clean()


def padded(step, n_seqs, n_tokens):
    """`step` padded to n_seqs requests and n_tokens tokens: the extra
    requests are empty (q_len 0, context 0, seq_len 0, table rows naming
    block 0) and the extra tokens belong to no request (slot -1: nothing is
    written for them)."""
    T, B = step.num_q_tokens, step.num_seqs

    def grow(t, n, fill=0):
        out = torch.full((n,) + tuple(t.shape[1:]), fill, dtype=t.dtype)
        out[:t.shape[0]] = t
        return out

    bt = torch.zeros((n_seqs, step.block_tables.shape[1]), dtype=torch.int32)
    bt[:B] = step.block_tables
    qsl = torch.full((n_seqs + 1,), T, dtype=torch.int32)
    qsl[:B + 1] = step.query_start_loc
    return dataclasses.replace(
        step, q=grow(step.q, n_tokens), k=grow(step.k, n_tokens), v=grow(step.v, n_tokens),
        slot_mapping=grow(step.slot_mapping, n_tokens, -1), block_tables=bt,
        query_start_loc=qsl, context_lens=grow(step.context_lens, n_seqs),
        seq_lens=grow(step.seq_lens, n_seqs))


def test_one_graph_serves_every_decode_batch_up_to_its_size():
    """One write + attention step captured at 64 decode requests replays
    batches of 1, 7, 33 and 64 rows: each smaller batch is padded with empty
    requests, and each replay is compared with the oracle on that batch; the
    padding rows of out are left untouched."""
    N = 64
    pool, (full,) = workloads.decode_heavy(seed=284095, num_seqs=N, lo=16, hi=1500,
                                           num_q_heads=8, num_kv_heads=2)
    kc, vc = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    st = StaticStep(full, kc, vc)
    st.run()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        st.run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st.run()
    torch.cuda.synchronize()
    kb, vb = oracle_write(full, bits(pool.k_cache), bits(pool.v_cache))
    for b in (1, 7, 33, N):
        step = workloads.subset(full, range(b))
        st.load(padded(step, N, N))
        st.out.fill_(float("nan"))
        st.lse.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        T = step.num_q_tokens
        ref_o, ref_l = oracle_attend(step, kb, vb)
        assert_attention_close(st.out[:T], st.lse[:T], ref_o, ref_l, f"graph replay, batch {b}")
        assert torch.isnan(st.out[T:].float()).all() and torch.isnan(st.lse[T:]).all()
    assert np.array_equal(bits(kc), kb) and np.array_equal(bits(vc), vb)
    assert_status_clean()
