"""A whole step (pa_write_kv + pa_attention) captured once in a CUDA graph and
replayed on new metadata.  Planning runs on the device, so nothing the host
passes depends on the metadata's contents: a graph captured for one step of
a given shape serves every later step of that shape, with the inputs copied
into the captured buffers in place."""
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
