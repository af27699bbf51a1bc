"""Seeded synthetic inputs for one continuous-batching attention step.

This module only draws random numbers and lays out metadata the way a
scheduler and block manager hand them to the attention step; it holds none of
the attention arithmetic.  Both the CUDA path and the CPU oracle consume what
it produces.

Shapes follow the scenarios on the pages:
  * tiny prefill -- 31/29/30-token prompts concatenated into one 90-token
    batch ("vLLM中如何实现大模型推理加速技术？", opening example);
  * chunked prefill (48 = 16+16+16) + prefix-cache hit (107 tokens, 48 cached)
    + decode rows (same page, chunked-prefill and prefix-caching sections);
  * decode-heavy, mixed continuous-batching and cascade shared-prefix steps
    sized as stated in the design notes.

Recipe: generator = torch.Generator('cpu').manual_seed(seed); every value is
an fp32 N(0,1) draw rounded to bf16 (round-to-nearest-even); physical blocks
are handed out from a seeded permutation of the pool, which is sized to the
blocks needed + 10% unless stated.  Every pool slot starts with an N(0,1)
value, so a read of a wrong slot shows up as a wrong result.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence, Tuple

import torch

SEED_BASE = 284000


@dataclasses.dataclass
class Step:
    """One step's inputs (CPU tensors)."""
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    scale: float
    q: torch.Tensor              # bf16 [T, Hq, d]
    k: torch.Tensor              # bf16 [T, Hkv, d]   new keys of this step
    v: torch.Tensor              # bf16 [T, Hkv, d]
    slot_mapping: torch.Tensor   # int64 [T]
    block_tables: torch.Tensor   # int32 [B, max_blocks]
    query_start_loc: torch.Tensor  # int32 [B+1]
    context_lens: torch.Tensor   # int32 [B]
    seq_lens: torch.Tensor       # int32 [B]
    # cascade layout (optional): shared prefix blocks and suffix-only metadata
    prefix_blocks: Optional[torch.Tensor] = None   # int32 [P / bs]
    prefix_len: int = 0
    suffix_block_tables: Optional[torch.Tensor] = None
    suffix_context_lens: Optional[torch.Tensor] = None
    suffix_seq_lens: Optional[torch.Tensor] = None
    label: str = ""

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_q_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def q_lens(self) -> torch.Tensor:
        return self.query_start_loc[1:] - self.query_start_loc[:-1]


@dataclasses.dataclass
class Pool:
    """The paged KV pool: bf16 [num_blocks, Hkv, bs, d] for K and for V."""
    k_cache: torch.Tensor
    v_cache: torch.Tensor

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])


def _randn_bf16(shape, gen: torch.Generator, chunk: int = 1 << 24) -> torch.Tensor:
    """N(0,1) fp32 draws rounded to bf16, generated in fixed-size pieces so
    large pools do not need an fp32 copy of the whole tensor."""
    numel = int(math.prod(shape))
    out = torch.empty(numel, dtype=torch.bfloat16)
    for s in range(0, numel, chunk):
        e = min(numel, s + chunk)
        out[s:e] = torch.randn(e - s, generator=gen, dtype=torch.float32).to(torch.bfloat16)
    return out.view(*shape)


def _uniform_int(lo: int, hi: int, n: int, gen: torch.Generator) -> List[int]:
    """n integers uniform in [lo, hi] inclusive."""
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]


def _blocks_for(length: int, bs: int) -> int:
    return (length + bs - 1) // bs


@dataclasses.dataclass
class Fp8Pool:
    """An e4m3 KV pool: uint8 codes [num_blocks, Hkv, bs, d] for K and V and
    one fp32 scale per kv head for each (an element is code value x scale)."""
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    k_scale: torch.Tensor
    v_scale: torch.Tensor

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])


def _random_e4m3_codes(shape, gen: torch.Generator) -> torch.Tensor:
    """Finite e4m3 codes with a random sign, an exponent field uniform in
    1..11 (magnitudes 2^-6 .. 30) and a uniform mantissa: log-uniform values,
    no NaN code."""
    sign = torch.randint(0, 2, shape, generator=gen, dtype=torch.int32) << 7
    e = torch.randint(1, 12, shape, generator=gen, dtype=torch.int32) << 3
    m = torch.randint(0, 8, shape, generator=gen, dtype=torch.int32)
    return (sign | e | m).to(torch.uint8)


def fp8_pool_like(pool: Pool, seed: int) -> Fp8Pool:
    """An e4m3 pool with the shape of `pool`: seeded random codes and per-kv-head
    scales uniform in [1/24, 1/12] (so new bf16 N(0,1) tokens divided by the
    scale stay far inside the e4m3 range)."""
    gen = torch.Generator().manual_seed(seed)
    shape = tuple(pool.k_cache.shape)
    hkv = shape[1]
    kc = _random_e4m3_codes(shape, gen)
    vc = _random_e4m3_codes(shape, gen)
    ks = 1.0 / torch.empty(hkv).uniform_(12.0, 24.0, generator=gen)
    vs = 1.0 / torch.empty(hkv).uniform_(12.0, 24.0, generator=gen)
    return Fp8Pool(kc, vc, ks.float(), vs.float())


def make_pool(num_blocks: int, num_kv_heads: int, block_size: int, head_dim: int,
              gen: torch.Generator) -> Pool:
    shape = (num_blocks, num_kv_heads, block_size, head_dim)
    return Pool(_randn_bf16(shape, gen), _randn_bf16(shape, gen))


def build_step(requests: Sequence[Tuple[int, int]], *, num_q_heads: int, num_kv_heads: int,
               head_dim: int, block_size: int, gen: torch.Generator,
               tables: Sequence[Sequence[int]], max_blocks: Optional[int] = None,
               label: str = "") -> Step:
    """Draw q/k/v for the new tokens of `requests` = [(context_len, q_len)] and
    lay out the metadata.  tables[b] lists request b's physical blocks in
    logical order (at least ceil((ctx+n)/bs) of them)."""
    B = len(requests)
    qlens = [n for _, n in requests]
    T = sum(qlens)
    qsl = [0]
    for n in qlens:
        qsl.append(qsl[-1] + n)
    if max_blocks is None:
        max_blocks = max([len(t) for t in tables] + [1])
    bt = torch.full((B, max_blocks), -1, dtype=torch.int32)
    for b, t in enumerate(tables):
        bt[b, :len(t)] = torch.tensor(list(t), dtype=torch.int32)
    slots = []
    for b, (ctx, n) in enumerate(requests):
        for i in range(n):
            pos = ctx + i
            slots.append(int(tables[b][pos // block_size]) * block_size + pos % block_size)
    q = _randn_bf16((T, num_q_heads, head_dim), gen)
    k = _randn_bf16((T, num_kv_heads, head_dim), gen)
    v = _randn_bf16((T, num_kv_heads, head_dim), gen)
    return Step(num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                block_size=block_size, scale=1.0 / math.sqrt(head_dim), q=q, k=k, v=v,
                slot_mapping=torch.tensor(slots, dtype=torch.int64),
                block_tables=bt,
                query_start_loc=torch.tensor(qsl, dtype=torch.int32),
                context_lens=torch.tensor([c for c, _ in requests], dtype=torch.int32),
                seq_lens=torch.tensor([c + n for c, n in requests], dtype=torch.int32),
                label=label)


def _assign_tables(requests, block_size, gen, slack=0.10, num_blocks=None,
                   prefix_blocks=0):
    """Hand out physical blocks from a seeded permutation of the pool.
    The first `prefix_blocks` permuted blocks are shared by every request."""
    need = [_blocks_for(c + n, block_size) - prefix_blocks for c, n in requests]
    total = prefix_blocks + sum(need)
    if num_blocks is None:
        num_blocks = max(1, math.ceil(total * (1.0 + slack)))
    assert num_blocks >= total
    perm = [int(x) for x in torch.randperm(num_blocks, generator=gen)]
    prefix = perm[:prefix_blocks]
    cursor = prefix_blocks
    tables = []
    for n_own in need:
        tables.append(prefix + perm[cursor:cursor + n_own])
        cursor += n_own
    return num_blocks, tables, prefix


# ---------------------------------------------------------------------------
# The five scenarios
# ---------------------------------------------------------------------------

def tiny_prefill(seed: int = SEED_BASE + 0):
    """3 prompts (31, 29, 30 tokens) as one 90-token batch, empty cache.
    4 q / 2 kv heads, d=64, bs=16, pool of 32 blocks; each request takes the
    next 2 entries of a seeded permutation of the pool."""
    gen = torch.Generator().manual_seed(seed)
    reqs = [(0, 31), (0, 29), (0, 30)]
    nb, tables, _ = _assign_tables(reqs, 16, gen, num_blocks=32)
    pool = make_pool(nb, 2, 16, 64, gen)
    step = build_step(reqs, num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=16,
                      gen=gen, tables=tables, label="tiny_prefill")
    return pool, [step]


def chunked_prefix_decode(seed: int = SEED_BASE + 1, num_decode: int = 4):
    """Three steps on one pool (8 q / 2 kv heads, d=128, bs=16):
      1. chunk 1 of a 48-token prompt (ctx 0, 16 tokens);
      2. chunk 2 (ctx 16, 16 tokens);
      3. chunk 3 (ctx 32, 16 tokens) + a 107-token prompt whose first 48 tokens
         hit the cache (its table starts with the 48-token prompt's 3 blocks;
         59 new tokens at positions 48..106) + decode rows with seq_len
         uniform in [60, 300]."""
    gen = torch.Generator().manual_seed(seed)
    bs, hq, hkv, d = 16, 8, 2, 128
    dec_lens = _uniform_int(60, 300, num_decode, gen)
    reqs_all = [(0, 48), (0, 107)] + [(L - 1, 1) for L in dec_lens]
    need = [_blocks_for(c + n, bs) for c, n in reqs_all]
    need[1] -= 3  # the hit request owns only the blocks after the shared prefix
    total = sum(need)
    nb = math.ceil(total * 1.1)
    perm = [int(x) for x in torch.randperm(nb, generator=gen)]
    cur = 0
    own = []
    for k in need:
        own.append(perm[cur:cur + k])
        cur += k
    table_a = own[0]
    table_b = table_a[:3] + own[1]
    dec_tables = own[2:]
    pool = make_pool(nb, hkv, bs, d, gen)
    mb = max(len(t) for t in [table_a, table_b] + dec_tables)
    kw = dict(num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs, gen=gen,
              max_blocks=mb)
    s1 = build_step([(0, 16)], tables=[table_a], label="chunk1", **kw)
    s2 = build_step([(16, 16)], tables=[table_a], label="chunk2", **kw)
    s3 = build_step([(32, 16), (48, 59)] + [(L - 1, 1) for L in dec_lens],
                    tables=[table_a, table_b] + dec_tables, label="chunk3+hit+decode", **kw)
    return pool, [s1, s2, s3]


def decode_heavy(seed: int = SEED_BASE + 2, num_seqs: int = 256, lo: int = 512,
                 hi: int = 4096, num_q_heads: int = 32, num_kv_heads: int = 8,
                 head_dim: int = 128, block_size: int = 16):
    """num_seqs decode rows (q_len 1) with seq_len uniform in [lo, hi]."""
    gen = torch.Generator().manual_seed(seed)
    lens = _uniform_int(lo, hi, num_seqs, gen)
    reqs = [(L - 1, 1) for L in lens]
    nb, tables, _ = _assign_tables(reqs, block_size, gen)
    pool = make_pool(nb, num_kv_heads, block_size, head_dim, gen)
    step = build_step(reqs, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                      head_dim=head_dim, block_size=block_size, gen=gen, tables=tables,
                      label=f"decode_heavy_{num_seqs}x[{lo},{hi}]")
    return pool, [step]


def _mixed_requests(gen, num_chunks, chunk_len, chunk_ctx, num_decode, decode_len, num_spec,
                    spec_len, spec_ctx):
    dec = _uniform_int(decode_len[0], decode_len[1], num_decode, gen)
    spec = _uniform_int(spec_ctx[0], spec_ctx[1], num_spec, gen)
    chunks = _uniform_int(chunk_ctx[0], chunk_ctx[1], num_chunks, gen)
    return ([(L - 1, 1) for L in dec] + [(c, spec_len) for c in spec]
            + [(c, chunk_len) for c in chunks])


def mixed_step_requests(seed: int = SEED_BASE + 3, num_chunks: int = 8, chunk_len: int = 512,
                        chunk_ctx: Tuple[int, int] = (0, 8192), num_decode: int = 192,
                        decode_len: Tuple[int, int] = (256, 8192), num_spec: int = 32,
                        spec_len: int = 5, spec_ctx: Tuple[int, int] = (256, 8192)):
    """The (context_len, q_len) list of mixed_step(seed) without building its
    pool: the same draws, in the same order."""
    gen = torch.Generator().manual_seed(seed)
    return _mixed_requests(gen, num_chunks, chunk_len, chunk_ctx, num_decode, decode_len,
                           num_spec, spec_len, spec_ctx)


def from_requests(requests: Sequence[Tuple[int, int]], seed: int, num_q_heads: int = 32,
                  num_kv_heads: int = 8, head_dim: int = 128, block_size: int = 16,
                  label: str = "requests"):
    """A pool and one step for a given [(context_len, q_len)] list, e.g. the
    requests a router sent to one replica: blocks from a seeded permutation
    of a pool sized to the blocks needed + 10 %, then q/k/v."""
    gen = torch.Generator().manual_seed(seed)
    reqs = list(requests)
    nb, tables, _ = _assign_tables(reqs, block_size, gen)
    pool = make_pool(nb, num_kv_heads, block_size, head_dim, gen)
    step = build_step(reqs, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                      head_dim=head_dim, block_size=block_size, gen=gen, tables=tables,
                      label=label)
    return pool, [step]


def mixed_step(seed: int = SEED_BASE + 3, num_chunks: int = 8, chunk_len: int = 512,
               chunk_ctx: Tuple[int, int] = (0, 8192), num_decode: int = 192,
               decode_len: Tuple[int, int] = (256, 8192), num_spec: int = 32,
               spec_len: int = 5, spec_ctx: Tuple[int, int] = (256, 8192),
               num_q_heads: int = 32, num_kv_heads: int = 8, head_dim: int = 128,
               block_size: int = 16):
    """One mixed continuous-batching step: decode rows first, then
    speculative-verify rows (1 + 4 drafts), then chunked-prefill chunks."""
    gen = torch.Generator().manual_seed(seed)
    reqs = _mixed_requests(gen, num_chunks, chunk_len, chunk_ctx, num_decode, decode_len,
                           num_spec, spec_len, spec_ctx)
    nb, tables, _ = _assign_tables(reqs, block_size, gen)
    pool = make_pool(nb, num_kv_heads, block_size, head_dim, gen)
    step = build_step(reqs, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                      head_dim=head_dim, block_size=block_size, gen=gen, tables=tables,
                      label=f"mixed_{num_chunks}x{chunk_len}+{num_decode}dec+{num_spec}spec")
    return pool, [step]


def cascade(seed: int = SEED_BASE + 4, num_seqs: int = 64, prefix_len: int = 8192,
            suffix: Tuple[int, int] = (128, 1024), num_q_heads: int = 32,
            num_kv_heads: int = 8, head_dim: int = 128, block_size: int = 16):
    """Cascade shared-prefix decode: every request's table starts with the same
    prefix_len / bs physical blocks, followed by its own suffix blocks; the
    new decode token is the last suffix token.  Also returns suffix-only
    metadata (tables without the prefix, lengths counted within the suffix)."""
    assert prefix_len % block_size == 0
    gen = torch.Generator().manual_seed(seed)
    sfx = _uniform_int(suffix[0], suffix[1], num_seqs, gen)
    reqs = [(prefix_len + s - 1, 1) for s in sfx]
    pblocks = prefix_len // block_size
    nb, tables, prefix = _assign_tables(reqs, block_size, gen, prefix_blocks=pblocks)
    pool = make_pool(nb, num_kv_heads, block_size, head_dim, gen)
    step = build_step(reqs, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                      head_dim=head_dim, block_size=block_size, gen=gen, tables=tables,
                      label=f"cascade_{num_seqs}x({prefix_len}+[{suffix[0]},{suffix[1]}])")
    smax = max(_blocks_for(s, block_size) for s in sfx)
    st = torch.full((num_seqs, smax), -1, dtype=torch.int32)
    for b, t in enumerate(tables):
        own = t[pblocks:]
        st[b, :len(own)] = torch.tensor(own, dtype=torch.int32)
    step.prefix_blocks = torch.tensor(prefix, dtype=torch.int32)
    step.prefix_len = prefix_len
    step.suffix_block_tables = st
    step.suffix_context_lens = torch.tensor([s - 1 for s in sfx], dtype=torch.int32)
    step.suffix_seq_lens = torch.tensor(sfx, dtype=torch.int32)
    return pool, [step]


def graph_replay_pair(seed: int = SEED_BASE + 5, num_decode: int = 12, num_spec: int = 2,
                      spec_len: int = 5, chunk_len: int = 40, ctx: Tuple[int, int] = (16, 1500),
                      num_q_heads: int = 8, num_kv_heads: int = 2, head_dim: int = 128,
                      block_size: int = 16):
    """Two steps with identical shapes on one pool -- the same request count,
    q_lens (decode rows, speculative-verify rows, one chunk long enough for
    the tensor-core path) and block-table width -- but their own context
    lengths, blocks and values: one step is captured in a CUDA graph, the
    other is replayed through it."""
    gen = torch.Generator().manual_seed(seed)

    def draw():
        dec = _uniform_int(ctx[0], ctx[1], num_decode, gen)
        spec = _uniform_int(ctx[0], ctx[1], num_spec, gen)
        chunk = _uniform_int(0, ctx[1], 1, gen)
        return ([(L - 1, 1) for L in dec] + [(c, spec_len) for c in spec]
                + [(c, chunk_len) for c in chunk])

    ra, rb = draw(), draw()
    nb, tables, _ = _assign_tables(ra + rb, block_size, gen)
    pool = make_pool(nb, num_kv_heads, block_size, head_dim, gen)
    mb = max(len(t) for t in tables)
    kw = dict(num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
              block_size=block_size, gen=gen, max_blocks=mb)
    sa = build_step(ra, tables=tables[:len(ra)], label="graph_capture", **kw)
    sb = build_step(rb, tables=tables[len(ra):], label="graph_replay", **kw)
    return pool, [sa, sb]


CONFIGS = {
    "tiny_prefill": tiny_prefill,
    "chunked_prefix_decode": chunked_prefix_decode,
    "decode_heavy": decode_heavy,
    "mixed_step": mixed_step,
    "cascade": cascade,
}


def subset(step: Step, idx: Sequence[int]) -> Step:
    """The sub-batch made of requests `idx` (same pool), e.g. to let the oracle
    check sampled requests of a large step one by one."""
    idx = list(idx)
    qsl = step.query_start_loc
    rows = torch.cat([torch.arange(int(qsl[b]), int(qsl[b + 1])) for b in idx]) \
        if idx else torch.zeros(0, dtype=torch.long)
    lens = [int(qsl[b + 1] - qsl[b]) for b in idx]
    nqsl = [0]
    for n in lens:
        nqsl.append(nqsl[-1] + n)
    return dataclasses.replace(
        step, q=step.q[rows].contiguous(), k=step.k[rows].contiguous(),
        v=step.v[rows].contiguous(), slot_mapping=step.slot_mapping[rows].contiguous(),
        block_tables=step.block_tables[idx].contiguous(),
        query_start_loc=torch.tensor(nqsl, dtype=torch.int32),
        context_lens=step.context_lens[idx].contiguous(),
        seq_lens=step.seq_lens[idx].contiguous(),
        suffix_block_tables=(None if step.suffix_block_tables is None
                             else step.suffix_block_tables[idx].contiguous()),
        suffix_context_lens=(None if step.suffix_context_lens is None
                             else step.suffix_context_lens[idx].contiguous()),
        suffix_seq_lens=(None if step.suffix_seq_lens is None
                         else step.suffix_seq_lens[idx].contiguous()),
        label=step.label + f"[subset {len(idx)}]")
