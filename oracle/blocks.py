"""Plain model of the paged-KV block manager with a prefix cache -- TEST
INFRASTRUCTURE ONLY (the tests compare the C++ block manager with it; the
product never imports it).

Rules, from "11. 推理加速(一):vLLM 原理" (chuoer47.github.io):
  §11.2 fixed-size blocks; per-request block table (logical -> physical);
        physical blocks need not be contiguous; a physical block is taken
        only when the request's tokens reach it; requests with the same
        prefix share physical blocks ([3,7,11] and [3,7,5]); a shared block
        that would be written is copied first (copy-on-write).
  §11.4 every full block is known by its token ids; a new request references
        cached blocks (ref_count += 1) instead of computing them again.
Readings where the page is silent (the same ones the C++ code takes):
  * a block's identity is the whole token prefix up to its end (its K/V
    depends on every earlier token); only full blocks are cached; here the
    identity is the prefix itself, as a tuple -- no hashing at all;
  * matching runs from block 0 and stops at the first miss, and never covers
    the prompt's last token;
  * a new block is the lowest-numbered free one, else the cached,
    unreferenced block released longest ago (evicted: it stops matching);
    a finished request releases its blocks from last to first;
  * a filled block whose prefix is already cached elsewhere stays uncached;
  * copy-on-write when a request writes into a partially filled block that
    other requests also reference.
Every operation is a direct, slow restatement (linear scans, dicts, lists).
"""
from __future__ import annotations

OK, INVALID, NO_BLOCKS = 0, 1, 3   # the library's PA_OK, PA_ERR_INVALID_ARG, PA_ERR_WORKSPACE


class Request:
    def __init__(self, tokens):
        self.tokens = list(tokens)
        self.computed = 0
        self.table = []


class BlockManagerModel:
    def __init__(self, num_blocks: int, block_size: int):
        self.n, self.bs = num_blocks, block_size
        self.ref = [0] * num_blocks
        self.key = [None] * num_blocks        # prefix tuple of a cached block
        self.released = [0] * num_blocks      # release order of unreferenced cached blocks
        self.cache = {}                       # prefix tuple -> block
        self.reqs = {}
        self.clock = 0

    # -- block pool ---------------------------------------------------------
    def free_blocks(self):
        return [b for b in range(self.n) if self.ref[b] == 0 and self.key[b] is None]

    def evictable_blocks(self):
        return [b for b in range(self.n) if self.ref[b] == 0 and self.key[b] is not None]

    def available(self):
        return len(self.free_blocks()) + len(self.evictable_blocks())

    def alloc(self):
        free = self.free_blocks()
        if free:
            b = min(free)
        else:
            b = min(self.evictable_blocks(), key=lambda x: self.released[x])
            del self.cache[self.key[b]]
            self.key[b] = None
        self.ref[b] = 1
        return b

    def release(self, b):
        self.ref[b] -= 1
        if self.ref[b] == 0 and self.key[b] is not None:
            self.clock += 1
            self.released[b] = self.clock

    def prefix(self, tokens, i):
        """Identity of block i of a sequence: its whole token prefix."""
        return tuple(tokens[:(i + 1) * self.bs])

    # -- requests -----------------------------------------------------------
    def add_request(self, rid, tokens):
        if rid in self.reqs or len(tokens) < 1:
            return INVALID, 0
        r = Request(tokens)
        for i in range((len(tokens) - 1) // self.bs):
            b = self.cache.get(self.prefix(tokens, i))
            if b is None:
                break
            self.ref[b] += 1
            r.table.append(b)
        r.computed = len(r.table) * self.bs
        self.reqs[rid] = r
        return OK, r.computed

    def append_tokens(self, rid, tokens):
        if rid not in self.reqs:
            return INVALID
        self.reqs[rid].tokens += list(tokens)
        return OK

    def fork(self, src, dst):
        if src == dst or dst in self.reqs or src not in self.reqs:
            return INVALID
        s = self.reqs[src]
        r = Request(s.tokens)
        r.computed, r.table = s.computed, list(s.table)
        for b in r.table:
            self.ref[b] += 1
        self.reqs[dst] = r
        return OK

    def free_request(self, rid):
        if rid not in self.reqs:
            return INVALID
        for b in reversed(self.reqs[rid].table):
            self.release(b)
        del self.reqs[rid]
        return OK

    def schedule(self, rids, num_new, max_blocks, max_copies):
        """Returns (code, metadata dict or None)."""
        bs = self.bs
        need = copies_needed = 0
        if len(set(rids)) != len(rids):
            return INVALID, None
        for rid, n in zip(rids, num_new):
            if rid not in self.reqs or n < 1:
                return INVALID, None
            r = self.reqs[rid]
            end = r.computed + n
            if end > len(r.tokens) or -(-end // bs) > max_blocks:
                return INVALID, None
            cow = r.computed % bs != 0 and self.ref[r.table[r.computed // bs]] > 1
            need += -(-end // bs) - len(r.table) + int(cow)
            copies_needed += int(cow)
        if copies_needed > max_copies:
            return INVALID, None
        if need > self.available():
            return NO_BLOCKS, None
        tables, qsl, ctx, sl, slots, copies = [], [0], [], [], [], []
        for rid, n in zip(rids, num_new):
            r = self.reqs[rid]
            if r.computed % bs != 0:
                i = r.computed // bs
                old = r.table[i]
                if self.ref[old] > 1:
                    new = self.alloc()
                    copies.append((old, new))
                    self.release(old)
                    r.table[i] = new
            end = r.computed + n
            while len(r.table) * bs < end:
                r.table.append(self.alloc())
            tables.append(r.table + [-1] * (max_blocks - len(r.table)))
            ctx.append(r.computed)
            sl.append(end)
            qsl.append(qsl[-1] + n)
            for p in range(r.computed, end):
                slots.append(r.table[p // bs] * bs + p % bs)
            first_new_full = r.computed // bs
            r.computed = end
            for i in range(first_new_full, end // bs):
                key = self.prefix(r.tokens, i)
                b = r.table[i]
                if self.key[b] is None and key not in self.cache:
                    self.cache[key] = b
                    self.key[b] = key
        return OK, {"block_tables": tables, "query_start_loc": qsl, "context_lens": ctx,
                    "seq_lens": sl, "slot_mapping": slots, "copies": copies}
