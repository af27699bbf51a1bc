"""Brute-force NumPy fp64 attention for tiny inputs -- TEST INFRASTRUCTURE ONLY.

An independent restatement of the step, used only to pin ``oracle.c``: it
walks every (request, query row, q head, key) with Python loops, builds the
key list position by position through the block table ([CH] "11. 推理加速(一):
vLLM 原理", §11.2 Block Table), and evaluates softmax without the max shift
(inputs are tiny, so exp never overflows).  Nothing here is shared with the
C oracle or the CUDA library.
"""
from __future__ import annotations

import math

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    u = bits.astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def attention(q_bits, kc_bits, vc_bits, block_tables, qsl, ctx, seq_lens, scale):
    return attention_values(bf16_bits_to_f64(np.asarray(q_bits)),
                            bf16_bits_to_f64(np.asarray(kc_bits)),
                            bf16_bits_to_f64(np.asarray(vc_bits)),
                            block_tables, qsl, ctx, seq_lens, scale)


def attention_values(q, kc, vc, block_tables, qsl, ctx, seq_lens, scale):
    """The same loops over float64 q [T,Hq,d] and caches [nb,Hkv,bs,d]."""
    T, hq, d = q.shape
    _, hkv, bs, _ = kc.shape
    per_kv = hq // hkv
    out = np.zeros((T, hq, d))
    lse = np.zeros((T, hq))
    for b in range(len(seq_lens)):
        start, stop = int(qsl[b]), int(qsl[b + 1])
        for i in range(stop - start):
            pos = int(ctx[b]) + i          # absolute position of this query token
            for h in range(hq):
                kvh = h // per_kv
                weights = []
                values = []
                for j in range(int(seq_lens[b])):
                    if j > pos:             # causal: a token sees itself and earlier ones
                        continue
                    phys = int(block_tables[b][j // bs])
                    key = kc[phys, kvh, j % bs]
                    s = scale * float(sum(q[start + i, h, e] * key[e] for e in range(d)))
                    weights.append(math.exp(s))
                    values.append(vc[phys, kvh, j % bs])
                z = sum(weights)
                lse[start + i, h] = math.log(z)
                acc = np.zeros(d)
                for w, val in zip(weights, values):
                    acc += (w / z) * val
                out[start + i, h] = acc
    return out, lse
