"""Bounded device waits that run out.

Every wait inside the kernels gives up after 2 s: the kernel raises
PA_DEV_WAIT_TIMEOUT in the status word, lets its copies in flight land and
returns, and the context stays usable.  The test hook pa_set_test_stall
makes one such wait run out on purpose (a stage that is never issued, or a
CTA that never existed); nothing faults or traps.  Each test checks that the
call returns, that the status word carries the timeout, that a read-and-clear
empties it, and that the next normal step is at parity with the oracle and
leaves a clean status.
"""
import time

import numpy as np
import pytest
import torch

import paged_kv_cache_284_gb300 as pk
from paged_kv_cache_284_gb300 import workloads
from gpu_helpers import (DEV, assert_attention_close, assert_status_clean, bits, gpu_attend,
                         gpu_write, oracle_attend, oracle_write)

pytestmark = pytest.mark.gpu


def stalled_call(step, kc, vc, which):
    pk.read_device_status(clear=True)
    pk.set_test_stall(which)
    try:
        t0 = time.perf_counter()
        out, lse = gpu_attend(step, kc, vc)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
    finally:
        pk.set_test_stall(pk.PA_TEST_STALL_NONE)
    status = pk.read_device_status(clear=True)
    return out, lse, dt, status


def check_next_step_clean(pool, step, kc, vc):
    kb, vb = oracle_write(step, bits(pool.k_cache), bits(pool.v_cache))
    out, lse = gpu_attend(step, kc, vc)
    torch.cuda.synchronize()
    assert_attention_close(out, lse, *oracle_attend(step, kb, vb), "after the timeout")
    assert_status_clean()


def test_split_kv_consumers_time_out_when_a_stage_never_comes():
    # 16 decode rows: the split-KV kernel waits for its plan (no tensor-core
    # grid beside it), so the hook applies
    pool, (step,) = workloads.decode_heavy(seed=284070, num_seqs=16, lo=100, hi=2000,
                                           num_q_heads=8, num_kv_heads=2)
    kc, vc = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    gpu_write(step, kc, vc)
    torch.cuda.synchronize()
    out, lse, dt, status = stalled_call(step, kc, vc, pk.PA_TEST_STALL_SPLIT_KV)
    assert status & pk.PA_DEV_WAIT_TIMEOUT, hex(status)
    assert 1.5 < dt < 60.0, dt            # the consumers' wait ran to its 2 s limit
    assert pk.read_device_status(clear=True) == 0   # read-and-clear emptied it
    check_next_step_clean(pool, step, kc, vc)


def test_last_tensor_core_grid_times_out_waiting_for_a_missing_cta():
    # a step of >= 512 tokens with chunks: split-KV and tensor-core kernels
    # side by side; the last grid waits for one first-grid CTA too many
    pool, (step,) = workloads.mixed_step(seed=284071, num_chunks=2, chunk_len=256,
                                         chunk_ctx=(0, 300), num_decode=16,
                                         decode_len=(100, 1500), num_spec=2,
                                         spec_ctx=(50, 600), num_q_heads=8, num_kv_heads=2)
    assert step.num_q_tokens >= 512
    kc, vc = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    gpu_write(step, kc, vc)
    torch.cuda.synchronize()
    out, lse, dt, status = stalled_call(step, kc, vc, pk.PA_TEST_STALL_LAST_GRID)
    assert status & pk.PA_DEV_WAIT_TIMEOUT, hex(status)
    assert 1.5 < dt < 60.0, dt
    # every item ran before the final wait: the stalled step's result is right
    kb, vb = oracle_write(step, bits(pool.k_cache), bits(pool.v_cache))
    assert_attention_close(out, lse, *oracle_attend(step, kb, vb), "stalled last grid")
    assert pk.read_device_status(clear=True) == 0
    check_next_step_clean(pool, step, kc, vc)
