"""Shared plumbing for the GPU parity tests: move a seeded step to the device,
run it through the C ABI, run the oracle on the same inputs, compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_cache_284_gb300 as pk

# Acceptance bar for attention outputs against the fp64 oracle (bf16 inputs,
# fp32 accumulation, bf16 output): element-wise max and mean absolute error,
# and the absolute error of the natural-log LSE.
OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-3

DEV = torch.device("cuda:0")


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def dev_meta(step):
    return dict(block_tables=step.block_tables.to(DEV), query_start_loc=step.query_start_loc.to(DEV),
                context_lens=step.context_lens.to(DEV), seq_lens=step.seq_lens.to(DEV))


def gpu_write(step, kc, vc):
    pk.pa_write_kv(step.k.to(DEV), step.v.to(DEV), step.slot_mapping.to(DEV), kc, vc)


def gpu_attend(step, kc, vc, **kw):
    q = step.q.to(DEV)
    out = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    pk.pa_attention(q, kc, vc, scale=step.scale, out=out, lse=lse, **dev_meta(step), **kw)
    return out, lse


def oracle_write(step, k_bits, v_bits):
    return oracle.write_kv(step.k, step.v, step.slot_mapping, k_bits, v_bits)


def oracle_attend(step, k_bits, v_bits):
    return oracle.attention(step.q, k_bits, v_bits, step.block_tables, step.query_start_loc,
                            step.context_lens, step.seq_lens, step.scale)


def assert_attention_close(out, lse, ref_o, ref_l, what=""):
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    err = np.abs(o - ref_o)
    lerr = np.abs(l - ref_l)
    msg = (f"{what}: max|dO|={err.max():.3e} mean|dO|={err.mean():.3e} "
           f"max|dLSE|={lerr.max():.3e}")
    assert err.max() <= OUT_MAX_ABS, msg
    assert err.mean() <= OUT_MEAN_ABS, msg
    assert lerr.max() <= LSE_MAX_ABS, msg
    return err.max(), err.mean(), lerr.max()


def assert_status_clean():
    st = pk.read_device_status(clear=True)
    assert st == 0, f"device status {st:#x}"


def run_and_check(pool, steps, **kw):
    """Write + attend each step in order on one pool (GPU and oracle), compare
    caches bit for bit and attention within tolerance."""
    kc, vc = pool.k_cache.to(DEV), pool.v_cache.to(DEV)
    kb, vb = bits(pool.k_cache), bits(pool.v_cache)
    for step in steps:
        gpu_write(step, kc, vc)
        kb, vb = oracle_write(step, kb, vb)
        out, lse = gpu_attend(step, kc, vc, **kw)
        torch.cuda.synchronize()
        assert np.array_equal(bits(kc), kb), f"{step.label}: K cache differs"
        assert np.array_equal(bits(vc), vb), f"{step.label}: V cache differs"
        ref_o, ref_l = oracle_attend(step, kb, vb)
        assert_attention_close(out, lse, ref_o, ref_l, f"{step.label} {kw}")
    assert_status_clean()
    return kc, vc


# ---- FP8 (e4m3) KV pool -------------------------------------------------------

def codes(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy()


def fp8_dev(pool8):
    """Device copies of an Fp8Pool: (k codes, v codes, k_scale, v_scale)."""
    return (pool8.k_cache.to(DEV), pool8.v_cache.to(DEV), pool8.k_scale.to(DEV),
            pool8.v_scale.to(DEV))


def gpu_write_fp8(step, kc, vc, ks, vs):
    pk.pa_write_kv(step.k.to(DEV), step.v.to(DEV), step.slot_mapping.to(DEV), kc, vc,
                   k_scale=ks, v_scale=vs)


def gpu_attend_fp8(step, kc, vc, ks, vs, **kw):
    q = step.q.to(DEV)
    out = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    ws = pk.pa_attention(q, kc, vc, scale=step.scale, out=out, lse=lse, k_scale=ks, v_scale=vs,
                         **dev_meta(step), **kw)
    gpu_attend_fp8.last_workspace = ws
    return out, lse


def plan_header(ws):
    """The step plan's header at the start of the workspace (white-box check):
    work items of the two kernels and the fp8 staging counts."""
    h = ws[:64].cpu().view(torch.int32).tolist()
    return {"short_items": h[0], "long_items": h[1], "split_stages": h[4], "num_staged": h[6],
            "staged_blocks": h[7]}


def long_requests(step, short_max_rows=64):
    """Requests whose q_len * group exceeds the split-KV kernel's rows."""
    group = step.num_q_heads // step.num_kv_heads
    return [b for b, n in enumerate(step.q_lens.tolist()) if n * group > short_max_rows]


def staging_blocks_for(step, reqs):
    bs = step.block_size
    return sum(-(-int(step.seq_lens[b]) // bs) for b in reqs)


def run_and_check_fp8(pool8, steps, **kw):
    """Write + attend each step on one e4m3 pool (GPU and oracle): caches equal
    byte for byte, attention within tolerance of the fp64 oracle over the
    dequantised codes."""
    kc, vc, ks, vs = fp8_dev(pool8)
    kb, vb = codes(pool8.k_cache), codes(pool8.v_cache)
    sk, sv = pool8.k_scale.numpy(), pool8.v_scale.numpy()
    for step in steps:
        gpu_write_fp8(step, kc, vc, ks, vs)
        kb, vb = oracle.write_kv_fp8(step.k, step.v, step.slot_mapping, kb, vb, sk, sv)
        out, lse = gpu_attend_fp8(step, kc, vc, ks, vs, **kw)
        torch.cuda.synchronize()
        assert np.array_equal(codes(kc), kb), f"{step.label}: fp8 K cache differs"
        assert np.array_equal(codes(vc), vb), f"{step.label}: fp8 V cache differs"
        ref_o, ref_l = oracle.attention_fp8(step.q, kb, vb, sk, sv, step.block_tables,
                                            step.query_start_loc, step.context_lens,
                                            step.seq_lens, step.scale)
        assert_attention_close(out, lse, ref_o, ref_l, f"fp8 {step.label} {kw}")
    assert_status_clean()
    return kc, vc, ks, vs
