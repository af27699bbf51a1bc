"""CPU oracle for paged-KV attention -- TEST INFRASTRUCTURE ONLY.

Plain fp64 definitions of the step's operations (see ``oracle.c`` for the
citations and readings).  Only the test suite, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline leg may import this package; the CUDA library
never does, and shares no code with it.

``oracle.c`` is compiled to ``liboracle.so`` next to this file by
``build_oracle()`` (gcc, -O2, OpenMP).  ``brute.py`` is an independent NumPy
triple loop used to pin the C code on tiny inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

ORC_OK, ORC_BAD_ARG, ORC_BAD_META, ORC_NO_MEM = 0, 1, 2, 3


def build_oracle(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain C, gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build_oracle()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.oracle_write_kv.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, P]
        lib.oracle_attention.argtypes = [P, P, P, i32, i32, i32, i32, P, i32, P, P, P, i32, i32,
                                         f64, P, P, P]
        lib.oracle_prefix_attention.argtypes = [P, P, P, i32, i32, i32, i32, P, i32, i32, i32,
                                                f64, P, P]
        lib.oracle_merge_states.argtypes = [P, P, P, P, i64, i32, i32, P, P]
        lib.oracle_e4m3_encode.argtypes = [P, i64, P]
        lib.oracle_e4m3_decode.argtypes = [P, i64, P]
        lib.oracle_write_kv_fp8.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, P, P, P]
        lib.oracle_attention_fp8.argtypes = [P, P, P, P, P, i32, i32, i32, i32, P, i32, P, P, P,
                                             i32, i32, f64, P, P, P]
        for fn in (lib.oracle_write_kv, lib.oracle_attention, lib.oracle_prefix_attention,
                   lib.oracle_merge_states, lib.oracle_e4m3_encode, lib.oracle_e4m3_decode,
                   lib.oracle_write_kv_fp8, lib.oracle_attention_fp8):
            fn.restype = ctypes.c_int
        _lib = lib
    return _lib


def _bits(a) -> np.ndarray:
    """bf16 data as a C-contiguous uint16 array (accepts torch bf16 or uint16)."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            assert a.dtype == torch.bfloat16, a.dtype
            return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.int16).numpy()
                                        .view(np.uint16))
    except ImportError:  # pragma: no cover
        pass
    a = np.asarray(a)
    assert a.dtype == np.uint16, a.dtype
    return np.ascontiguousarray(a)


def _u8(a) -> np.ndarray:
    """e4m3 codes as a C-contiguous uint8 array (accepts torch uint8 /
    float8_e4m3fn tensors or numpy)."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            t = a.detach().cpu().contiguous()
            if t.dtype != torch.uint8:
                t = t.view(torch.uint8)
            return np.ascontiguousarray(t.numpy())
    except ImportError:  # pragma: no cover
        pass
    a = np.asarray(a)
    assert a.dtype == np.uint8, a.dtype
    return np.ascontiguousarray(a)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(_np(a), dtype=np.float32))


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(_np(a), dtype=np.int32))


def _i64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(_np(a), dtype=np.int64))


def _np(a):
    try:
        import torch
        if isinstance(a, torch.Tensor):
            return a.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != ORC_OK:
        raise ValueError(f"{what}: oracle status {rc}")


def write_kv(k, v, slot_mapping, k_cache, v_cache):
    """Return (k_cache', v_cache') as uint16 bit arrays after reshape_and_cache.

    k, v: bf16 [T, Hkv, d]; slot_mapping: int64 [T]; caches: bf16
    [num_blocks, Hkv, block_size, d].  Inputs are not modified.
    """
    kb, vb = _bits(k), _bits(v)
    kc, vc = _bits(k_cache).copy(), _bits(v_cache).copy()
    slots = _i64(slot_mapping)
    nb, hkv, bs, d = kc.shape
    T = slots.shape[0]
    _check(_load().oracle_write_kv(_ptr(kb), _ptr(vb), _ptr(slots), T, hkv, d, bs, nb,
                                   _ptr(kc), _ptr(vc)), "write_kv")
    return kc, vc


def attention(q, k_cache, v_cache, block_tables, query_start_loc, context_lens, seq_lens,
              scale, return_visible=False):
    """fp64 varlen paged attention.  Returns (out [T,Hq,d], lse [T,Hq]) float64
    (and per-row visible key counts int32 [T] if return_visible)."""
    qb = _bits(q)
    kc, vc = _bits(k_cache), _bits(v_cache)
    nb, hkv, bs, d = kc.shape
    T, hq, dq = qb.shape
    assert dq == d
    bt = _i32(block_tables)
    if bt.ndim == 1:
        bt = bt.reshape(1, -1)
    qsl, ctx, sl = _i32(query_start_loc), _i32(context_lens), _i32(seq_lens)
    B = sl.shape[0]
    out = np.zeros((T, hq, d), dtype=np.float64)
    lse = np.zeros((T, hq), dtype=np.float64)
    vis = np.zeros((T,), dtype=np.int32)
    _check(_load().oracle_attention(_ptr(qb), _ptr(kc), _ptr(vc), nb, bs, hkv, d, _ptr(bt),
                                    bt.shape[1], _ptr(qsl), _ptr(ctx), _ptr(sl), B, hq,
                                    float(scale), _ptr(out), _ptr(lse), _ptr(vis)),
           "attention")
    if return_visible:
        return out, lse, vis
    return out, lse


def prefix_attention(q, k_cache, v_cache, prefix_blocks, prefix_len, scale):
    """fp64 non-causal attention of every q row over the shared prefix."""
    qb = _bits(q)
    kc, vc = _bits(k_cache), _bits(v_cache)
    nb, hkv, bs, d = kc.shape
    T, hq, _ = qb.shape
    pb = _i32(prefix_blocks)
    out = np.zeros((T, hq, d), dtype=np.float64)
    lse = np.zeros((T, hq), dtype=np.float64)
    _check(_load().oracle_prefix_attention(_ptr(qb), _ptr(kc), _ptr(vc), nb, bs, hkv, d,
                                           _ptr(pb), int(prefix_len), T, hq, float(scale),
                                           _ptr(out), _ptr(lse)), "prefix_attention")
    return out, lse


def merge_states(o_a, lse_a, o_b, lse_b):
    """fp64 merge of two attention states (arrays of float64)."""
    oa = np.ascontiguousarray(np.asarray(_np(o_a), dtype=np.float64))
    ob = np.ascontiguousarray(np.asarray(_np(o_b), dtype=np.float64))
    la = np.ascontiguousarray(np.asarray(_np(lse_a), dtype=np.float64))
    lb = np.ascontiguousarray(np.asarray(_np(lse_b), dtype=np.float64))
    assert oa.shape == ob.shape and la.shape == lb.shape == oa.shape[:-1]
    d = oa.shape[-1]
    h = oa.shape[-2] if oa.ndim >= 3 else 1
    n = int(np.prod(oa.shape[:-2])) if oa.ndim >= 3 else oa.shape[0]
    out = np.zeros_like(oa)
    lse = np.zeros_like(la)
    _check(_load().oracle_merge_states(_ptr(oa), _ptr(la), _ptr(ob), _ptr(lb), n, h, d,
                                       _ptr(out), _ptr(lse)), "merge_states")
    return out, lse


# ---------------------------------------------------------------------------
# FP8 (e4m3) KV cache
# ---------------------------------------------------------------------------

def e4m3_encode(x):
    """float32 values -> e4m3 codes (uint8), nearest-even, saturating at 448."""
    xa = _f32(x)
    out = np.zeros(xa.shape, dtype=np.uint8)
    _check(_load().oracle_e4m3_encode(_ptr(xa), xa.size, _ptr(out)), "e4m3_encode")
    return out


def e4m3_decode(codes):
    """e4m3 codes -> float64 values (NaN for the NaN codes)."""
    ca = _u8(codes)
    out = np.zeros(ca.shape, dtype=np.float64)
    _check(_load().oracle_e4m3_decode(_ptr(ca), ca.size, _ptr(out)), "e4m3_decode")
    return out


def write_kv_fp8(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale):
    """Return (k_cache', v_cache') as uint8 code arrays after reshape_and_cache
    into an e4m3 cache with per-kv-head scales (fp32 [Hkv])."""
    kb, vb = _bits(k), _bits(v)
    kc, vc = _u8(k_cache).copy(), _u8(v_cache).copy()
    ks, vs = _f32(k_scale), _f32(v_scale)
    slots = _i64(slot_mapping)
    nb, hkv, bs, d = kc.shape
    assert ks.shape == vs.shape == (hkv,)
    _check(_load().oracle_write_kv_fp8(_ptr(kb), _ptr(vb), _ptr(slots), slots.shape[0], hkv, d,
                                       bs, nb, _ptr(ks), _ptr(vs), _ptr(kc), _ptr(vc)),
           "write_kv_fp8")
    return kc, vc


def attention_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, query_start_loc,
                  context_lens, seq_lens, scale, return_visible=False):
    """fp64 varlen paged attention over an e4m3 cache (values = code x scale)."""
    qb = _bits(q)
    kc, vc = _u8(k_cache), _u8(v_cache)
    ks, vs = _f32(k_scale), _f32(v_scale)
    nb, hkv, bs, d = kc.shape
    T, hq, dq = qb.shape
    assert dq == d and ks.shape == vs.shape == (hkv,)
    bt = _i32(block_tables)
    if bt.ndim == 1:
        bt = bt.reshape(1, -1)
    qsl, ctx, sl = _i32(query_start_loc), _i32(context_lens), _i32(seq_lens)
    B = sl.shape[0]
    out = np.zeros((T, hq, d), dtype=np.float64)
    lse = np.zeros((T, hq), dtype=np.float64)
    vis = np.zeros((T,), dtype=np.int32)
    _check(_load().oracle_attention_fp8(_ptr(qb), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), nb, bs,
                                        hkv, d, _ptr(bt), bt.shape[1], _ptr(qsl), _ptr(ctx),
                                        _ptr(sl), B, hq, float(scale), _ptr(out), _ptr(lse),
                                        _ptr(vis)), "attention_fp8")
    if return_visible:
        return out, lse, vis
    return out, lse
