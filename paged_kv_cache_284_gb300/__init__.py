"""paged_kv_cache_284_gb300 -- attention over a paged KV cache for one
continuous-batching step, on one GB300 (sm_103a).

Thin ctypes binding over the C ABI of ``libpa.so`` (declared in
``include/pa.h``).  The functions below only marshal arguments (check dtypes,
shapes and devices, pass raw pointers and the current CUDA stream); every
step of the path runs in the library's CUDA kernels.  If ``libpa.so`` is
missing the import of the binding fails loudly -- there is no fallback.

Calls (same names as the C ABI):
  pa_write_kv          reshape_and_cache through a slot mapping
  pa_attention         varlen paged attention (decode, chunks, prefix hits,
                       speculative verify in one batch)
  pa_merge_states      the cascade merge operator
  pa_prefix_attention  cascade shared-prefix (multi-query) pass
  pa_cascade_decode    prefix pass + suffix decode + merge in one call
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpa.so")

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_CUDA, \
    PA_ERR_BAD_METADATA = range(6)
PA_DEV_BAD_METADATA, PA_DEV_BAD_BLOCK, PA_DEV_BAD_SLOT, PA_DEV_WAIT_TIMEOUT, \
    PA_DEV_PLAN_OVERFLOW = 0x1, 0x2, 0x4, 0x8, 0x10

EXPORTED = ["pa_write_kv", "pa_attention_workspace_size", "pa_attention", "pa_attention_ex",
            "pa_write_kv_attention", "pa_cascade_fp8_staging_bytes",
            "pa_merge_states", "pa_cascade_workspace_size", "pa_prefix_attention",
            "pa_cascade_decode", "pa_validate_metadata", "pa_last_error_message",
            "pa_status_string", "pa_read_device_status", "pa_set_profile_events",
            "pa_attention_no_alloc", "pa_fp8_staging_bytes", "pa_kernel_launches",
            # block manager (include/pa_blocks.h)
            "pa_bm_create", "pa_bm_destroy", "pa_bm_add_request", "pa_bm_append_tokens",
            "pa_bm_fork", "pa_bm_schedule", "pa_bm_free_request", "pa_bm_num_free_blocks",
            "pa_bm_num_cached_blocks", "pa_bm_block_ref_count", "pa_bm_request_blocks",
            "pa_bm_num_computed",
            "pa_set_test_stall", "pa_set_tile_counter",
            # request router for sharded replicas (include/pa_shard.h)
            "pa_partition_requests"]
PA_KERNEL_WRITE_KV, PA_KERNEL_PLAN, PA_KERNEL_SPLIT_KV, PA_KERNEL_TENSOR_CORE = range(4)


class PaError(RuntimeError):
    def __init__(self, code: int, what: str, msg: str):
        super().__init__(f"{what}: {_STATUS.get(code, code)}: {msg}")
        self.code = code


_STATUS = {0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED", 3: "PA_ERR_WORKSPACE",
           4: "PA_ERR_CUDA", 5: "PA_ERR_BAD_METADATA"}


PA_KV_BF16, PA_KV_FP8_E4M3 = 0, 1


class KVDesc(ctypes.Structure):
    _fields_ = [("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p)]


def _declare(lib):
    P, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    i64 = ctypes.c_int64
    KV = ctypes.POINTER(KVDesc)
    sig = {
        "pa_write_kv": ([P, P, P, i32, KV, P], ctypes.c_int),
        "pa_attention_workspace_size": ([i32, i32, i32, i32, i32], sz),
        "pa_attention": ([P, KV, P, i32, P, P, P, i32, i32, i32, f32, P, P, P, sz, P],
                         ctypes.c_int),
        "pa_attention_ex": ([P, KV, P, i32, P, P, P, i32, i32, i32, f32, P, P, P, sz, i32, i32,
                             P], ctypes.c_int),
        "pa_write_kv_attention": ([P, P, P, i32, P, KV, P, i32, P, P, P, i32, i32, i32, f32, P, P,
                                   P, sz, P], ctypes.c_int),
        "pa_merge_states": ([P, P, P, P, i32, i32, i32, P, P, P], ctypes.c_int),
        "pa_cascade_workspace_size": ([i32, i32, i32, i32, i32, i32], sz),
        "pa_cascade_fp8_staging_bytes": ([i32, i32, i32, i32], sz),
        "pa_prefix_attention": ([P, KV, P, i32, i32, i32, f32, P, P, P, sz, P], ctypes.c_int),
        "pa_cascade_decode": ([P, KV, P, i32, P, i32, P, P, P, i32, i32, i32, f32, P, P, P, sz,
                               P], ctypes.c_int),
        "pa_validate_metadata": ([P, i32, P, P, P, i32, i32, P, i32, i32], ctypes.c_int),
        "pa_last_error_message": ([], ctypes.c_char_p),
        "pa_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "pa_read_device_status": ([ctypes.POINTER(ctypes.c_uint32), ctypes.c_int, P],
                                  ctypes.c_int),
        "pa_set_profile_events": ([i32, P, P], ctypes.c_int),
        "pa_attention_no_alloc": ([P, KV, P, i32, P, P, P, i32, i32, i32, f32, P, P, P],
                                  ctypes.c_int),
        "pa_fp8_staging_bytes": ([i32, i32, i32, i64], sz),
        "pa_kernel_launches": ([], ctypes.c_uint64),
        "pa_bm_create": ([i32, i32], P),
        "pa_bm_destroy": ([P], None),
        "pa_bm_add_request": ([P, i64, P, i32, P], ctypes.c_int),
        "pa_bm_append_tokens": ([P, i64, P, i32], ctypes.c_int),
        "pa_bm_fork": ([P, i64, i64], ctypes.c_int),
        "pa_bm_schedule": ([P, i32, P, P, i32, P, P, P, P, P, i32, P, P], ctypes.c_int),
        "pa_bm_free_request": ([P, i64], ctypes.c_int),
        "pa_bm_num_free_blocks": ([P], i32),
        "pa_bm_num_cached_blocks": ([P], i32),
        "pa_bm_block_ref_count": ([P, i32], i32),
        "pa_bm_request_blocks": ([P, i64, P, i32], i32),
        "pa_bm_num_computed": ([P, i64], i32),
        "pa_partition_requests": ([P, i32, i32, P, P], ctypes.c_int),
        "pa_set_test_stall": ([i32], ctypes.c_int),
        "pa_set_tile_counter": ([P], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


def load_library(path: str = LIB_PATH):
    if not os.path.exists(path):
        raise ImportError(f"libpa.so not built at {path}: run "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    return _declare(ctypes.CDLL(path))


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = load_library()
    return _lib


def _check(rc: int, what: str):
    if rc != PA_OK:
        raise PaError(rc, what, lib().pa_last_error_message().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, device=True):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


_FP8_DTYPES = (torch.uint8,) + ((torch.float8_e4m3fn,) if hasattr(torch, "float8_e4m3fn") else ())


def kv_desc(k_cache: torch.Tensor, v_cache: torch.Tensor, k_scale=None, v_scale=None) -> KVDesc:
    """Descriptor of a paged KV pool.  bf16 caches: k_scale / v_scale must be
    None.  e4m3 caches (torch.uint8 codes or torch.float8_e4m3fn): k_scale and
    v_scale are fp32 CUDA tensors [num_kv_heads]."""
    if k_cache.dtype in _FP8_DTYPES:
        for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
            if t.dtype not in _FP8_DTYPES or not t.is_contiguous() or not t.is_cuda:
                raise TypeError(f"{name} must be a contiguous CUDA uint8 / float8_e4m3fn tensor")
        if k_scale is None or v_scale is None:
            raise ValueError("an fp8 KV pool needs k_scale and v_scale")
        _need(k_scale, "k_scale", torch.float32)
        _need(v_scale, "v_scale", torch.float32)
        dtype = PA_KV_FP8_E4M3
    else:
        _need(k_cache, "k_cache", torch.bfloat16)
        _need(v_cache, "v_cache", torch.bfloat16)
        if k_scale is not None or v_scale is not None:
            raise ValueError("scales are for fp8 KV pools only")
        dtype = PA_KV_BF16
    if k_cache.shape != v_cache.shape or k_cache.dim() != 4:
        raise ValueError("caches must both be [num_blocks, num_kv_heads, block_size, head_dim]")
    nb, hkv, bs, d = k_cache.shape
    if dtype == PA_KV_FP8_E4M3 and (k_scale.numel() != hkv or v_scale.numel() != hkv):
        raise ValueError("k_scale / v_scale must hold num_kv_heads values")
    return KVDesc(k_cache.data_ptr(), v_cache.data_ptr(), nb, bs, hkv, d, dtype, 0,
                  None if k_scale is None else k_scale.data_ptr(),
                  None if v_scale is None else v_scale.data_ptr())


def pa_write_kv(k, v, slot_mapping, k_cache, v_cache, stream=None, k_scale=None, v_scale=None):
    """reshape_and_cache: k/v bf16 [T, Hkv, d], slot_mapping int64 [T]; an fp8
    pool quantises with k_scale / v_scale (fp32 [Hkv])."""
    _need(k, "k", torch.bfloat16)
    _need(v, "v", torch.bfloat16)
    _need(slot_mapping, "slot_mapping", torch.int64)
    kv = kv_desc(k_cache, v_cache, k_scale, v_scale)
    _check(lib().pa_write_kv(_ptr(k), _ptr(v), _ptr(slot_mapping), int(k.shape[0]),
                             ctypes.byref(kv), _stream(stream)), "pa_write_kv")


def workspace_size(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim) -> int:
    return int(lib().pa_attention_workspace_size(num_seqs, num_q_tokens, num_q_heads,
                                                 num_kv_heads, head_dim))


def cascade_workspace_size(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim,
                           prefix_len) -> int:
    return int(lib().pa_cascade_workspace_size(num_seqs, num_q_tokens, num_q_heads, num_kv_heads,
                                               head_dim, prefix_len))


def cascade_fp8_staging_bytes(num_kv_heads, head_dim, block_size, prefix_len) -> int:
    return int(lib().pa_cascade_fp8_staging_bytes(num_kv_heads, head_dim, block_size,
                                                  int(prefix_len)))


def _cascade_need(kv, num_seqs, T, hq, prefix_len) -> int:
    need = cascade_workspace_size(num_seqs, T, hq, kv.num_kv_heads, kv.head_dim, prefix_len)
    if kv.kv_dtype == PA_KV_FP8_E4M3:
        # the workspace's tail holds the prefix decoded to bf16
        need = ((need + 255) // 256) * 256 + cascade_fp8_staging_bytes(
            kv.num_kv_heads, kv.head_dim, kv.block_size, prefix_len)
    return need


def alloc_workspace(nbytes: int, device=None) -> torch.Tensor:
    """Device workspace owned by torch (256-byte aligned by the allocator)."""
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device or "cuda")


def fp8_staging_bytes(num_kv_heads, head_dim, block_size, num_blocks) -> int:
    return int(lib().pa_fp8_staging_bytes(num_kv_heads, head_dim, block_size, int(num_blocks)))


def pa_attention(q, k_cache, v_cache, block_tables, query_start_loc, context_lens, seq_lens,
                 scale, out, lse=None, workspace=None, stream=None, short_q_max_rows=-1,
                 split_keys=0, k_scale=None, v_scale=None, staging_blocks=0):
    """Varlen paged attention for one step; writes out (bf16 [T,Hq,d]) and lse
    (fp32 [T,Hq], optional).  An fp8 pool takes k_scale / v_scale (fp32
    [Hkv]); a workspace allocated here gets room to stage staging_blocks
    blocks of its long requests for the tensor-core kernel (a caller's
    workspace is used as given).  Returns the workspace tensor used."""
    _need(q, "q", torch.bfloat16)
    _need(out, "out", torch.bfloat16)
    for name, t in (("block_tables", block_tables), ("query_start_loc", query_start_loc),
                    ("context_lens", context_lens), ("seq_lens", seq_lens)):
        _need(t, name, torch.int32)
    if lse is not None:
        _need(lse, "lse", torch.float32)
    kv = kv_desc(k_cache, v_cache, k_scale, v_scale)
    T, hq, _ = q.shape
    B = int(seq_lens.shape[0])
    need = workspace_size(B, T, hq, kv.num_kv_heads, kv.head_dim)
    if kv.kv_dtype == PA_KV_FP8_E4M3 and staging_blocks > 0:
        need += fp8_staging_bytes(kv.num_kv_heads, kv.head_dim, kv.block_size, staging_blocks)
    if workspace is None or workspace.numel() < need:
        workspace = alloc_workspace(need, q.device)
    _check(lib().pa_attention_ex(_ptr(q), ctypes.byref(kv), _ptr(block_tables),
                                 int(block_tables.shape[1]), _ptr(query_start_loc),
                                 _ptr(context_lens), _ptr(seq_lens), B, T, hq, float(scale),
                                 _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
                                 int(short_q_max_rows), int(split_keys), _stream(stream)),
           "pa_attention")
    return workspace


def pa_write_kv_attention(k, v, slot_mapping, q, k_cache, v_cache, block_tables,
                          query_start_loc, context_lens, seq_lens, scale, out, lse=None,
                          workspace=None, stream=None, k_scale=None, v_scale=None,
                          staging_blocks=0):
    """pa_write_kv then pa_attention in one call (same arguments, same
    results); the cache write runs beside the step's planner.  Returns the
    workspace tensor used."""
    _need(k, "k", torch.bfloat16)
    _need(v, "v", torch.bfloat16)
    _need(slot_mapping, "slot_mapping", torch.int64)
    _need(q, "q", torch.bfloat16)
    _need(out, "out", torch.bfloat16)
    for name, t in (("block_tables", block_tables), ("query_start_loc", query_start_loc),
                    ("context_lens", context_lens), ("seq_lens", seq_lens)):
        _need(t, name, torch.int32)
    if lse is not None:
        _need(lse, "lse", torch.float32)
    kv = kv_desc(k_cache, v_cache, k_scale, v_scale)
    T, hq, _ = q.shape
    B = int(seq_lens.shape[0])
    need = workspace_size(B, T, hq, kv.num_kv_heads, kv.head_dim)
    if kv.kv_dtype == PA_KV_FP8_E4M3 and staging_blocks > 0:
        need += fp8_staging_bytes(kv.num_kv_heads, kv.head_dim, kv.block_size, staging_blocks)
    if workspace is None or workspace.numel() < need:
        workspace = alloc_workspace(need, q.device)
    _check(lib().pa_write_kv_attention(_ptr(k), _ptr(v), _ptr(slot_mapping), int(k.shape[0]),
                                       _ptr(q), ctypes.byref(kv), _ptr(block_tables),
                                       int(block_tables.shape[1]), _ptr(query_start_loc),
                                       _ptr(context_lens), _ptr(seq_lens), B, T, hq,
                                       float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                       workspace.numel(), _stream(stream)),
           "pa_write_kv_attention")
    return workspace


def pa_merge_states(o_a, lse_a, o_b, lse_b, out, lse_out=None, stream=None):
    for name, t in (("o_a", o_a), ("o_b", o_b), ("out", out)):
        _need(t, name, torch.bfloat16)
    for name, t in (("lse_a", lse_a), ("lse_b", lse_b)):
        _need(t, name, torch.float32)
    if lse_out is not None:
        _need(lse_out, "lse_out", torch.float32)
    n, h, d = o_a.shape
    _check(lib().pa_merge_states(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), n, h, d,
                                 _ptr(out), _ptr(lse_out), _stream(stream)), "pa_merge_states")


def pa_prefix_attention(q, k_cache, v_cache, prefix_blocks, prefix_len, scale, out, lse=None,
                        workspace=None, stream=None, k_scale=None, v_scale=None):
    """Shared-prefix attention; an fp8 pool takes k_scale / v_scale (fp32
    [Hkv]) and a workspace with room for the prefix's bf16 copy."""
    _need(q, "q", torch.bfloat16)
    _need(out, "out", torch.bfloat16)
    _need(prefix_blocks, "prefix_blocks", torch.int32)
    kv = kv_desc(k_cache, v_cache, k_scale, v_scale)
    T, hq, _ = q.shape
    need = _cascade_need(kv, 1, T, hq, prefix_len)
    if workspace is None or workspace.numel() < need:
        workspace = alloc_workspace(need, q.device)
    _check(lib().pa_prefix_attention(_ptr(q), ctypes.byref(kv), _ptr(prefix_blocks),
                                     int(prefix_len), T, hq, float(scale), _ptr(out), _ptr(lse),
                                     _ptr(workspace), workspace.numel(), _stream(stream)),
           "pa_prefix_attention")
    return workspace


def pa_cascade_decode(q, k_cache, v_cache, prefix_blocks, prefix_len, block_tables,
                      query_start_loc, context_lens, seq_lens, scale, out, lse=None,
                      workspace=None, stream=None, k_scale=None, v_scale=None):
    """Cascade decode; an fp8 pool takes k_scale / v_scale (fp32 [Hkv]) and a
    workspace with room for the prefix's bf16 copy."""
    _need(q, "q", torch.bfloat16)
    _need(out, "out", torch.bfloat16)
    for name, t in (("prefix_blocks", prefix_blocks), ("block_tables", block_tables),
                    ("query_start_loc", query_start_loc), ("context_lens", context_lens),
                    ("seq_lens", seq_lens)):
        _need(t, name, torch.int32)
    kv = kv_desc(k_cache, v_cache, k_scale, v_scale)
    T, hq, _ = q.shape
    B = int(seq_lens.shape[0])
    need = _cascade_need(kv, B, T, hq, prefix_len)
    if workspace is None or workspace.numel() < need:
        workspace = alloc_workspace(need, q.device)
    _check(lib().pa_cascade_decode(_ptr(q), ctypes.byref(kv), _ptr(prefix_blocks),
                                   int(prefix_len), _ptr(block_tables), int(block_tables.shape[1]),
                                   _ptr(query_start_loc), _ptr(context_lens), _ptr(seq_lens), B,
                                   T, hq, float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                   workspace.numel(), _stream(stream)), "pa_cascade_decode")
    return workspace


def pa_validate_metadata(block_tables, query_start_loc, context_lens, seq_lens, num_blocks,
                         block_size, slot_mapping=None):
    """Host-side metadata check (CPU tensors).  Raises PaError on a problem."""
    bt = block_tables.detach().cpu().to(torch.int32).contiguous()
    qsl = query_start_loc.detach().cpu().to(torch.int32).contiguous()
    ctx = context_lens.detach().cpu().to(torch.int32).contiguous()
    sl = seq_lens.detach().cpu().to(torch.int32).contiguous()
    sm = None if slot_mapping is None else slot_mapping.detach().cpu().to(torch.int64).contiguous()
    T = int(qsl[-1]) if qsl.numel() else 0
    _check(lib().pa_validate_metadata(_ptr(bt), int(bt.shape[1]), _ptr(qsl), _ptr(ctx), _ptr(sl),
                                      int(sl.shape[0]), T, _ptr(sm), int(num_blocks),
                                      int(block_size)), "pa_validate_metadata")


def partition_requests(seq_lens, num_ranks: int):
    """Request router for request-sharded replicas (host only): the rank of
    each request, balancing KV tokens greedily longest first, and the KV
    tokens each rank receives.  seq_lens: sequence of ints or a tensor."""
    sl = torch.as_tensor(seq_lens, dtype=torch.int32).detach().cpu().contiguous()
    n = int(sl.numel())
    rank_of = torch.empty(n, dtype=torch.int32)
    loads = torch.empty(max(int(num_ranks), 1), dtype=torch.int64)
    rc = lib().pa_partition_requests(_ptr(sl) if n else None, n, int(num_ranks),
                                     _ptr(rank_of) if n else None, _ptr(loads))
    if rc != PA_OK:
        raise PaError(rc, "pa_partition_requests", "bad sizes or a negative length")
    return rank_of.tolist(), loads[:int(num_ranks)].tolist()


PA_TEST_STALL_NONE, PA_TEST_STALL_SPLIT_KV, PA_TEST_STALL_LAST_GRID = 0, 1, 2


def set_test_stall(which: int):
    """Test hook: make one bounded device wait run out (see pa.h)."""
    _check(lib().pa_set_test_stall(int(which)), "pa_set_test_stall")


def set_tile_counter(counter=None):
    """Count the tensor-core kernel's 128-key tiles into `counter` (a CUDA
    int64 tensor of one element) until called with None."""
    if counter is not None and (counter.dtype != torch.int64 or not counter.is_cuda):
        raise TypeError("counter must be a CUDA int64 tensor")
    _check(lib().pa_set_tile_counter(_ptr(counter)), "pa_set_tile_counter")


def read_device_status(clear: bool = True, stream=None) -> int:
    v = ctypes.c_uint32(0)
    _check(lib().pa_read_device_status(ctypes.byref(v), 1 if clear else 0, _stream(stream)),
           "pa_read_device_status")
    return int(v.value)


def kernel_launches() -> int:
    """Kernels the library has enqueued in this process so far."""
    return int(lib().pa_kernel_launches())


def set_profile_events(which: int, start=None, end=None):
    """Bracket every launch of kernel `which` with the given torch.cuda.Event
    records (None clears)."""
    s = None if start is None else ctypes.c_void_p(start.cuda_event)
    e = None if end is None else ctypes.c_void_p(end.cuda_event)
    _check(lib().pa_set_profile_events(int(which), s, e), "pa_set_profile_events")


def pa_attention_no_alloc(q, k_cache, v_cache, block_tables, query_start_loc, context_lens,
                          seq_lens, scale, out, lse=None, stream=None, k_scale=None,
                          v_scale=None):
    """pa_attention without a workspace, for callers that cannot allocate
    device memory: the library's own fixed scratch array is used.  Calls that
    overlap on the GPU share that array and must be ordered."""
    _need(q, "q", torch.bfloat16)
    _need(out, "out", torch.bfloat16)
    for name, t in (("block_tables", block_tables), ("query_start_loc", query_start_loc),
                    ("context_lens", context_lens), ("seq_lens", seq_lens)):
        _need(t, name, torch.int32)
    if lse is not None:
        _need(lse, "lse", torch.float32)
    kv = kv_desc(k_cache, v_cache, k_scale, v_scale)
    T, hq, _ = q.shape
    _check(lib().pa_attention_no_alloc(_ptr(q), ctypes.byref(kv), _ptr(block_tables),
                                       int(block_tables.shape[1]), _ptr(query_start_loc),
                                       _ptr(context_lens), _ptr(seq_lens), int(seq_lens.shape[0]),
                                       T, hq, float(scale), _ptr(out), _ptr(lse), _stream(stream)),
           "pa_attention_no_alloc")
