"""Python binding of the host block manager (include/pa_blocks.h): argument
marshalling only; every decision is made by the C++ code in libpa."""
from __future__ import annotations

import ctypes
from typing import Dict, List, Optional, Sequence

import numpy as np

from . import PaError, _STATUS, PA_OK, lib


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class BlockManager:
    """Paged-KV block manager with a content-hash prefix cache."""

    def __init__(self, num_blocks: int, block_size: int):
        self._h = lib().pa_bm_create(int(num_blocks), int(block_size))
        if not self._h:
            raise ValueError("pa_bm_create failed (bad sizes or out of memory)")
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)

    def close(self):
        if self._h:
            lib().pa_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # interpreter shutdown
            pass

    def _check(self, rc: int, what: str):
        if rc != PA_OK:
            raise PaError(rc, what, _STATUS.get(rc, str(rc)))

    def add_request(self, req_id: int, tokens: Sequence[int]) -> int:
        """Admit a request; returns the number of prompt tokens already cached."""
        t = _i32(tokens)
        cached = ctypes.c_int32(0)
        self._check(lib().pa_bm_add_request(self._h, int(req_id), _ptr(t), t.size,
                                            ctypes.byref(cached)), "pa_bm_add_request")
        return cached.value

    def append_tokens(self, req_id: int, tokens: Sequence[int]):
        t = _i32(tokens)
        self._check(lib().pa_bm_append_tokens(self._h, int(req_id), _ptr(t) if t.size else None,
                                              t.size), "pa_bm_append_tokens")

    def fork(self, src: int, dst: int):
        self._check(lib().pa_bm_fork(self._h, int(src), int(dst)), "pa_bm_fork")

    def free_request(self, req_id: int):
        self._check(lib().pa_bm_free_request(self._h, int(req_id)), "pa_bm_free_request")

    def schedule(self, req_ids: Sequence[int], num_new: Sequence[int], max_blocks_per_seq: int,
                 max_copies: Optional[int] = None) -> Dict[str, np.ndarray]:
        """One step's metadata: block_tables, query_start_loc, context_lens,
        seq_lens, slot_mapping and the (src, dst) block copies to do first."""
        ids = np.ascontiguousarray(np.asarray(req_ids, dtype=np.int64))
        n = _i32(num_new)
        B, T = ids.size, int(n.sum()) if n.size else 0
        if max_copies is None:
            max_copies = B
        bt = np.empty((B, max_blocks_per_seq), np.int32)
        qsl = np.empty(B + 1, np.int32)
        ctx = np.empty(B, np.int32)
        sl = np.empty(B, np.int32)
        slots = np.empty(T, np.int64)
        copies = np.empty((max(max_copies, 1), 2), np.int32)
        nc = ctypes.c_int32(0)
        self._check(lib().pa_bm_schedule(self._h, B, _ptr(ids), _ptr(n), int(max_blocks_per_seq),
                                         _ptr(bt), _ptr(qsl), _ptr(ctx), _ptr(sl), _ptr(slots),
                                         int(max_copies), _ptr(copies), ctypes.byref(nc)),
                    "pa_bm_schedule")
        return {"block_tables": bt, "query_start_loc": qsl, "context_lens": ctx,
                "seq_lens": sl, "slot_mapping": slots, "copies": copies[:nc.value].copy()}

    def try_schedule(self, *a, **kw):
        """schedule(), or the PA_* error code instead of an exception."""
        try:
            return self.schedule(*a, **kw)
        except PaError as e:
            return e.code

    @property
    def num_free_blocks(self) -> int:
        return int(lib().pa_bm_num_free_blocks(self._h))

    @property
    def num_cached_blocks(self) -> int:
        return int(lib().pa_bm_num_cached_blocks(self._h))

    def ref_count(self, block: int) -> int:
        return int(lib().pa_bm_block_ref_count(self._h, int(block)))

    def blocks_of(self, req_id: int) -> Optional[List[int]]:
        cap = self.num_blocks
        out = np.empty(cap, np.int32)
        k = int(lib().pa_bm_request_blocks(self._h, int(req_id), _ptr(out), cap))
        return None if k < 0 else out[:k].tolist()

    def num_computed(self, req_id: int) -> int:
        return int(lib().pa_bm_num_computed(self._h, int(req_id)))
