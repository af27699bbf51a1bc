"""C-ABI checks that need no GPU: the library loads, exports every entry
point declared in include/*.h, rejects bad scalar arguments before touching
the device, and the host-side metadata validator catches each kind of bad
metadata."""
import ctypes
import os
import re

import pytest
import torch

import paged_kv_cache_284_gb300 as pk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    """Every function declared by the headers under include/."""
    names = set()
    inc = os.path.join(ROOT, "include")
    for h in sorted(os.listdir(inc)):
        if h.endswith(".h"):
            src = re.sub(r"/\*.*?\*/", "", open(os.path.join(inc, h)).read(), flags=re.S)
            names.update(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_library_exports_every_declared_function():
    lib = pk.lib()
    names = declared_functions()
    assert len(names) >= 10
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(pk.EXPORTED)


def test_test_stall_hook_rejects_unknown_values():
    assert pk.lib().pa_set_test_stall(7) == pk.PA_ERR_INVALID_ARG
    assert pk.lib().pa_set_test_stall(pk.PA_TEST_STALL_NONE) == pk.PA_OK


def test_status_strings():
    assert pk.lib().pa_status_string(0) == b"PA_OK"
    assert pk.lib().pa_status_string(3) == b"PA_ERR_WORKSPACE"


def test_workspace_size():
    ws = pk.workspace_size(256, 256, 32, 8, 128)
    assert ws > 0 and ws % 256 == 0
    assert pk.workspace_size(1, 1, 30, 8, 128) == 0     # 30 % 8 != 0
    assert pk.workspace_size(1, 1, 32, 8, 96) == 0      # head_dim not built
    assert pk.cascade_workspace_size(64, 64, 32, 8, 128, 8192) > ws // 100


def call_attention(head_dim=128, block_size=16, hq=32, hkv=8, scale=0.1, ws_bytes=1 << 30,
                   short_rows=-1, split_keys=0):
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: arguments fail first
    kv = pk.KVDesc(1 << 20, 1 << 21, 100, block_size, hkv, head_dim)
    return pk.lib().pa_attention_ex(fake, ctypes.byref(kv), fake, 4, fake, fake, fake, 2, 3, hq,
                                    scale, fake, None, ctypes.c_void_p(1 << 22), ws_bytes,
                                    short_rows, split_keys, None)


def test_attention_rejects_bad_arguments_on_host():
    assert call_attention(head_dim=96) == pk.PA_ERR_UNSUPPORTED
    assert call_attention(block_size=24) == pk.PA_ERR_UNSUPPORTED
    assert call_attention(block_size=512) == pk.PA_ERR_UNSUPPORTED
    assert call_attention(hq=30) == pk.PA_ERR_INVALID_ARG
    assert call_attention(scale=float("nan")) == pk.PA_ERR_INVALID_ARG
    assert call_attention(short_rows=65) == pk.PA_ERR_INVALID_ARG
    assert call_attention(split_keys=100) == pk.PA_ERR_INVALID_ARG
    assert call_attention(ws_bytes=1024) == pk.PA_ERR_WORKSPACE
    assert b"workspace" in pk.lib().pa_last_error_message()


def test_write_kv_rejects_bad_arguments_on_host():
    kv = pk.KVDesc(1 << 20, 1 << 21, 100, 16, 8, 80)
    f = ctypes.c_void_p(1 << 20)
    assert pk.lib().pa_write_kv(f, f, f, 4, ctypes.byref(kv), None) == pk.PA_ERR_UNSUPPORTED
    kv = pk.KVDesc(1 << 20, (1 << 21) + 8, 100, 16, 8, 128)   # misaligned cache
    assert pk.lib().pa_write_kv(f, f, f, 4, ctypes.byref(kv), None) == pk.PA_ERR_INVALID_ARG


def call_fused(k=1 << 20, slots=1 << 20, n_new=4, head_dim=128, ws_bytes=1 << 30):
    """pa_write_kv_attention with pointers that are never dereferenced: every
    case below fails its host checks before any CUDA call."""
    f = ctypes.c_void_p(1 << 20)
    kv = pk.KVDesc(1 << 20, 1 << 21, 100, 16, 8, head_dim)
    return pk.lib().pa_write_kv_attention(
        ctypes.c_void_p(k), f, ctypes.c_void_p(slots) if slots else None, n_new, f,
        ctypes.byref(kv), f, 4, f, f, f, 2, 3, 32, 0.1, f, None, ctypes.c_void_p(1 << 22),
        ws_bytes, None)


def test_write_kv_attention_rejects_bad_arguments_on_host():
    assert call_fused(k=(1 << 20) + 8) == pk.PA_ERR_INVALID_ARG    # misaligned new K rows
    assert call_fused(slots=0) == pk.PA_ERR_INVALID_ARG            # no slot mapping
    assert call_fused(n_new=-1) == pk.PA_ERR_INVALID_ARG
    assert call_fused(head_dim=96) == pk.PA_ERR_UNSUPPORTED
    assert call_fused(ws_bytes=1024) == pk.PA_ERR_WORKSPACE
    assert b"workspace" in pk.lib().pa_last_error_message()


def good_meta():
    bt = torch.tensor([[3, 7, 11], [3, 7, 5]], dtype=torch.int32)
    qsl = torch.tensor([0, 5, 6], dtype=torch.int32)
    ctx = torch.tensor([30, 40], dtype=torch.int32)
    sl = torch.tensor([35, 41], dtype=torch.int32)
    slots = torch.tensor([11 * 16 + 14, 11 * 16 + 15, -1, 2, 3, 5 * 16 + 8], dtype=torch.int64)
    return bt, qsl, ctx, sl, slots


def test_validate_metadata_accepts_good_metadata():
    bt, qsl, ctx, sl, slots = good_meta()
    pk.pa_validate_metadata(bt, qsl, ctx, sl, num_blocks=12, block_size=16, slot_mapping=slots)


@pytest.mark.parametrize("mutate,needle", [
    (lambda m: m[3].__setitem__(0, 36), b"seq_lens"),
    (lambda m: m[1].__setitem__(2, 4), b"decreases"),
    (lambda m: m[0].__setitem__((1, 2), 12), b"out of range"),
    (lambda m: m[0].__setitem__((0, 0), -1), b"out of range"),
    (lambda m: m[4].__setitem__(3, 12 * 16), b"outside pool"),
    (lambda m: m[4].__setitem__(4, 2), b"twice"),
])
def test_validate_metadata_rejects(mutate, needle):
    m = list(good_meta())
    mutate(m)
    with pytest.raises(pk.PaError) as e:
        pk.pa_validate_metadata(m[0], m[1], m[2], m[3], num_blocks=12, block_size=16,
                                slot_mapping=m[4])
    assert e.value.code == pk.PA_ERR_BAD_METADATA
    assert needle in pk.lib().pa_last_error_message()


def test_fp8_descriptor_is_checked_on_host():
    """The fp8 pool's descriptor fields are validated before any CUDA call."""
    lib = pk.lib()
    fake = ctypes.c_void_p(1 << 20)
    cases = [
        (pk.KVDesc(1 << 20, 1 << 21, 100, 16, 8, 128, 7, 0, 1 << 22, 1 << 22), pk.PA_ERR_UNSUPPORTED),
        (pk.KVDesc(1 << 20, 1 << 21, 100, 16, 8, 64, pk.PA_KV_FP8_E4M3, 0, 1 << 22, 1 << 22),
         pk.PA_ERR_UNSUPPORTED),                                       # fp8 needs head_dim 128
        (pk.KVDesc(1 << 20, 1 << 21, 100, 16, 8, 128, pk.PA_KV_FP8_E4M3, 0, None, 1 << 22),
         pk.PA_ERR_INVALID_ARG),                                       # missing k_scale
        (pk.KVDesc(1 << 20, 1 << 21, 100, 16, 8, 128, pk.PA_KV_FP8_E4M3, 0, (1 << 22) + 2,
                   1 << 22), pk.PA_ERR_INVALID_ARG),                   # misaligned scale
        (pk.KVDesc(1 << 20, 1 << 21, 100, 16, 8, 128, pk.PA_KV_BF16, 3, None, None),
         pk.PA_ERR_INVALID_ARG),                                       # reserved != 0
    ]
    for kv, want in cases:
        assert lib.pa_write_kv(fake, fake, fake, 4, ctypes.byref(kv), None) == want
    # on an fp8 pool, prefix attention and cascade decode need room for the
    # prefix's bf16 copy beyond their layout: refused on the host without it
    kv = pk.KVDesc(1 << 20, 1 << 21, 100, 16, 8, 128, pk.PA_KV_FP8_E4M3, 0, 1 << 22, 1 << 22)
    base = pk.cascade_workspace_size(1, 4, 32, 8, 128, 64)
    extra = pk.cascade_fp8_staging_bytes(8, 128, 16, 64)
    assert base > 0 and extra >= 4 * 2 * (8 * 16 * 128 * 2)   # 4 blocks of K and V in bf16
    rc = lib.pa_prefix_attention(fake, ctypes.byref(kv), fake, 64, 4, 32, 0.1, fake, None,
                                 ctypes.c_void_p(1 << 23), base, None)
    assert rc == pk.PA_ERR_WORKSPACE
    rc = lib.pa_cascade_decode(fake, ctypes.byref(kv), fake, 64, fake, 8, fake, fake, fake, 4, 4,
                               32, 0.1, fake, None, ctypes.c_void_p(1 << 23),
                               pk.cascade_workspace_size(4, 4, 32, 8, 128, 64), None)
    assert rc == pk.PA_ERR_WORKSPACE
    assert pk.cascade_fp8_staging_bytes(8, 128, 16, 0) == 0


def test_kv_descriptor_layout():
    """Python's ctypes mirror of pa_kv_desc: two pointers, six int32, two
    pointers (56 bytes, pointer-aligned)."""
    assert ctypes.sizeof(pk.KVDesc) == 56
    assert pk.KVDesc.k_scale.offset == 40 and pk.KVDesc.v_scale.offset == 48
