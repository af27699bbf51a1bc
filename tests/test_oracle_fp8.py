"""Pins of the oracle's FP8 (e4m3) KV-cache functions, against things other
than the oracle itself: torch's float8_e4m3fn conversion (a library routine
for the same format), closed forms of the format, the already-pinned bf16
attention path, and the brute-force loops.

The pages only name KV-cache quantisation (2048ai.net page on the vLLM V1
engine, §02 推理优化); the format (OCP E4M3: bias 7, 3 mantissa bits, no
infinity, max 448), round-to-nearest-even with saturation, and one fp32 scale
per kv head for K and for V are the readings the oracle and the kernels share.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import brute

E4M3_MAX = 448.0


def torch_encode(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def torch_decode(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()


def all_codes():
    return np.arange(256, dtype=np.uint8)


def finite_codes():
    c = all_codes()
    return c[(c & 0x7F) != 0x7F]


def test_decode_matches_torch_for_every_code():
    c = all_codes()
    ours, ref = oracle.e4m3_decode(c), torch_decode(c)
    nan = (c & 0x7F) == 0x7F
    assert np.isnan(ours[nan]).all() and np.isnan(ref[nan]).all()
    assert np.array_equal(ours[~nan], ref[~nan])


def test_decode_closed_forms():
    v = oracle.e4m3_decode(np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x7E, 0xFE, 0x80], np.uint8))
    assert list(v) == [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 448.0, -448.0, 0.0]
    assert math.copysign(1.0, v[-1]) == -1.0  # negative zero


def test_every_finite_value_encodes_to_itself():
    c = finite_codes()
    vals = oracle.e4m3_decode(c).astype(np.float32)
    enc = oracle.e4m3_encode(vals)
    # +0 and -0 are distinct codes of equal value
    assert np.array_equal(enc, c)


def test_midpoints_round_to_even_mantissa():
    c = finite_codes()
    pos = np.sort(oracle.e4m3_decode(c[c < 0x80]))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    assert np.array_equal((mids.astype(np.float64) * 2).astype(np.float32) / 2, mids)  # exact
    enc = oracle.e4m3_encode(mids)
    lo = oracle.e4m3_encode(pos[:-1].astype(np.float32))
    hi = oracle.e4m3_encode(pos[1:].astype(np.float32))
    want = np.where((lo & 1) == 0, lo, hi)  # the neighbour with the even mantissa
    assert np.array_equal(enc, want)
    assert np.array_equal(enc, torch_encode(mids))


def test_encode_matches_torch_on_random_values():
    rng = np.random.default_rng(5)
    mag = np.exp2(rng.uniform(-14, math.log2(E4M3_MAX), 200_000))
    x = (mag * rng.choice([-1.0, 1.0], mag.size)).astype(np.float32)
    x = x[np.abs(x) <= E4M3_MAX]
    assert np.array_equal(oracle.e4m3_encode(x), torch_encode(x))


def test_encode_saturates_and_keeps_nan():
    x = np.array([448.0, 449.0, 463.9, 464.0, 1e30, np.inf, -500.0, -np.inf, np.nan],
                 np.float32)
    assert list(oracle.e4m3_encode(x)) == [0x7E] * 6 + [0xFE, 0xFE, 0x7F]


def random_codes(gen, shape, max_exp=11):
    """Finite codes with exponent field 1..max_exp (magnitudes 2^-6 .. ~2^(max_exp-6))."""
    sign = torch.randint(0, 2, shape, generator=gen, dtype=torch.int32) << 7
    e = torch.randint(1, max_exp + 1, shape, generator=gen, dtype=torch.int32) << 3
    m = torch.randint(0, 8, shape, generator=gen, dtype=torch.int32)
    return (sign | e | m).to(torch.uint8).numpy()


def bf16_bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_write_kv_fp8_places_scaled_codes_and_skips_padding():
    gen = torch.Generator().manual_seed(11)
    nb, hkv, bs, d, T = 6, 2, 4, 8, 5
    k = torch.randn(T, hkv, d, generator=gen).to(torch.bfloat16)
    v = torch.randn(T, hkv, d, generator=gen).to(torch.bfloat16)
    ks = np.array([0.0371, 0.0125], np.float32)
    vs = np.array([0.0213, 0.0490], np.float32)
    slots = np.array([5, -1, 17, 0, 23], np.int64)
    kc0 = random_codes(gen, (nb, hkv, bs, d))
    vc0 = random_codes(gen, (nb, hkv, bs, d))
    kc, vc = oracle.write_kv_fp8(k, v, slots, kc0, vc0, ks, vs)
    want_k, want_v = kc0.copy(), vc0.copy()
    kf, vf = k.float().numpy(), v.float().numpy()
    for t, s in enumerate(slots):
        if s < 0:
            continue
        # binary32 quotient, then torch's e4m3 conversion
        want_k[s // bs, :, s % bs] = torch_encode((kf[t] / ks[:, None]).astype(np.float32))
        want_v[s // bs, :, s % bs] = torch_encode((vf[t] / vs[:, None]).astype(np.float32))
    assert np.array_equal(kc, want_k) and np.array_equal(vc, want_v)


def small_fp8_case(gen, k_scale, v_scale, hq=4, hkv=2, d=8, bs=4):
    reqs = [(0, 5), (6, 1), (3, 4)]  # (context, q_len)
    tables = [[0, 1], [2, 3], [5, 4]]
    nb = 6
    kc = random_codes(gen, (nb, hkv, bs, d), max_exp=8)
    vc = random_codes(gen, (nb, hkv, bs, d), max_exp=8)
    T = sum(n for _, n in reqs)
    q = torch.randn(T, hq, d, generator=gen).to(torch.bfloat16)
    qsl = np.cumsum([0] + [n for _, n in reqs]).astype(np.int32)
    ctx = np.array([c for c, _ in reqs], np.int32)
    sl = np.array([c + n for c, n in reqs], np.int32)
    bt = np.array(tables, np.int32)
    return q, kc, vc, np.asarray(k_scale, np.float32), np.asarray(v_scale, np.float32), bt, qsl, \
        ctx, sl


def test_fp8_attention_with_power_of_two_scales_equals_bf16_attention():
    """With power-of-two scales every dequantised element is a bf16 value, so
    attention over the fp8 cache must equal the (pinned) bf16 attention over
    a bf16 cache holding those values."""
    gen = torch.Generator().manual_seed(12)
    q, kc, vc, ks, vs, bt, qsl, ctx, sl = small_fp8_case(gen, [2.0 ** -4, 2.0 ** -3],
                                                         [2.0 ** -2, 2.0 ** -5])
    kd = torch_decode(kc) * ks[None, :, None, None]
    vd = torch_decode(vc) * vs[None, :, None, None]
    kb = torch.from_numpy(kd).to(torch.bfloat16)
    vb = torch.from_numpy(vd).to(torch.bfloat16)
    assert np.array_equal(kb.double().numpy(), kd) and np.array_equal(vb.double().numpy(), vd)
    scale = 1 / math.sqrt(q.shape[-1])
    o8, l8 = oracle.attention_fp8(q, kc, vc, ks, vs, bt, qsl, ctx, sl, scale)
    o16, l16 = oracle.attention(q, kb, vb, bt, qsl, ctx, sl, scale)
    assert np.allclose(o8, o16, rtol=0, atol=1e-12) and np.allclose(l8, l16, rtol=0, atol=1e-12)


def test_fp8_attention_matches_brute_force_with_arbitrary_scales():
    gen = torch.Generator().manual_seed(13)
    q, kc, vc, ks, vs, bt, qsl, ctx, sl = small_fp8_case(gen, [0.0173, 0.0611], [0.0297, 0.0089])
    scale = 1 / math.sqrt(q.shape[-1])
    o8, l8 = oracle.attention_fp8(q, kc, vc, ks, vs, bt, qsl, ctx, sl, scale)
    kd = torch_decode(kc) * ks.astype(np.float64)[None, :, None, None]
    vd = torch_decode(vc) * vs.astype(np.float64)[None, :, None, None]
    qd = q.double().numpy()
    ob, lb = brute.attention_values(qd, kd, vd, bt, qsl, ctx, sl, scale)
    assert np.allclose(o8, ob, rtol=0, atol=1e-10) and np.allclose(l8, lb, rtol=0, atol=1e-10)


def test_fp8_write_then_attend_is_close_to_bf16_attention():
    """Quantisation error bound: e4m3 keeps 4 significant bits, so each
    dequantised element is within 2^-4 relative (half an ulp) of the scaled
    bf16 input when no element is subnormal or saturated; attention over the
    fp8 cache then stays close to attention over the exact values."""
    gen = torch.Generator().manual_seed(14)
    hkv, hq, d, bs, L = 2, 4, 16, 4, 12
    k = torch.randn(L, hkv, d, generator=gen).to(torch.bfloat16)
    v = torch.randn(L, hkv, d, generator=gen).to(torch.bfloat16)
    q = torch.randn(1, hq, d, generator=gen).to(torch.bfloat16)
    ks = np.array([1 / 16, 1 / 24], np.float32)
    vs = np.array([1 / 20, 1 / 16], np.float32)
    slots = np.arange(L, dtype=np.int64)
    nb = L // bs
    kc, vc = oracle.write_kv_fp8(k, v, slots, np.zeros((nb, hkv, bs, d), np.uint8),
                                 np.zeros((nb, hkv, bs, d), np.uint8), ks, vs)
    kd = oracle.e4m3_decode(kc) * ks[None, :, None, None]
    kx = k.double().numpy().reshape(nb, bs, hkv, d).transpose(0, 2, 1, 3)
    normal = np.abs(kx) >= 2.0 ** -6 * ks[None, :, None, None]
    assert np.all(np.abs(kd - kx)[normal] <= 2.0 ** -4 * np.abs(kx)[normal] + 1e-12)
    bt = np.arange(nb, dtype=np.int32)[None]
    qsl, ctx, sl = np.array([0, 1], np.int32), np.array([L - 1], np.int32), np.array([L], np.int32)
    o8, _ = oracle.attention_fp8(q, kc, vc, ks, vs, bt, qsl, ctx, sl, 0.25)
    kb = torch.from_numpy(kx.astype(np.float32)).to(torch.bfloat16)
    vb = torch.from_numpy(v.double().numpy().reshape(nb, bs, hkv, d).transpose(0, 2, 1, 3)
                          .astype(np.float32)).to(torch.bfloat16)
    o16, _ = oracle.attention(q, kb, vb, bt, qsl, ctx, sl, 0.25)
    assert np.abs(o8 - o16).max() < 0.1
