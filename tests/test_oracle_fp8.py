"""Pins of the oracle's fp8 (E4M3) KV-cache quantization and of decode over
the dequantized cache: a library routine (torch's float8_e4m3fn), closed forms
and exactly representable cases that reduce fp8 decode to the bf16 oracle."""
import numpy as np
import pytest
import torch

from oracle import attention as oracle
from paged_kv_cache_86_gb300.workloads import bf16_to_u16


def test_every_code_value_matches_torch_float8_e4m3fn():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = np.array([oracle.e4m3_value(c) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got)) and nan.sum() == 2          # 0x7F, 0xFF
    assert np.array_equal(got[~nan], ref[~nan])
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0x01) == 2.0 ** -9
    assert oracle.e4m3_value(0x08) == 2.0 ** -6                           # smallest normal


def test_encoding_matches_torch_round_to_nearest_even():
    rng = np.random.default_rng(1)
    finite = np.array([oracle.e4m3_value(c) for c in range(0x7F)])
    mids = (finite[:-1] + finite[1:]) / 2                                  # every tie
    x = np.concatenate([rng.uniform(-448, 448, 3000), rng.normal(0, 1, 2000),
                        rng.normal(0, 0.01, 1000), mids, -mids, finite, -finite]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(v) for v in x], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_encoding_saturates_and_keeps_nan():
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(449.0) == 0x7E and oracle.e4m3_encode(1e30) == 0x7E
    assert oracle.e4m3_encode(-1e30) == 0xFE
    assert oracle.e4m3_encode(float("nan")) == 0x7F
    assert oracle.e4m3_encode(2.0 ** -11) == 0x00                         # below half the smallest step
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00                         # tie: to the even code 0
    assert oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02                     # tie between 1 and 2: even


def bf16_rows(rng, shape, sigma=1.0):
    return bf16_to_u16(torch.from_numpy(rng.normal(0, sigma, shape).astype(np.float32)).to(torch.bfloat16))


def test_row_quantization_closed_forms_and_error_bound():
    rng = np.random.default_rng(2)
    x = bf16_rows(rng, (64, 128), sigma=3.0)
    codes, scales = oracle.quantize_rows_fp8(x)
    xf = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)
    amax = np.abs(xf).max(axis=1)
    # the largest element of each row lands on +-448 exactly; scale = amax / 448 in float32
    arg = np.abs(xf).argmax(axis=1)
    assert all(codes[i, arg[i]] & 0x7F == 0x7E for i in range(64))
    assert np.array_equal(scales, (amax.astype(np.float32) / np.float32(448.0)).astype(np.float32))
    # dequantization error: half a step of a 3-bit mantissa for normal codes,
    # half the subnormal step for the rest (both times the row scale)
    deq = np.vectorize(oracle.e4m3_value)(codes) * scales[:, None].astype(np.float64)
    bound = np.maximum(2.0 ** -4 * np.abs(xf), 2.0 ** -10 * scales[:, None]) * (1 + 1e-6)
    assert (np.abs(deq - xf) <= bound).all()


def test_zero_row_quantizes_to_zero_codes_and_zero_scale():
    codes, scales = oracle.quantize_rows_fp8(np.zeros((2, 128), np.uint16))
    assert not codes.any() and not scales.any()


def representable_cache(rng, nb, bs, hkv, d):
    """bf16 caches whose every (slot, head) row is exactly representable after
    quantization: E4M3 values times a power-of-two row scale, with one element
    at +-448 so that the row scale comes out as exactly that power of two. The
    E4M3 values come from torch's float8_e4m3fn, not from the oracle."""
    finite = torch.arange(0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    vals = rng.choice(np.concatenate([finite, -finite]), size=(nb, bs, hkv, d))
    vals[..., 0] = np.where(rng.random((nb, bs, hkv)) < 0.5, 448.0, -448.0)
    pow2 = 2.0 ** rng.integers(-12, -6, size=(nb, bs, hkv, 1))
    f = (vals * pow2).astype(np.float32)
    return bf16_to_u16(torch.from_numpy(f).to(torch.bfloat16))


def test_fp8_decode_equals_bf16_decode_when_quantization_is_exact():
    rng = np.random.default_rng(3)
    nb, bs, hkv, hq, d = 24, 4, 2, 6, 128
    kc, vc = representable_cache(rng, nb, bs, hkv, d), representable_cache(rng, nb, bs, hkv, d)
    # quantize the whole pool through the oracle's store, one token per slot
    k8 = np.zeros((nb, bs, hkv, d), np.uint8)
    v8 = np.zeros_like(k8)
    ks = np.zeros((nb * bs, hkv), np.float32)
    vs = np.zeros_like(ks)
    slots = np.arange(nb * bs, dtype=np.int32)
    oracle.store_kvcache_fp8(kc.reshape(-1, hkv, d), vc.reshape(-1, hkv, d), k8, v8, ks, vs, slots, bs)
    assert set(np.unique(np.log2(ks))) <= set(range(-12, -6))           # powers of two
    tables = rng.permutation(nb).astype(np.int32).reshape(4, 6)
    lens = np.array([1, 7, 24, 13], np.int32)
    q = bf16_rows(rng, (4, hq, d))
    ref = oracle.paged_decode(q, kc, vc, tables, lens, 0.3)
    got = oracle.paged_decode_fp8(q, k8, v8, ks, vs, tables, lens, 0.3)
    assert np.array_equal(got, ref)


def test_fp8_store_writes_only_named_slots():
    rng = np.random.default_rng(4)
    nb, bs, hkv, d = 6, 4, 2, 128
    k8 = np.full((nb, bs, hkv, d), 0x5A, np.uint8)
    v8 = k8.copy()
    ks = np.full((nb * bs, hkv), -1.0, np.float32)
    vs = ks.copy()
    key, val = bf16_rows(rng, (3, hkv, d)), bf16_rows(rng, (3, hkv, d))
    slots = np.array([5, -1, 22], np.int32)
    oracle.store_kvcache_fp8(key, val, k8, v8, ks, vs, slots, bs)
    for t, s in ((0, 5), (2, 22)):
        c, sc = oracle.quantize_rows_fp8(key[t])
        assert np.array_equal(k8.reshape(-1, hkv, d)[s], c) and np.array_equal(ks[s], sc)
        c, sc = oracle.quantize_rows_fp8(val[t])
        assert np.array_equal(v8.reshape(-1, hkv, d)[s], c) and np.array_equal(vs[s], sc)
    untouched = [s for s in range(nb * bs) if s not in (5, 22)]
    assert (k8.reshape(-1, hkv, d)[untouched] == 0x5A).all() and (ks[untouched] == -1).all()


def test_fp8_decode_context_one_returns_the_dequantized_value():
    rng = np.random.default_rng(5)
    nb, bs, hkv, hq, d = 4, 4, 2, 4, 128
    k8 = rng.integers(0, 0x7F, size=(nb, bs, hkv, d), dtype=np.uint8)
    v8 = rng.integers(0, 0x7F, size=(nb, bs, hkv, d), dtype=np.uint8) | (rng.integers(0, 2, size=(nb, bs, hkv, d), dtype=np.uint8) << 7)
    ks = rng.uniform(0.001, 0.01, (nb * bs, hkv)).astype(np.float32)
    vs = rng.uniform(0.001, 0.01, (nb * bs, hkv)).astype(np.float32)
    tables = np.array([[2], [0]], np.int32)
    q = bf16_rows(rng, (2, hq, d))
    out = oracle.paged_decode_fp8(q, k8, v8, ks, vs, tables, np.array([1, 1], np.int32), 0.1)
    for i, blk in enumerate((2, 0)):
        slot = blk * bs
        for g in range(hq):
            h = g // (hq // hkv)
            want = np.array([oracle.e4m3_value(c) for c in v8[blk, 0, h]]) * float(vs[slot, h])
            assert np.allclose(out[i, g], want, rtol=0, atol=1e-15)
