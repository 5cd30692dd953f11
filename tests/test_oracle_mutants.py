"""The pins catch plausible mistakes: each test plants one in a copy of the C
oracle (on the CPU), rebuilds it, and checks that at least one pin now fails
while the unmodified oracle passes them all."""
import math
import os
import shutil

import numpy as np
import pytest

from oracle import attention as oracle
from test_oracle_attention import SCALE128, _sdpa, bits_to_f64, paged_pool, to_bf16_bits

SRC = os.path.join(os.path.dirname(oracle.__file__), "pkv_oracle.c")

# (name, original text, planted mistake); each original occurs in the source.
MUTANTS = [
    ("gqa_head_map", "g / group", "g % group"),
    ("gather_offset", "(physical_block * block_size + offset) * row;",
     "(physical_block + offset) * row;"),
    ("kv_head_stride", "k_seq + p * row + kv_head * head_dim", "k_seq + p * row + kv_head"),
    ("dropped_scale", "scores_buf[p] = scale * dot;", "scores_buf[p] = dot;"),
    ("unnormalised", "const double weight = scores_buf[p] / denom;",
     "const double weight = scores_buf[p];"),
    ("mask_off_by_one", "causal ? prefix + r + 1 : k_len", "causal ? prefix + r : k_len"),
    ("top_left_mask", "causal ? prefix + r + 1 : k_len", "causal ? r + 1 : k_len"),
    ("store_swaps_operand", "v_cache[dst + e] = value[t * row + e];",
     "v_cache[dst + e] = key[t * row + e];"),
    ("context_excludes_new_token", "const int64_t n = context_lens[i];",
     "const int64_t n = context_lens[i] > 0 ? context_lens[i] - 1 : 0;"),
    ("fp8_v_uses_k_scale", "const double vs = v_scales[slot * num_kv_heads + h];",
     "const double vs = k_scales[slot * num_kv_heads + h];"),
    ("fp8_ties_to_odd", "(err == best_err && (c & 1) == 0)", "(err == best_err && (c & 1) == 1)"),
    ("fp8_exponent_bias", "ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)"),
    ("fp8_subnormal_step", "ldexp((double)m, -9)", "ldexp((double)m, -10)"),
    ("fp8_scale_inverted", "volatile float sc = amax / 448.0f;", "volatile float sc = 448.0f / amax;"),
    ("fp8_amax_not_abs", "const float a = fabsf(bf16_bits_to_float(x[d]));",
     "const float a = bf16_bits_to_float(x[d]);"),
]


def _build(tmp_path, name, before=None, after=None):
    src = open(SRC).read()
    if before is not None:
        assert before in src, f"mutation anchor missing: {before}"
        src = src.replace(before, after)
    c_path = tmp_path / f"{name}.c"
    c_path.write_text(src)
    return oracle.load_library(oracle.build(force=True, src=str(c_path),
                                            out=str(tmp_path / f"lib{name}.so")))


def _pin_store(lib):
    rng = np.random.default_rng(1)
    nb, bs, hkv, d, t = 6, 4, 2, 8, 9
    k = np.zeros((nb, bs, hkv, d), np.uint16)
    v = k.copy()
    slots = rng.choice(nb * bs, size=t, replace=False).astype(np.int32)
    key = rng.integers(1, 1 << 16, size=(t, hkv, d), dtype=np.uint16)
    val = rng.integers(1, 1 << 16, size=(t, hkv, d), dtype=np.uint16)
    oracle.store_kvcache(key, val, k, v, slots, bs, lib=lib)
    return all(np.array_equal(k[s // bs, s % bs], key[i]) and np.array_equal(v[s // bs, s % bs], val[i])
               for i, s in enumerate(slots))


def _pin_ctx_one(lib):
    rng = np.random.default_rng(3)
    hkv, g, d, bs, s = 2, 4, 16, 4, 4
    lk = [to_bf16_bits(rng.standard_normal((1, hkv, d))) for _ in range(s)]
    lv = [to_bf16_bits(rng.standard_normal((1, hkv, d))) for _ in range(s)]
    kp, tab = paged_pool(lk, bs, 9, np.random.default_rng(2))
    vp, _ = paged_pool(lv, bs, 9, np.random.default_rng(2))
    q = to_bf16_bits(rng.standard_normal((s, hkv * g, d)))
    out = oracle.paged_decode(q, kp, vp, tab, np.ones(s, np.int32), 0.3, lib=lib)
    return all(np.array_equal(out[i, h], bits_to_f64(lv[i][0, h // g]))
               for i in range(s) for h in range(hkv * g))


def _pin_equal_keys(lib):
    rng = np.random.default_rng(4)
    hkv, hq, d, bs, lens = 2, 4, 16, 4, [3, 9, 14]
    lk = [np.repeat(to_bf16_bits(rng.standard_normal((1, hkv, d))), n, axis=0) for n in lens]
    lv = [to_bf16_bits(rng.standard_normal((n, hkv, d))) for n in lens]
    kp, tab = paged_pool(lk, bs, 12, np.random.default_rng(5))
    vp, _ = paged_pool(lv, bs, 12, np.random.default_rng(5))
    q = to_bf16_bits(rng.standard_normal((len(lens), hq, d)))
    out = oracle.paged_decode(q, kp, vp, tab, np.array(lens, np.int32), 0.5, lib=lib)
    return all(np.allclose(out[i, h], bits_to_f64(lv[i]).mean(0)[h // 2], atol=1e-12, rtol=0)
               for i in range(len(lens)) for h in range(hq))


def _pin_two_keys(lib):
    d = 128
    q = np.zeros((1, 1, d), np.float32)
    q[0, 0, 3] = 2.0
    k = np.zeros((2, 1, d), np.float32)
    k[0, 0, 3], k[1, 0, 3] = 1.5, -3.0
    v = np.random.default_rng(6).standard_normal((2, 1, d))
    kb, vb, qb = to_bf16_bits(k), to_bf16_bits(v), to_bf16_bits(q)
    kp, tab = paged_pool([kb], 4, 2, np.random.default_rng(1))
    vp, _ = paged_pool([vb], 4, 2, np.random.default_rng(1))
    out = oracle.paged_decode(qb, kp, vp, tab, np.array([2], np.int32), SCALE128, lib=lib)
    w1 = 1.0 / (1.0 + math.exp(SCALE128 * 2.0 * (1.5 + 3.0)))
    exp = (1 - w1) * bits_to_f64(vb[0, 0]) + w1 * bits_to_f64(vb[1, 0])
    return np.allclose(out[0, 0], exp, atol=1e-13, rtol=0)


def _pin_prefill_equal_keys(lib):
    rng = np.random.default_rng(7)
    hkv, hq, d, bs = 1, 2, 8, 4
    q_lens, prefixes = [4, 3], [5, 0]
    k_lens = [a + b for a, b in zip(q_lens, prefixes)]
    lk = [np.repeat(to_bf16_bits(rng.standard_normal((1, hkv, d))), n, axis=0) for n in k_lens]
    lv = [to_bf16_bits(rng.standard_normal((n, hkv, d))) for n in k_lens]
    kp, tab = paged_pool(lk, bs, 6, np.random.default_rng(8))
    vp, _ = paged_pool(lv, bs, 6, np.random.default_rng(8))
    cu_q = np.array([0, 4, 7], np.int32)
    cu_k = np.array([0, k_lens[0], k_lens[0] + k_lens[1]], np.int32)
    q = to_bf16_bits(rng.standard_normal((7, hq, d)))
    out = oracle.paged_prefill(q, kp, vp, cu_q, cu_k, tab, 0.5, lib=lib)
    ok = True
    for i in range(2):
        v = bits_to_f64(lv[i])
        for r in range(q_lens[i]):
            for h in range(hq):
                ok &= np.allclose(out[cu_q[i] + r, h], v[: prefixes[i] + r + 1].mean(0)[0],
                                  atol=1e-12, rtol=0)
    return ok


def _pin_sdpa_decode(lib):
    rng = np.random.default_rng(9)
    hkv, hq, d, bs, lens = 2, 4, 16, 4, [7, 20]
    lk = [to_bf16_bits(rng.standard_normal((n, hkv, d))) for n in lens]
    lv = [to_bf16_bits(rng.standard_normal((n, hkv, d))) for n in lens]
    kp, tab = paged_pool(lk, bs, 10, np.random.default_rng(10))
    vp, _ = paged_pool(lv, bs, 10, np.random.default_rng(10))
    q = to_bf16_bits(rng.standard_normal((len(lens), hq, d)))
    out = oracle.paged_decode(q, kp, vp, tab, np.array(lens, np.int32), 0.35, lib=lib)
    ok = True
    for i in range(len(lens)):
        ref = _sdpa(bits_to_f64(q[i])[:, None, :], bits_to_f64(lk[i]).transpose(1, 0, 2).copy(),
                    bits_to_f64(lv[i]).transpose(1, 0, 2).copy(), 0.35)[:, 0, :]
        ok &= np.allclose(out[i], ref, atol=1e-12, rtol=1e-12)
    return ok


def _pin_fp8_codes_match_torch(lib):
    import torch
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = np.array([oracle.e4m3_value(c, lib=lib) for c in codes])
    nan = np.isnan(ref)
    if not (np.array_equal(nan, np.isnan(got)) and np.array_equal(got[~nan], ref[~nan])):
        return False
    x = np.concatenate([np.random.default_rng(11).uniform(-448, 448, 500),
                        (ref[1:0x7E] + ref[2:0x7F]) / 2]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return np.array_equal(np.array([oracle.e4m3_encode(v, lib=lib) for v in x], np.uint8), want)


def _pin_fp8_row_quantization(lib):
    import torch
    rng = np.random.default_rng(12)
    x = to_bf16_bits(rng.normal(0, 3.0, (16, 64)))
    codes, scales = oracle.quantize_rows_fp8(x, lib=lib)
    xf = bits_to_f64(x)
    amax = np.abs(xf).max(axis=1)
    if not np.array_equal(scales, (amax.astype(np.float32) / np.float32(448.0)).astype(np.float32)):
        return False
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    deq = vals * scales[:, None].astype(np.float64)
    bound = np.maximum(2.0 ** -4 * np.abs(xf), 2.0 ** -10 * scales[:, None]) * (1 + 1e-6)
    return bool((np.abs(deq - xf) <= bound).all())


def _pin_fp8_exact_decode(lib):
    from test_oracle_fp8 import representable_cache
    rng = np.random.default_rng(13)
    nb, bs, hkv, hq, d = 12, 4, 2, 4, 32
    kc, vc = representable_cache(rng, nb, bs, hkv, d), representable_cache(rng, nb, bs, hkv, d)
    k8 = np.zeros((nb, bs, hkv, d), np.uint8)
    v8 = np.zeros_like(k8)
    ks = np.zeros((nb * bs, hkv), np.float32)
    vs = np.zeros_like(ks)
    oracle.store_kvcache_fp8(kc.reshape(-1, hkv, d), vc.reshape(-1, hkv, d), k8, v8, ks, vs,
                             np.arange(nb * bs, dtype=np.int32), bs, lib=lib)
    tables = rng.permutation(nb).astype(np.int32).reshape(3, 4)
    lens = np.array([3, 16, 9], np.int32)
    q = to_bf16_bits(rng.standard_normal((3, hq, d)))
    ref = oracle.paged_decode(q, kc, vc, tables, lens, 0.3, lib=lib)
    got = oracle.paged_decode_fp8(q, k8, v8, ks, vs, tables, lens, 0.3, lib=lib)
    return np.array_equal(got, ref)


PINS = [_pin_sdpa_decode, _pin_store, _pin_ctx_one, _pin_equal_keys, _pin_two_keys, _pin_prefill_equal_keys,
        _pin_fp8_codes_match_torch, _pin_fp8_row_quantization, _pin_fp8_exact_decode]


def _run_pins(lib):
    results = {}
    for pin in PINS:
        try:
            results[pin.__name__] = bool(pin(lib))
        except oracle.OracleError:
            results[pin.__name__] = False
    return results


def test_unmodified_oracle_passes_every_pin(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc missing")
    results = _run_pins(_build(tmp_path, "original"))
    assert all(results.values()), results


@pytest.mark.parametrize("name,before,after", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(tmp_path, name, before, after):
    if shutil.which("gcc") is None:
        pytest.skip("gcc missing")
    results = _run_pins(_build(tmp_path, name, before, after))
    assert not all(results.values()), f"mutant {name} passed every pin: {results}"
