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


PINS = [_pin_sdpa_decode, _pin_store, _pin_ctx_one, _pin_equal_keys, _pin_two_keys, _pin_prefill_equal_keys]


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
