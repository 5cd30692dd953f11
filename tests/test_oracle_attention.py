"""Pins of the attention oracle against closed forms, invariants and a library routine.

Every test builds its own tiny paged inputs: logical per-sequence K/V first,
then a scatter into a shuffled block pool with numpy fancy indexing, so that
the expected values never pass through the oracle's own gather.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as oracle

SCALE128 = 1.0 / math.sqrt(128.0)


def to_bf16_bits(x) -> np.ndarray:
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bits_to_f64(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def paged_pool(logical, block_size, num_blocks, rng, fill_value=None):
    """Scatter each sequence's logical [n, Hkv, D] rows into a shuffled pool.

    Returns (pool [NB, bs, Hkv, D] uint16, block_tables [S, MB] int32)."""
    hkv, d = logical[0].shape[1:]
    if fill_value is None:
        pool = to_bf16_bits(rng.standard_normal((num_blocks, block_size, hkv, d)))
    else:
        pool = np.full((num_blocks, block_size, hkv, d), fill_value, dtype=np.uint16)
    need = [-(-x.shape[0] // block_size) for x in logical]
    mb = max(max(need), 1)
    perm = rng.permutation(num_blocks)
    tables = np.full((len(logical), mb), -1, dtype=np.int32)
    flat = pool.reshape(num_blocks * block_size, hkv, d)
    taken = 0
    for i, x in enumerate(logical):
        ids = perm[taken:taken + need[i]]
        taken += need[i]
        tables[i, :need[i]] = ids
        pos = np.arange(x.shape[0])
        flat[ids[pos // block_size] * block_size + pos % block_size] = x
    return pool, tables


def same_pool_layout(pool_k, pool_v):
    assert pool_k.shape == pool_v.shape


# ------------------------------------------------------------ store pins --

def test_store_then_read_back_by_slot():
    rng = np.random.default_rng(1)
    nb, bs, hkv, d, t = 9, 4, 2, 16, 13
    k_cache = np.full((nb, bs, hkv, d), 0xFFFF, dtype=np.uint16)
    v_cache = k_cache.copy()
    slots = rng.choice(nb * bs, size=t, replace=False).astype(np.int32)
    slots[3] = -1  # padded token: no write
    key = rng.integers(0, 1 << 16, size=(t, hkv, d), dtype=np.uint16)
    value = rng.integers(0, 1 << 16, size=(t, hkv, d), dtype=np.uint16)
    oracle.store_kvcache(key, value, k_cache, v_cache, slots, bs)
    for i, s in enumerate(slots):
        if s < 0:
            continue
        assert np.array_equal(k_cache[s // bs, s % bs], key[i])
        assert np.array_equal(v_cache[s // bs, s % bs], value[i])
    written = set(int(s) for s in slots if s >= 0)
    for s in range(nb * bs):
        if s not in written:
            assert (k_cache[s // bs, s % bs] == 0xFFFF).all()
            assert (v_cache[s // bs, s % bs] == 0xFFFF).all()


def test_store_rejects_out_of_range_slot():
    k = np.zeros((2, 4, 1, 8), dtype=np.uint16)
    v = k.copy()
    with pytest.raises(oracle.OracleError):
        oracle.store_kvcache(np.ones((1, 1, 8), np.uint16), np.ones((1, 1, 8), np.uint16), k, v,
                             np.array([8], np.int32), 4)


def test_store_mid_block_chunk_matches_logical_positions():
    """A chunk that starts mid-block lands after its prefix in logical order."""
    rng = np.random.default_rng(2)
    bs, hkv, d, prefix, chunk = 4, 1, 8, 6, 7
    table = np.array([5, 0, 3, 1], np.int32)
    nb = 6
    k = np.zeros((nb, bs, hkv, d), np.uint16)
    v = k.copy()
    new = rng.integers(1, 1 << 16, size=(chunk, hkv, d), dtype=np.uint16)
    pos = prefix + np.arange(chunk)
    slots = (table[pos // bs] * bs + pos % bs).astype(np.int32)
    oracle.store_kvcache(new, new, k, v, slots, bs)
    flat = k.reshape(nb * bs, hkv, d)
    for r in range(chunk):
        p = prefix + r
        assert np.array_equal(flat[table[p // bs] * bs + p % bs], new[r])


# ----------------------------------------------------------- decode pins --

@pytest.mark.parametrize("group", [1, 2, 4])
def test_decode_context_one_returns_own_value(group):
    """softmax over one key is 1: every query head of a group returns that V."""
    rng = np.random.default_rng(3)
    hkv, d, bs, nb, s = 2, 128, 16, 40, 5
    hq = hkv * group
    logical_k = [to_bf16_bits(rng.standard_normal((1, hkv, d))) for _ in range(s)]
    logical_v = [to_bf16_bits(rng.standard_normal((1, hkv, d))) for _ in range(s)]
    k_pool, tables = paged_pool(logical_k, bs, nb, np.random.default_rng(7))
    v_pool, tables_v = paged_pool(logical_v, bs, nb, np.random.default_rng(7))
    assert np.array_equal(tables, tables_v)
    q = to_bf16_bits(rng.standard_normal((s, hq, d)) * 3)
    out = oracle.paged_decode(q, k_pool, v_pool, tables, np.ones(s, np.int32), SCALE128)
    for i in range(s):
        for g in range(hq):
            assert np.array_equal(out[i, g], bits_to_f64(logical_v[i][0, g // group]))


def test_decode_equal_keys_give_mean_value():
    rng = np.random.default_rng(4)
    hkv, hq, d, bs = 2, 8, 128, 16
    lens = [1, 15, 16, 17, 300]
    logical_k, logical_v = [], []
    for n in lens:
        one = to_bf16_bits(rng.standard_normal((1, hkv, d)))
        logical_k.append(np.repeat(one, n, axis=0))
        logical_v.append(to_bf16_bits(rng.standard_normal((n, hkv, d))))
    k_pool, tables = paged_pool(logical_k, bs, 64, np.random.default_rng(9))
    v_pool, _ = paged_pool(logical_v, bs, 64, np.random.default_rng(9))
    q = to_bf16_bits(rng.standard_normal((len(lens), hq, d)))
    out = oracle.paged_decode(q, k_pool, v_pool, tables, np.array(lens, np.int32), SCALE128)
    for i, n in enumerate(lens):
        mean = bits_to_f64(logical_v[i]).mean(axis=0)  # [Hkv, D]
        for g in range(hq):
            np.testing.assert_allclose(out[i, g], mean[g // (hq // hkv)], rtol=0, atol=1e-13)


def test_decode_two_keys_closed_form():
    """Two keys with known dot products: weights are a logistic of the score gap."""
    d, bs = 128, 4
    a, b0, b1 = 2.0, 1.5, -3.0
    q = np.zeros((1, 1, d), np.float32)
    q[0, 0, 5] = a
    k = np.zeros((2, 1, d), np.float32)
    k[0, 0, 5], k[1, 0, 5] = b0, b1
    v = np.random.default_rng(5).standard_normal((2, 1, d))
    kb, vb, qb = to_bf16_bits(k), to_bf16_bits(v), to_bf16_bits(q)
    k_pool, tables = paged_pool([kb], bs, 3, np.random.default_rng(1))
    v_pool, _ = paged_pool([vb], bs, 3, np.random.default_rng(1))
    out = oracle.paged_decode(qb, k_pool, v_pool, tables, np.array([2], np.int32), SCALE128)
    s0, s1 = SCALE128 * a * b0, SCALE128 * a * b1
    w1 = 1.0 / (1.0 + math.exp(s0 - s1))
    expected = (1 - w1) * bits_to_f64(vb[0, 0]) + w1 * bits_to_f64(vb[1, 0])
    np.testing.assert_allclose(out[0, 0], expected, rtol=0, atol=1e-14)


def test_decode_zero_context_is_zero_row():
    k_pool = np.ones((2, 4, 1, 8), np.uint16)
    out = oracle.paged_decode(np.ones((2, 2, 8), np.uint16), k_pool, k_pool,
                              np.array([[0], [1]], np.int32), np.array([0, 3], np.int32), 0.3)
    assert (out[0] == 0).all()
    assert np.isfinite(out[1]).all()


def _random_decode_case(rng, lens, hkv, hq, d, bs, nb):
    logical_k = [to_bf16_bits(rng.standard_normal((n, hkv, d))) for n in lens]
    logical_v = [to_bf16_bits(rng.standard_normal((n, hkv, d))) for n in lens]
    q = to_bf16_bits(rng.standard_normal((len(lens), hq, d)))
    return logical_k, logical_v, q


def test_decode_block_permutation_invariance():
    rng = np.random.default_rng(6)
    lens = [37, 5, 64, 1]
    lk, lv, q = _random_decode_case(rng, lens, 2, 4, 32, 8, 40)
    outs = []
    for seed in (11, 12, 13):
        k_pool, tables = paged_pool(lk, 8, 40, np.random.default_rng(seed))
        v_pool, _ = paged_pool(lv, 8, 40, np.random.default_rng(seed))
        outs.append(oracle.paged_decode(q, k_pool, v_pool, tables, np.array(lens, np.int32), 0.2))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_decode_block_size_invariance():
    rng = np.random.default_rng(8)
    lens = [33, 7, 16]
    lk, lv, q = _random_decode_case(rng, lens, 2, 4, 16, 1, 1)
    outs = []
    for bs in (1, 4, 16, 64):
        nb = sum(-(-n // bs) for n in lens) + 3
        k_pool, tables = paged_pool(lk, bs, nb, np.random.default_rng(bs))
        v_pool, _ = paged_pool(lv, bs, nb, np.random.default_rng(bs))
        outs.append(oracle.paged_decode(q, k_pool, v_pool, tables, np.array(lens, np.int32), 0.25))
    for o in outs[1:]:
        assert np.array_equal(outs[0], o)


def _sdpa(q, k, v, scale, mask=None):
    """torch's scaled_dot_product_attention in fp64; q [H, L, D], k/v [Hkv, n, D]."""
    group = q.shape[0] // k.shape[0]
    kk = torch.from_numpy(k).repeat_interleave(group, dim=0)
    vv = torch.from_numpy(v).repeat_interleave(group, dim=0)
    m = None if mask is None else torch.from_numpy(mask)
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], kk[None], vv[None], attn_mask=m, scale=scale)[0].numpy()


def test_decode_matches_library_sdpa():
    rng = np.random.default_rng(10)
    lens = [300, 5000, 70]  # the pages' example requests A, B, C
    hkv, hq, d, bs = 2, 8, 128, 16
    lk, lv, q = _random_decode_case(rng, lens, hkv, hq, d, bs, 512)
    k_pool, tables = paged_pool(lk, bs, 512, np.random.default_rng(3))
    v_pool, _ = paged_pool(lv, bs, 512, np.random.default_rng(3))
    out = oracle.paged_decode(q, k_pool, v_pool, tables, np.array(lens, np.int32), SCALE128)
    for i in range(len(lens)):
        qi = bits_to_f64(q[i])[:, None, :]                      # [Hq, 1, D]
        ki = bits_to_f64(lk[i]).transpose(1, 0, 2).copy()       # [Hkv, n, D]
        vi = bits_to_f64(lv[i]).transpose(1, 0, 2).copy()
        ref = _sdpa(qi, ki, vi, SCALE128)[:, 0, :]
        np.testing.assert_allclose(out[i], ref, rtol=1e-12, atol=1e-12)


def test_decode_seq_mask_computes_only_selected():
    rng = np.random.default_rng(12)
    lens = [5, 9, 3]
    lk, lv, q = _random_decode_case(rng, lens, 1, 2, 8, 4, 10)
    k_pool, tables = paged_pool(lk, 4, 10, np.random.default_rng(1))
    v_pool, _ = paged_pool(lv, 4, 10, np.random.default_rng(1))
    full = oracle.paged_decode(q, k_pool, v_pool, tables, np.array(lens, np.int32), 0.3)
    part = oracle.paged_decode(q, k_pool, v_pool, tables, np.array(lens, np.int32), 0.3,
                               seq_mask=[0, 1, 0])
    assert np.isnan(part[0]).all() and np.isnan(part[2]).all()
    assert np.array_equal(part[1], full[1])


# ---------------------------------------------------------- prefill pins --

def _prefill_case(rng, q_lens, prefixes, hkv, hq, d, bs, extra_blocks=5, equal_keys=False):
    k_lens = [c + n for c, n in zip(prefixes, q_lens)]
    if equal_keys:
        lk = [np.repeat(to_bf16_bits(rng.standard_normal((1, hkv, d))), n, axis=0) for n in k_lens]
    else:
        lk = [to_bf16_bits(rng.standard_normal((n, hkv, d))) for n in k_lens]
    lv = [to_bf16_bits(rng.standard_normal((n, hkv, d))) for n in k_lens]
    nb = sum(-(-n // bs) for n in k_lens) + extra_blocks
    k_pool, tables = paged_pool(lk, bs, nb, np.random.default_rng(21))
    v_pool, _ = paged_pool(lv, bs, nb, np.random.default_rng(21))
    cu_q = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(k_lens)]).astype(np.int32)
    q = to_bf16_bits(rng.standard_normal((int(cu_q[-1]), hq, d)))
    return lk, lv, k_pool, v_pool, tables, cu_q, cu_k, q


def test_prefill_equal_keys_bottom_right_causal():
    """With equal keys, row r of a chunk after a c-token prefix averages V[0..c+r]."""
    rng = np.random.default_rng(13)
    q_lens, prefixes = [5, 1, 9, 4], [0, 7, 13, 16]
    hkv, hq, d, bs = 2, 4, 16, 4
    lk, lv, kp, vp, tables, cu_q, cu_k, q = _prefill_case(rng, q_lens, prefixes, hkv, hq, d, bs,
                                                         equal_keys=True)
    out = oracle.paged_prefill(q, kp, vp, cu_q, cu_k, tables, 0.4, causal=True)
    for i, (n, c) in enumerate(zip(q_lens, prefixes)):
        v = bits_to_f64(lv[i])
        for r in range(n):
            mean = v[: c + r + 1].mean(axis=0)
            for g in range(hq):
                np.testing.assert_allclose(out[cu_q[i] + r, g], mean[g // (hq // hkv)], atol=1e-13, rtol=0)


def test_prefill_noncausal_sees_all_keys():
    rng = np.random.default_rng(14)
    q_lens, prefixes = [3, 6], [4, 0]
    lk, lv, kp, vp, tables, cu_q, cu_k, q = _prefill_case(rng, q_lens, prefixes, 1, 2, 8, 4,
                                                         equal_keys=True)
    out = oracle.paged_prefill(q, kp, vp, cu_q, cu_k, tables, 0.4, causal=False)
    for i, n in enumerate(q_lens):
        mean = bits_to_f64(lv[i]).mean(axis=0)
        for r in range(n):
            for g in range(2):
                np.testing.assert_allclose(out[cu_q[i] + r, g], mean[0], atol=1e-13, rtol=0)


def test_prefill_matches_library_sdpa_with_bottom_right_mask():
    rng = np.random.default_rng(15)
    q_lens, prefixes = [40, 17, 64], [0, 23, 100]
    hkv, hq, d, bs = 2, 8, 128, 16
    lk, lv, kp, vp, tables, cu_q, cu_k, q = _prefill_case(rng, q_lens, prefixes, hkv, hq, d, bs)
    out = oracle.paged_prefill(q, kp, vp, cu_q, cu_k, tables, SCALE128, causal=True)
    for i, (n, c) in enumerate(zip(q_lens, prefixes)):
        qi = bits_to_f64(q[cu_q[i]:cu_q[i + 1]]).transpose(1, 0, 2).copy()  # [Hq, n, D]
        ki = bits_to_f64(lk[i]).transpose(1, 0, 2).copy()
        vi = bits_to_f64(lv[i]).transpose(1, 0, 2).copy()
        mask = np.arange(c + n)[None, :] <= (c + np.arange(n))[:, None]
        ref = _sdpa(qi, ki, vi, SCALE128, mask).transpose(1, 0, 2)
        np.testing.assert_allclose(out[cu_q[i]:cu_q[i + 1]], ref, rtol=1e-12, atol=1e-12)


def test_prefill_last_row_equals_decode():
    rng = np.random.default_rng(16)
    q_lens, prefixes = [8, 3, 20], [11, 0, 45]
    hkv, hq, d, bs = 2, 4, 32, 8
    lk, lv, kp, vp, tables, cu_q, cu_k, q = _prefill_case(rng, q_lens, prefixes, hkv, hq, d, bs)
    out = oracle.paged_prefill(q, kp, vp, cu_q, cu_k, tables, 0.2, causal=True)
    last_rows = cu_q[1:] - 1
    dec = oracle.paged_decode(q[last_rows], kp, vp, tables, (cu_k[1:] - cu_k[:-1]).astype(np.int32), 0.2)
    assert np.array_equal(out[last_rows], dec)


def test_prefill_row_mask_and_permutation_invariance():
    rng = np.random.default_rng(17)
    q_lens, prefixes = [9, 4], [3, 30]
    lk, lv, kp, vp, tables, cu_q, cu_k, q = _prefill_case(rng, q_lens, prefixes, 2, 4, 16, 4)
    full = oracle.paged_prefill(q, kp, vp, cu_q, cu_k, tables, 0.3)
    mask = np.zeros(int(cu_q[-1]), np.uint8)
    mask[[0, 5, 11]] = 1
    part = oracle.paged_prefill(q, kp, vp, cu_q, cu_k, tables, 0.3, row_mask=mask)
    assert np.array_equal(part[mask == 1], full[mask == 1])
    assert np.isnan(part[mask == 0]).all()
    # re-place the same logical K/V into a differently shuffled pool
    nb = kp.shape[0]
    kp2, t2 = paged_pool(lk, 4, nb, np.random.default_rng(99))
    vp2, _ = paged_pool(lv, 4, nb, np.random.default_rng(99))
    assert not np.array_equal(t2, tables)
    assert np.array_equal(oracle.paged_prefill(q, kp2, vp2, cu_q, cu_k, t2, 0.3), full)


def test_prefill_rejects_bad_metadata():
    kp = np.zeros((4, 4, 1, 8), np.uint16)
    q = np.zeros((3, 1, 8), np.uint16)
    with pytest.raises(oracle.OracleError):  # causal chunk longer than its keys
        oracle.paged_prefill(q, kp, kp, np.array([0, 3], np.int32), np.array([0, 2], np.int32),
                             np.array([[0]], np.int32), 1.0)
    with pytest.raises(oracle.OracleError):  # block id beyond the pool
        oracle.paged_prefill(q, kp, kp, np.array([0, 3], np.int32), np.array([0, 3], np.int32),
                             np.array([[9]], np.int32), 1.0)
