"""The seeded input generator: shapes, determinism, and block tables / slots
consistent with the oracle's block arithmetic (no GPU)."""
import numpy as np
import pytest

from oracle import blocks
from paged_kv_cache_86_gb300 import workloads as W


def _check_tables(w):
    bs = w.block_size
    used = []
    for i, n in enumerate(w.context_lens):
        nb = blocks.num_blocks(int(n), bs)
        row = w.block_tables[i]
        assert (row[:nb] >= 0).all() and (row[:nb] < w.num_blocks).all()
        assert (row[nb:] == W.PAD_BLOCK).all()
        used.extend(row[:nb].tolist())
    assert len(used) == len(set(used)), "a physical block is shared between sequences"
    assert w.block_tables.shape[1] % 32 == 0


def test_decode_3seq_matches_recipe():
    w = W.decode_3seq()
    assert w.context_lens.tolist() == [300, 5000, 70]
    assert (w.num_q_heads, w.num_kv_heads, w.block_size, w.num_blocks) == (8, 2, 16, 512)
    assert sum(blocks.num_blocks(int(n), 16) for n in w.context_lens) == 337
    _check_tables(w)
    # the step's new token of sequence i sits at position ctx_i - 1
    for i, n in enumerate(w.context_lens):
        assert w.slot_mapping[i] == blocks.slot_of(w.block_tables[i], int(n) - 1, 16)


def test_generator_is_deterministic():
    a, b = W.decode_64seq(num_seqs=8, max_len=600), W.decode_64seq(num_seqs=8, max_len=600)
    assert np.array_equal(a.block_tables, b.block_tables)
    assert np.array_equal(a.context_lens, b.context_lens)
    for k in a.tensors:
        assert (a.tensors[k] == b.tensors[k]).all()


def test_fragmented_pool_recipe():
    w = W.decode_512seq(num_seqs=64, hi=4096)
    need = sum(blocks.num_blocks(int(n), 16) for n in w.context_lens)
    assert w.num_blocks == int(np.ceil(need / 0.3))
    assert w.context_lens.min() >= 16 and w.context_lens.max() <= 4096
    _check_tables(w)


def test_lognormal_lengths_full_size_statistics():
    lens = W.lognormal_lengths(np.random.default_rng(86003 + 1000), 512)
    assert lens.min() >= 16 and lens.max() <= 4096
    assert 700 < np.median(lens) < 900          # median 800
    assert 0.01 < (lens == 4096).mean() < 0.12  # a few percent clipped at max_model_len


def test_longtail_recipe():
    w = W.decode_longtail(num_long=2, long_len=3000, num_short=20, short_len=200)
    assert sorted(w.context_lens.tolist()) == [200] * 20 + [3000] * 2
    _check_tables(w)


def test_prefill_chunks_slots_follow_prefix():
    w = W.prefill_chunks(num_seqs=6, q_len=40, max_prefix=300)
    assert np.array_equal(np.diff(w.cu_seqlens_q), np.full(6, 40))
    k_lens = np.diff(w.cu_seqlens_k)
    prefixes = k_lens - 40
    assert (prefixes >= 0).all() and (prefixes <= 300).all()
    _check_tables(w)
    t = 0
    for i in range(6):
        for r in range(40):
            assert w.slot_mapping[t] == blocks.slot_of(w.block_tables[i], int(prefixes[i]) + r, 16)
            t += 1
    assert len(set(w.slot_mapping.tolist())) == w.slot_mapping.shape[0]


@pytest.mark.parametrize("name", sorted(W.NAMED))
def test_full_size_metadata(name):
    w = W.NAMED[name](fill="none")
    _check_tables(w)
    if w.kind == "prefill":
        assert w.num_q_rows == 16384 and w.num_new_tokens == 16384
        assert np.diff(w.cu_seqlens_k).max() <= 4096
    else:
        assert w.num_new_tokens == int((w.context_lens > 0).sum())
    expected = {"decode_3seq": 3, "decode_64seq": 64, "decode_512seq": 512,
                "decode_longtail": 256, "prefill_chunks": 32}[name]
    assert w.num_seqs == expected
