"""Host block manager with prefix caching and copy-on-write (CPU only): the
pages' worked examples, sharing and release rules, COW pairs, cache-key
separation, and bookkeeping invariants under a random workload."""
import random

import pytest

from paged_kv_cache_86_gb300.block_manager import (BlockManager, CacheKey, CopyOp, Sequence,
                                                   chain_hash)


def seq(sid, toks, bs):
    return Sequence(sid, toks, bs)


def test_block_split_of_a_ten_token_sequence():
    # nano vllm代码详解 §3.2.1: seq_len 10 at block_size 4 -> blocks of 4, 4, 2
    s = seq("a", range(10), 4)
    assert s.num_blocks == 3
    assert [len(s.block(i)) for i in range(3)] == [4, 4, 2]
    assert s.last_block_num_tokens == 2


def test_fresh_pool_allocation_takes_the_head_of_the_free_list():
    # LLM Infra 101 v0.5 "KV Block Manager": 33 tokens at block 16 from a pool of 5
    m = BlockManager(5, 16)
    s = m.allocate(seq("a", range(33), 16))
    assert s.block_table == [0, 1, 2]
    assert list(m.free_block_ids) == [3, 4]


def test_shared_prefix_reuses_the_full_block_and_misses_after():
    # nano vllm代码详解 §3.2 example: seq1 A B C D | E F, seq2 A B C D | X Y
    A, B, C, D, E, F, X, Y = range(8)
    m = BlockManager(8, 4)
    s1 = m.allocate(seq(1, [A, B, C, D, E, F], 4))
    s2 = m.allocate(seq(2, [A, B, C, D, X, Y], 4))
    assert s1.block_table[0] == s2.block_table[0]
    assert s1.block_table[1] != s2.block_table[1]
    assert s2.num_cached_tokens == 4 and s1.num_cached_tokens == 0
    assert m.blocks[s1.block_table[0]].ref_count == 2
    # once a block misses, later blocks miss too even if their own tokens match
    s3 = m.allocate(seq(3, [A, B, C, X, E, F, A, B], 4))
    assert s3.num_cached_tokens == 0 and s3.block_table[0] != s1.block_table[0]


def test_release_is_last_to_first_and_keeps_hashes_for_reuse():
    m = BlockManager(6, 2)
    s = m.allocate(seq("a", [1, 2, 3, 4, 5], 2))        # blocks 0, 1 full; 2 partial
    assert s.block_table == [0, 1, 2]
    m.deallocate("a")
    assert list(m.free_block_ids) == [3, 4, 5, 2, 1, 0]
    # the full blocks are still found by hash and taken back from the free list
    t = m.allocate(seq("b", [1, 2, 3, 4, 9], 2))
    assert t.block_table[:2] == [0, 1] and t.num_cached_tokens == 4
    assert 0 not in m.free_block_ids and 1 not in m.free_block_ids


def test_append_starts_and_completes_blocks():
    # nano vllm代码详解 §3.2.3 / §3.2.4: a token that starts a block takes one free
    # block; a token that fills a block gets the block hashed and cached
    m = BlockManager(4, 4)
    s = m.allocate(seq("a", [10, 11, 12, 13], 4))
    assert m.blocks[s.block_table[0]].hash != -1
    assert m.can_append(s)
    assert m.append_token("a", 14) == [] and len(s.block_table) == 2     # len 5: 5 % 4 == 1
    last = m.blocks[s.block_table[1]]
    for t in (15, 16):
        m.append_token("a", t)
        assert last.hash == -1                                          # still partial
    m.append_token("a", 17)                                             # len 8: full
    assert last.hash == chain_hash([14, 15, 16, 17], m.blocks[s.block_table[0]].hash)
    assert m.hash_to_block_id[last.hash] == last.block_id


def test_fork_then_write_into_the_shared_partial_block_copies_it():
    # 推理运行时 §Prefix cache 与 copy-on-write: a branch must not write into a
    # shared block that is not yet full
    m = BlockManager(8, 4)
    m.allocate(seq("p", [1, 2, 3, 4, 5, 6], 4))                        # blocks [0, 1], 1 partial
    c = m.fork("p", "c")
    assert c.block_table == [0, 1] and m.blocks[1].ref_count == 2 and m.blocks[0].ref_count == 2
    ops = m.append_token("c", 7)
    assert ops == [CopyOp(src=1, dst=c.block_table[1], rows=2)]
    assert c.block_table[1] != 1 and m.blocks[1].ref_count == 1
    assert m.append_token("p", 8) == []                                 # the parent owns block 1 now
    # a shared FULL block is never copied: the next token starts a new block
    m.append_token("c", 9)                                              # c: [1..6, 7, 9] full
    assert m.append_token("c", 10) == []


def test_different_cache_keys_never_share():
    toks = list(range(8))
    a = BlockManager(8, 4, CacheKey(model="m", tenant="t1"))
    s1 = a.allocate(seq(1, toks, 4))
    h_t1 = a.blocks[s1.block_table[0]].hash
    b = BlockManager(8, 4, CacheKey(model="m", tenant="t2"))
    s2 = b.allocate(seq(1, toks, 4))
    assert b.blocks[s2.block_table[0]].hash != h_t1
    # one manager, one key: the same tokens are shared
    s3 = a.allocate(seq(2, toks, 4))
    assert s3.num_cached_tokens == 8


def test_chain_hash_depends_on_prefix_and_order():
    assert chain_hash([1, 2], 0) != chain_hash([2, 1], 0)
    assert chain_hash([1, 2], 0) != chain_hash([1, 2], 1)
    assert chain_hash([1, 2], 5) == chain_hash([1, 2], 5)


def test_slots_follow_the_block_table():
    m = BlockManager(10, 4)
    m.allocate(seq("x", range(3), 4))
    s = m.allocate(seq("a", range(100, 110), 4))
    assert [s.slot(p) for p in range(10)] == [
        s.block_table[p // 4] * 4 + p % 4 for p in range(10)]
    with pytest.raises(IndexError):
        s.slot(10)


def test_errors():
    m = BlockManager(2, 4)
    m.allocate(seq("a", range(8), 4))
    with pytest.raises(MemoryError):
        m.allocate(seq("b", range(100, 101), 4))
    with pytest.raises(ValueError):
        m.allocate(seq("a", range(1), 4))
    with pytest.raises(KeyError):
        m.deallocate("zzz")
    with pytest.raises(MemoryError):
        m.append_token("a", 1)                   # len 9 needs a ninth-token block


def test_bookkeeping_invariants_under_random_workload():
    rng = random.Random(86)
    bs, nb = 4, 64
    m = BlockManager(nb, bs)
    live = {}
    for step in range(3000):
        op = rng.random()
        if op < 0.25 and len(live) < 12:
            sid = f"s{step}"
            base = rng.choice([[1, 2, 3, 4, 5, 6, 7, 8], [1, 2, 3, 4, 9, 9, 9, 9], []])
            toks = base[: rng.randint(0, len(base))] + [rng.randint(0, 5) for _ in range(rng.randint(1, 9))]
            s = seq(sid, toks, bs)
            if m.can_allocate(s):
                m.allocate(s)
                live[sid] = s
        elif op < 0.35 and live and len(live) < 12:
            parent = rng.choice(list(live))
            cid = f"f{step}"
            live[cid] = m.fork(parent, cid)
        elif op < 0.85 and live:
            sid = rng.choice(list(live))
            if m.can_append(live[sid]):
                m.append_token(sid, rng.randint(0, 5))
        elif live:
            sid = rng.choice(list(live))
            m.deallocate(sid)
            del live[sid]
        # every block's count equals the number of live tables holding it
        counts = [0] * nb
        for s in live.values():
            assert len(s.block_table) == s.num_blocks
            for b in s.block_table:
                counts[b] += 1
        assert counts == [b.ref_count for b in m.blocks]
        free = set(m.free_block_ids)
        assert len(free) == len(m.free_block_ids)
        assert free.isdisjoint(m.used_block_ids) and len(free) + len(m.used_block_ids) == nb
        assert all((counts[b] > 0) == (b in m.used_block_ids) for b in range(nb))
        # a block reachable by hash holds exactly the tokens it was cached with
        for h, b in m.hash_to_block_id.items():
            assert m.blocks[b].hash == h and len(m.blocks[b].token_ids) == bs
        # no two live sequences write into a shared partial last block
        for s in live.values():
            last = m.blocks[s.block_table[-1]]
            if len(s) % bs and last.ref_count > 1:
                holders = [t for t in live.values() if t.block_table[-1] == last.block_id]
                lens = {len(t) for t in holders}
                assert len(lens) == 1    # shared only while the contents are identical
