"""Mixed-batch host logic (CPU only): the round builder against the pages'
worked example and budget rules, and the flattened metadata it produces."""
import numpy as np
import pytest

from paged_kv_cache_86_gb300.block_manager import BlockManager, Sequence
from paged_kv_cache_86_gb300.scheduler import Scheduled, build_batch, mixed_metadata


def test_pages_example_decode_first_then_one_chunk():
    # 推理运行时 §build_batch baseline: two decodes and a prompt of 6 under a token
    # budget of 5, 3 sequences and chunks of 3 -> d0, d1, then 3 tokens of p0
    reqs = [{"id": "d0", "phase": "decode", "prompt_left": 0},
            {"id": "p0", "phase": "prefill", "prompt_left": 6},
            {"id": "d1", "phase": "decode", "prompt_left": 0}]
    batch = build_batch(reqs, token_budget=5, max_sequences=3, prefill_chunk=3)
    assert [b.request_id for b in batch] == ["d0", "d1", "p0"]
    assert [b.tokens for b in batch] == [1, 1, 3]


def test_budgets_bound_the_round():
    reqs = [{"id": f"d{i}", "phase": "decode", "prompt_left": 0} for i in range(3)] + \
           [{"id": "w0", "phase": "waiting", "prompt_left": 100},
            {"id": "p1", "phase": "prefill", "prompt_left": 2}]
    b = build_batch(reqs, token_budget=10, max_sequences=8, prefill_chunk=4)
    assert [(x.request_id, x.tokens) for x in b] == [("d0", 1), ("d1", 1), ("d2", 1), ("w0", 4), ("p1", 2)]
    b = build_batch(reqs, token_budget=5, max_sequences=8, prefill_chunk=4)   # chunk cut by budget
    assert [(x.request_id, x.tokens) for x in b] == [("d0", 1), ("d1", 1), ("d2", 1), ("w0", 2)]
    b = build_batch(reqs, token_budget=100, max_sequences=2, prefill_chunk=4)  # sequence cap
    assert [x.request_id for x in b] == ["d0", "d1"]
    b = build_batch(reqs, token_budget=2, max_sequences=8, prefill_chunk=4)    # decodes alone fill it
    assert [x.request_id for x in b] == ["d0", "d1"]
    # N_scheduled = N_decode + N_prefill_chunk never exceeds the token budget
    for budget in range(1, 20):
        b = build_batch(reqs, token_budget=budget, max_sequences=8, prefill_chunk=4)
        assert sum(x.tokens for x in b) <= budget


def test_budget_errors():
    with pytest.raises(ValueError):
        build_batch([], 0, 1, 1)
    with pytest.raises(ValueError):
        build_batch([{"id": 1, "phase": "decode", "prompt_left": 0}] * 2, 4, 4, 4)
    assert build_batch([{"id": 1, "phase": "finished", "prompt_left": 0}], 4, 4, 4) == []


def test_mixed_metadata_flattens_decode_then_chunks():
    bs = 4
    m = BlockManager(32, bs)
    d = m.allocate(Sequence("d", list(range(10)), bs))          # 10 tokens cached, the 11th arrives
    m.append_token("d", 99)
    p = m.allocate(Sequence("p", list(range(100, 109)), bs))   # 9-token prompt, 3 already computed
    items = [Scheduled("d", "decode", 1), Scheduled("p", "prefill", 4)]
    md = mixed_metadata(items, {"d": d, "p": p}, {"d": 10, "p": 3}, bs)
    assert md.num_decode_seqs == 1
    assert md.cu_seqlens_q.tolist() == [0, 1, 5]
    assert md.cu_seqlens_k.tolist() == [0, 11, 18]            # decode sees 11, the chunk 3 + 4
    assert md.positions.tolist() == [10, 3, 4, 5, 6]
    assert md.slot_mapping.tolist() == [d.slot(10)] + [p.slot(i) for i in range(3, 7)]
    assert md.max_seqlen_q == 4 and md.max_seqlen_k == 11
    assert (md.block_tables[0, :len(d.block_table)] == d.block_table).all()
    with pytest.raises(ValueError):
        mixed_metadata(list(reversed(items)), {"d": d, "p": p}, {"d": 10, "p": 3}, bs)
