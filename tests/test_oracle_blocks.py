"""Pins of the host-side block arithmetic against the numbers the pages print."""
import json
import os

import pytest

from oracle import blocks

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


ARITH = _load("block_arithmetic.json")


@pytest.mark.parametrize("tokens,expected", ARITH["ceil_blocks"]["cases"])
def test_ceil_blocks(tokens, expected):
    assert blocks.num_blocks(tokens, ARITH["ceil_blocks"]["block_size"]) == expected


def test_sequence_split_fills():
    case = ARITH["sequence_split"]
    n, bs = case["num_tokens"], case["block_size"]
    nb = blocks.num_blocks(n, bs)
    fills = [end - begin for begin, end in (blocks.block_token_span(i, n, bs) for i in range(nb))]
    assert fills == case["block_fills"]
    assert blocks.last_block_num_tokens(n, bs) == case["block_fills"][-1]


@pytest.mark.parametrize("n", range(0, 70))
@pytest.mark.parametrize("bs", [1, 4, 16, 256])
def test_last_block_fill_closed_form(n, bs):
    nb = blocks.num_blocks(n, bs)
    # brute force: walk the tokens block by block
    walked, filled = 0, 0
    while filled < n:
        filled += min(bs, n - filled)
        walked += 1
    assert nb == walked
    if n:
        assert blocks.last_block_num_tokens(n, bs) == n - (nb - 1) * bs
        assert 1 <= blocks.last_block_num_tokens(n, bs) <= bs
    assert blocks.num_cached_blocks(n, bs) == n // bs


def test_fresh_pool_allocation():
    case = ARITH["fresh_pool_allocation"]
    m = blocks.BlockManager(case["total_blocks"], case["block_size"])
    t = m.allocate("req-a", case["tokens"])
    assert t.block_ids == case["block_ids"]
    assert list(m.free_block_ids) == case["free_after"]


def test_append_crosses_boundary():
    case = ARITH["append_crosses_boundary"]
    m = blocks.BlockManager(16, case["block_size"])
    assert len(m.allocate("req-a", case["before"]).block_ids) == case["blocks_before"]
    assert len(m.append_tokens("req-a", case["after"] - case["before"]).block_ids) == case["blocks_after"]


@pytest.mark.parametrize("length,case", ARITH["append_cases"]["cases"])
def test_append_cases(length, case):
    assert blocks.append_case(length, ARITH["append_cases"]["block_size"]) == case


def test_append_only_grows_on_boundary():
    m = blocks.BlockManager(64, 16)
    m.allocate("r", 1)
    for n in range(2, 200):
        before = len(m.snapshot("r").block_ids)
        after = len(m.append_tokens("r", 1).block_ids)
        assert after - before == (1 if blocks.needs_new_block_on_append(n, 16) else 0)


def test_release_returns_blocks_fifo():
    m = blocks.BlockManager(6, 4)
    m.allocate("a", 8)   # 0, 1
    m.allocate("b", 5)   # 2, 3
    assert m.release("a") == [0, 1]
    assert list(m.free_block_ids) == [4, 5, 0, 1]
    assert m.allocate("c", 12).block_ids == [4, 5, 0]


def test_manager_errors():
    with pytest.raises(ValueError):
        blocks.BlockManager(0)
    with pytest.raises(ValueError):
        blocks.BlockManager(4, 0)
    m = blocks.BlockManager(2, 16)
    m.allocate("a", 16)
    with pytest.raises(ValueError):
        m.allocate("a", 1)
    with pytest.raises(ValueError):
        m.allocate("b", -1)
    with pytest.raises(KeyError):
        m.append_tokens("zz", 1)
    with pytest.raises(KeyError):
        m.release("zz")
    with pytest.raises(MemoryError):
        m.allocate("c", 17)  # over-allocation: 2 blocks wanted, 1 free


def test_block_usage_bench_matches_page():
    g = _load("block_usage_bench.json")
    inp = g["input"]
    rep = blocks.block_usage_report(inp["request_tokens"], inp["block_size"], inp["total_blocks"])
    exp = g["expected"]
    assert rep["block_usage"]["allocated_tokens"] == exp["block_usage"]["allocated_tokens"]
    assert rep["block_usage"]["reserved_tokens"] == exp["block_usage"]["reserved_tokens"]
    assert rep["block_usage"]["used_blocks"] == exp["block_usage"]["used_blocks"]
    assert rep["block_usage"]["free_blocks"] == exp["block_usage"]["free_blocks"]
    assert (rep["block_usage"]["internal_fragmentation_tokens"]
            == exp["block_usage"]["internal_fragmentation_tokens"])
    assert rep["block_usage"]["block_utilization"] == pytest.approx(
        exp["block_usage"]["block_utilization"], abs=1e-15)
    base, ebase = rep["contiguous_fixed_slot_baseline"], exp["contiguous_fixed_slot_baseline"]
    assert base["reserved_tokens"] == ebase["reserved_tokens"]
    assert base["internal_fragmentation_tokens"] == ebase["internal_fragmentation_tokens"]
    assert base["utilization"] == pytest.approx(ebase["utilization"], abs=1e-15)
    assert (rep["fragmentation_tokens_saved_vs_contiguous"]
            == exp["fragmentation_tokens_saved_vs_contiguous"])
    one = g["single_request_example"]
    single = blocks.block_usage_report([one["tokens"]], one["block_size"], 4)["block_usage"]
    assert single["reserved_tokens"] == one["reserved_tokens"]
    assert single["internal_fragmentation_tokens"] == one["internal_fragmentation_tokens"]
    assert single["block_utilization"] == one["utilization"]


def test_make_2d_indices_example():
    case = ARITH["make_2d_indices"]
    assert blocks.make_2d_indices([tuple(r) for r in case["ranges"]], case["stride"]) == case["expected"]


def test_slot_is_flat_2d_index():
    # A slot is the make_2d_indices index of (physical block, offset) in a
    # [num_blocks, block_size] table: the same flat arithmetic, both pinned.
    table = [7, 2, 5]
    bs = 4
    for pos in range(12):
        row = table[pos // bs]
        assert blocks.slot_of(table, pos, bs) == blocks.make_2d_indices([(row, pos % bs, pos % bs + 1)], bs)[0]


@pytest.mark.parametrize("n,expected", ARITH["align_up_32"]["cases"])
def test_align_up_32(n, expected):
    assert blocks.align_up_32(n) == expected


def test_cache_per_page_llama7b():
    c = ARITH["cache_per_page"]
    per_page = blocks.cache_bytes_per_page(c["head_dim"], c["num_kv_heads"], c["page_size"],
                                           c["dtype_bytes"], c["num_layers"])
    assert per_page == c["bytes"]
    assert c["available_bytes"] // per_page == c["num_pages"]


def test_kv_size_qwen3_32b():
    c = ARITH["kv_size_qwen3_32b"]
    mha = blocks.kv_cache_bytes(c["num_layers"], c["num_tokens"], c["mha_width"], c["dtype_bytes"])
    assert mha / 1024 ** 3 == c["mha_gib"]
    gqa = blocks.kv_cache_bytes(c["num_layers"], c["num_tokens"], c["gqa_width"], c["dtype_bytes"])
    assert gqa / 1e9 == pytest.approx(c["gqa_gb_decimal_approx"], abs=0.1)  # "about 33.5 GB"
    assert gqa * 5 == mha  # 8 KV heads x 128 = 1024 of a 5120-wide hidden state
