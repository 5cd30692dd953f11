"""Host-side block arithmetic of a paged KV cache, as the pages define it.

TEST INFRASTRUCTURE (part of the oracle). Plain Python restatements of the
closed forms and the block-manager behaviour the pages describe, used to pin
the index arithmetic that the CUDA kernels and the input generator rely on.

Sources (page title, section):
* LLM Infra 101 v0.5 (ifuryst.com feed), sections "KV Block", "KV Block
  Manager" and the block-usage bench under "推理".
* LLM Infra 101 v0.2 summary: KV size ~ 2 * L * T * H * dtype.
* Mini-SGLang 源码解析（二）: §6.8 `_make_2d_indices`, §7.3 KV capacity per
  page, §7.7 `_align_up_32`.
* nano vllm代码详解 (lpnh.cn): §2 Sequence (`num_blocks`,
  `last_block_num_tokens`, `num_cached_blocks`, `block(i)`), §3.2.1 allocate
  example, §3.2.3 `can_append`, §3.2.4 `may_append` cases.
"""
from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field


# ----------------------------------------------------------- closed forms --

def num_blocks(num_tokens: int, block_size: int) -> int:
    """Blocks that cover ``num_tokens``: ceil(num_tokens / block_size)."""
    if num_tokens < 0 or block_size < 1:
        raise ValueError("num_tokens must be >= 0 and block_size >= 1")
    return -(-num_tokens // block_size)


def last_block_num_tokens(num_tokens: int, block_size: int) -> int:
    """Tokens held by the last block: num_tokens - (num_blocks - 1) * block_size."""
    return num_tokens - (num_blocks(num_tokens, block_size) - 1) * block_size


def num_cached_blocks(num_cached_tokens: int, block_size: int) -> int:
    """Full blocks already holding KV: num_cached_tokens // block_size."""
    return num_cached_tokens // block_size


def block_token_span(i: int, num_tokens: int, block_size: int) -> tuple[int, int]:
    """Token index range [begin, end) of logical block ``i`` of a sequence."""
    if not 0 <= i < num_blocks(num_tokens, block_size):
        raise IndexError("block index out of range")
    return i * block_size, min((i + 1) * block_size, num_tokens)


def slot_of(block_table_row, position: int, block_size: int) -> int:
    """Flat cache slot of logical token ``position``: the row-major index of
    (physical block, offset) in a [num_blocks, block_size] table."""
    physical_block = int(block_table_row[position // block_size])
    offset = position % block_size
    return physical_block * block_size + offset


def make_2d_indices(ranges, stride: int) -> list[int]:
    """Flat indices of (row, begin, end) ranges of a 2-D table with row stride
    ``stride``: row * stride + col for col in [begin, end), ranges concatenated."""
    out: list[int] = []
    for row, begin, end in ranges:
        out.extend(row * stride + col for col in range(begin, end))
    return out


def align_up_32(n: int) -> int:
    """Round up to a multiple of 32 (32 int32 = 128 bytes per page-table row)."""
    return (n + 31) // 32 * 32


def kv_cache_bytes(num_layers: int, num_tokens: int, kv_width: int, dtype_bytes: int) -> int:
    """KV bytes of ``num_tokens`` tokens: 2 (K and V) * layers * tokens * width * dtype,
    where width = num_kv_heads * head_dim."""
    return 2 * num_layers * num_tokens * kv_width * dtype_bytes


def cache_bytes_per_page(head_dim: int, num_kv_heads: int, page_size: int, dtype_bytes: int,
                         num_layers: int) -> int:
    """Bytes of KV one page holds over all layers."""
    return 2 * head_dim * num_kv_heads * page_size * dtype_bytes * num_layers


def needs_new_block_on_append(seq_len_after_append: int, block_size: int) -> bool:
    """A sequence that has just grown to ``seq_len_after_append`` tokens opens a
    new block exactly when the new token is the first of a block."""
    if seq_len_after_append < 1 or block_size < 1:
        raise ValueError("sequence length and block_size must be >= 1")
    return (seq_len_after_append - 1) % block_size == 0


def append_case(seq_len_after_append: int, block_size: int) -> str:
    """Which of the three append cases a decode step hits: 'new_block' (the new
    token starts a block), 'block_filled' (it completes one), or 'middle'."""
    if needs_new_block_on_append(seq_len_after_append, block_size):
        return "new_block"
    if seq_len_after_append % block_size == 0:
        return "block_filled"
    return "middle"


# -------------------------------------------------------- block manager --

@dataclass
class RequestBlocks:
    request_id: str
    block_ids: list[int] = field(default_factory=list)
    token_count: int = 0


class BlockManager:
    """A fixed pool of ``total_blocks`` blocks with a FIFO free list.

    allocate(request, n): takes ceil(n / bs) blocks from the head of the free list.
    append_tokens(request, n): takes only the extra blocks the longer sequence needs.
    release(request): returns the request's blocks to the tail of the free list.
    Invalid counts and duplicate requests raise ValueError, unknown requests
    KeyError, and a pool that cannot cover a request raises MemoryError.
    """

    def __init__(self, total_blocks: int, block_size: int = 16):
        if total_blocks < 1:
            raise ValueError("total_blocks must be at least 1")
        if block_size < 1:
            raise ValueError("block_size must be at least 1")
        self.total_blocks = total_blocks
        self.block_size = block_size
        self.free_block_ids: deque[int] = deque(range(total_blocks))
        self.tables: dict[str, RequestBlocks] = {}

    def _take(self, count: int) -> list[int]:
        if count > len(self.free_block_ids):
            raise MemoryError(f"need {count} blocks, {len(self.free_block_ids)} free")
        return [self.free_block_ids.popleft() for _ in range(count)]

    def allocate(self, request_id: str, token_count: int) -> RequestBlocks:
        if request_id in self.tables:
            raise ValueError(f"request already holds blocks: {request_id}")
        if token_count < 0:
            raise ValueError("token_count must be non-negative")
        blocks = self._take(num_blocks(token_count, self.block_size))
        self.tables[request_id] = RequestBlocks(request_id, blocks, token_count)
        return self.snapshot(request_id)

    def append_tokens(self, request_id: str, token_count: int = 1) -> RequestBlocks:
        if token_count < 0:
            raise ValueError("token_count must be non-negative")
        if request_id not in self.tables:
            raise KeyError(f"request holds no blocks: {request_id}")
        table = self.tables[request_id]
        grown = table.token_count + token_count
        extra = num_blocks(grown, self.block_size) - num_blocks(table.token_count, self.block_size)
        table.block_ids.extend(self._take(extra))
        table.token_count = grown
        return self.snapshot(request_id)

    def release(self, request_id: str) -> list[int]:
        if request_id not in self.tables:
            raise KeyError(f"request holds no blocks: {request_id}")
        table = self.tables.pop(request_id)
        self.free_block_ids.extend(table.block_ids)
        return list(table.block_ids)

    def snapshot(self, request_id: str) -> RequestBlocks:
        t = self.tables[request_id]
        return RequestBlocks(t.request_id, list(t.block_ids), t.token_count)

    def usage(self) -> dict:
        """Block-usage figures of the live requests."""
        allocated = sum(t.token_count for t in self.tables.values())
        used = sum(len(t.block_ids) for t in self.tables.values())
        reserved = used * self.block_size
        return {
            "allocated_tokens": allocated,
            "reserved_tokens": reserved,
            "internal_fragmentation_tokens": reserved - allocated,
            "block_utilization": allocated / reserved if reserved else 0.0,
            "used_blocks": used,
            "free_blocks": len(self.free_block_ids),
        }


def contiguous_baseline(request_tokens) -> dict:
    """Every request reserves one contiguous slot as long as the longest request."""
    request_tokens = list(request_tokens)
    allocated = sum(request_tokens)
    reserved = len(request_tokens) * max(request_tokens, default=0)
    return {
        "reserved_tokens": reserved,
        "internal_fragmentation_tokens": reserved - allocated,
        "utilization": allocated / reserved if reserved else 0.0,
    }


def block_usage_report(request_tokens, block_size: int, total_blocks: int) -> dict:
    """Allocate every request in a fresh pool and compare with the contiguous baseline."""
    manager = BlockManager(total_blocks, block_size)
    for i, n in enumerate(request_tokens):
        manager.allocate(f"req-{i}", n)
    usage = manager.usage()
    baseline = contiguous_baseline(request_tokens)
    return {
        "block_size": block_size,
        "block_usage": usage,
        "contiguous_fixed_slot_baseline": baseline,
        "fragmentation_tokens_saved_vs_contiguous":
            baseline["internal_fragmentation_tokens"] - usage["internal_fragmentation_tokens"],
        "request_tokens": list(request_tokens),
    }
