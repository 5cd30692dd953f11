"""Host block manager with prefix caching, reference counts and copy-on-write.

Decides which physical cache block each logical block of a sequence uses; the
GPU side only ever sees the results (block tables, slots, copy pairs for
``pkv_copy_blocks``). The bookkeeping follows nano-vllm's BlockManager as the
pages describe it (nano vllm代码详解 §3.1 Block, §3.2 BlockManager):

* a block holds ``block_size`` tokens; a FULL block gets a chained hash of its
  token ids and the previous block's hash, and is entered in a hash -> block
  table so that a later sequence with the same prefix reuses it (§3.2.1
  allocate: once one block misses, every later block of that sequence misses,
  because the prefix already differs); partially filled blocks are never shared
  through the cache;
* blocks are shared by reference count; releasing a sequence walks its blocks
  from the last to the first and returns a block to the free list when its
  count reaches zero, keeping its hash so that it can still be found (§3.2.2);
* a decode step appends one token: when the new token starts a block, one
  free block is taken; when it fills a block, that block's hash is computed
  and cached (§3.2.3 can_append, §3.2.4 may_append).

Added here, as the runtime page requires (推理运行时 §Prefix cache 与
copy-on-write): ``fork`` makes a branch (beam search, parallel sampling) that
shares ALL of its parent's blocks, including a partly filled last block; before
either side writes a token into a shared block that is not full, the writer
gets its own copy (a (src, dst, rows) pair for ``pkv_copy_blocks``), so the
other request's history never changes. The same page lists what a cache key
must cover besides the token ids -- model and weights, adapter, position / rope
configuration, cache dtype, tenant; ``CacheKey`` carries those and seeds the
hash chain, so blocks are only reused under an identical key.
"""
from __future__ import annotations

import hashlib
from collections import deque
from dataclasses import dataclass, field


@dataclass(frozen=True)
class CacheKey:
    """Everything besides the token ids that must match for a block to be reused."""
    model: str = ""
    adapter: str = ""
    rope: str = ""
    cache_dtype: str = "bf16"
    tenant: str = ""

    def seed(self) -> int:
        text = "\x1f".join((self.model, self.adapter, self.rope, self.cache_dtype, self.tenant))
        return int.from_bytes(hashlib.blake2b(text.encode(), digest_size=8).digest(), "little")


def chain_hash(token_ids, prefix: int) -> int:
    """64-bit hash of a full block's token ids chained to the previous block's hash."""
    h = hashlib.blake2b(digest_size=8)
    h.update(prefix.to_bytes(8, "little", signed=False))
    for t in token_ids:
        h.update(int(t).to_bytes(8, "little", signed=True))
    return int.from_bytes(h.digest(), "little")


@dataclass
class Block:
    block_id: int
    ref_count: int = 0
    hash: int = -1              # -1 until the block is full and cached
    token_ids: list = field(default_factory=list)


@dataclass(frozen=True)
class CopyOp:
    """Rows [0, rows) of block src must be copied to block dst (pkv_copy_blocks)."""
    src: int
    dst: int
    rows: int


class Sequence:
    """A request's tokens and the physical blocks that hold their K/V."""

    def __init__(self, seq_id, token_ids, block_size: int):
        self.seq_id = seq_id
        self.token_ids = list(token_ids)
        self.block_size = block_size
        self.block_table: list[int] = []
        self.num_cached_tokens = 0      # tokens whose K/V were already in the cache

    def __len__(self):
        return len(self.token_ids)

    @property
    def num_blocks(self) -> int:
        return (len(self.token_ids) + self.block_size - 1) // self.block_size

    @property
    def last_block_num_tokens(self) -> int:
        return len(self.token_ids) - (self.num_blocks - 1) * self.block_size

    def block(self, i: int) -> list:
        if not 0 <= i < self.num_blocks:
            raise IndexError(i)
        return self.token_ids[i * self.block_size:(i + 1) * self.block_size]

    def slot(self, position: int) -> int:
        """Flat cache slot of a token position: block_id * block_size + offset."""
        if not 0 <= position < len(self.token_ids):
            raise IndexError(position)
        return self.block_table[position // self.block_size] * self.block_size + position % self.block_size


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int, key: CacheKey = CacheKey()):
        if num_blocks < 1 or block_size < 1:
            raise ValueError("num_blocks and block_size must be at least 1")
        self.block_size = block_size
        self.blocks = [Block(i) for i in range(num_blocks)]
        self.free_block_ids: deque[int] = deque(range(num_blocks))
        self.used_block_ids: set[int] = set()
        self.hash_to_block_id: dict[int, int] = {}
        self.key = key
        self._seed = key.seed()
        self.seqs: dict = {}

    # ---------------------------------------------------------------- pool --
    def _take(self, block_id: int | None = None) -> Block:
        """Mark a free block used (the head of the free list unless one is named)."""
        if block_id is None:
            if not self.free_block_ids:
                raise MemoryError("no free block")
            block_id = self.free_block_ids.popleft()
        else:
            self.free_block_ids.remove(block_id)
        b = self.blocks[block_id]
        if b.hash != -1 and self.hash_to_block_id.get(b.hash) == block_id:
            del self.hash_to_block_id[b.hash]   # its old content is about to be overwritten
        b.ref_count, b.hash, b.token_ids = 1, -1, []
        self.used_block_ids.add(block_id)
        return b

    def _drop(self, block_id: int) -> None:
        b = self.blocks[block_id]
        b.ref_count -= 1
        if b.ref_count < 0:
            raise RuntimeError(f"block {block_id} released more often than taken")
        if b.ref_count == 0:
            self.used_block_ids.discard(block_id)
            self.free_block_ids.append(block_id)

    def num_free_blocks(self) -> int:
        return len(self.free_block_ids)

    # ------------------------------------------------------------ sequences --
    def can_allocate(self, seq: Sequence) -> bool:
        return len(self.free_block_ids) >= seq.num_blocks

    def allocate(self, seq: Sequence) -> Sequence:
        """Give a new sequence its blocks, reusing cached full blocks of an equal
        prefix; seq.num_cached_tokens counts the tokens whose K/V are already there."""
        if seq.seq_id in self.seqs:
            raise ValueError(f"sequence already allocated: {seq.seq_id}")
        if seq.block_size != self.block_size:
            raise ValueError("sequence block_size differs from the manager's")
        if not self.can_allocate(seq):
            raise MemoryError(f"need {seq.num_blocks} blocks, {len(self.free_block_ids)} free")
        prefix, miss = self._seed, False
        for i in range(seq.num_blocks):
            toks = seq.block(i)
            full = len(toks) == self.block_size
            h = chain_hash(toks, prefix) if full else -1
            hit_id = self.hash_to_block_id.get(h, -1) if full else -1
            if hit_id == -1 or self.blocks[hit_id].token_ids != toks:
                miss = True
            if miss:
                b = self._take()
            else:
                seq.num_cached_tokens += self.block_size
                if hit_id in self.used_block_ids:
                    b = self.blocks[hit_id]
                    b.ref_count += 1
                else:                               # cached but free: take it back
                    b = self._take(hit_id)
            if full:
                b.hash, b.token_ids = h, list(toks)
                self.hash_to_block_id[h] = b.block_id
                prefix = h
            seq.block_table.append(b.block_id)
        self.seqs[seq.seq_id] = seq
        return seq

    def fork(self, parent_id, child_id) -> Sequence:
        """A branch sharing every block of its parent (the last one possibly partial)."""
        if child_id in self.seqs:
            raise ValueError(f"sequence already allocated: {child_id}")
        parent = self.seqs[parent_id]
        child = Sequence(child_id, parent.token_ids, self.block_size)
        child.block_table = list(parent.block_table)
        child.num_cached_tokens = len(parent)
        for bid in child.block_table:
            self.blocks[bid].ref_count += 1
        self.seqs[child_id] = child
        return child

    def deallocate(self, seq_id) -> None:
        seq = self.seqs.pop(seq_id)
        for bid in reversed(seq.block_table):
            self._drop(bid)
        seq.block_table = []
        seq.num_cached_tokens = 0

    def can_append(self, seq: Sequence) -> bool:
        """Room for one more token: a new block when it starts one, or a copy of a
        shared partial last block."""
        n = len(seq) + 1
        needs = 1 if (n % self.block_size == 1 or self.block_size == 1) else 0
        if not needs and self.blocks[seq.block_table[-1]].ref_count > 1:
            needs = 1
        return len(self.free_block_ids) >= needs

    def append_token(self, seq_id, token_id) -> list[CopyOp]:
        """Append one generated token. Returns the block copies that must run on the
        GPU (pkv_copy_blocks) before the token's K/V is written."""
        seq = self.seqs[seq_id]
        seq.token_ids.append(int(token_id))
        n, bs = len(seq), self.block_size
        ops: list[CopyOp] = []
        if (n - 1) % bs == 0:                       # the token starts a new block
            if seq.block_table:
                last = self.blocks[seq.block_table[-1]]
                if last.hash == -1:
                    raise RuntimeError("previous block should be full and cached")
            seq.block_table.append(self._take().block_id)
        else:
            last = self.blocks[seq.block_table[-1]]
            if last.ref_count > 1:                  # shared partial block: copy on write
                fresh = self._take()
                ops.append(CopyOp(last.block_id, fresh.block_id, (n - 1) % bs))
                last.ref_count -= 1
                seq.block_table[-1] = fresh.block_id
        if n % bs == 0:                             # the token fills its block: cache it
            b = self.blocks[seq.block_table[-1]]
            prefix = self.blocks[seq.block_table[-2]].hash if len(seq.block_table) > 1 else self._seed
            toks = seq.block(seq.num_blocks - 1)
            b.hash, b.token_ids = chain_hash(toks, prefix), list(toks)
            self.hash_to_block_id[b.hash] = b.block_id
        return ops

    # ------------------------------------------------------------- metadata --
    def block_table_rows(self, seq_ids, width: int | None = None, pad: int = -1):
        """Block tables of the given sequences as equal-length rows (padded)."""
        rows = [self.seqs[s].block_table for s in seq_ids]
        width = width if width is not None else max((len(r) for r in rows), default=0)
        return [list(r) + [pad] * (width - len(r)) for r in rows]
