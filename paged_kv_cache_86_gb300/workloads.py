"""Seeded synthetic inputs for paged KV-cache attention.

This module only draws inputs: request lengths, a block pool and the block
tables that place each sequence in it, the slots of the tokens a step writes,
and N(0, 1) bf16 values for q, the new K/V and the cache. It holds none of the
attention arithmetic and imports neither the CUDA library nor the oracle, so
both sides can be fed from it.

Workloads (shapes from the pages' examples and nano-vllm's defaults:
max_num_seqs 512, max_num_batched_tokens 16384, max_model_len 4096, block
size 16 or 256; nano vllm代码详解 §1 Config; request lengths 300 / 5000 / 70
from LLM Infra 101 v0.5's opening example):

  decode_3seq_ctx300_5000_70_bs16     3 sequences, Hq 8 / Hkv 2, block 16,
                                      a 512-block pool assigned by permutation
  decode_64seq_u128_4096_bs256        64 sequences, lengths U[128, 4096],
                                      Hq 16 / Hkv 8, block 256, pool 1.25x need
  decode_512seq_lognormal_bs16        512 sequences, lengths
                                      clip(rint(exp(ln 800 + N(0,1))), 16, 4096),
                                      Hq 32 / Hkv 8, block 16, fragmented pool:
                                      ceil(need / 0.3) blocks, a random 30 %
                                      freed in random order, drawn FIFO
  decode_8x32768_248x200_bs256        8 sequences of 32768 + 248 of 200 in a
                                      seeded order, Hq 32 / Hkv 8, block 256
  prefill_32x512_prefix_u0_3584_bs16  32 chunks of 512 new tokens after a
                                      cached prefix U[0, 3584], Hq 32 / Hkv 8,
                                      block 16, pool 1.25x need

A decode step writes one new token per sequence at position context_lens[i]-1
(the token counts in its own context); a prefill step writes its chunk at
positions prefix .. prefix+q_len-1. Block tables are padded with -1 past each
sequence's last block and to a row length rounded up to 32 entries.

Values: metadata comes from numpy's default_rng(seed). bf16 values are
fp32 N(0, 1) draws rounded to nearest even, from torch's generator seeded
with seed + a per-tensor offset, on the host ("host" fill) or on the GPU
("device" fill, for pools too large to draw on the host quickly); "none"
draws metadata only.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

PAD_BLOCK = -1

_VALUE_STREAMS = {"q": 1, "key": 2, "value": 3, "k_cache": 4, "v_cache": 5}


@dataclass
class Workload:
    name: str
    kind: str                      # "decode" or "prefill"
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    block_tables: np.ndarray       # [S, MB] int32
    context_lens: np.ndarray       # [S] int32: tokens each sequence attends to (decode) / k_len (prefill)
    slot_mapping: np.ndarray       # [T] int32: slots of the tokens this step stores
    cu_seqlens_q: np.ndarray | None = None   # [S+1] int32 (prefill)
    cu_seqlens_k: np.ndarray | None = None   # [S+1] int32 (prefill)
    tensors: dict = field(default_factory=dict)  # bf16 torch tensors: q, key, value, k_cache, v_cache

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def num_new_tokens(self) -> int:
        return int(self.slot_mapping.shape[0])

    @property
    def num_q_rows(self) -> int:
        return int(self.cu_seqlens_q[-1]) if self.kind == "prefill" else self.num_seqs

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max(initial=0))

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_q).astype(np.int32)

    def meta(self) -> dict:
        return {"name": self.name, "kind": self.kind, "seed": self.seed, "num_seqs": self.num_seqs,
                "num_q_heads": self.num_q_heads, "num_kv_heads": self.num_kv_heads,
                "head_dim": self.head_dim, "block_size": self.block_size,
                "num_blocks": self.num_blocks, "total_context": int(self.context_lens.sum()),
                "new_tokens": self.num_new_tokens}


def bf16_to_u16(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a bf16 tensor as a host numpy uint16 array."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _normal_bf16(shape, seed: int, device) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(tuple(int(s) for s in shape), generator=g, device=device, dtype=torch.float32)
    return x.to(torch.bfloat16)


def fp8_pool(num_blocks: int, block_size: int, num_kv_heads: int, seed: int, head_dim: int = 128,
             device=None):
    """A random pre-filled fp8 cache for one of K or V: uint8 codes uniform over
    the 254 finite E4M3 codes (every byte except 0x7F and 0xFF) and fp32 row
    scales |N(0,1)| * 2 / 448 + 1e-3 per (slot, KV head). Plain seeded random
    bytes and floats; nothing here quantizes anything."""
    dev = device or "cuda"
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    codes = torch.randint(0, 254, (num_blocks, block_size, num_kv_heads, head_dim),
                          generator=g, device=dev, dtype=torch.int32)
    codes = torch.where(codes >= 0x7F, codes + 1, codes).to(torch.uint8)  # 0..126, 128..254
    scales = torch.randn((num_blocks * block_size, num_kv_heads), generator=g, device=dev)
    scales = scales.abs() * (2.0 / 448.0) + 1e-3
    return codes, scales.float()


def _align32(n: int) -> int:
    return (n + 31) // 32 * 32


def _blocks_needed(lengths, bs):
    return [-(-int(n) // bs) for n in lengths]


def _assign(lengths, bs, order, mb=None):
    """Hand out blocks from ``order`` (a sequence of physical ids) in request order."""
    need = _blocks_needed(lengths, bs)
    mb = mb or _align32(max(max(need, default=1), 1))
    tables = np.full((len(lengths), mb), PAD_BLOCK, dtype=np.int32)
    taken = 0
    for i, n in enumerate(need):
        tables[i, :n] = order[taken:taken + n]
        taken += n
    if taken > len(order):
        raise ValueError("pool too small")
    return tables


def pool_permuted(rng, lengths, bs, num_blocks):
    """Blocks drawn in the order of one seeded permutation of the pool."""
    return _assign(lengths, bs, rng.permutation(num_blocks).astype(np.int32))


def pool_fragmented(rng, lengths, bs, free_fraction=0.3):
    """A pool of ceil(need / free_fraction) blocks, all in use, of which a random
    ``free_fraction`` is freed in random order; sequences then take blocks from
    that free list first-in first-out. Returns (tables, num_blocks)."""
    need = sum(_blocks_needed(lengths, bs))
    num_blocks = max(1, math.ceil(need / free_fraction))
    freed = rng.permutation(num_blocks)[: math.ceil(free_fraction * num_blocks)].astype(np.int32)
    return _assign(lengths, bs, freed), num_blocks


def _slots(tables, positions_per_seq, bs):
    out = []
    for i, positions in enumerate(positions_per_seq):
        positions = np.asarray(positions, dtype=np.int64)
        out.append(tables[i, positions // bs].astype(np.int64) * bs + positions % bs)
    return np.concatenate(out).astype(np.int32) if out else np.zeros(0, np.int32)


def _fill_values(w: Workload, fill: str, device: str | None):
    if fill == "none":  # metadata only
        w.tensors = {}
        return w
    dev = "cpu" if fill == "host" else (device or "cuda")
    hq, hkv, d = w.num_q_heads, w.num_kv_heads, w.head_dim
    shapes = {
        "q": (w.num_q_rows, hq, d),
        "key": (w.num_new_tokens, hkv, d),
        "value": (w.num_new_tokens, hkv, d),
        "k_cache": (w.num_blocks, w.block_size, hkv, d),
        "v_cache": (w.num_blocks, w.block_size, hkv, d),
    }
    w.tensors = {k: _normal_bf16(s, w.seed * 16 + _VALUE_STREAMS[k], dev) for k, s in shapes.items()}
    return w


def decode_workload(name, lengths, num_q_heads, num_kv_heads, block_size, seed, *,
                    pool="permuted", num_blocks=None, pool_factor=1.25, head_dim=128,
                    fill="host", device=None) -> Workload:
    rng = np.random.default_rng(seed)
    lengths = np.asarray(lengths, dtype=np.int32)
    need = sum(_blocks_needed(lengths, block_size))
    if pool == "fragmented":
        tables, num_blocks = pool_fragmented(rng, lengths, block_size)
    else:
        num_blocks = num_blocks or max(1, math.ceil(pool_factor * need))
        tables = pool_permuted(rng, lengths, block_size, num_blocks)
    new_pos = [[n - 1] if n > 0 else [] for n in lengths]
    slots = _slots(tables, new_pos, block_size)
    w = Workload(name=name, kind="decode", seed=seed, num_q_heads=num_q_heads,
                 num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=block_size,
                 num_blocks=int(num_blocks), scale=1.0 / math.sqrt(head_dim),
                 block_tables=tables, context_lens=lengths, slot_mapping=slots)
    return _fill_values(w, fill, device)


def prefill_workload(name, q_lens, prefixes, num_q_heads, num_kv_heads, block_size, seed, *,
                     pool_factor=1.25, head_dim=128, fill="host", device=None) -> Workload:
    rng = np.random.default_rng(seed)
    q_lens = np.asarray(q_lens, dtype=np.int32)
    prefixes = np.asarray(prefixes, dtype=np.int32)
    k_lens = (q_lens + prefixes).astype(np.int32)
    need = sum(_blocks_needed(k_lens, block_size))
    num_blocks = max(1, math.ceil(pool_factor * need))
    tables = pool_permuted(rng, k_lens, block_size, num_blocks)
    positions = [np.arange(c, c + n) for c, n in zip(prefixes, q_lens)]
    slots = _slots(tables, positions, block_size)
    cu_q = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(k_lens)]).astype(np.int32)
    w = Workload(name=name, kind="prefill", seed=seed, num_q_heads=num_q_heads,
                 num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=block_size,
                 num_blocks=int(num_blocks), scale=1.0 / math.sqrt(head_dim),
                 block_tables=tables, context_lens=k_lens, slot_mapping=slots,
                 cu_seqlens_q=cu_q, cu_seqlens_k=cu_k)
    return _fill_values(w, fill, device)


# ------------------------------------------------------------ named sets --

def decode_3seq(seed=86001, **kw):
    return decode_workload("decode_3seq_ctx300_5000_70_bs16", [300, 5000, 70], 8, 2, 16, seed,
                           num_blocks=512, **kw)


def decode_64seq(seed=86002, num_seqs=64, max_len=4096, **kw):
    rng = np.random.default_rng(seed + 1000)
    lengths = rng.integers(128, max_len + 1, size=num_seqs)
    return decode_workload(f"decode_{num_seqs}seq_u128_{max_len}_bs256", lengths, 16, 8, 256,
                           seed, **kw)


def lognormal_lengths(rng, num_seqs, median=800.0, sigma=1.0, lo=16, hi=4096):
    x = np.rint(np.exp(np.log(median) + sigma * rng.standard_normal(num_seqs)))
    return np.clip(x, lo, hi).astype(np.int32)


def decode_512seq(seed=86003, num_seqs=512, hi=4096, **kw):
    lengths = lognormal_lengths(np.random.default_rng(seed + 1000), num_seqs, hi=hi)
    return decode_workload(f"decode_{num_seqs}seq_lognormal_bs16", lengths, 32, 8, 16, seed,
                           pool="fragmented", **kw)


def decode_longtail(seed=86004, num_long=8, long_len=32768, num_short=248, short_len=200, **kw):
    rng = np.random.default_rng(seed + 1000)
    lengths = np.array([long_len] * num_long + [short_len] * num_short, dtype=np.int32)
    lengths = lengths[rng.permutation(lengths.shape[0])]
    return decode_workload(f"decode_{num_long}x{long_len}_{num_short}x{short_len}_bs256",
                           lengths, 32, 8, 256, seed, **kw)


def prefill_chunks(seed=86005, num_seqs=32, q_len=512, max_prefix=3584, **kw):
    rng = np.random.default_rng(seed + 1000)
    prefixes = rng.integers(0, max_prefix + 1, size=num_seqs)
    return prefill_workload(f"prefill_{num_seqs}x{q_len}_prefix_u0_{max_prefix}_bs16",
                            [q_len] * num_seqs, prefixes, 32, 8, 16, seed, **kw)


NAMED = {
    "decode_3seq": decode_3seq,
    "decode_64seq": decode_64seq,
    "decode_512seq": decode_512seq,
    "decode_longtail": decode_longtail,
    "prefill_chunks": prefill_chunks,
}
