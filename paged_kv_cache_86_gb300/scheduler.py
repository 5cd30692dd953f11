"""Host side of a mixed batch: which requests run in a scheduling round, and the
flattened metadata one ``pkv_mixed_step`` call takes.

Per round there are three budgets -- tokens, sequences and the size of a
prefill chunk. Every decode request gets its one token first; what is left of
the token budget goes to waiting / prefill requests in order, each taking at
most one chunk, so that a long prompt never stalls the decodes behind it
(推理运行时 §build_batch baseline; §Chunked prefill: N_scheduled = N_decode +
N_prefill_chunk). The result puts decode requests first, which is the layout
``pkv_mixed_step`` wants (decode sequences 0..D-1, one query row each).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

DECODE = "decode"
PREFILL_PHASES = ("waiting", "prefill")


@dataclass(frozen=True)
class Scheduled:
    request_id: object
    phase: str
    tokens: int


def build_batch(requests, token_budget: int, max_sequences: int, prefill_chunk: int) -> list:
    """requests: dicts with "id", "phase" ("decode", "waiting" or "prefill") and
    "prompt_left" (prompt tokens still to prefill). Returns Scheduled items,
    decode requests first, in request order within each phase."""
    if token_budget <= 0 or max_sequences <= 0 or prefill_chunk <= 0:
        raise ValueError("scheduler budgets must be positive")
    ids = [r["id"] for r in requests]
    if len(set(ids)) != len(ids):
        raise ValueError("request ids must be unique within a scheduling round")
    ordered = [r for r in requests if r["phase"] == DECODE] + \
              [r for r in requests if r["phase"] in PREFILL_PHASES]
    out: list[Scheduled] = []
    left = token_budget
    for r in ordered:
        if len(out) >= max_sequences or left == 0:
            break
        want = 1 if r["phase"] == DECODE else min(int(r["prompt_left"]), prefill_chunk, left)
        if 0 < want <= left:
            out.append(Scheduled(r["id"], r["phase"], want))
            left -= want
    return out


@dataclass
class MixedMetadata:
    """Flattened inputs of one pkv_mixed_step call (host numpy arrays)."""
    num_decode_seqs: int
    cu_seqlens_q: np.ndarray     # [S + 1] int32
    cu_seqlens_k: np.ndarray     # [S + 1] int32
    slot_mapping: np.ndarray     # [total_q] int32: cache slot of each query row's token
    block_tables: np.ndarray     # [S, MB] int32, padded with -1
    positions: np.ndarray        # [total_q] int32: absolute position of each query row
    max_seqlen_q: int
    max_seqlen_k: int


def mixed_metadata(items, seqs, computed, block_size: int, table_width: int | None = None):
    """items: Scheduled (decode first); seqs[id]: its block manager Sequence (token
    ids and block table, already holding every token scheduled this round);
    computed[id]: tokens whose K/V are already in the cache before this round.
    A decode item schedules the sequence's newest token; a prefill item the next
    ``tokens`` prompt tokens after the computed ones."""
    cu_q, cu_k, slots, pos, rows = [0], [0], [], [], []
    num_decode = 0
    seen_prefill = False
    for it in items:
        s = seqs[it.request_id]
        done = int(computed[it.request_id])
        if it.phase == DECODE:
            if seen_prefill:
                raise ValueError("decode items must come before prefill items")
            num_decode += 1
            if it.tokens != 1 or done != len(s) - 1:
                raise ValueError("a decode item schedules exactly the newest token")
        else:
            seen_prefill = True
        start, stop = done, done + it.tokens
        if stop > len(s):
            raise ValueError("scheduled tokens beyond the sequence")
        for p in range(start, stop):
            slots.append(s.slot(p))
            pos.append(p)
        cu_q.append(cu_q[-1] + it.tokens)
        cu_k.append(cu_k[-1] + stop)
        rows.append(list(s.block_table))
    width = table_width if table_width is not None else max((len(r) for r in rows), default=0)
    tables = np.full((len(rows), max(width, 1)), -1, np.int32)
    for i, r in enumerate(rows):
        tables[i, :len(r)] = r
    q_lens = np.diff(cu_q)
    k_lens = np.diff(cu_k)
    return MixedMetadata(num_decode, np.asarray(cu_q, np.int32), np.asarray(cu_k, np.int32),
                         np.asarray(slots, np.int32), tables, np.asarray(pos, np.int32),
                         int(q_lens.max(initial=0)), int(k_lens.max(initial=0)))
