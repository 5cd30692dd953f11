"""Helpers shared by the GPU parity tests: move a workload to the device, build
the oracle's expected values for chosen sequences, and compare with the
stated tolerance |gpu - oracle| <= 1e-2 * max(1, |oracle|)."""
from __future__ import annotations

import numpy as np
import torch

from oracle import attention as oracle
from paged_kv_cache_86_gb300.workloads import Workload, bf16_to_u16

RTOL = 1e-2  # |gpu - oracle| <= RTOL * max(1, |oracle|), elementwise

# Every comparison's worst |err| / bound, with the test that made it; the
# conftest prints them at the end of the session so the margin to the
# tolerance can be read from the log.
MARGINS: list = []
CURRENT_TEST = {"id": ""}


def device_meta(w: Workload, device="cuda") -> dict:
    d = {
        "block_tables": torch.from_numpy(w.block_tables).to(device),
        "context_lens": torch.from_numpy(w.context_lens).to(device),
        "slot_mapping": torch.from_numpy(w.slot_mapping).to(device),
    }
    if w.cu_seqlens_q is not None:
        d["cu_seqlens_q"] = torch.from_numpy(w.cu_seqlens_q).to(device)
        d["cu_seqlens_k"] = torch.from_numpy(w.cu_seqlens_k).to(device)
    return d


def device_tensors(w: Workload, device="cuda") -> dict:
    return {k: v.to(device) for k, v in w.tensors.items()}


def compact_inputs(w: Workload, seq_ids, k_cache, v_cache):
    """The blocks of the chosen sequences only, copied to the host, with block
    tables and new-token slots renumbered into the compact pool. Valid input for
    the oracle because its result does not depend on where blocks sit."""
    seq_ids = np.asarray(seq_ids)
    bs = w.block_size
    rows = w.block_tables[seq_ids]
    nblk = [-(-int(w.context_lens[i]) // bs) for i in seq_ids]
    used = np.unique(np.concatenate([rows[j, :n] for j, n in enumerate(nblk)] + [np.zeros(0, np.int32)]))
    remap = {int(b): k for k, b in enumerate(used)}
    tables = np.full_like(rows, -1)
    for j, n in enumerate(nblk):
        tables[j, :n] = [remap[int(b)] for b in rows[j, :n]]
    idx = torch.from_numpy(used.astype(np.int64)).to(k_cache.device)
    kc = bf16_to_u16(k_cache.index_select(0, idx)) if len(used) else np.zeros((1,) + tuple(k_cache.shape[1:]), np.uint16)
    vc = bf16_to_u16(v_cache.index_select(0, idx)) if len(used) else kc.copy()
    return used, remap, tables, kc.copy(), vc.copy()


def per_sequence_rows(w: Workload, t: dict):
    """New-token rows indexed by sequence, on the device: row i is sequence i's
    new token (the workload keeps one key/value row per non-empty sequence);
    zeros for empty ones. The input layout of the fused decode steps."""
    tok = np.cumsum(w.context_lens > 0) - 1
    kn = torch.zeros((w.num_seqs, w.num_kv_heads, w.head_dim), dtype=torch.bfloat16,
                     device=t["key"].device)
    vn = torch.zeros_like(kn)
    nz = np.nonzero(w.context_lens > 0)[0]
    if len(nz):
        dst = torch.from_numpy(nz).to(kn.device)
        src = torch.from_numpy(tok[nz]).to(kn.device)
        kn[dst] = t["key"][src]
        vn[dst] = t["value"][src]
    return kn, vn


def decode_step_reference(w: Workload, seq_ids, k_cache, v_cache, q, key, value):
    """Oracle store of the chosen sequences' new tokens, then oracle decode.

    k_cache/v_cache are the caches BEFORE the step's store (device or host
    tensors); q/key/value the step's inputs. Returns float64 [len(seq_ids), Hq, D]."""
    assert w.kind == "decode"
    seq_ids = np.asarray(seq_ids)
    used, remap, tables, kc, vc = compact_inputs(w, seq_ids, k_cache, v_cache)
    bs = w.block_size
    # new token of sequence i is token index (number of non-empty sequences before i)
    token_of_seq = np.cumsum(w.context_lens > 0) - 1
    sel = [i for i in seq_ids if w.context_lens[i] > 0]
    if sel:
        slots = []
        for i in sel:
            s = int(w.slot_mapping[token_of_seq[i]])
            slots.append(remap[s // bs] * bs + s % bs)
        toks = torch.from_numpy(token_of_seq[sel].astype(np.int64))
        oracle.store_kvcache(bf16_to_u16(key.cpu()[toks]), bf16_to_u16(value.cpu()[toks]), kc, vc,
                             np.array(slots, np.int32), bs)
    qsel = bf16_to_u16(q.cpu()[torch.from_numpy(seq_ids.astype(np.int64))])
    return oracle.paged_decode(qsel, kc, vc, tables, w.context_lens[seq_ids], w.scale)


def assert_close(gpu: torch.Tensor, ref: np.ndarray, what: str = ""):
    g = gpu.float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite GPU output"
    err = np.abs(g - ref)
    bound = RTOL * np.maximum(1.0, np.abs(ref))
    ratio = float((err / bound).max()) if err.size else 0.0
    MARGINS.append({"test": CURRENT_TEST["id"], "what": what, "elements": int(err.size),
                    "max_err": float(err.max()) if err.size else 0.0, "ratio": ratio})
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements beyond tolerance; "
                             f"max err {err.max():.3e}; worst |err|/bound {ratio:.3f}; "
                             f"first at {idx.tolist()}")
    return float(err.max())


def prefill_step_reference(w: Workload, k_cache, v_cache, q, key, value, row_mask=None):
    """Oracle store of the chunk tokens, then oracle prefill (selected rows).

    k_cache/v_cache are the caches before the step's store. Returns float64
    [total_q, Hq, D] (NaN in rows not selected)."""
    assert w.kind == "prefill"
    kc, vc = bf16_to_u16(k_cache).copy(), bf16_to_u16(v_cache).copy()
    oracle.store_kvcache(bf16_to_u16(key), bf16_to_u16(value), kc, vc, w.slot_mapping, w.block_size)
    return oracle.paged_prefill(bf16_to_u16(q), kc, vc, w.cu_seqlens_q, w.cu_seqlens_k,
                                w.block_tables, w.scale, causal=True, row_mask=row_mask)
