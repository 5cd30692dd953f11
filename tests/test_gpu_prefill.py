"""GPU parity of a chunked-prefill step (store of the chunk, then paged varlen
causal prefill on tcgen05) against the oracle, within
|gpu - oracle| <= 1e-2 * max(1, |oracle|)."""
import numpy as np
import pytest
import torch

import paged_kv_cache_86_gb300 as pkv
from paged_kv_cache_86_gb300 import workloads as W
from pkv_testutil import assert_close, device_meta, prefill_step_reference

pytestmark = pytest.mark.gpu


def run_prefill_step(w, t, causal=True):
    m = device_meta(w)
    pkv.store_kvcache(t["key"], t["value"], t["k_cache"], t["v_cache"], m["slot_mapping"])
    out = pkv.paged_prefill(t["q"], t["k_cache"], t["v_cache"], m["cu_seqlens_q"], m["cu_seqlens_k"],
                            m["block_tables"], w.scale, max_seqlen_q=int(w.q_lens.max()),
                            max_seqlen_k=int(w.context_lens.max()), causal=causal)
    assert pkv.get_device_errors() == 0
    return out


def check(w, rows=None, what=""):
    t = {k: v.cuda() for k, v in w.tensors.items()}
    mask = None
    if rows is not None:
        mask = np.zeros(w.num_q_rows, np.uint8)
        mask[rows] = 1
    ref = prefill_step_reference(w, t["k_cache"], t["v_cache"], t["q"], t["key"], t["value"], mask)
    out = run_prefill_step(w, t)
    sel = np.arange(w.num_q_rows) if rows is None else np.asarray(rows)
    return assert_close(out[torch.from_numpy(sel).cuda()], ref[sel], what or w.name)


def test_prefill_small_chunks_ragged_tiles():
    check(W.prefill_chunks(num_seqs=4, q_len=200, max_prefix=300))


def test_prefill_single_tile_no_prefix():
    check(W.prefill_workload("p_one", [128], [0], 32, 8, 16, seed=1))


def test_prefill_empty_chunks_between_others():
    # sequences with no new rows, with and without a cached prefix, between
    # chunks: they claim no work item and own no output row
    check(W.prefill_workload("p_empty", [0, 130, 0, 5, 0], [40, 100, 0, 3, 0], 16, 8, 16, seed=77))


def test_prefill_with_no_rows_is_a_noop():
    w = W.prefill_workload("p_none", [0, 0], [40, 0], 16, 8, 16, seed=78)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    kc, vc = t["k_cache"].clone(), t["v_cache"].clone()
    out = run_prefill_step(w, t)
    torch.cuda.synchronize()
    assert tuple(out.shape) == (0, 16, 128)
    assert torch.equal(t["k_cache"], kc) and torch.equal(t["v_cache"], vc)


@pytest.mark.parametrize("q_lens,prefixes", [
    ([1, 5, 128, 129, 300], [0, 17, 64, 3, 250]),
    ([64, 64], [1000, 1]),
    ([257], [0]),
])
def test_prefill_varlen(q_lens, prefixes):
    check(W.prefill_workload("p_varlen", q_lens, prefixes, 32, 8, 16, seed=sum(q_lens)))


@pytest.mark.parametrize("bs", [1, 2, 4, 8, 12, 16, 20, 24, 32, 128, 256])
def test_prefill_block_sizes(bs):
    # block sizes that are not a multiple of 8 gather K/V rows with cp.async
    # instead of TMA boxes; ragged last tiles in both chunks
    check(W.prefill_workload(f"p_bs{bs}", [130, 77], [300, 45], 16, 8, bs, seed=300 + bs))


@pytest.mark.parametrize("hkv,group,bs", [(3, 3, 1), (8, 4, 1), (2, 8, 4), (1, 4, 6)])
def test_prefill_gathered_rows_with_head_groups(hkv, group, bs):
    # the gather path with an odd group (paired query tiles), GQA groups up to
    # 8 and a single KV head, chunks over several 128-key tiles
    check(W.prefill_workload(f"p_gather_h{hkv}g{group}b{bs}", [300, 129, 40], [500, 0, 1000],
                             hkv * group, hkv, bs, seed=700 + hkv * 10 + group + bs))


def test_prefill_page_size_one_chunks_every_row():
    # token-level paging (one token per block, shuffled over the pool), the
    # shape of the benchmark's chunks at a smaller count
    prefixes = np.random.default_rng(87001).integers(0, 1501, size=6)
    check(W.prefill_workload("p_page1", [512] * 6, prefixes, 32, 8, 1, seed=87001))


@pytest.mark.parametrize("hkv,group", [(3, 3), (2, 5), (4, 1), (1, 3)])
def test_prefill_odd_groups_pair_query_tiles(hkv, group):
    # odd GQA groups run two consecutive 128-row query tiles of one head per
    # work item: ragged pairs (300 = 256 + 44 rows, 257, 33) and a full one (512)
    check(W.prefill_workload(f"p_odd_h{hkv}g{group}", [300, 512, 33, 257], [100, 0, 700, 31],
                             hkv * group, hkv, 16, seed=500 + hkv * 10 + group))


@pytest.mark.parametrize("hkv,group", [(8, 1), (4, 2), (8, 4), (2, 8), (1, 4)])
def test_prefill_head_groups(hkv, group):
    check(W.prefill_workload(f"p_h{hkv}g{group}", [140, 33], [200, 7], hkv * group, hkv, 16,
                             seed=400 + hkv * 10 + group))


def test_prefill_noncausal_matches_oracle():
    from oracle import attention as oracle
    from paged_kv_cache_86_gb300.workloads import bf16_to_u16
    w = W.prefill_workload("p_noncausal", [100, 60], [40, 0], 16, 8, 16, seed=9)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    kc, vc = bf16_to_u16(t["k_cache"]).copy(), bf16_to_u16(t["v_cache"]).copy()
    oracle.store_kvcache(bf16_to_u16(t["key"]), bf16_to_u16(t["value"]), kc, vc, w.slot_mapping,
                         w.block_size)
    ref = oracle.paged_prefill(bf16_to_u16(t["q"]), kc, vc, w.cu_seqlens_q, w.cu_seqlens_k,
                               w.block_tables, w.scale, causal=False)
    out = run_prefill_step(w, t, causal=False)
    assert_close(out, ref, "noncausal")


def test_prefill_last_row_matches_decode():
    w = W.prefill_chunks(num_seqs=6, q_len=150, max_prefix=700)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    out = run_prefill_step(w, t)
    m = device_meta(w)
    last = torch.from_numpy((w.cu_seqlens_q[1:] - 1).astype(np.int64)).cuda()
    dec = pkv.paged_decode(t["q"][last].contiguous(), t["k_cache"], t["v_cache"], m["block_tables"],
                           m["context_lens"], w.scale)
    diff = (out[last].float() - dec.float()).abs()
    assert diff.max().item() <= 2e-2 * max(1.0, dec.float().abs().max().item())


def test_prefill_full_size_whole_chunks_and_every_tile_boundary():
    """The 32 x 512 chunked workload at full size: every row of 8 of its chunks
    (the 4 longest and 4 shortest prefixes), and in all 32 chunks the first and
    last row of every 128-row query tile."""
    w = W.prefill_chunks()
    assert w.num_q_rows == 16384
    cu = w.cu_seqlens_q
    order = np.argsort(w.context_lens)
    whole = list(order[:4]) + list(order[-4:])
    rows = set()
    for i in whole:
        rows |= set(range(int(cu[i]), int(cu[i + 1])))
    for i in range(w.num_seqs):
        for r0 in range(int(cu[i]), int(cu[i + 1]), 128):
            rows |= {r0, min(r0 + 127, int(cu[i + 1]) - 1)}
    check(w, rows=sorted(rows))
