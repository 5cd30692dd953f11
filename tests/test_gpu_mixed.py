"""GPU parity of pkv_mixed_step (decode requests and prefill chunks of one
round, decode first) against the oracle's store + prefill over the whole
flattened batch, and of its decode rows against pkv_paged_decode."""
import numpy as np
import pytest
import torch

import paged_kv_cache_86_gb300 as pkv
from paged_kv_cache_86_gb300 import workloads as W
from pkv_testutil import assert_close, device_meta, prefill_step_reference

pytestmark = pytest.mark.gpu


def mixed_workload(name, decode_lens, chunk_q, chunk_prefix, hq, hkv, bs, seed):
    """Decode sequences first (one query row at position len - 1), then chunks."""
    q_lens = [1] * len(decode_lens) + list(chunk_q)
    prefixes = [n - 1 for n in decode_lens] + list(chunk_prefix)
    return W.prefill_workload(name, q_lens, prefixes, hq, hkv, bs, seed), len(decode_lens)


def run_mixed(w, d, t):
    m = device_meta(w)
    out = pkv.mixed_step(t["q"], t["key"], t["value"], m["slot_mapping"], t["k_cache"], t["v_cache"],
                         m["cu_seqlens_q"], m["cu_seqlens_k"], m["block_tables"], d, w.scale,
                         max_seqlen_q=int(w.q_lens.max()), max_seqlen_k=int(w.context_lens.max()))
    torch.cuda.synchronize()
    return out, m


@pytest.mark.parametrize("hkv,group,bs", [(8, 4, 16), (2, 4, 16), (8, 2, 32), (4, 3, 16), (8, 4, 1),
                                          (2, 2, 4)])
def test_mixed_step_matches_the_oracle(hkv, group, bs):
    w, d = mixed_workload(f"mixed_{hkv}x{group}_bs{bs}", [1, 2, 17, 300, 1000], [3, 130, 64],
                          [0, 70, 500], hkv * group, hkv, bs, seed=400 + hkv + group + bs)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    ref = prefill_step_reference(w, t["k_cache"], t["v_cache"], t["q"], t["key"], t["value"])
    out, m = run_mixed(w, d, t)
    assert pkv.get_device_errors() == 0
    assert_close(out, ref, w.name)
    # the decode rows came from the decode path: identical to pkv_paged_decode
    # on the same (already stored) cache
    lens = (m["cu_seqlens_k"][1:d + 1] - m["cu_seqlens_k"][:d]).contiguous()
    dec = pkv.paged_decode(t["q"][:d].contiguous(), t["k_cache"], t["v_cache"],
                           m["block_tables"][:d].contiguous(), lens, w.scale,
                           max_context_len=int(w.context_lens.max()))
    assert torch.equal(out[:d], dec)


def test_mixed_step_only_decodes_and_only_chunks():
    for dl, cq, cp in (([5, 40, 9], [], []), ([], [7, 129], [3, 0])):
        w, d = mixed_workload("mixed_edge", dl, cq, cp, 16, 4, 16, seed=11)
        t = {k: v.cuda() for k, v in w.tensors.items()}
        ref = prefill_step_reference(w, t["k_cache"], t["v_cache"], t["q"], t["key"], t["value"])
        out, _ = run_mixed(w, d, t)
        assert pkv.get_device_errors() == 0
        assert_close(out, ref, "mixed_edge")


def test_mixed_step_with_empty_chunks():
    # chunks with no new rows (with and without a cached prefix) among the
    # round's chunks add no work and no output row
    w, d = mixed_workload("mixed_empty", [4, 300], [0, 33, 0, 140], [10, 5, 0, 60], 16, 4, 16,
                          seed=15)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    ref = prefill_step_reference(w, t["k_cache"], t["v_cache"], t["q"], t["key"], t["value"])
    out, _ = run_mixed(w, d, t)
    assert pkv.get_device_errors() == 0
    assert_close(out, ref, "mixed_empty")


def test_mixed_step_flags_a_decode_sequence_with_two_rows():
    w, d = mixed_workload("mixed_bad", [5, 9], [4], [2], 8, 2, 16, seed=12)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    # claim three decode sequences: the third one has four query rows
    m = device_meta(w)
    pkv.mixed_step(t["q"], t["key"], t["value"], m["slot_mapping"], t["k_cache"], t["v_cache"],
                   m["cu_seqlens_q"], m["cu_seqlens_k"], m["block_tables"], 3, w.scale,
                   max_seqlen_q=4, max_seqlen_k=int(w.context_lens.max()))
    torch.cuda.synchronize()
    assert pkv.get_device_errors() & pkv._lib.DEVERR_LENGTH


def test_mixed_step_full_size_decode_rows_and_chunk_tiles():
    """A full-size round: every decode row, every row of two of the chunks, and
    the first and last row of every 128-row tile of the others."""
    rng = np.random.default_rng(13)
    dec = np.clip(np.rint(np.exp(np.log(800) + rng.standard_normal(256))), 16, 4096).astype(int)
    w, d = mixed_workload("mixed_256d_8x512", dec.tolist(), [512] * 8,
                          rng.integers(0, 3585, 8).tolist(), 32, 8, 16, seed=14)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    mask = np.zeros(w.num_q_rows, np.uint8)
    cu = w.cu_seqlens_q
    rows = set(range(d))
    for i in range(d, w.num_seqs):
        if i < d + 2:
            rows |= set(range(int(cu[i]), int(cu[i + 1])))
        for r0 in range(int(cu[i]), int(cu[i + 1]), 128):
            rows |= {r0, min(r0 + 127, int(cu[i + 1]) - 1)}
    rows = np.array(sorted(rows))
    mask[rows] = 1
    ref = prefill_step_reference(w, t["k_cache"], t["v_cache"], t["q"], t["key"], t["value"], row_mask=mask)
    out, _ = run_mixed(w, d, t)
    assert pkv.get_device_errors() == 0
    sel = np.sort(rows)
    assert_close(out[torch.from_numpy(sel).cuda()], ref[sel], w.name)


def test_mixed_step_with_side_prefill_replays_from_a_cuda_graph():
    """A round whose prefill also runs beside the decode kernel on the library's
    second stream (forked from and joined into the caller's stream): captured
    in a CUDA graph and replayed, it gives the eager call's output bit for bit
    (which items each prefill launch claims varies, their arithmetic does not),
    and the eager call matches the oracle."""
    rng = np.random.default_rng(21)
    dec = np.clip(np.rint(np.exp(np.log(800) + rng.standard_normal(128))), 16, 4096).astype(int)
    w, d = mixed_workload("mixed_graph", dec.tolist(), [512] * 4, rng.integers(0, 3585, 4).tolist(),
                          32, 8, 16, seed=22)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    m = device_meta(w)
    kc0, vc0 = t["k_cache"].clone(), t["v_cache"].clone()
    mq, mk = int(w.q_lens.max()), int(w.context_lens.max())
    ws = torch.empty(pkv.mixed_workspace_size(d, 32, 8), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(t["q"])

    def call():
        pkv.mixed_step(t["q"], t["key"], t["value"], m["slot_mapping"], t["k_cache"], t["v_cache"],
                       m["cu_seqlens_q"], m["cu_seqlens_k"], m["block_tables"], d, w.scale, mq, mk,
                       out=out, workspace=ws)

    call()
    torch.cuda.synchronize()
    eager = out.clone()
    mask = np.zeros(w.num_q_rows, np.uint8)
    cu = w.cu_seqlens_q
    rows = set(range(d))
    for i in range(d, w.num_seqs):
        for r0 in range(int(cu[i]), int(cu[i + 1]), 128):
            rows |= {r0, min(r0 + 127, int(cu[i + 1]) - 1)}
    rows = np.array(sorted(rows))
    mask[rows] = 1
    ref = prefill_step_reference(w, kc0, vc0, t["q"], t["key"], t["value"], row_mask=mask)
    assert_close(eager[torch.from_numpy(rows).cuda()], ref[rows], w.name)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()                      # warm-up on the capture stream
        torch.cuda.synchronize()
        out.zero_()
        with torch.cuda.graph(g, stream=s):
            call()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    assert pkv.get_device_errors() == 0
