"""GPU parity of pkv_decode_step -- the store of each sequence's newest token
and the paged decode in one call -- against the oracle; its bit-for-bit
equivalence with pkv_store_kvcache followed by pkv_paged_decode; and replays of
the step from a CUDA graph captured at a padded batch size."""
import dataclasses

import numpy as np
import pytest
import torch

import paged_kv_cache_86_gb300 as pkv
from paged_kv_cache_86_gb300 import workloads as W
from pkv_testutil import assert_close, decode_step_reference, device_meta, per_sequence_rows

pytestmark = pytest.mark.gpu


def run_step(w, t, m):
    kn, vn = per_sequence_rows(w, t)
    out = pkv.decode_step(t["q"], kn, vn, t["k_cache"], t["v_cache"], m["block_tables"],
                          m["context_lens"], w.scale)
    assert pkv.get_device_errors() == 0
    return out


# (Hkv, G, bs) covering the all-heads tcgen05 kernel (which plans the call and
# writes the new rows itself), the per-head tcgen05 kernel and the CUDA-core
# kernel (behind the step's planning launch; blocks 3, 1 and 5)
SHAPES = [(8, 4, 16), (8, 4, 256), (4, 8, 32), (16, 2, 16), (8, 1, 16), (2, 4, 16),
          (3, 5, 32), (8, 4, 3), (4, 2, 1), (2, 2, 5)]


@pytest.mark.parametrize("hkv,group,bs", SHAPES)
def test_decode_step_matches_oracle(hkv, group, bs):
    lens = [1, 2, 16, 17, 0, 300, 1023, 5, 129, 2000, 0, 64]
    w = W.decode_workload(f"step_{hkv}x{group}_bs{bs}", lens, hkv * group, hkv, bs,
                          seed=700 + hkv * 13 + group * 5 + bs)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    m = device_meta(w)
    ref = decode_step_reference(w, np.arange(w.num_seqs), t["k_cache"], t["v_cache"], t["q"],
                                t["key"], t["value"])
    out = run_step(w, t, m)
    assert_close(out, ref, w.name)
    for i in np.nonzero(w.context_lens == 0)[0]:
        assert (out[int(i)] == 0).all()


@pytest.mark.parametrize("hkv,group,bs", [(8, 4, 16), (2, 4, 16), (8, 4, 3)])
def test_decode_step_equals_store_then_decode(hkv, group, bs):
    lens = np.random.default_rng(3).integers(1, 900, size=70)
    w = W.decode_workload(f"eq_{hkv}x{group}_bs{bs}", lens, hkv * group, hkv, bs, seed=31 + bs)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    m = device_meta(w)
    kc2, vc2 = t["k_cache"].clone(), t["v_cache"].clone()
    pkv.store_kvcache(t["key"], t["value"], kc2, vc2, m["slot_mapping"])
    two_calls = pkv.paged_decode(t["q"], kc2, vc2, m["block_tables"], m["context_lens"], w.scale)
    fused = run_step(w, t, m)
    assert torch.equal(fused, two_calls)
    assert torch.equal(t["k_cache"], kc2) and torch.equal(t["v_cache"], vc2)


def test_decode_step_512seq_full_size_every_sequence():
    w = W.decode_512seq(fill="device")
    t = {k: v.cuda() for k, v in w.tensors.items()}
    m = device_meta(w)
    ids = np.arange(w.num_seqs)
    ref = decode_step_reference(w, ids, t["k_cache"], t["v_cache"], t["q"], t["key"], t["value"])
    out = run_step(w, t, m)
    assert_close(out[torch.from_numpy(ids).cuda()], ref, w.name)
    # every new token landed in its slot
    slots = torch.from_numpy(w.slot_mapping.astype(np.int64)).cuda()
    flat_k = t["k_cache"].view(-1, w.num_kv_heads, w.head_dim)
    flat_v = t["v_cache"].view(-1, w.num_kv_heads, w.head_dim)
    assert torch.equal(flat_k[slots], t["key"]) and torch.equal(flat_v[slots], t["value"])


@pytest.mark.parametrize("hkv,group", [(8, 4), (2, 4)])
def test_decode_step_replays_from_a_cuda_graph_at_a_padded_batch(hkv, group):
    """37 live sequences padded to a captured batch of 64 with empty rows; the
    graph is replayed for three consecutive steps (context_lens grows by one
    and new q / K / V rows arrive each step, all through the same buffers).
    Eight KV heads run the all-heads kernel, two the per-head kernel (its
    launches chained as programmatic dependents inside the graph)."""
    live, padded, bs = 37, 64, 16
    rng = np.random.default_rng(9)
    lens0 = (rng.integers(0, 40, size=live) * bs + rng.integers(1, bs - 3, size=live)).astype(np.int32)
    grown = np.concatenate([lens0 + 3, np.zeros(padded - live, np.int32)])  # blocks for 3 steps
    w0 = W.decode_workload("graph_pad", grown, hkv * group, hkv, bs, seed=77)
    t = {k: v.cuda() for k, v in w0.tensors.items()}
    bt = torch.from_numpy(w0.block_tables).cuda()
    cl = torch.zeros(padded, dtype=torch.int32, device="cuda")
    q = torch.zeros_like(t["q"])
    kn = torch.zeros((padded, hkv, 128), dtype=torch.bfloat16, device="cuda")
    vn = torch.zeros_like(kn)
    out = torch.empty_like(q)
    ws = torch.empty(pkv.decode_workspace_size(padded, hkv * group, hkv), dtype=torch.uint8,
                     device="cuda")
    max_ctx = int(w0.block_tables.shape[1] * bs)

    def step():
        pkv.decode_step(q, kn, vn, t["k_cache"], t["v_cache"], bt, cl, w0.scale,
                        max_context_len=max_ctx, out=out, workspace=ws)

    step()  # eager call first: one-time function attributes are set outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()

    gen = torch.Generator(device="cuda").manual_seed(5)
    for k in range(3):
        lens = np.concatenate([lens0 + k, np.zeros(padded - live, np.int32)]).astype(np.int32)
        cl.copy_(torch.from_numpy(lens))
        q.normal_(generator=gen)
        kn.normal_(generator=gen)
        vn.normal_(generator=gen)
        q[live:] = 0
        kn[live:] = 0
        vn[live:] = 0
        # the oracle's view of this step: same tables, grown lengths, new-token slots
        pos = [[n - 1] for n in lens[:live]] + [[] for _ in range(padded - live)]
        slots = np.array([w0.block_tables[i, p[0] // bs] * bs + p[0] % bs
                          for i, p in enumerate(pos) if p], dtype=np.int32)
        wk = dataclasses.replace(w0, context_lens=lens, slot_mapping=slots)
        ids = np.arange(live)
        ref = decode_step_reference(wk, ids, t["k_cache"], t["v_cache"], q, kn[:live], vn[:live])
        g.replay()
        torch.cuda.synchronize()
        assert pkv.get_device_errors() == 0
        assert_close(out[:live], ref, f"graph step {k}")
        assert (out[live:] == 0).all()


def test_decode_step_on_all_heads_kernel_reports_bad_metadata_and_skips_it():
    """The all-heads kernel plans the call itself: a length beyond max_context_len
    is clamped and reported, and a new row whose block id is out of range is not
    written anywhere (and reported); the other sequences are still correct."""
    lens = [40, 40, 300, 17]
    w = W.decode_workload("step_bad_meta", lens, 32, 8, 16, seed=77)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    m = device_meta(w)
    kn, vn = per_sequence_rows(w, t)
    # sequence 1's last block id out of range: its new row must not be written
    bt = m["block_tables"].clone()
    bt[1, (lens[1] - 1) // 16] = w.num_blocks + 5
    kc0, vc0 = t["k_cache"].clone(), t["v_cache"].clone()
    pkv.decode_step(t["q"], kn, vn, t["k_cache"], t["v_cache"], bt, m["context_lens"], w.scale)
    assert pkv.get_device_errors() & pkv._lib.DEVERR_BLOCK_ID
    # every cache row other than the three good sequences' new rows is unchanged
    slots = [int(w.slot_mapping[k]) for k in (0, 2, 3)]
    flat0, flat = kc0.view(-1, 8, 128), t["k_cache"].view(-1, 8, 128)
    mask = torch.ones(flat.shape[0], dtype=torch.bool, device="cuda")
    mask[torch.tensor(slots, device="cuda")] = False
    assert torch.equal(flat[mask], flat0[mask])
    assert torch.equal(t["v_cache"].view(-1, 8, 128)[mask], vc0.view(-1, 8, 128)[mask])
    # a length beyond the bound: clamped and reported
    lens_t = m["context_lens"].clone()
    lens_t[2] = 10_000
    pkv.decode_step(t["q"], kn, vn, t["k_cache"], t["v_cache"], m["block_tables"], lens_t, w.scale,
                    max_context_len=512)
    assert pkv.get_device_errors() & pkv._lib.DEVERR_LENGTH


def test_decode_step_on_all_heads_kernel_with_empty_and_many_sequences():
    """Thousands of sequences (the per-CTA plan takes several passes over the
    lengths), a fifth of them empty, on the all-heads kernel: every non-empty
    sequence matches the oracle and every empty one gives a zero row."""
    rng = np.random.default_rng(91)
    lens = rng.integers(1, 60, size=2500)
    lens[rng.choice(2500, 500, replace=False)] = 0
    w = W.decode_workload("step_many", lens, 32, 8, 16, seed=92)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    m = device_meta(w)
    ids = np.arange(w.num_seqs)
    ref = decode_step_reference(w, ids, t["k_cache"], t["v_cache"], t["q"], t["key"], t["value"])
    out = run_step(w, t, m)
    assert_close(out, ref, w.name)
    for i in np.nonzero(w.context_lens == 0)[0]:
        assert (out[int(i)] == 0).all()
