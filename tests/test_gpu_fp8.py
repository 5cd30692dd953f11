"""GPU parity of the fp8 (E4M3, per token-head scale) KV path against the
oracle: the quantizing store bit for bit (codes and scales), decode over the
quantized cache within |gpu - oracle| <= 1e-2 * max(1, |oracle|), and the fused
fp8 decode step (store of each sequence's newest token + decode in one call)
against both the oracle and the two separate calls."""
import numpy as np
import pytest
import torch

import paged_kv_cache_86_gb300 as pkv
from oracle import attention as oracle
from paged_kv_cache_86_gb300 import workloads as W
from paged_kv_cache_86_gb300.workloads import bf16_to_u16
from pkv_testutil import assert_close, per_sequence_rows

pytestmark = pytest.mark.gpu


def fp8_case(w, seed):
    kc, ks = W.fp8_pool(w.num_blocks, w.block_size, w.num_kv_heads, seed * 16 + 7)
    vc, vs = W.fp8_pool(w.num_blocks, w.block_size, w.num_kv_heads, seed * 16 + 8)
    return kc, vc, ks, vs


def step_fp8(w, t, kc, vc, ks, vs):
    """GPU store of the step's new tokens, then fp8 decode."""
    sm = torch.from_numpy(w.slot_mapping).cuda()
    pkv.store_kvcache_fp8(t["key"], t["value"], kc, vc, ks, vs, sm)
    out = pkv.paged_decode_fp8(t["q"], kc, vc, ks, vs, torch.from_numpy(w.block_tables).cuda(),
                               torch.from_numpy(w.context_lens).cuda(), w.scale)
    torch.cuda.synchronize()
    assert pkv.get_device_errors() == 0
    return out


def oracle_step_fp8(w, seq_ids, kc, vc, ks, vs, t):
    """Oracle store + fp8 decode on host copies of the pool taken BEFORE the GPU step."""
    k8, v8 = kc.cpu().numpy().copy(), vc.cpu().numpy().copy()
    k_s, v_s = ks.cpu().numpy().copy(), vs.cpu().numpy().copy()
    oracle.store_kvcache_fp8(bf16_to_u16(t["key"]), bf16_to_u16(t["value"]), k8, v8, k_s, v_s,
                             w.slot_mapping, w.block_size)
    mask = np.zeros(w.num_seqs, np.uint8)
    mask[np.asarray(seq_ids)] = 1
    out = oracle.paged_decode_fp8(bf16_to_u16(t["q"]), k8, v8, k_s, v_s, w.block_tables,
                                  w.context_lens, w.scale, seq_mask=mask)
    return out[np.asarray(seq_ids)], (k8, v8, k_s, v_s)


# the all-heads tcgen05 kernel (Hkv 4 or 8, 128/Hkv dividing the block size),
# else the CUDA-core kernel (2 x 4 at 16, 8 x 4 at 1, 1 x 8 at 4, 4 x 2 at 12)
@pytest.mark.parametrize("hkv,group,bs", [(8, 4, 16), (8, 1, 16), (8, 2, 32), (4, 8, 32),
                                          (4, 2, 64), (8, 2, 256), (8, 8, 16), (2, 4, 16),
                                          (8, 4, 1), (1, 8, 4), (4, 2, 12), (1, 4, 1)])
def test_fp8_store_and_decode_match_the_oracle(hkv, group, bs):
    lens = [1, 2, 15, 16, 17, 0, 300, 1025, 77, 2000]
    w = W.decode_workload(f"fp8_{hkv}x{group}_bs{bs}", lens, hkv * group, hkv, bs,
                          seed=900 + hkv * 7 + group * 3 + bs)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    kc, vc, ks, vs = fp8_case(w, w.seed)
    ids = np.arange(w.num_seqs)
    ref, (k8, v8, k_s, v_s) = oracle_step_fp8(w, ids, kc, vc, ks, vs, t)
    out = step_fp8(w, t, kc, vc, ks, vs)
    # the store: codes and scales bit for bit, everywhere in the pool
    assert np.array_equal(kc.cpu().numpy(), k8) and np.array_equal(vc.cpu().numpy(), v8)
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), k_s.view(np.uint32))
    assert np.array_equal(vs.cpu().numpy().view(np.uint32), v_s.view(np.uint32))
    assert_close(out, ref, w.name)
    assert (out[5] == 0).all()


def test_fp8_store_zero_and_large_rows():
    w = W.decode_workload("fp8_rows", [3, 9], 32, 8, 16, seed=31)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    t["key"][0].zero_()                              # an all-zero row: codes 0, scale 0
    t["value"][1] *= 1000.0                          # large values: scale grows, codes saturate at 448
    kc, vc, ks, vs = fp8_case(w, 31)
    ids = np.arange(w.num_seqs)
    ref, (k8, v8, k_s, v_s) = oracle_step_fp8(w, ids, kc, vc, ks, vs, t)
    out = step_fp8(w, t, kc, vc, ks, vs)
    assert np.array_equal(kc.cpu().numpy(), k8) and np.array_equal(vc.cpu().numpy(), v8)
    assert np.array_equal(ks.cpu().numpy(), k_s) and np.array_equal(vs.cpu().numpy(), v_s)
    s0 = int(w.slot_mapping[0])
    assert (kc.view(-1, 8, 128)[s0] == 0).all() and (ks[s0] == 0).all()
    assert_close(out, ref, w.name)


def test_fp8_decode_512seq_full_size_every_sequence():
    w = W.decode_512seq(fill="device")
    t = {k: v.cuda() for k, v in w.tensors.items()}
    kc, vc, ks, vs = fp8_case(w, w.seed)
    ids = np.arange(w.num_seqs)
    ref, _ = oracle_step_fp8(w, ids, kc, vc, ks, vs, t)
    out = step_fp8(w, t, kc, vc, ks, vs)
    assert_close(out[torch.from_numpy(ids).cuda()], ref, w.name)


def test_fp8_decode_rejects_shapes_without_the_kernel():
    w = W.decode_workload("fp8_bad", [5, 9], 6, 2, 16, seed=32)     # 3 query heads per KV head: no fp8 kernel
    t = {k: v.cuda() for k, v in w.tensors.items()}
    kc, vc, ks, vs = fp8_case(w, 32)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_fp8(t["q"], kc, vc, ks, vs, torch.from_numpy(w.block_tables).cuda(),
                             torch.from_numpy(w.context_lens).cuda(), w.scale)
    assert e.value.status == -2


def test_fp8_decode_late_maximum_rescales_the_accumulator():
    # the new token of each sequence is a key aligned with one query head: its
    # logit exceeds the reference maximum of the segment's first stage by far
    # more than the lazy-rescale threshold, in the last stage of the context
    hkv, group, bs = 8, 4, 16
    lens = [300, 2000, 700, 64, 17]
    w = W.decode_workload("fp8_late_max", lens, hkv * group, hkv, bs, seed=4321)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    for i in range(len(lens)):
        for h, logit in ((0, 30.0), (3, 12.0), (5, 9.0), (7, 20.0)):
            q = t["q"][i, h * group + (i % group)].float()
            t["key"][i, h] = (q * (logit * 128 ** 0.5 / float((q * q).sum()))).to(torch.bfloat16)
    kc, vc, ks, vs = fp8_case(w, w.seed)
    ids = np.arange(w.num_seqs)
    ref, _ = oracle_step_fp8(w, ids, kc, vc, ks, vs, t)
    out = step_fp8(w, t, kc, vc, ks, vs)
    assert_close(out, ref, w.name)


def run_step_fp8(w, t, kc, vc, ks, vs):
    kn, vn = per_sequence_rows(w, t)
    out = pkv.decode_step_fp8(t["q"], kn, vn, kc, vc, ks, vs,
                              torch.from_numpy(w.block_tables).cuda(),
                              torch.from_numpy(w.context_lens).cuda(), w.scale)
    torch.cuda.synchronize()
    assert pkv.get_device_errors() == 0
    return out


@pytest.mark.parametrize("hkv,group,bs", [(8, 4, 16), (8, 1, 16), (4, 8, 32), (8, 2, 256),
                                          (8, 8, 32), (2, 2, 5), (8, 4, 3)])
def test_fp8_decode_step_matches_the_oracle(hkv, group, bs):
    lens = [1, 2, 16, 17, 0, 300, 1023, 5, 129, 2000, 0, 64]
    w = W.decode_workload(f"fp8_step_{hkv}x{group}_bs{bs}", lens, hkv * group, hkv, bs,
                          seed=1700 + hkv * 13 + group * 5 + bs)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    kc, vc, ks, vs = fp8_case(w, w.seed)
    ids = np.arange(w.num_seqs)
    ref, (k8, v8, k_s, v_s) = oracle_step_fp8(w, ids, kc, vc, ks, vs, t)
    out = run_step_fp8(w, t, kc, vc, ks, vs)
    assert np.array_equal(kc.cpu().numpy(), k8) and np.array_equal(vc.cpu().numpy(), v8)
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), k_s.view(np.uint32))
    assert np.array_equal(vs.cpu().numpy().view(np.uint32), v_s.view(np.uint32))
    assert_close(out, ref, w.name)
    for i in np.nonzero(w.context_lens == 0)[0]:
        assert (out[int(i)] == 0).all()


def test_fp8_decode_step_equals_store_then_decode():
    lens = np.random.default_rng(13).integers(1, 900, size=70)
    w = W.decode_workload("fp8_step_eq", lens, 32, 8, 16, seed=1313)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    kc, vc, ks, vs = fp8_case(w, w.seed)
    kc2, vc2, ks2, vs2 = kc.clone(), vc.clone(), ks.clone(), vs.clone()
    two_calls = step_fp8(w, t, kc2, vc2, ks2, vs2)
    fused = run_step_fp8(w, t, kc, vc, ks, vs)
    assert torch.equal(fused, two_calls)
    assert torch.equal(kc, kc2) and torch.equal(vc, vc2)
    assert torch.equal(ks.view(torch.int32), ks2.view(torch.int32))
    assert torch.equal(vs.view(torch.int32), vs2.view(torch.int32))


def test_fp8_decode_step_512seq_full_size_every_sequence():
    w = W.decode_512seq(fill="device")
    t = {k: v.cuda() for k, v in w.tensors.items()}
    kc, vc, ks, vs = fp8_case(w, w.seed)
    ids = np.arange(w.num_seqs)
    ref, _ = oracle_step_fp8(w, ids, kc, vc, ks, vs, t)
    out = run_step_fp8(w, t, kc, vc, ks, vs)
    assert_close(out[torch.from_numpy(ids).cuda()], ref, w.name)


def test_fp8_decode_extreme_query_magnitudes():
    # per query head the kernel scales Q by a power of two before splitting it
    # into two E4M3 terms: rows far above the E4M3 range (448) and far below
    # its normal range must come out as with a plain Q
    hkv, group, bs = 8, 4, 16
    lens = [300, 2000, 700, 64, 17, 1]
    w = W.decode_workload("fp8_q_range", lens, hkv * group, hkv, bs, seed=4242)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    big = torch.tensor([3.0e4, 1.0, 1.0e-4, 5.0e3, 1.0, 2.0e-5], device="cuda")
    t["q"] = (t["q"].float() * big[:, None, None] / 128 ** 0.5 * 0.05).to(torch.bfloat16)
    t["q"][1, 5] *= 1.0e4          # one head of an ordinary row far above the rest
    kc, vc, ks, vs = fp8_case(w, w.seed)
    ids = np.arange(w.num_seqs)
    ref, _ = oracle_step_fp8(w, ids, kc, vc, ks, vs, t)
    out = step_fp8(w, t, kc, vc, ks, vs)
    assert torch.isfinite(out.float()).all()
    assert_close(out, ref, w.name)


def test_fp8_decode_step_replays_from_a_cuda_graph_at_a_padded_batch():
    """29 live sequences padded to a captured batch of 48 with empty rows; the
    fp8 step is replayed for three consecutive steps (context_lens grows by one
    and new q / K / V rows arrive each step, all through the same buffers)."""
    live, padded, hkv, group, bs = 29, 48, 8, 4, 16
    rng = np.random.default_rng(19)
    lens0 = (rng.integers(0, 30, size=live) * bs + rng.integers(1, bs - 3, size=live)).astype(np.int32)
    grown = np.concatenate([lens0 + 3, np.zeros(padded - live, np.int32)])  # blocks for 3 steps
    w0 = W.decode_workload("graph_pad_fp8", grown, hkv * group, hkv, bs, seed=78)
    kc, vc, ks, vs = fp8_case(w0, w0.seed)
    bt = torch.from_numpy(w0.block_tables).cuda()
    cl = torch.zeros(padded, dtype=torch.int32, device="cuda")
    q = torch.zeros((padded, hkv * group, 128), dtype=torch.bfloat16, device="cuda")
    kn = torch.zeros((padded, hkv, 128), dtype=torch.bfloat16, device="cuda")
    vn = torch.zeros_like(kn)
    out = torch.empty_like(q)
    ws = torch.empty(pkv.decode_workspace_size(padded, hkv * group, hkv), dtype=torch.uint8,
                     device="cuda")
    max_ctx = int(w0.block_tables.shape[1] * bs)

    def step():
        pkv.decode_step_fp8(q, kn, vn, kc, vc, ks, vs, bt, cl, w0.scale, max_context_len=max_ctx,
                            out=out, workspace=ws)

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

    gen = torch.Generator(device="cuda").manual_seed(6)
    mask = np.zeros(padded, np.uint8)
    mask[:live] = 1
    for k in range(3):
        lens = np.concatenate([lens0 + k, np.zeros(padded - live, np.int32)]).astype(np.int32)
        cl.copy_(torch.from_numpy(lens))
        q.normal_(generator=gen)
        kn.normal_(generator=gen)
        vn.normal_(generator=gen)
        q[live:] = 0
        kn[live:] = 0
        vn[live:] = 0
        # the oracle's view of this step: host copies of the pool before the replay
        k8, v8 = kc.cpu().numpy().copy(), vc.cpu().numpy().copy()
        k_s, v_s = ks.cpu().numpy().copy(), vs.cpu().numpy().copy()
        slots = np.array([w0.block_tables[i, (n - 1) // bs] * bs + (n - 1) % bs
                          for i, n in enumerate(lens[:live])], dtype=np.int32)
        oracle.store_kvcache_fp8(bf16_to_u16(kn[:live]), bf16_to_u16(vn[:live]), k8, v8, k_s, v_s,
                                 slots, bs)
        ref = oracle.paged_decode_fp8(bf16_to_u16(q), k8, v8, k_s, v_s, w0.block_tables, lens,
                                      w0.scale, seq_mask=mask)[:live]
        g.replay()
        torch.cuda.synchronize()
        assert pkv.get_device_errors() == 0
        assert np.array_equal(kc.cpu().numpy(), k8) and np.array_equal(vc.cpu().numpy(), v8)
        assert np.array_equal(ks.cpu().numpy().view(np.uint32), k_s.view(np.uint32))
        assert np.array_equal(vs.cpu().numpy().view(np.uint32), v_s.view(np.uint32))
        assert_close(out[:live], ref, f"fp8 graph step {k}")
        assert (out[live:] == 0).all()
