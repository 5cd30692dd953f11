"""GPU parity of a decode step (store of the new tokens, then paged decode)
against the oracle, within |gpu - oracle| <= 1e-2 * max(1, |oracle|)."""
import numpy as np
import pytest
import torch

import paged_kv_cache_86_gb300 as pkv
from paged_kv_cache_86_gb300 import workloads as W
from pkv_testutil import assert_close, decode_step_reference, device_meta

pytestmark = pytest.mark.gpu


def run_decode_step(w, t=None):
    """GPU store + decode through the C ABI; returns (out, tensors before store)."""
    t = t or {k: v.cuda() for k, v in w.tensors.items()}
    m = device_meta(w)
    pkv.store_kvcache(t["key"], t["value"], t["k_cache"], t["v_cache"], m["slot_mapping"])
    out = pkv.paged_decode(t["q"], t["k_cache"], t["v_cache"], m["block_tables"],
                           m["context_lens"], w.scale)
    assert pkv.get_device_errors() == 0
    return out


def check(w, seq_ids=None, what=""):
    t = {k: v.cuda() for k, v in w.tensors.items()}
    seq_ids = np.arange(w.num_seqs) if seq_ids is None else np.asarray(seq_ids)
    ref = decode_step_reference(w, seq_ids, t["k_cache"], t["v_cache"], t["q"], t["key"], t["value"])
    out = run_decode_step(w, t)
    return assert_close(out[torch.from_numpy(seq_ids).cuda()], ref, what or w.name)


def test_decode_3seq_pages_example():
    check(W.decode_3seq())


def test_decode_64seq_reduced():
    check(W.decode_64seq(num_seqs=12, max_len=1500))


def test_decode_512seq_reduced():
    check(W.decode_512seq(num_seqs=40, hi=900))


def test_decode_longtail_reduced():
    check(W.decode_longtail(num_long=2, long_len=6000, num_short=30, short_len=200))


@pytest.mark.parametrize("hkv", [1, 2, 4, 8])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_decode_head_configurations(hkv, group):
    lens = [1, 2, 15, 16, 17, 63, 200, 777]
    w = W.decode_workload(f"heads_{hkv}x{group}", lens, hkv * group, hkv, 16, seed=100 + hkv * 10 + group)
    check(w)


@pytest.mark.parametrize("hkv,group,bs", [(16, 1, 16), (3, 5, 32), (2, 16, 16), (1, 12, 8),
                                           (8, 4, 12), (4, 4, 6), (4, 4, 32), (32, 2, 16),
                                           (8, 3, 16), (16, 8, 16), (64, 1, 16), (2, 4, 3),
                                           (1, 2, 8), (2, 8, 1), (1, 1, 5), (1, 2, 1)])
def test_decode_more_head_shapes(hkv, group, bs):
    # all-heads tcgen05 kernel when Hkv is 4, 8 or 16, G is 1, 2, 4 or 8 and
    # 128/Hkv divides the block size; per-head tcgen05 kernel for other block
    # sizes that are multiples of 16 (of 8 when the CUDA-core kernel cannot
    # take the heads: 1 x 12 at 8); the CUDA-core split kernel for the rest
    # (8 x 4 at 12, 4 x 4 at 6, 2 x 4 at 3, 1 x 2 at 8, 2 x 8 at 1, 1 x 1 at 5;
    # at blocks shorter than a stage its stages span several blocks)
    lens = [1, 9, 128, 129, 700, 2000]
    w = W.decode_workload(f"shape_{hkv}x{group}_bs{bs}", lens, hkv * group, hkv, bs,
                          seed=500 + hkv * 31 + group * 7 + bs)
    check(w)


@pytest.mark.parametrize("bs", [1, 3, 8, 64, 256, 1024])
def test_decode_block_sizes(bs):
    w = W.decode_workload(f"bs{bs}", [5, 300, 1, 1024, 77], 32, 8, bs, seed=200 + bs)
    check(w)


def test_decode_one_long_sequence_splits_over_every_cta():
    # one 60000-token context is cut into many ranges: exercises the combine pass
    w = W.decode_workload("one_long", [60000], 32, 8, 16, seed=11)
    check(w)


def test_decode_many_tiny_sequences():
    rng = np.random.default_rng(5)
    lens = rng.integers(1, 9, size=3000)
    w = W.decode_workload("tiny_many", lens, 32, 8, 16, seed=12)
    check(w, seq_ids=np.concatenate([np.arange(0, 3000, 97), [2999]]))


def test_decode_zero_context_rows_are_zero():
    w = W.decode_workload("with_empty", [0, 40, 0, 3, 0], 8, 2, 16, seed=13)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    ref = decode_step_reference(w, np.arange(5), t["k_cache"], t["v_cache"], t["q"], t["key"], t["value"])
    out = run_decode_step(w, t)
    for i in (0, 2, 4):
        assert (out[i] == 0).all()
    assert_close(out, ref, "with_empty")


def test_decode_context_one_returns_stored_value():
    w = W.decode_workload("ctx1", [1] * 37, 32, 8, 16, seed=14)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    out = run_decode_step(w, t)
    g = 4
    for i in range(37):
        for h in range(32):
            assert torch.equal(out[i, h], t["value"][i, h // g])


def test_decode_repeat_calls_are_deterministic_and_reuse_workspace():
    w = W.decode_512seq(num_seqs=64, hi=2000)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    m = device_meta(w)
    pkv.store_kvcache(t["key"], t["value"], t["k_cache"], t["v_cache"], m["slot_mapping"])
    ws = torch.empty(pkv.decode_workspace_size(w.num_seqs, 32, 8), dtype=torch.uint8, device="cuda")
    a = pkv.paged_decode(t["q"], t["k_cache"], t["v_cache"], m["block_tables"], m["context_lens"],
                         w.scale, workspace=ws)
    b = pkv.paged_decode(t["q"], t["k_cache"], t["v_cache"], m["block_tables"], m["context_lens"],
                         w.scale, workspace=ws)
    assert torch.equal(a, b)


def test_decode_flags_bad_block_id_and_length():
    w = W.decode_workload("bad_meta", [40, 40], 8, 2, 16, seed=15)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    m = device_meta(w)
    bt = m["block_tables"].clone()
    bt[0, 1] = w.num_blocks + 3
    pkv.paged_decode(t["q"], t["k_cache"], t["v_cache"], bt, m["context_lens"], w.scale)
    assert pkv.get_device_errors() & pkv._lib.DEVERR_BLOCK_ID
    lens = m["context_lens"].clone()
    lens[1] = 10_000
    pkv.paged_decode(t["q"], t["k_cache"], t["v_cache"], m["block_tables"], lens, w.scale,
                     max_context_len=64)
    assert pkv.get_device_errors() & pkv._lib.DEVERR_LENGTH


def test_decode_rejects_small_workspace():
    w = W.decode_workload("ws", [4, 4], 8, 2, 16, seed=16)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    m = device_meta(w)
    with pytest.raises(pkv.PkvError):
        pkv.paged_decode(t["q"], t["k_cache"], t["v_cache"], m["block_tables"], m["context_lens"],
                         w.scale, workspace=torch.empty(256, dtype=torch.uint8, device="cuda"))


# ---- full-size workloads, in the launch configuration the bench times: every
# sequence against the oracle

def test_decode_64seq_full_size_every_sequence():
    check(W.decode_64seq(fill="device"))


def test_decode_512seq_full_size_every_sequence():
    check(W.decode_512seq(fill="device"))


def test_decode_longtail_full_size_every_sequence():
    check(W.decode_longtail(fill="device"))


def test_decode_full_size_all_rows_within_convex_hull():
    """Any size: each output coordinate is a convex combination of the V values
    it attends to, so it is finite and no larger in magnitude than max |V|."""
    w = W.decode_512seq(fill="device")
    t = {k: v.cuda() for k, v in w.tensors.items()}
    out = run_decode_step(w, t)
    vmax = max(t["v_cache"].abs().max().item(), t["value"].abs().max().item())
    assert torch.isfinite(out.float()).all()
    assert out.float().abs().max().item() <= vmax * (1 + 1e-2)


def test_decode_rejects_shapes_no_kernel_covers():
    # block size not a multiple of 8 with 3 KV heads: neither tensor-core kernel
    # applies and the CUDA-core kernel needs Hkv dividing 8 -> PKV_ERR_SHAPE
    w = W.decode_workload("unsupported", [5, 9], 6, 3, 3, seed=17)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    m = device_meta(w)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode(t["q"], t["k_cache"], t["v_cache"], m["block_tables"], m["context_lens"],
                         w.scale)
    assert e.value.status == -2


def aligned_key(q_row, logit):
    """A key whose scaled dot product with q_row (scale 1/sqrt(D)) is `logit`."""
    q = q_row.float()
    d = q.shape[0]
    return (q * (logit * d ** 0.5 / float((q * q).sum()))).to(torch.bfloat16)


@pytest.mark.parametrize("hkv,group", [(8, 4), (4, 8), (16, 2)])
def test_decode_late_maximum_rescales_the_accumulator(hkv, group):
    # keys aligned with one query head far into the context: a later stage's
    # logit exceeds the reference maximum of the segment's first stage by much
    # more than the lazy-rescale threshold, in heads handled by different
    # softmax warps, twice in one sequence, and once at the new token itself
    lens = [300, 2000, 700, 64, 4000, 17]
    w = W.decode_workload(f"late_max_{hkv}x{group}", lens, hkv * group, hkv, 16, seed=321 + hkv)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    bs = w.block_size
    # (logit 100 puts exp2 of the gap beyond bf16's range: without the rescale
    # the P^T values would overflow)
    spikes = [(0, 0.7, 30.0), (hkv // 2 - 1, 0.5, 12.0), (hkv - 3, 0.9, 9.0), (hkv - 3, 0.95, 40.0),
              (hkv - 1, 0.3, 15.0), (1, 0.6, 100.0)]
    for i, n in enumerate(lens):
        for h, frac, logit in spikes:
            pos = int(frac * (n - 1))           # an already cached position (< n - 1)
            blk, off = int(w.block_tables[i, pos // bs]), pos % bs
            g = (i + h) % group
            t["k_cache"][blk, off, h] = aligned_key(t["q"][i, h * group + g], logit)
        # the new token of this step is a spike too (quantized and stored first)
        t["key"][i, hkv - 2] = aligned_key(t["q"][i, (hkv - 2) * group], 25.0)
    ids = np.arange(w.num_seqs)
    ref = decode_step_reference(w, ids, t["k_cache"], t["v_cache"], t["q"], t["key"], t["value"])
    out = run_decode_step(w, t)
    assert_close(out, ref, w.name)
