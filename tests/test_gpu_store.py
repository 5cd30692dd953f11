"""GPU parity of pkv_store_kvcache against the oracle store: bit-exact caches."""
import numpy as np
import pytest
import torch

import paged_kv_cache_86_gb300 as pkv
from oracle import attention as oracle
from paged_kv_cache_86_gb300 import workloads as W
from paged_kv_cache_86_gb300.workloads import bf16_to_u16
from pkv_testutil import device_meta

pytestmark = pytest.mark.gpu


def _run_and_compare(w, key=None, value=None):
    t = {k: v.cuda() for k, v in w.tensors.items()}
    key = t["key"] if key is None else key
    value = t["value"] if value is None else value
    ref_k, ref_v = bf16_to_u16(t["k_cache"]).copy(), bf16_to_u16(t["v_cache"]).copy()
    oracle.store_kvcache(bf16_to_u16(key), bf16_to_u16(value), ref_k, ref_v, w.slot_mapping,
                         w.block_size)
    m = device_meta(w)
    pkv.store_kvcache(key, value, t["k_cache"], t["v_cache"], m["slot_mapping"])
    assert pkv.get_device_errors() == 0
    assert np.array_equal(bf16_to_u16(t["k_cache"]), ref_k)
    assert np.array_equal(bf16_to_u16(t["v_cache"]), ref_v)


def test_store_decode_3seq():
    _run_and_compare(W.decode_3seq())


def test_store_small_chunked_prefill_mid_block():
    w = W.prefill_chunks(num_seqs=5, q_len=37, max_prefix=200)
    assert (w.cu_seqlens_k[1:] - w.cu_seqlens_k[:-1] - 37).min() >= 0
    _run_and_compare(w)


def test_store_full_chunked_prefill_16384_tokens():
    w = W.prefill_chunks()
    assert w.num_new_tokens == 16384
    _run_and_compare(w)


@pytest.mark.parametrize("hkv", [1, 2, 4, 8])
def test_store_head_counts_and_block_sizes(hkv):
    for bs in (1, 16, 256):
        w = W.decode_workload(f"store_h{hkv}_bs{bs}", [1, 17, 300, 5], 8 * hkv, hkv, bs,
                              seed=7 + hkv + bs)
        _run_and_compare(w)


def test_store_strided_rows_from_fused_qkv():
    """K and V as views into one [T, Hq + 2 Hkv, D] projection output."""
    w = W.prefill_chunks(num_seqs=3, q_len=20, max_prefix=50)
    hq, hkv, d = w.num_q_heads, w.num_kv_heads, w.head_dim
    fused = torch.zeros(w.num_new_tokens, hq + 2 * hkv, d, dtype=torch.bfloat16, device="cuda")
    fused[:, hq:hq + hkv] = w.tensors["key"].cuda()
    fused[:, hq + hkv:] = w.tensors["value"].cuda()
    key, value = fused[:, hq:hq + hkv], fused[:, hq + hkv:]
    assert key.stride(0) == (hq + 2 * hkv) * d
    _run_and_compare(w, key=key, value=value)


def test_store_skips_negative_slots_and_flags_out_of_range():
    w = W.decode_workload("store_edges", [10, 20, 30, 40], 8, 2, 16, seed=3)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    before_k = t["k_cache"].clone()
    slots = w.slot_mapping.copy()
    slots[0] = -1                                  # padded token
    slots[2] = w.num_blocks * w.block_size + 5     # beyond the pool
    pkv.store_kvcache(t["key"], t["value"], t["k_cache"], t["v_cache"],
                      torch.from_numpy(slots).cuda())
    bits = pkv.get_device_errors()
    assert bits & pkv._lib.DEVERR_SLOT
    assert pkv.get_device_errors() == 0            # cleared
    flat_before = before_k.view(-1, 2, 128)
    flat_after = t["k_cache"].view(-1, 2, 128)
    bs = w.block_size
    assert torch.equal(flat_after[w.slot_mapping[0]], flat_before[w.slot_mapping[0]])
    assert torch.equal(flat_after[slots[1]], t["key"][1])
    assert torch.equal(flat_after[slots[3]], t["key"][3])
    changed = (flat_after != flat_before).any(dim=(1, 2)).nonzero().flatten().tolist()
    assert sorted(changed) == sorted([int(slots[1]), int(slots[3])])
    assert bs == 16


def test_store_zero_tokens_is_noop():
    w = W.decode_workload("store_none", [4], 8, 2, 16, seed=5)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    before = t["k_cache"].clone()
    empty = torch.zeros(0, 2, 128, dtype=torch.bfloat16, device="cuda")
    pkv.store_kvcache(empty, empty, t["k_cache"], t["v_cache"],
                      torch.zeros(0, dtype=torch.int32, device="cuda"))
    assert torch.equal(before, t["k_cache"])
