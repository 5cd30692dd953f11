"""The binding refuses tensors whose memory is not the dense row-major layout the
kernels read through raw pointers (a transposed q, a sliced block table or
cache, strided cu_seqlens). These checks run before any device check, so they
are exercised here on CPU tensors; a dense CPU tensor gets past them and is then
refused for not being on the GPU."""
import pytest
import torch

import paged_kv_cache_86_gb300 as pkv

BF16, I32 = torch.bfloat16, torch.int32


def prefill_args():
    # two sequences of 4 query rows over 20 keys, 8 query / 2 KV heads, block 16
    q = torch.zeros(8, 8, 128, dtype=BF16)
    kc = torch.zeros(6, 16, 2, 128, dtype=BF16)
    vc = torch.zeros_like(kc)
    cu_q = torch.tensor([0, 4, 8], dtype=I32)
    cu_k = torch.tensor([0, 20, 40], dtype=I32)
    bt = torch.tensor([[0, 1], [2, 3]], dtype=I32)
    return dict(q=q, k_cache=kc, v_cache=vc, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, block_tables=bt)


def call_prefill(a):
    return pkv.paged_prefill(a["q"], a["k_cache"], a["v_cache"], a["cu_seqlens_q"],
                             a["cu_seqlens_k"], a["block_tables"], 0.088, 4, 20)


def strided_views(a):
    """One non-contiguous view per argument, of the same shape and dtype."""
    return {
        "q": a["q"].transpose(0, 1).contiguous().transpose(0, 1),
        "k_cache": torch.zeros(6, 16, 4, 128, dtype=BF16)[:, :, :2],
        "v_cache": torch.zeros(6, 16, 2, 256, dtype=BF16)[..., :128],
        "cu_seqlens_q": torch.tensor([0, 9, 4, 9, 8, 9], dtype=I32)[::2],
        "cu_seqlens_k": torch.tensor([0, 9, 20, 9, 40, 9], dtype=I32)[::2],
        "block_tables": torch.tensor([[0, 1, 9, 9], [2, 3, 9, 9]], dtype=I32)[:, :2],
    }


@pytest.mark.parametrize("name", ["q", "k_cache", "v_cache", "cu_seqlens_q", "cu_seqlens_k",
                                  "block_tables"])
def test_prefill_rejects_a_strided_view(name):
    a = prefill_args()
    view = strided_views(a)[name]
    assert view.shape == a[name].shape and not view.is_contiguous()
    a[name] = view
    with pytest.raises(ValueError, match=f"{name} must be contiguous"):
        call_prefill(a)


def test_prefill_dense_cpu_tensors_pass_layout_then_fail_device():
    with pytest.raises(TypeError, match="CUDA tensor"):
        call_prefill(prefill_args())


def mixed_args():
    a = prefill_args()
    a["key"] = torch.zeros(8, 2, 128, dtype=BF16)
    a["value"] = torch.zeros(8, 2, 128, dtype=BF16)
    a["slot_mapping"] = torch.arange(8, dtype=I32)
    return a


def call_mixed(a):
    return pkv.mixed_step(a["q"], a["key"], a["value"], a["slot_mapping"], a["k_cache"],
                          a["v_cache"], a["cu_seqlens_q"], a["cu_seqlens_k"], a["block_tables"],
                          0, 0.088, 4, 20)


@pytest.mark.parametrize("name", ["q", "k_cache", "v_cache", "cu_seqlens_q", "cu_seqlens_k",
                                  "block_tables", "slot_mapping"])
def test_mixed_step_rejects_a_strided_view(name):
    a = mixed_args()
    views = strided_views(a)
    views["slot_mapping"] = torch.arange(16, dtype=I32)[::2]
    view = views[name]
    assert view.shape == a[name].shape and not view.is_contiguous()
    a[name] = view
    with pytest.raises(ValueError, match=f"{name} must be contiguous"):
        call_mixed(a)


def test_mixed_step_rejects_split_key_rows():
    # a key whose [Hkv, D] row is not one dense block (heads interleaved)
    a = mixed_args()
    a["key"] = torch.zeros(8, 128, 2, dtype=BF16).transpose(1, 2)
    with pytest.raises(ValueError, match="key rows must be contiguous"):
        call_mixed(a)


def test_mixed_step_dense_cpu_tensors_pass_layout_then_fail_device():
    with pytest.raises(TypeError, match="CUDA tensor"):
        call_mixed(mixed_args())
