"""pkv_paged_decode_static_ws, the decode entry point for callers that cannot
give the library device memory (e.g. a plug-in whose host framework owns all
device memory, or a runtime that only passes its input and output buffers).
It must give the same result as pkv_paged_decode with a caller workspace, call
after call, while allocating nothing itself; its scratch is a fixed 16 MiB
array inside the library.

Kept in a file that sorts last so that a run stopping at the first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_86_gb300 as pkv
from oracle import attention as oracle
from paged_kv_cache_86_gb300 import workloads as W
from paged_kv_cache_86_gb300.workloads import bf16_to_u16
from pkv_testutil import RTOL, assert_close, compact_inputs, device_meta

pytestmark = pytest.mark.gpu

STATIC_CAPACITY = 16 << 20


def _entry_point():
    lib = pkv.load()
    f = lib.pkv_paged_decode_static_ws
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    f.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i32, ctypes.c_float,
                  ctypes.c_int, vp]
    f.restype = ctypes.c_int
    return f


def _call_static(f, w, t, m, out):
    stream = torch.cuda.current_stream()
    return f(ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(t["q"].data_ptr()),
             ctypes.c_void_p(t["k_cache"].data_ptr()), ctypes.c_void_p(t["v_cache"].data_ptr()),
             ctypes.c_void_p(m["block_tables"].data_ptr()), w.max_blocks_per_seq,
             ctypes.c_void_p(m["context_lens"].data_ptr()), w.num_seqs,
             w.max_blocks_per_seq * w.block_size, w.num_q_heads, w.num_kv_heads, w.head_dim,
             w.block_size, w.num_blocks, w.scale, 0, ctypes.c_void_p(stream.cuda_stream))


def _within_tolerance(got, ref):
    g, r = got.double(), ref.double()
    return bool(((g - r).abs() <= RTOL * torch.clamp(r.abs(), min=1.0)).all())


def _oracle_decode(w, t):
    """The oracle's decode of every sequence over the caches as they are."""
    ids = np.arange(w.num_seqs)
    _, _, tables, kc, vc = compact_inputs(w, ids, t["k_cache"], t["v_cache"])
    return oracle.paged_decode(bf16_to_u16(t["q"]), kc, vc, tables, w.context_lens, w.scale)


def _device_memory_in_use():
    """Free device memory as the driver sees it and the count of torch allocations."""
    free, _ = torch.cuda.mem_get_info()
    return free, torch.cuda.memory_stats().get("allocation.all.allocated", 0)


@pytest.mark.parametrize("make", [
    lambda: W.decode_512seq(num_seqs=96, hi=3000),     # sequences cut across CTA ranges
    lambda: W.decode_3seq(),                           # 2 KV heads: every sequence combined
])
def test_static_workspace_decode_matches_workspace_decode(make):
    w = make()
    t = {k: v.cuda() for k, v in w.tensors.items()}
    m = device_meta(w)
    assert pkv.decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads) <= STATIC_CAPACITY
    ref = pkv.paged_decode(t["q"], t["k_cache"], t["v_cache"], m["block_tables"],
                           m["context_lens"], w.scale)
    f = _entry_point()
    outs = [torch.full_like(t["q"], float("nan")) for _ in range(3)]
    # the first call on this device may look up the scratch array's address;
    # after it, further calls must not allocate device memory of any kind
    assert _call_static(f, w, t, m, outs[0]) == 0
    torch.cuda.synchronize()
    before = _device_memory_in_use()
    for out in outs[1:]:  # two calls in a row share (and reuse) the static scratch
        assert _call_static(f, w, t, m, out) == 0
        torch.cuda.synchronize()
    assert _device_memory_in_use() == before
    assert pkv.get_device_errors() == 0
    expected = _oracle_decode(w, t)
    for out in outs:
        assert _within_tolerance(out, ref)
        assert torch.equal(out, ref)  # the same deterministic kernels as the workspace call
        assert_close(out, expected, w.name + " (static scratch) vs oracle")


def test_static_workspace_rejects_batch_beyond_capacity():
    # enough sequences that the partial records outgrow the 16 MiB array
    num_seqs = 5000
    lens = np.full(num_seqs, 4, np.int32)
    w = W.decode_workload("too_big", lens, 8, 2, 16, seed=3)
    assert pkv.decode_workspace_size(num_seqs, 8, 2) > STATIC_CAPACITY
    t = {k: v.cuda() for k, v in w.tensors.items()}
    m = device_meta(w)
    out = torch.empty_like(t["q"])
    assert _call_static(_entry_point(), w, t, m, out) == -4  # PKV_ERR_WORKSPACE
