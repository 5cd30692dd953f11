"""On-GPU failure path, without a fault: a bounded mbarrier wait on a barrier
that nothing arrives on runs out, reports PKV_DEVERR_TIMEOUT, and the two warps
that meet once per step on an OR-reducing hardware barrier (the decode softmax
warps' protocol) leave in the same step; the context stays usable."""
import pytest
import torch

import paged_kv_cache_86_gb300 as pkv
from paged_kv_cache_86_gb300 import workloads as W
from pkv_testutil import assert_close, decode_step_reference, device_meta

pytestmark = pytest.mark.gpu


def test_no_wait_runs_out_without_a_failure():
    assert pkv.get_device_errors() == 0
    res = pkv.selftest_bounded_wait(8)
    assert res == [8, 8, 0, 8]
    assert pkv.get_device_errors() == 0


@pytest.mark.parametrize("fail_step", [0, 3, 7])
def test_a_wait_that_runs_out_reports_and_both_warps_leave_together(fail_step):
    res = pkv.selftest_bounded_wait(fail_step)
    assert res[0] == fail_step and res[1] == fail_step   # same step, no warp left behind
    assert res[2] == 1                                   # the timeout was seen
    assert res[3] == fail_step                           # steps before it completed
    assert pkv.get_device_errors() & pkv._lib.DEVERR_TIMEOUT


def test_context_is_usable_after_a_reported_timeout():
    pkv.selftest_bounded_wait(2)
    assert pkv.get_device_errors() & pkv._lib.DEVERR_TIMEOUT
    w = W.decode_workload("after_timeout", [5, 300, 40], 32, 8, 16, seed=3)
    t = {k: v.cuda() for k, v in w.tensors.items()}
    ref = decode_step_reference(w, list(range(w.num_seqs)), t["k_cache"], t["v_cache"], t["q"],
                                t["key"], t["value"])
    m = device_meta(w)
    pkv.store_kvcache(t["key"], t["value"], t["k_cache"], t["v_cache"], m["slot_mapping"])
    out = pkv.paged_decode(t["q"], t["k_cache"], t["v_cache"], m["block_tables"], m["context_lens"], w.scale)
    assert pkv.get_device_errors() == 0
    assert_close(out, ref, w.name)
