"""The bench's CPU-baseline leg (no GPU): the oracle timed on a bounded sample,
on all host cores or on a chosen number of threads, which it restores."""
import bench
from oracle import attention as oracle
from paged_kv_cache_86_gb300 import workloads as W


def test_cpu_leg_on_one_thread_restores_the_thread_count():
    before = oracle.max_threads()
    r = bench.cpu_oracle_sample(W.decode_3seq(), target_s=0.2, max_seqs=3, threads=1)
    assert r["cores"] == 1 and r["kind"] == "oracle" and r["value"] > 0
    assert "1 thread(s)" in r["sample"]
    assert oracle.max_threads() == before


def test_cpu_leg_on_all_threads():
    r = bench.cpu_oracle_sample(W.decode_3seq(), target_s=0.2, max_seqs=3)
    assert r["cores"] == oracle.max_threads() and r["value"] > 0
