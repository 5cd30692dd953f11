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


def test_reference_line_carries_the_gpu_arms_config(monkeypatch):
    """The reference arm's JSON line names the same workload and sizes as the
    GPU arm's (both come from bench.workload_config)."""
    from types import SimpleNamespace
    w = W.decode_3seq()
    monkeypatch.setattr(bench, "make_workload", lambda name, **kw: w)
    monkeypatch.setattr(bench, "cpu_oracle_sample",
                        lambda *a, **kw: {"value": 10.0, "unit": bench.UNIT, "cores": 1,
                                          "kind": "oracle", "sample": "stub", "seconds": 0.1})
    line = bench.run_reference(SimpleNamespace(steps=2, warmup=0, workload="decode_3seq"), 0)
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["config"] == bench.workload_config(w)
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert bench.run_reference(SimpleNamespace(steps=2, warmup=0, workload="decode_3seq"), 1) is None
