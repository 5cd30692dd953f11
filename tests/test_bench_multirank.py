"""The host side of bench.py's N > 1 path on CPU: two gloo ranks on 127.0.0.1.
Each rank builds its own replica workload (same shape, its own seed), the job
time is the maximum over ranks, and the reported value counts every rank's
sequences (weak scaling)."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = bench.make_workload("decode_512seq", seed_offset=rank, fill="none")
        my_ms = 1.0 + rank                       # rank 1 is the slow one
        job_ms = bench.max_over_ranks(my_ms, world, torch.device("cpu"))
        value = bench.job_throughput(world, w.num_seqs, job_ms)
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), lens=w.context_lens,
                 num_seqs=w.num_seqs, job_ms=job_ms, value=value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_replicas_weak_scaling(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    r = [np.load(tmp_path / f"rank{i}.npz") for i in range(world)]
    # replicas: same per-rank work, different seeded data
    assert int(r[0]["num_seqs"]) == int(r[1]["num_seqs"]) == 512
    assert not np.array_equal(r[0]["lens"], r[1]["lens"])
    # barrier + max-over-ranks timing, identical on every rank
    assert float(r[0]["job_ms"]) == float(r[1]["job_ms"]) == 2.0
    # whole-job throughput: all ranks' sequences over the slowest rank's time
    assert float(r[0]["value"]) == pytest.approx(2 * 512 / 2.0e-3)


def test_single_rank_reduction_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1, None) == 3.25
    assert bench.job_throughput(1, 512, 0.5) == pytest.approx(1.024e6)
