#!/usr/bin/env python
"""Benchmark of one decode step over a block-paged KV cache on GB300.

A step is the whole hot path for one batch: store each sequence's new K/V token
into the cache, then paged decode attention over every sequence's cached
context, both through one pkv_decode_step call (the attention kernel, which
plans the call and writes the new tokens, then the combine). The two-call path
(pkv_store_kvcache + pkv_paged_decode) is timed beside it for the breakdown.

Default workload: 512 sequences, context lengths clip(rint(exp(ln 800 +
N(0,1))), 16, 4096), 32 query / 8 KV heads, head_dim 128, block size 16, a
fragmented pool; bf16, synthetic (seeded). One JSON line is printed by rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--workload decode_512seq|decode_64seq|decode_longtail|decode_3seq]

Under torchrun (N > 1) every rank runs its own replica of the workload (weak
scaling, no collective on the data path); the timed region is bracketed by a
barrier and the max over ranks is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode tokens/s + KV GB/s (% of GB300 HBM peak) at 512 seqs"
UNIT = "tokens/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--workload", default="decode_512seq")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="smaller case of the same workload recipe (profiling captures)")
    ap.add_argument("--quick", action="store_true",
                    help="warm-up and timed steps only: no per-op, e2e, clocks or CPU legs")
    ap.add_argument("--only-prefill", action="store_true",
                    help="time only the chunked-prefill row (store + prefill), for profiling")
    ap.add_argument("--only-row", default=None,
                    choices=["fp8", "copy", "mixed", "store", "decode_3seq", "decode_64seq",
                             "decode_longtail", "small_blocks"],
                    help="time only one row (fp8 decode, block copy, mixed round, sustained "
                         "store, or another decode workload), for profiling (--num-seqs applies "
                         "to the fp8 row, --store-copies to the store row)")
    ap.add_argument("--store-copies", type=int, default=16,
                    help="back-to-back disjoint store launches of the sustained store row")
    return ap.parse_args()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_bf16_peak():
    """Dense bf16 GEMM TFLOP/s: the measured burst figure, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"])
    return 1900.0


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, enabled: bool = True):
        self.enabled = enabled
        self.idx = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        if not self.enabled:
            return self
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.path is None:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for _, _, flags in rows for k, v in enumerate(flags)
                          if v.lower() == "active"})
        sm = [r[0] for r in rows]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# -------------------------------------------------------------- workloads --

def make_workload(name, seed_offset=0, fill="device", num_seqs=None):
    import inspect
    from paged_kv_cache_86_gb300 import workloads as W
    fn = W.NAMED[name]
    params = inspect.signature(fn).parameters
    kw = {"seed": params["seed"].default + seed_offset, "fill": fill}
    if num_seqs is not None:
        if "num_seqs" not in params:
            raise SystemExit(f"--num-seqs is not supported for {name}")
        kw["num_seqs"] = num_seqs
    return fn(**kw)


def decode_step_launches(w) -> int:
    """Kernels one pkv_decode_step launches on the all-heads tcgen05 path: the
    attention kernel (which plans the call and writes the new tokens) and the
    combine."""
    return 2


def max_over_ranks(x, world, device):
    """The slowest rank's value (the job's time); a no-op on one rank."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, units_per_rank, ms):
    """Whole-job units per second: every rank processed units_per_rank in ms."""
    return world * units_per_rank / (ms * 1e-3)


def decode_bytes(w) -> int:
    """Algorithmic HBM bytes of one decode launch: K and V of every cached token
    once per KV head, q in, out, block-table entries and context lengths."""
    hkv, hq, d, bs = w.num_kv_heads, w.num_q_heads, w.head_dim, w.block_size
    ctx = w.context_lens.astype(np.int64)
    return int((ctx * hkv * d * 2 * 2).sum() + w.num_seqs * hq * d * 2 * 2
               + 4 * ((ctx + bs - 1) // bs).sum() + 4 * w.num_seqs)


def workload_config(w, world=1) -> dict:
    """The JSON line's config: the workload and its sizes (both arms print it)."""
    kv = int((w.context_lens.astype(np.int64) * w.num_kv_heads * w.head_dim * 4).sum())
    return {"workload": w.name, "num_seqs": w.num_seqs, "num_q_heads": w.num_q_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
            "block_size": w.block_size, "num_blocks": w.num_blocks,
            "total_context_tokens": int(w.context_lens.sum()),
            "kv_bytes_read_per_step": kv,
            "l2": "inputs larger than L2: every step streams the whole KV context "
                  f"({kv / 1e9:.2f} GB > 129 MB L2)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def store_bytes(w) -> int:
    """K and V rows read from the new-token buffers and written to the cache, plus slots."""
    return int(w.num_new_tokens * (2 * w.num_kv_heads * w.head_dim * 2 * 2 + 4))


def source_hash(paths):
    """Hash of the code of the given sources with comments and blank space
    stripped, so that editing a comment does not orphan a recorded profile."""
    m = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        m.update(" ".join(text.split()).encode())
    return m.hexdigest()[:16]


def profiled_traffic(name):
    """DRAM bytes (read + write) per decode call from the committed ncu launch
    list, if it was taken on the current kernel sources; otherwise None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(name)
    if not rec or rec.get("source_sha256_16") != source_hash(rec.get("sources", [])):
        return None
    return rec.get("dram_bytes_per_launch")


# ------------------------------------------------------------ cpu oracle --

def cpu_oracle_sample(w, target_s=15.0, max_seqs=None, threads=None):
    """Time the oracle (store of the new tokens + decode) on a bounded sample of
    the workload's sequences, on this host's cores (or on `threads` of them).
    Returns a cpu_baseline dict."""
    import torch
    from oracle import attention as oracle
    from paged_kv_cache_86_gb300.workloads import bf16_to_u16

    prev_threads = oracle.max_threads()
    if threads:
        oracle.set_threads(threads)
    cores = oracle.max_threads()
    order = np.random.default_rng(0).permutation(w.num_seqs)
    t = w.tensors
    done_tokens, done_seqs, elapsed = 0, 0, 0.0
    token_of_seq = np.cumsum(w.context_lens > 0) - 1
    bs = w.block_size
    batch = 8
    passes = 0
    while elapsed < target_s and (max_seqs is None or done_seqs < max_seqs):
        start = done_seqs % w.num_seqs
        if start == 0 and done_seqs:
            passes += 1
        ids = np.sort(order[start:start + batch])
        rows = w.block_tables[ids]
        nblk = [-(-int(w.context_lens[i]) // bs) for i in ids]
        used = np.unique(np.concatenate([rows[j, :n] for j, n in enumerate(nblk)]))
        remap = {int(b): k for k, b in enumerate(used)}
        tables = np.full_like(rows, -1)
        for j, n in enumerate(nblk):
            tables[j, :n] = [remap[int(b)] for b in rows[j, :n]]
        idx = torch.from_numpy(used.astype(np.int64)).to(t["k_cache"].device)
        kc = bf16_to_u16(t["k_cache"].index_select(0, idx)).copy()
        vc = bf16_to_u16(t["v_cache"].index_select(0, idx)).copy()
        toks = token_of_seq[ids]
        slots = np.array([remap[int(w.slot_mapping[k]) // bs] * bs + int(w.slot_mapping[k]) % bs
                          for k in toks], np.int32)
        key = bf16_to_u16(t["key"][torch.from_numpy(toks.astype(np.int64)).to(t["key"].device)])
        val = bf16_to_u16(t["value"][torch.from_numpy(toks.astype(np.int64)).to(t["value"].device)])
        q = bf16_to_u16(t["q"][torch.from_numpy(ids.astype(np.int64)).to(t["q"].device)])
        lens = w.context_lens[ids].copy()
        t0 = time.perf_counter()
        oracle.store_kvcache(key, val, kc, vc, slots, bs)
        oracle.paged_decode(q, kc, vc, tables, lens, w.scale)
        elapsed += time.perf_counter() - t0
        done_seqs += len(ids)
        done_tokens += int(lens.sum())
    if threads:
        oracle.set_threads(prev_threads)
    value = done_seqs / elapsed if elapsed > 0 else None
    return {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{done_seqs} sequences of the {w.num_seqs}-sequence batch in seeded random "
                      f"order, cycling ({done_tokens} cached tokens), store + decode in fp64 C "
                      f"with OpenMP on {cores} thread(s), {elapsed:.1f} s",
            "seconds": elapsed}


# --------------------------------------------------------------- GPU arm --

def run_pkv(args, rank, world, device):
    import torch
    import torch.distributed as dist
    import paged_kv_cache_86_gb300 as pkv
    from paged_kv_cache_86_gb300 import _lib

    torch.cuda.set_device(device)
    w = make_workload(args.workload, seed_offset=rank, fill="device", num_seqs=args.num_seqs)
    t = {k: v.to(device) for k, v in w.tensors.items()}
    bt = torch.from_numpy(w.block_tables).to(device)
    cl = torch.from_numpy(w.context_lens).to(device)
    sm = torch.from_numpy(w.slot_mapping).to(device)
    out = torch.empty_like(t["q"])
    ws = torch.empty(pkv.decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads),
                     dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    # the step's new K/V rows indexed by sequence (the workload keeps one row per
    # non-empty sequence, in order)
    if w.num_new_tokens == w.num_seqs:
        kn, vn = t["key"], t["value"]
    else:
        kn = torch.zeros((w.num_seqs,) + tuple(t["key"].shape[1:]), dtype=t["key"].dtype, device=device)
        vn = torch.zeros_like(kn)
        nz = torch.from_numpy(np.nonzero(w.context_lens > 0)[0]).to(device)
        kn[nz] = t["key"]
        vn[nz] = t["value"]

    def step():
        # one decode step: store of each sequence's new token + paged decode
        pkv.decode_step(t["q"], kn, vn, t["k_cache"], t["v_cache"], bt, cl, w.scale, out=out,
                        workspace=ws)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if pkv.get_device_errors() != 0:
        raise RuntimeError("device-side range check fired during warm-up")

    def barrier():
        if world > 1:
            dist.barrier()

    clocks = ClockSampler(device.index if device.index is not None else 0,
                          enabled=(rank == 0 and not args.no_clocks))
    with clocks:
        barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        step_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, device)
        if args.quick:
            return {"metric": METRIC, "value": job_throughput(world, w.num_seqs, step_ms), "unit": UNIT,
                    "n_gpus": world, "steps": args.steps, "ms_per_step": step_ms,
                    "config": {"workload": w.name, "num_seqs": w.num_seqs}, "quick": True}

        # per-call durations over the same number of steps, events on the launching
        # stream: the decode step call (the roofline's launch), then the two-call
        # path (store, paged decode) for the breakdown
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for a, b in evs:
            a.record(stream)
            step()
            b.record(stream)
        evs2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
                 torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for a, b, c in evs2:
            a.record(stream)
            pkv.store_kvcache(t["key"], t["value"], t["k_cache"], t["v_cache"], sm)
            b.record(stream)
            pkv.paged_decode(t["q"], t["k_cache"], t["v_cache"], bt, cl, w.scale, out=out,
                             workspace=ws)
            c.record(stream)
        torch.cuda.synchronize()
    call_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    store_ms = statistics.mean(a.elapsed_time(b) for a, b, _ in evs2)
    decode_ms = statistics.mean(b.elapsed_time(c) for _, b, c in evs2)
    if pkv.get_device_errors() != 0:
        raise RuntimeError("device-side range check fired during the timed region")


    # end to end through the public API with host buffers: every step copies its
    # inputs from pinned host memory (q, new K, new V, block tables, lengths as one
    # packed buffer at 256-byte aligned offsets), runs the decode step, and copies
    # its output back to pinned host memory. The copies run on two copy streams
    # with double-buffered device inputs and outputs, ordered by events, so step
    # k+1's upload and step k-1's download overlap step k's compute; every copy is
    # inside the timed region.
    e2e_ms, h2d, d2h = measure_e2e(w, t, kn, vn, bt, cl, ws, out, args.steps, device, barrier)
    e2e_ms = max_over_ranks(e2e_ms, world, device)

    peak, peak_kind = measured_peaks()
    dbytes = decode_bytes(w) + store_bytes(w)
    achieved = dbytes / (call_ms * 1e-3) / 1e9
    result = {
        "metric": METRIC, "value": job_throughput(world, w.num_seqs, step_ms), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16 values, lognormal context lengths)",
        "config": workload_config(w, world),
        "kv_gbs": achieved,
        "roofline": {"bound": "hbm",
                     "kernel": "pkv_decode_step (plan + new-token store, tcgen05 decode, combine)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs",
                     "traffic": profiled_traffic(w.name),
                     "algorithmic_bytes_per_launch": dbytes, "launch_ms": call_ms},
        "ops": {"decode_step_ms": call_ms, "store_ms": store_ms,
                "store_gbs": store_bytes(w) / (store_ms * 1e-3) / 1e9, "decode_ms": decode_ms,
                "decode_gbs": decode_bytes(w) / (decode_ms * 1e-3) / 1e9},
        "e2e": {"value": job_throughput(world, w.num_seqs, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms},
        "gpu_launches": args.steps * decode_step_launches(w),
        "clocks": clocks.summary(),
    }
    result["prefill_row"] = measure_prefill(args, device, steps=max(5, min(args.steps, 20)))
    result["gpu_launches_prefill_row"] = 2 * max(5, min(args.steps, 20))
    result["copy_blocks_row"] = measure_copy_blocks(device, steps=max(5, min(args.steps, 20)))
    result["fp8_decode_row"] = measure_fp8_decode(device, steps=max(5, min(args.steps, 20)))
    result["mixed_batch_row"] = measure_mixed(device, steps=max(5, min(args.steps, 20)))
    result["store_row"] = measure_store_sustained(device)
    result["decode_config_rows"] = [measure_decode_config(n, device, steps=max(5, min(args.steps, 20)))
                                    for n in ("decode_3seq", "decode_64seq", "decode_longtail")]
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_oracle_sample(w)
        one = cpu_oracle_sample(w, target_s=5.0, threads=1)   # the same oracle on one core
        result["cpu_baseline"]["single_thread"] = {k: one[k] for k in ("value", "unit", "cores", "sample")}
    return result


def measure_e2e(w, t, kn, vn, bt, cl, ws, out, steps, device, barrier=lambda: None):
    """Mean ms per decode step end to end through the public API with host
    buffers (see run_pkv), and the bytes copied in and out per step."""
    import torch
    import paged_kv_cache_86_gb300 as pkv
    parts = [("q", t["q"]), ("key", kn), ("value", vn), ("bt", bt), ("cl", cl)]
    offs, off = {}, 0
    for k, v in parts:
        offs[k] = off
        off += (v.numel() * v.element_size() + 255) // 256 * 256
    host_pack = torch.empty(off, dtype=torch.uint8).pin_memory()

    def view(buf, k, like):
        n = like.numel() * like.element_size()
        return buf[offs[k]:offs[k] + n].view(like.dtype).view(like.shape)

    for k, v in parts:
        view(host_pack, k, v).copy_(v.cpu())
    dev_packs = [torch.empty(off, dtype=torch.uint8, device=device) for _ in range(2)]
    devs = [{k: view(p, k, v) for k, v in parts} for p in dev_packs]
    outs = [out, torch.empty_like(out)]
    host_outs = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for _, v in parts)
    d2h = host_outs[0].numel() * host_outs[0].element_size()
    comp = torch.cuda.current_stream(device)
    up, down = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def ev():
        return torch.cuda.Event()

    def run(n, start=None, end=None):
        uploaded = [ev(), ev()]     # H2D of step k into pack k % 2 done
        computed = [ev(), ev()]     # step k (reads pack k % 2, writes outs[k % 2]) done
        downloaded = [ev(), ev()]   # D2H of outs[k % 2] done
        fresh = [True, True]
        if start is not None:
            start.record(up)
        with torch.cuda.stream(up):
            dev_packs[0].copy_(host_pack, non_blocking=True)
            uploaded[0].record(up)
        for k in range(n):
            b = k % 2
            if k + 1 < n:           # upload step k+1 while step k computes
                nb = (k + 1) % 2
                if k >= 1:          # pack nb was read by step k-1
                    up.wait_event(computed[nb])
                with torch.cuda.stream(up):
                    dev_packs[nb].copy_(host_pack, non_blocking=True)
                    uploaded[nb].record(up)
            comp.wait_event(uploaded[b])
            if not fresh[b]:        # outs[b] is still being downloaded (step k-2)
                comp.wait_event(downloaded[b])
            d = devs[b]
            pkv.decode_step(d["q"], d["key"], d["value"], t["k_cache"], t["v_cache"], d["bt"],
                            d["cl"], w.scale, out=outs[b], workspace=ws)
            computed[b].record(comp)
            fresh[b] = False
            down.wait_event(computed[b])
            with torch.cuda.stream(down):
                host_outs[b].copy_(outs[b], non_blocking=True)
                downloaded[b].record(down)
        comp.wait_stream(up)
        comp.wait_stream(down)
        if end is not None:
            end.record(comp)

    run(3)
    torch.cuda.synchronize()
    barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    run(steps, a, b)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps, h2d, d2h


def decode_kernel_path(w) -> str:
    """Which attention kernel the library's dispatch picks for this shape (its
    documented rule: all-heads tcgen05 kernel when Hkv is a power of two >= 4 and
    128 / Hkv tokens divide the block size; per-head tcgen05 kernel when the block
    size is a multiple of 8; CUDA-core split kernel otherwise)."""
    hkv, bs = w.num_kv_heads, w.block_size
    if hkv >= 4 and hkv & (hkv - 1) == 0 and bs % (128 // hkv) == 0:
        return "decode_tcg_kernel (tcgen05, all KV heads per stage)"
    if bs % 8 == 0:
        return "decode_tc_kernel (tcgen05, one KV head per CTA)"
    return "decode_split_kernel (CUDA cores)"


def measure_decode_config(name, device, steps):
    """A decode-step row for another decode workload: pkv_decode_step (the new
    token of every sequence stored, then paged decode) timed with CUDA events.
    Workloads whose K/V exceed L2 run back to back (every step streams more than
    L2); smaller ones are timed launch by launch after a clean L2 refill."""
    import torch
    import paged_kv_cache_86_gb300 as pkv
    w = make_workload(name, fill="device")
    t = {k: v.to(device) for k, v in w.tensors.items()}
    bt = torch.from_numpy(w.block_tables).to(device)
    cl = torch.from_numpy(w.context_lens).to(device)
    assert (w.context_lens > 0).all() and w.num_new_tokens == w.num_seqs
    out = torch.empty_like(t["q"])
    ws = torch.empty(pkv.decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads),
                     dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def step():
        pkv.decode_step(t["q"], t["key"], t["value"], t["k_cache"], t["v_cache"], bt, cl, w.scale,
                        out=out, workspace=ws)

    for _ in range(5):
        step()
    torch.cuda.synchronize()
    nbytes = decode_bytes(w) + store_bytes(w)
    kv = int((w.context_lens.astype(np.int64) * w.num_kv_heads * w.head_dim * 4).sum())
    if kv > (256 << 20):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            step()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / steps
        how = f"back to back, mean of {steps} steps; {kv / 1e9:.2f} GB of K/V per step > L2"
    else:
        ms = timed_after_clean_flush(step, steps, device)
        how = (f"{kv / 1e6:.1f} MB of K/V fits in L2: each step after a clean 256 MiB L2 "
               f"refill, median of {steps}")
    if pkv.get_device_errors() != 0:
        raise RuntimeError(f"device-side range check fired in the {name} measurement")
    hpeak, kind = measured_peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": w.name, "num_seqs": w.num_seqs, "num_q_heads": w.num_q_heads,
            "num_kv_heads": w.num_kv_heads, "block_size": w.block_size,
            "total_context_tokens": int(w.context_lens.sum()),
            "kernel": decode_kernel_path(w), "ms": ms,
            "tokens_per_s": w.num_seqs / (ms * 1e-3),
            "algorithmic_bytes_per_launch": nbytes, "gbs": gbs, "frac_of_hbm": gbs / hpeak,
            "peak_source": f"{kind} hbm_gbs", "timing": how}


def measure_store_sustained(device, copies=16, reps=5):
    """The store row in the regime where its writes must reach HBM: `copies`
    disjoint repetitions of the chunked-prefill store (16384 tokens at the
    workload's slots, each copy in its own region of one large pool, each with
    its own input rows) launched back to back. Per-launch time is the slope
    between a run of copies/4 launches and a run of all copies (each run after
    a clean L2 refill), so the dirty lines a run leaves in L2 at its end event
    cancel out; the mean over the long run is reported beside it."""
    import torch
    import paged_kv_cache_86_gb300 as pkv
    w = make_workload("prefill_chunks", fill="none")
    hkv, d, bs = w.num_kv_heads, w.head_dim, w.block_size
    slots_per_copy = w.num_blocks * bs
    nb = w.num_blocks * copies
    kc = torch.empty((nb, bs, hkv, d), dtype=torch.bfloat16, device=device)
    vc = torch.empty_like(kc)
    base = torch.from_numpy(w.slot_mapping.astype(np.int64)).to(device)
    sms = [(base + j * slots_per_copy).to(torch.int32) for j in range(copies)]
    g = torch.Generator(device=device).manual_seed(86021)
    keys = torch.empty((copies, w.num_new_tokens, hkv, d), dtype=torch.bfloat16,
                       device=device).normal_(generator=g)
    vals = torch.empty_like(keys).normal_(generator=g)
    stream = torch.cuda.current_stream(device)

    def run(n):
        for j in range(n):
            pkv.store_kvcache(keys[j], vals[j], kc, vc, sms[j])

    run(copies)
    torch.cuda.synchronize()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    flush_rd = torch.ones(64 << 20, dtype=torch.float32, device=device)
    short = max(1, copies // 4)
    times = {short: [], copies: []}
    for _ in range(reps):
        for n in (short, copies):
            flush.zero_()
            flush_rd.sum()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            run(n)
            b.record(stream)
            torch.cuda.synchronize()
            times[n].append(a.elapsed_time(b))
    if pkv.get_device_errors() != 0:
        raise RuntimeError("device-side range check fired in the store measurement")
    t_short, t_long = statistics.median(times[short]), statistics.median(times[copies])
    slope = (t_long - t_short) / (copies - short)
    sb = store_bytes(w)
    hpeak, kind = measured_peaks()
    return {"workload": f"{copies} x store of {w.num_new_tokens} chunk tokens "
                        f"({w.name} slots) into disjoint pool regions",
            "algorithmic_bytes_per_launch": sb,
            "ms_per_launch": slope, "gbs": sb / (slope * 1e-3) / 1e9,
            "frac_of_hbm": sb / (slope * 1e-3) / 1e9 / hpeak,
            "ms_per_launch_mean_of_long_run": t_long / copies,
            "frac_of_hbm_mean_of_long_run": sb / (t_long / copies * 1e-3) / 1e9 / hpeak,
            "peak_source": f"{kind} hbm_gbs",
            "timing": f"slope between {short} and {copies} back-to-back launches, medians of "
                      f"{reps} runs, each run after a clean 256 MiB L2 refill; "
                      f"{copies * sb / 2e9:.2f} GB written per long run (> L2)"}


def fp8_decode_bytes(w) -> int:
    """Algorithmic HBM bytes of one fp8 decode launch: one-byte K and V codes of
    every cached token once per KV head plus their fp32 row scales, q in, out,
    block-table entries and context lengths."""
    ctx = w.context_lens.astype(np.int64)
    kv = int((ctx * w.num_kv_heads * (w.head_dim + 4) * 2).sum())
    qo = 2 * w.num_seqs * w.num_q_heads * w.head_dim * 2
    tables = int((4 * ((ctx + w.block_size - 1) // w.block_size)).sum()) + 4 * w.num_seqs
    return kv + qo + tables


def measure_fp8_decode(device, steps, num_seqs=None):
    """The fp8 KV row: the 512-sequence decode batch over an fp8 E4M3 cache
    (per token-head scales): the quantizing store of the 512 new tokens, then
    pkv_paged_decode_fp8, each timed with CUDA events; and the same step as one
    pkv_decode_step_fp8 call."""
    import torch
    import paged_kv_cache_86_gb300 as pkv
    from paged_kv_cache_86_gb300 import workloads as W
    w = make_workload("decode_512seq", fill="device", num_seqs=num_seqs)
    t = {k: v.to(device) for k, v in w.tensors.items() if k in ("q", "key", "value")}
    kc, ks = W.fp8_pool(w.num_blocks, w.block_size, w.num_kv_heads, w.seed * 16 + 7, device=device)
    vc, vs = W.fp8_pool(w.num_blocks, w.block_size, w.num_kv_heads, w.seed * 16 + 8, device=device)
    bt = torch.from_numpy(w.block_tables).to(device)
    cl = torch.from_numpy(w.context_lens).to(device)
    sm = torch.from_numpy(w.slot_mapping).to(device)
    out = torch.empty_like(t["q"])
    ws = torch.empty(pkv.decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads),
                     dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def store():
        pkv.store_kvcache_fp8(t["key"], t["value"], kc, vc, ks, vs, sm)

    def decode():
        pkv.paged_decode_fp8(t["q"], kc, vc, ks, vs, bt, cl, w.scale, out=out, workspace=ws)

    for _ in range(3):
        store()
        decode()
    torch.cuda.synchronize()
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps)]
    for a, b, c in evs:
        a.record(stream)
        store()
        b.record(stream)
        decode()
        c.record(stream)
    torch.cuda.synchronize()
    if pkv.get_device_errors() != 0:
        raise RuntimeError("device-side range check fired in the fp8 measurement")
    store_ms = statistics.mean(a.elapsed_time(b) for a, b, _ in evs)
    decode_ms = statistics.mean(b.elapsed_time(c) for _, b, c in evs)
    # the same step as one call: every sequence of the batch is non-empty, so
    # new-token row i is sequence i's
    assert (w.context_lens > 0).all()

    def fused():
        pkv.decode_step_fp8(t["q"], t["key"], t["value"], kc, vc, ks, vs, bt, cl, w.scale,
                            out=out, workspace=ws)

    for _ in range(3):
        fused()
    torch.cuda.synchronize()
    fevs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(2)) for _ in range(steps)]
    for a, b in fevs:
        a.record(stream)
        fused()
        b.record(stream)
    torch.cuda.synchronize()
    if pkv.get_device_errors() != 0:
        raise RuntimeError("device-side range check fired in the fp8 step measurement")
    fused_ms = statistics.mean(a.elapsed_time(b) for a, b in fevs)
    hpeak, _ = measured_peaks()
    nbytes = fp8_decode_bytes(w)
    step_ms = store_ms + decode_ms
    return {"workload": w.name + "_fp8_e4m3", "decode_ms": decode_ms, "store_ms": store_ms,
            "fused_step_ms": fused_ms,
            "fused_step_tokens_per_s": w.num_seqs / (fused_ms * 1e-3),
            "tokens_per_s": w.num_seqs / (step_ms * 1e-3),
            "algorithmic_bytes_per_launch": nbytes,
            "gbs": nbytes / (decode_ms * 1e-3) / 1e9,
            "frac_of_hbm": nbytes / (decode_ms * 1e-3) / 1e9 / hpeak,
            "l2": f"inputs larger than L2 ({nbytes / 1e9:.2f} GB of codes and scales per launch)"}


def measure_mixed(device, steps):
    """The mixed-batch row: one round of 256 decode requests (lengths as the
    512-sequence batch's distribution) and 8 prefill chunks of 512 after prefixes
    U[0, 3584] -- 4352 scheduled tokens -- through pkv_mixed_step, and the same
    round through pkv_store_kvcache + pkv_paged_prefill over every sequence."""
    import torch
    import paged_kv_cache_86_gb300 as pkv
    from paged_kv_cache_86_gb300 import workloads as W
    rng = np.random.default_rng(86011)
    dec = np.clip(np.rint(np.exp(np.log(800) + rng.standard_normal(256))), 16, 4096).astype(int)
    prefixes = rng.integers(0, 3585, 8)
    q_lens = [1] * len(dec) + [512] * 8
    w = W.prefill_workload("mixed_256decode_8x512chunks_bs16", q_lens,
                           [int(n) - 1 for n in dec] + [int(x) for x in prefixes], 32, 8, 16,
                           seed=86011, fill="device", device=device)
    t = {k: v.to(device) for k, v in w.tensors.items()}
    bt = torch.from_numpy(w.block_tables).to(device)
    sm = torch.from_numpy(w.slot_mapping).to(device)
    cq = torch.from_numpy(w.cu_seqlens_q).to(device)
    ck = torch.from_numpy(w.cu_seqlens_k).to(device)
    out = torch.empty_like(t["q"])
    d = len(dec)
    mq, mk = int(w.q_lens.max()), int(w.context_lens.max())
    ws = torch.empty(max(pkv.mixed_workspace_size(d, 32, 8), 256), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def mixed():
        pkv.mixed_step(t["q"], t["key"], t["value"], sm, t["k_cache"], t["v_cache"], cq, ck, bt, d,
                       w.scale, mq, mk, out=out, workspace=ws)

    def prefill_all():
        pkv.store_kvcache(t["key"], t["value"], t["k_cache"], t["v_cache"], sm)
        pkv.paged_prefill(t["q"], t["k_cache"], t["v_cache"], cq, ck, bt, w.scale, mq, mk, out=out)

    res = {}
    for name, fn in (("mixed_step", mixed), ("store_plus_prefill_kernel_for_all", prefill_all)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        res[name] = timed_after_clean_flush(fn, steps, device)
    if pkv.get_device_errors() != 0:
        raise RuntimeError("device-side range check fired in the mixed-batch measurement")
    tokens = int(w.num_q_rows)
    # the round's floors: decode rows are HBM-bound (K/V once per KV head, q,
    # out, tables), chunk rows tensor-bound (causal-region FLOPs), and every new
    # token is stored (its K/V rows read and written)
    hkv, hq, dd, bs = w.num_kv_heads, w.num_q_heads, w.head_dim, w.block_size
    ctx = w.context_lens[:d].astype(np.int64)
    dec_bytes = int((ctx * hkv * dd * 4).sum() + d * hq * dd * 4
                    + (4 * ((ctx + bs - 1) // bs)).sum() + 4 * d)
    q_lens, k_lens = w.q_lens[d:].astype(np.int64), w.context_lens[d:].astype(np.int64)
    chunk_flops = sum(4 * dd * hq * int(((k - q) + np.arange(1, q + 1)).sum())
                      for q, k in zip(q_lens, k_lens))
    chunk_bytes = int((k_lens * hkv * dd * 4).sum() + q_lens.sum() * hq * dd * 4)
    st_bytes = store_bytes(w)
    hpeak, _ = measured_peaks()
    tpeak = measured_bf16_peak()
    hbm_ms = (dec_bytes + st_bytes) / (hpeak * 1e9) * 1e3
    tensor_ms = chunk_flops / (tpeak * 1e12) * 1e3
    floor_serial = hbm_ms + tensor_ms
    floor_overlap = max((dec_bytes + st_bytes + chunk_bytes) / (hpeak * 1e9) * 1e3, tensor_ms)
    ms = res["mixed_step"]
    return {"workload": w.name, "scheduled_tokens": tokens, "ms": ms,
            "tokens_per_s": tokens / (ms * 1e-3),
            "ms_all_through_prefill_kernel": res["store_plus_prefill_kernel_for_all"],
            "roofline": {"decode_bytes": dec_bytes, "store_bytes": st_bytes,
                         "chunk_flops": chunk_flops, "chunk_kv_q_out_bytes": chunk_bytes,
                         "floor_ms_serial": floor_serial, "frac_serial": floor_serial / ms,
                         "floor_ms_overlapped": floor_overlap,
                         "frac_overlapped": floor_overlap / ms,
                         "how": "serial floor: decode rows' and stores' bytes at the measured HBM "
                                "peak, then the chunks' causal FLOPs at the measured bf16 burst "
                                "peak; overlapped floor: the larger of all bytes at the HBM peak "
                                "and the FLOPs at the bf16 peak"},
            "l2": "K/V of the round larger than L2 (~1 GB); each launch after a clean 256 MiB "
                  "L2 refill; median of launches"}


def measure_copy_blocks(device, steps, launches=8):
    """The copy-on-write row: 4096 whole-block copies (random distinct source and
    destination blocks of a 16-token, 8-KV-head pool), K and V: 512 MiB moved per
    launch. Timed two ways: one launch after a clean L2 refill (median of
    `steps`), and per launch as the slope between 2 and `launches` back-to-back
    launches over disjoint block pairs, where every launch's writes must reach
    HBM (the dirty lines left in L2 at a run's end event cancel out)."""
    import torch
    import paged_kv_cache_86_gb300 as pkv
    bs, hkv, d, pairs = 16, 8, 128, 4096
    nb = 2 * pairs * launches
    g = torch.Generator(device=device).manual_seed(86009)
    kc = torch.empty((nb, bs, hkv, d), dtype=torch.bfloat16, device=device).normal_(generator=g)
    vc = torch.empty_like(kc).normal_(generator=g)
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(86010)).to(torch.int32)
    srcs = [perm[2 * j * pairs:(2 * j + 1) * pairs].to(device) for j in range(launches)]
    dsts = [perm[(2 * j + 1) * pairs:(2 * j + 2) * pairs].to(device) for j in range(launches)]
    for j in range(launches):
        pkv.copy_blocks(kc, vc, srcs[j], dsts[j])
    torch.cuda.synchronize()
    ms = timed_after_clean_flush(lambda: pkv.copy_blocks(kc, vc, srcs[0], dsts[0]), steps, device)
    stream = torch.cuda.current_stream(device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    flush_rd = torch.ones(64 << 20, dtype=torch.float32, device=device)
    runs = {2: [], launches: []}
    for _ in range(5):
        for n in runs:
            flush.zero_()
            flush_rd.sum()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for j in range(n):
                pkv.copy_blocks(kc, vc, srcs[j], dsts[j])
            b.record(stream)
            torch.cuda.synchronize()
            runs[n].append(a.elapsed_time(b))
    if pkv.get_device_errors() != 0:
        raise RuntimeError("device-side range check fired in the block-copy measurement")
    slope = (statistics.median(runs[launches]) - statistics.median(runs[2])) / (launches - 2)
    nbytes = pairs * 2 * 2 * bs * hkv * d * 2      # K and V, read and write
    hpeak, _ = measured_peaks()
    return {"workload": f"copy_{pairs}_blocks_bs{bs}_hkv{hkv}", "bytes_per_launch": nbytes,
            "ms_per_launch": slope, "gbs": nbytes / (slope * 1e-3) / 1e9,
            "frac_of_hbm": nbytes / (slope * 1e-3) / 1e9 / hpeak,
            "timing": f"slope between 2 and {launches} back-to-back launches over disjoint block "
                      "pairs, medians of 5 runs, each run after a clean 256 MiB L2 refill",
            "ms_single_launch_after_clean_l2": ms,
            "frac_of_hbm_single_launch": nbytes / (ms * 1e-3) / 1e9 / hpeak}


def prefill_flops(w) -> int:
    """Causal-region FLOPs of one prefill launch: 2 contractions x 2 flops per
    multiply-add x D x Hq x (keys each query row sees)."""
    q_lens = np.diff(w.cu_seqlens_q).astype(np.int64)
    k_lens = np.diff(w.cu_seqlens_k).astype(np.int64)
    vis = sum(int(((k - q) + np.arange(1, q + 1)).sum()) for q, k in zip(q_lens, k_lens))
    return 4 * w.head_dim * w.num_q_heads * vis


def timed_after_clean_flush(fn, steps, device):
    """Median CUDA-event time of fn() over `steps` launches, each started right
    after L2 has been refilled with clean, unrelated lines (256 MiB written, then
    256 MiB read). The flush also keeps the GPU busy while the host submits fn(),
    so the events time the GPU work, not the host-side launch latency."""
    import torch
    stream = torch.cuda.current_stream(device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    flush_rd = torch.ones(64 << 20, dtype=torch.float32, device=device)
    times = []
    for _ in range(steps):
        flush.zero_()
        flush_rd.sum()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    return statistics.median(times)


def measure_small_blocks(device, steps):
    """Block sizes below a stage or tile (token-level paging among them): the
    512-sequence decode (lognormal lengths, Hq 32 / Hkv 8; bf16 and fp8 E4M3) at
    block sizes 16, 8 and 1, and with Hq 8 / Hkv 2 at 16; the 32 x 512 chunked
    prefill over the same prefixes as the prefill row at 16, 8, 4 and 1; each
    call timed with CUDA events after a clean L2 refill. Not part of the
    default run."""
    import torch
    import paged_kv_cache_86_gb300 as pkv
    from paged_kv_cache_86_gb300 import workloads as W
    res = {}
    lens = W.lognormal_lengths(np.random.default_rng(86003 + 1000), 512)
    for bs in (16, 8, 1):
        w = W.decode_workload(f"decode_512seq_bs{bs}", lens, 32, 8, bs, 86003, pool="fragmented",
                              fill="device", device=device)
        t = {k: v.to(device) for k, v in w.tensors.items() if k in ("q", "k_cache", "v_cache")}
        bt = torch.from_numpy(w.block_tables).to(device)
        cl = torch.from_numpy(w.context_lens).to(device)
        res[f"decode_512seq_bs{bs}_ms"] = timed_after_clean_flush(
            lambda: pkv.paged_decode(t["q"], t["k_cache"], t["v_cache"], bt, cl, w.scale), steps, device)
        del t
        kc, ks = W.fp8_pool(w.num_blocks, w.block_size, w.num_kv_heads, 7, device=device)
        vc, vs = W.fp8_pool(w.num_blocks, w.block_size, w.num_kv_heads, 8, device=device)
        q = torch.randn(w.num_seqs, 32, 128, device=device).to(torch.bfloat16)
        res[f"fp8_decode_512seq_bs{bs}_ms"] = timed_after_clean_flush(
            lambda: pkv.paged_decode_fp8(q, kc, vc, ks, vs, bt, cl, w.scale), steps, device)
        del kc, vc, ks, vs
    # two KV heads (Hq 8): the fp8 decode runs on the CUDA-core kernel at every
    # block size, the bf16 one on the per-head tcgen05 kernel at 16
    w = W.decode_workload("decode_512seq_hkv2_bs16", lens, 8, 2, 16, 86003, pool="fragmented",
                          fill="device", device=device)
    t = {k: v.to(device) for k, v in w.tensors.items() if k in ("q", "k_cache", "v_cache")}
    bt = torch.from_numpy(w.block_tables).to(device)
    cl = torch.from_numpy(w.context_lens).to(device)
    res["decode_512seq_hkv2_bs16_ms"] = timed_after_clean_flush(
        lambda: pkv.paged_decode(t["q"], t["k_cache"], t["v_cache"], bt, cl, w.scale), steps, device)
    del t
    kc, ks = W.fp8_pool(w.num_blocks, w.block_size, w.num_kv_heads, 7, device=device)
    vc, vs = W.fp8_pool(w.num_blocks, w.block_size, w.num_kv_heads, 8, device=device)
    q = torch.randn(w.num_seqs, 8, 128, device=device).to(torch.bfloat16)
    res["fp8_decode_512seq_hkv2_bs16_ms"] = timed_after_clean_flush(
        lambda: pkv.paged_decode_fp8(q, kc, vc, ks, vs, bt, cl, w.scale), steps, device)
    del kc, vc, ks, vs
    prefixes = np.random.default_rng(86005 + 1000).integers(0, 3584 + 1, size=32)
    for bs in (16, 8, 4, 1):
        w = W.prefill_workload(f"prefill_32x512_bs{bs}", [512] * 32, prefixes, 32, 8, bs, 86005,
                               fill="device", device=device)
        t = {k: v.to(device) for k, v in w.tensors.items() if k in ("q", "k_cache", "v_cache")}
        cq = torch.from_numpy(w.cu_seqlens_q).to(device)
        ck = torch.from_numpy(w.cu_seqlens_k).to(device)
        bt = torch.from_numpy(w.block_tables).to(device)
        res[f"prefill_32x512_bs{bs}_ms"] = timed_after_clean_flush(
            lambda: pkv.paged_prefill(t["q"], t["k_cache"], t["v_cache"], cq, ck, bt, w.scale,
                                      max_seqlen_q=512, max_seqlen_k=int(w.context_lens.max())),
            steps, device)
        del t
    res["kernels"] = ("decode: all-heads tcgen05 at 16, CUDA-core with stages over several blocks "
                      "below; two KV heads: per-head tcgen05 (bf16) and CUDA-core (fp8) at 16; "
                      "prefill: TMA boxes at 16 and 8, rows gathered with cp.async below 8")
    return res


def measure_prefill(args, device, steps):
    """The chunked-prefill row: store of 16384 chunk tokens, then causal paged
    prefill of 32 chunks of 512 over cached prefixes, each timed with CUDA events."""
    import torch
    import paged_kv_cache_86_gb300 as pkv
    w = make_workload("prefill_chunks", fill="device")
    t = {k: v.to(device) for k, v in w.tensors.items()}
    bt = torch.from_numpy(w.block_tables).to(device)
    sm = torch.from_numpy(w.slot_mapping).to(device)
    cq = torch.from_numpy(w.cu_seqlens_q).to(device)
    ck = torch.from_numpy(w.cu_seqlens_k).to(device)
    out = torch.empty_like(t["q"])
    mq, mk = int(w.q_lens.max()), int(w.context_lens.max())
    stream = torch.cuda.current_stream(device)

    def store():
        pkv.store_kvcache(t["key"], t["value"], t["k_cache"], t["v_cache"], sm)

    def prefill():
        pkv.paged_prefill(t["q"], t["k_cache"], t["v_cache"], cq, ck, bt, w.scale, mq, mk, out=out)

    for _ in range(3):
        store()
        prefill()
    torch.cuda.synchronize()
    # L2 (129 MB) is flushed before every timed launch by writing 256 MiB and
    # then reading 256 MiB, so the launch starts with clean, unrelated lines: a
    # write-only flush leaves ~129 MB of dirty lines whose write-back would be
    # charged to the next kernel. The store is also timed after the write-only
    # flush and reported beside it.
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    flush_rd = torch.ones(64 << 20, dtype=torch.float32, device=device)
    res = {}
    for name, fn, clean in (("store", store, True), ("prefill", prefill, True),
                            ("store_dirty_l2", store, False)):
        times = []
        for _ in range(steps):
            flush.zero_()
            if clean:
                flush_rd.sum()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        res[name] = statistics.median(times)
    if pkv.get_device_errors() != 0:
        raise RuntimeError("device-side range check fired in the prefill measurement")
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    tpeak = float(peaks.get("bf16_tflops", 1900.0))
    hpeak, _ = measured_peaks()
    fl = prefill_flops(w)
    sb = store_bytes(w)
    return {"workload": w.name,
            "l2": "256 MiB written then 256 MiB read before each launch (clean L2); median of launches",
            "store_note": "one 16384-token store launch: its 67 MB of writes fit in L2, so a "
                          "clean-L2 launch can end before they reach HBM; store_row gives the "
                          "sustained figure",
            "store_ms_single_launch_clean_l2": res["store"],
            "store_frac_of_hbm_single_launch_clean_l2": sb / (res["store"] * 1e-3) / 1e9 / hpeak,
            "store_ms_after_write_only_flush": res["store_dirty_l2"],
            "store_frac_of_hbm_after_write_only_flush": sb / (res["store_dirty_l2"] * 1e-3) / 1e9 / hpeak,
            "prefill_ms": res["prefill"], "prefill_tflops": fl / (res["prefill"] * 1e-3) / 1e12,
            "prefill_frac_of_bf16": fl / (res["prefill"] * 1e-3) / 1e12 / tpeak,
            "prefill_flops": fl, "peak_bf16_tflops": tpeak, "peak_source": "measured bf16_tflops (burst)"}


def run_reference(args, rank):
    """The oracle, as it stands, on the host cores: the reference arm."""
    if rank != 0:
        return None
    import torch
    w = make_workload(args.workload, fill="device" if torch.cuda.is_available() else "host")
    per_step = []
    for _ in range(max(args.warmup, 0)):
        cpu_oracle_sample(w, target_s=0.5, max_seqs=8)
    samples = []
    for _ in range(args.steps):
        r = cpu_oracle_sample(w, target_s=max(1.0, 60.0 / max(args.steps, 1)), max_seqs=None)
        samples.append(r)
        per_step.append(r["value"])
    value = statistics.mean(per_step)
    secs = sum(r["seconds"] for r in samples)
    cpu = {"value": value, "unit": UNIT, "cores": samples[0]["cores"], "kind": "oracle",
           "sample": samples[0]["sample"] + f"; {len(samples)} steps, {secs:.1f} s total"}
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * w.num_seqs / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) bf16 values, lognormal context lengths)",
            "config": workload_config(w),
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    device = torch.device("cuda", local)
    from paged_kv_cache_86_gb300.build import build
    if rank == 0:
        build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    if args.only_prefill:
        torch.cuda.set_device(device)
        res = {"prefill_row": measure_prefill(args, device, steps=max(1, args.steps))}
    elif args.only_row is not None:
        torch.cuda.set_device(device)
        steps = max(1, args.steps)
        if args.only_row == "fp8":
            res = {"fp8_decode_row": measure_fp8_decode(device, steps, num_seqs=args.num_seqs)}
        elif args.only_row == "copy":
            res = {"copy_blocks_row": measure_copy_blocks(device, steps)}
        elif args.only_row == "store":
            res = {"store_row": measure_store_sustained(device, copies=args.store_copies)}
        elif args.only_row == "small_blocks":
            res = {"small_blocks_row": measure_small_blocks(device, steps)}
        elif args.only_row.startswith("decode_"):
            res = {"decode_config_row": measure_decode_config(args.only_row, device, steps)}
        else:
            res = {"mixed_batch_row": measure_mixed(device, steps)}
    else:
        res = run_pkv(args, rank, world, device)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
