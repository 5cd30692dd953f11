"""Prefix sharing and copy-on-write on the GPU: pkv_copy_blocks against a plain
index copy, and decode over blocks shared through the host block manager
against the same sequences laid out in private blocks (bit for bit) and
against the oracle."""
import hashlib

import numpy as np
import pytest
import torch

import paged_kv_cache_86_gb300 as pkv
from oracle import attention as oracle
from paged_kv_cache_86_gb300.block_manager import BlockManager, Sequence
from paged_kv_cache_86_gb300.workloads import bf16_to_u16

pytestmark = pytest.mark.gpu

HKV, G, D, BS = 8, 4, 128, 16


def test_copy_blocks_matches_an_index_copy():
    nb, bs = 40, 16
    g = torch.Generator(device="cuda").manual_seed(1)
    kc = torch.randn((nb, bs, HKV, D), generator=g, device="cuda").to(torch.bfloat16)
    vc = torch.randn((nb, bs, HKV, D), generator=g, device="cuda").to(torch.bfloat16)
    src = [3, 7, 0, 39, 12]
    dst = [20, 21, 30, 1, 5]
    rows = [16, 5, 0, 1, 15]
    for use_rows in (False, True):
        k2, v2 = kc.clone(), vc.clone()
        exp_k, exp_v = kc.clone(), vc.clone()
        for s, d, r in zip(src, dst, rows if use_rows else [bs] * len(src)):
            exp_k[d, :r] = kc[s, :r]
            exp_v[d, :r] = vc[s, :r]
        pkv.copy_blocks(k2, v2, torch.tensor(src, dtype=torch.int32, device="cuda"),
                        torch.tensor(dst, dtype=torch.int32, device="cuda"),
                        torch.tensor(rows, dtype=torch.int32, device="cuda") if use_rows else None)
        torch.cuda.synchronize()
        assert pkv.get_device_errors() == 0
        assert torch.equal(k2, exp_k) and torch.equal(v2, exp_v)


def test_copy_blocks_skips_bad_ids_and_reports_them():
    nb, bs = 8, 16
    kc = torch.zeros((nb, bs, HKV, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.ones_like(kc)
    k2, v2 = kc.clone(), vc.clone()
    pkv.copy_blocks(k2, v2, torch.tensor([1, 9], dtype=torch.int32, device="cuda"),
                    torch.tensor([-1, 2], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert pkv.get_device_errors() & pkv._lib.DEVERR_BLOCK_ID
    assert torch.equal(k2, kc) and torch.equal(v2, vc)


def kv_of_prefix(tokens):
    """K and V rows [Hkv, D] of the last token of a prefix: a deterministic draw
    seeded by the whole prefix (as a model's K/V depend only on the prefix)."""
    h = hashlib.blake2b(np.asarray(tokens, np.int64).tobytes(), digest_size=8).digest()
    rng = np.random.default_rng(int.from_bytes(h, "little"))
    k = torch.from_numpy(rng.standard_normal((HKV, D), dtype=np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((HKV, D), dtype=np.float32)).to(torch.bfloat16)
    return k, v


def write_positions(kc, vc, positions_by_seq):
    """Store the K/V of (sequence tokens, position, slot) triples through pkv_store_kvcache."""
    keys, vals, slots = [], [], []
    for toks, pos, slot in positions_by_seq:
        k, v = kv_of_prefix(toks[:pos + 1])
        keys.append(k)
        vals.append(v)
        slots.append(slot)
    if not slots:
        return
    pkv.store_kvcache(torch.stack(keys).cuda(), torch.stack(vals).cuda(), kc, vc,
                      torch.tensor(slots, dtype=torch.int32, device="cuda"))


class Private:
    """Each sequence in its own fresh blocks (no sharing)."""

    def __init__(self, num_blocks):
        self.next = 0
        self.tables = {}
        self.num_blocks = num_blocks

    def table(self, sid, n_tokens):
        t = self.tables.setdefault(sid, [])
        while len(t) * BS < n_tokens:
            t.append(self.next)
            self.next += 1
        assert self.next <= self.num_blocks
        return t


def decode(kc, vc, q, tables, lens):
    width = max(len(t) for t in tables)
    bt = torch.tensor([t + [-1] * (width - len(t)) for t in tables], dtype=torch.int32, device="cuda")
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = pkv.paged_decode(q, kc, vc, bt, cl, 1.0 / np.sqrt(D))
    torch.cuda.synchronize()
    assert pkv.get_device_errors() == 0
    return out, bt.cpu().numpy(), np.asarray(lens, np.int32)


def test_shared_prefix_and_copy_on_write_match_private_blocks():
    rng = np.random.default_rng(86)
    p1 = rng.integers(0, 1000, 40).tolist()
    p2 = rng.integers(0, 1000, 70).tolist()
    prompts = {"s1": p1 + [1, 2, 3, 4, 5], "s2": p1 + rng.integers(0, 1000, 20).tolist(),
               "s3": p2 + [7, 8, 9], "s4": p1[:32] + rng.integers(0, 1000, 10).tolist(), "s5": list(p2)}
    nb = 256
    shp = (nb, BS, HKV, D)
    kc_s = torch.zeros(shp, dtype=torch.bfloat16, device="cuda")
    vc_s = torch.zeros_like(kc_s)
    kc_p, vc_p = torch.zeros_like(kc_s), torch.zeros_like(kc_s)
    m = BlockManager(nb, BS)
    priv = Private(nb)

    # prefill: the shared layout writes only what its cache lacks
    for sid, toks in prompts.items():
        s = m.allocate(Sequence(sid, toks, BS))
        write_positions(kc_s, vc_s, [(toks, p, s.slot(p)) for p in range(s.num_cached_tokens, len(toks))])
        t = priv.table(sid, len(toks))
        write_positions(kc_p, vc_p, [(toks, p, t[p // BS] * BS + p % BS) for p in range(len(toks))])
    assert m.seqs["s2"].num_cached_tokens == 32 and m.seqs["s4"].num_cached_tokens == 32
    assert m.seqs["s5"].num_cached_tokens == 64
    assert m.seqs["s1"].block_table[:2] == m.seqs["s2"].block_table[:2]

    # a branch of s1 (parallel sampling), then three decode steps on both branches
    m.fork("s1", "s1b")
    priv.tables["s1b"] = []
    write_positions(kc_p, vc_p, [(prompts["s1"], p, priv.table("s1b", len(prompts["s1"]))[p // BS] * BS + p % BS)
                                 for p in range(len(prompts["s1"]))])
    copies = 0
    for step in range(3):
        for sid, tok in (("s1b", 500 + step), ("s1", 600 + step)):
            ops = m.append_token(sid, tok)
            copies += len(ops)
            if ops:
                pkv.copy_blocks(kc_s, vc_s,
                                torch.tensor([o.src for o in ops], dtype=torch.int32, device="cuda"),
                                torch.tensor([o.dst for o in ops], dtype=torch.int32, device="cuda"),
                                torch.tensor([o.rows for o in ops], dtype=torch.int32, device="cuda"))
            s = m.seqs[sid]
            n = len(s)
            write_positions(kc_s, vc_s, [(s.token_ids, n - 1, s.slot(n - 1))])
            t = priv.table(sid, n)
            write_positions(kc_p, vc_p, [(s.token_ids, n - 1, t[(n - 1) // BS] * BS + (n - 1) % BS)])
    assert copies == 1                      # s1b's first write into the shared partial block

    sids = ["s1", "s1b", "s2", "s3", "s4", "s5"]
    lens = [len(m.seqs[s]) for s in sids]
    g = torch.Generator(device="cuda").manual_seed(2)
    q = torch.randn((len(sids), HKV * G, D), generator=g, device="cuda").to(torch.bfloat16)
    out_s, bt_s, cl = decode(kc_s, vc_s, q, [m.seqs[s].block_table for s in sids], lens)
    out_p, _, _ = decode(kc_p, vc_p, q, [priv.tables[s] for s in sids], lens)
    assert torch.equal(out_s, out_p)
    # the two branches diverged after the fork
    assert not torch.equal(out_s[0], out_s[1])
    # and the shared layout agrees with the oracle
    ref = oracle.paged_decode(bf16_to_u16(q.cpu()), bf16_to_u16(kc_s.cpu()), bf16_to_u16(vc_s.cpu()),
                              bt_s, cl, 1.0 / np.sqrt(D))
    got = out_s.float().cpu().numpy().astype(np.float64)
    assert (np.abs(got - ref) <= 1e-2 * np.maximum(1.0, np.abs(ref))).all()
