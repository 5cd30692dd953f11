"""The C-ABI library builds, loads without a GPU, and exports every entry point
that include/pkv.h declares (no compute calls here)."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_86_gb300 as pkv
from paged_kv_cache_86_gb300 import _lib
from paged_kv_cache_86_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.load()


def test_header_declares_the_three_operations():
    names = declared_functions()
    for n in ("pkv_store_kvcache", "pkv_paged_decode", "pkv_paged_prefill"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(_lib.EXPORTED) <= set(declared_functions())


def test_status_strings_and_version(lib):
    assert lib.pkv_status_string(0) == b"ok"
    for code in range(-6, 0):
        assert lib.pkv_status_string(code) != b"unknown status"
    assert pkv.version() >= 100


def test_host_validation_needs_no_gpu(lib):
    # Argument checks run before any CUDA call, so they answer on a CPU-only host.
    vp, null = ctypes.c_void_p, ctypes.c_void_p(0)
    assert lib.pkv_store_kvcache(null, null, null, null, null, 1, 8, 128, 16, 4, 1024, 1024,
                                 7, null) == -3            # dtype
    assert lib.pkv_store_kvcache(null, null, null, null, null, -1, 8, 128, 16, 4, 1024, 1024,
                                 0, null) == -1            # negative token count
    assert lib.pkv_store_kvcache(null, null, null, null, null, 0, 8, 128, 16, 4, 1024, 1024,
                                 0, null) == 0             # nothing to do
    assert lib.pkv_store_kvcache(null, null, null, null, null, 3, 8, 128, 16, 4, 1024, 1024,
                                 0, null) == -1            # null pointers
    assert lib.pkv_store_kvcache(vp(16), vp(16), vp(16), vp(16), vp(16), 3, 1, 12, 16, 4, 12, 12,
                                 0, null) == -2            # row not a multiple of 8 elements
    assert lib.pkv_store_kvcache(vp(18), vp(16), vp(16), vp(16), vp(16), 3, 8, 128, 16, 4, 1024,
                                 1024, 0, null) == -1      # misaligned key
    assert lib.pkv_paged_decode(null, null, null, null, null, 4, null, 2, 64, 8, 2, 64, 16, 8,
                                 0.1, null, 0, 0, null) == -2   # head_dim 64
    assert lib.pkv_paged_decode(null, null, null, null, null, 4, null, 2, 65, 8, 2, 128, 16, 8,
                                 0.1, null, 0, 0, null) == -1   # max_context_len > 4 * 16
    assert lib.pkv_paged_decode(null, null, null, null, null, 4, null, 0, 64, 8, 2, 128, 16, 8,
                                 0.1, null, 0, 0, null) == 0    # no sequences
    assert lib.pkv_paged_decode(null, null, null, null, null, 4, null, 2, 64, 8, 2, 128, 16, 8,
                                 float("nan"), null, 0, 0, null) == -1
    assert lib.pkv_paged_prefill(null, null, null, null, null, null, 8, 8, null, 4, 1, 8, 8, 2,
                                 128, 16, 8, 0.1, 1, null, 0, 1, null) == -3
    # 65535 chunks of up to 2048 query tiles, 32 head pairs: 2^32 work items,
    # more than the prefill kernel can number (32 bits)
    assert lib.pkv_paged_prefill(null, null, null, null, null, null, 2048 * 128, 2048 * 128, null,
                                 16384, 65535, 1 << 30, 64, 8, 128, 16, 8, 0.1, 1, null, 0, 0,
                                 null) == -1


def test_decode_step_host_validation_needs_no_gpu(lib):
    vp, null = ctypes.c_void_p, ctypes.c_void_p(0)
    a = vp(256)  # aligned dummy addresses: never dereferenced, checks fail first

    def step(key_new, value_new, ks, vs, num_seqs=2, head_dim=128, dtype=0, scale=0.1):
        return lib.pkv_decode_step(a, a, key_new, value_new, ks, vs, a, a, a, 4, a, num_seqs, 64,
                                   8, 2, head_dim, 16, 8, scale, a, 1 << 20, dtype, null)

    assert step(a, a, 256, 256, dtype=7) == -3          # dtype
    assert step(null, a, 256, 256) == -1                # missing new-token rows
    assert step(a, null, 256, 256) == -1
    assert step(a, a, 256, 256, head_dim=64) == -2      # head_dim 64
    assert step(vp(264), a, 256, 256) == -1             # misaligned key_new
    assert step(a, a, 255, 256) == -1                   # stride not a multiple of 8
    assert step(a, a, 128, 256) == -1                   # stride shorter than a row (2 x 128)
    assert step(a, a, 256, 256, scale=float("inf")) == -1
    assert step(null, null, 0, 0, num_seqs=0) == 0      # nothing to do


def test_copy_blocks_host_validation_needs_no_gpu(lib):
    vp, null = ctypes.c_void_p, ctypes.c_void_p(0)
    a = vp(256)
    assert lib.pkv_copy_blocks(a, a, a, a, null, 3, 8, 128, 16, 64, 7, null) == -3   # dtype
    assert lib.pkv_copy_blocks(a, a, a, a, null, -1, 8, 128, 16, 64, 0, null) == -1  # count
    assert lib.pkv_copy_blocks(a, a, a, a, null, 65536, 8, 128, 16, 64, 0, null) == -1
    assert lib.pkv_copy_blocks(a, a, a, a, null, 3, 1, 12, 16, 64, 0, null) == -2    # row of 12
    assert lib.pkv_copy_blocks(a, a, null, a, null, 3, 8, 128, 16, 64, 0, null) == -1  # no src
    assert lib.pkv_copy_blocks(vp(264), a, a, a, null, 3, 8, 128, 16, 64, 0, null) == -1  # align
    assert lib.pkv_copy_blocks(null, null, null, null, null, 0, 8, 128, 16, 64, 0, null) == 0


def test_fp8_host_validation_needs_no_gpu(lib):
    vp, null = ctypes.c_void_p, ctypes.c_void_p(0)
    a = vp(256)
    # store: head_dim other than 128, null scales, misaligned scales, short stride
    assert lib.pkv_store_kvcache_fp8(a, a, a, a, a, a, a, 3, 8, 64, 16, 8, 1024, 1024, null) == -2
    assert lib.pkv_store_kvcache_fp8(a, a, a, a, null, a, a, 3, 8, 128, 16, 8, 1024, 1024, null) == -1
    assert lib.pkv_store_kvcache_fp8(a, a, a, a, vp(260), a, a, 3, 8, 128, 16, 8, 1024, 1024, null) == -1
    assert lib.pkv_store_kvcache_fp8(a, a, a, a, a, a, a, 3, 8, 128, 16, 8, 512, 1024, null) == -1
    assert lib.pkv_store_kvcache_fp8(null, null, null, null, null, null, null, 0, 8, 128, 16, 8,
                                     1024, 1024, null) == 0
    # decode: missing scales, head_dim, no sequences
    assert lib.pkv_paged_decode_fp8(a, a, a, a, null, a, a, 4, a, 2, 64, 32, 8, 128, 16, 8, 0.1,
                                    a, 1 << 20, null) == -1
    assert lib.pkv_paged_decode_fp8(a, a, a, a, a, a, a, 4, a, 2, 64, 32, 8, 64, 16, 8, 0.1,
                                    a, 1 << 20, null) == -2
    assert lib.pkv_paged_decode_fp8(null, null, null, null, null, null, null, 4, null, 0, 64, 32,
                                    8, 128, 16, 8, 0.1, null, 0, null) == 0

    # decode step: missing new-token rows or scales, misaligned scales, head_dim,
    # short stride, no sequences
    def step(key_new, ks, k_scales, num_seqs=2, head_dim=128):
        return lib.pkv_decode_step_fp8(a, a, key_new, a, ks, 256, a, a, k_scales, a, a, 4, a,
                                       num_seqs, 64, 32, 8, head_dim, 16, 8, 0.1, a, 1 << 20, null)

    assert step(null, 256, a) == -1
    assert step(a, 256, null) == -1
    assert step(a, 256, vp(260)) == -1
    assert step(a, 256, a, head_dim=64) == -2
    assert step(a, 128, a) == -1
    assert lib.pkv_decode_step_fp8(null, null, null, null, 0, 0, null, null, null, null, null, 4,
                                   null, 0, 64, 32, 8, 128, 16, 8, 0.1, null, 0, null) == 0


def test_mixed_step_host_validation_needs_no_gpu(lib):
    vp, null = ctypes.c_void_p, ctypes.c_void_p(0)
    a = vp(256)

    def step(num_seqs=4, num_decode=2, total_q=10, head_dim=128, dtype=0, ws=a, ks=1024):
        return lib.pkv_mixed_step(a, a, a, a, a, ks, 1024, a, a, a, a, 8, 64, a, 4, num_seqs,
                                  num_decode, total_q, 32, 8, head_dim, 16, 8, 0.1, ws, 1 << 20,
                                  dtype, null)

    assert step(dtype=7) == -3
    assert step(num_decode=5) == -1            # more decode sequences than sequences
    assert step(total_q=1) == -1               # fewer rows than decode sequences
    assert step(head_dim=64) == -2
    assert step(ws=null) == -1
    assert step(ks=100) == -1                  # key stride shorter than a row
    assert step(num_seqs=0, num_decode=0, total_q=0) == 0
