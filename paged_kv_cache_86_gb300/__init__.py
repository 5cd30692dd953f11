"""Attention over a block-paged KV cache on one GB300 GPU.

The compute path is the C-ABI library ``libpkv.so`` (hand-written sm_103a
CUDA kernels, declared in ``include/pkv.h``); this package is its thin ctypes
binding plus the seeded synthetic workload generator used by tests and the
bench. Importing the package does not load the library; the first call does,
and fails loudly if it has not been built.
"""
from ._lib import (PkvError, copy_blocks, decode_step, decode_step_fp8, decode_workspace_size,
                   get_device_errors,
                   load, mixed_step, mixed_workspace_size, paged_decode, paged_decode_fp8,
                   paged_prefill, prefill_workspace_size, selftest_bounded_wait, store_kvcache,
                   store_kvcache_fp8, version)

__all__ = ["PkvError", "copy_blocks", "decode_step", "decode_step_fp8", "decode_workspace_size",
           "get_device_errors",
           "load", "mixed_step", "mixed_workspace_size", "paged_decode", "paged_decode_fp8",
           "paged_prefill", "prefill_workspace_size", "selftest_bounded_wait", "store_kvcache",
           "store_kvcache_fp8", "version"]
