"""CPU oracle for attention over a block-paged KV cache.

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg import this package. It shares no code with the CUDA
library in ``paged_kv_cache_86_gb300`` and never imports it.

* :mod:`oracle.attention` -- store / decode / prefill, a ctypes front end to the
  plain C implementation in ``pkv_oracle.c`` (double precision).
* :mod:`oracle.blocks` -- the host-side block arithmetic and block-manager
  model the pages print (block counts, slots, usage metrics, flat 2-D indices).
"""
