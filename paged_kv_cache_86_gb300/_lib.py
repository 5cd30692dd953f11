"""ctypes binding of libpkv (include/pkv.h): argument marshalling only.

Every function here takes torch tensors that already live on the GPU, checks
their dtype/shape/contiguity, passes raw device pointers and sizes to the C
entry point of the same name on the tensors' current CUDA stream, and turns a
non-zero status into :class:`PkvError`. No attention arithmetic happens here.
The library is built in-tree (``paged_kv_cache_86_gb300/libpkv.so``); if it is
missing, loading raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

PKV_BF16 = 0
STATUS = {0: "ok", -1: "invalid argument", -2: "unsupported shape", -3: "unsupported dtype",
          -4: "workspace missing, misaligned or too small", -5: "CUDA runtime error",
          -6: "device-side range check fired"}
DEVERR_SLOT, DEVERR_BLOCK_ID, DEVERR_LENGTH, DEVERR_TIMEOUT = 0x1, 0x2, 0x4, 0x8

EXPORTED = ("pkv_store_kvcache", "pkv_decode_workspace_size", "pkv_paged_decode",
            "pkv_prefill_workspace_size", "pkv_paged_prefill", "pkv_get_device_errors",
            "pkv_status_string", "pkv_version")


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)} ({status})")
        self.status = status


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load libpkv.so and declare the C signatures. Raises if it is not built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise ImportError(f"libpkv.so is not built ({path}); run "
                              "`python -m paged_kv_cache_86_gb300.build`")
        lib = ctypes.CDLL(path)
        vp, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                 ctypes.c_size_t)
        lib.pkv_store_kvcache.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i64, i64,
                                          ctypes.c_int, vp]
        lib.pkv_decode_workspace_size.argtypes = [i32, i32, i32, i32]
        lib.pkv_decode_workspace_size.restype = sz
        lib.pkv_paged_decode.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32,
                                         i32, i32, f32, vp, sz, ctypes.c_int, vp]
        lib.pkv_decode_step.argtypes = [vp, vp, vp, vp, i64, i64, vp, vp, vp, i32, vp, i32, i32,
                                        i32, i32, i32, i32, i32, f32, vp, sz, ctypes.c_int, vp]
        lib.pkv_store_kvcache_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                              i64, i64, vp]
        lib.pkv_paged_decode_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32,
                                             i32, i32, i32, i32, f32, vp, sz, vp]
        lib.pkv_decode_step_fp8.argtypes = [vp, vp, vp, vp, i64, i64, vp, vp, vp, vp, vp, i32, vp,
                                            i32, i32, i32, i32, i32, i32, i32, f32, vp, sz, vp]
        lib.pkv_mixed_workspace_size.argtypes = [i32, i32, i32, i32]
        lib.pkv_mixed_workspace_size.restype = sz
        lib.pkv_mixed_step.argtypes = [vp, vp, vp, vp, vp, i64, i64, vp, vp, vp, vp, i32, i32, vp,
                                       i32, i32, i32, i32, i32, i32, i32, i32, i32, f32, vp, sz,
                                       ctypes.c_int, vp]
        lib.pkv_copy_blocks.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_int,
                                        vp]
        lib.pkv_prefill_workspace_size.argtypes = [i32, i32, i32, i32]
        lib.pkv_prefill_workspace_size.restype = sz
        lib.pkv_paged_prefill.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, vp, i32, i32, i32,
                                          i32, i32, i32, i32, i32, f32, i32, vp, sz, ctypes.c_int,
                                          vp]
        lib.pkv_get_device_errors.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
        lib.pkv_selftest_bounded_wait.argtypes = [i32, vp, vp]
        lib.pkv_status_string.argtypes = [ctypes.c_int]
        lib.pkv_status_string.restype = ctypes.c_char_p
        lib.pkv_version.restype = i32
        for name in ("pkv_store_kvcache", "pkv_paged_decode", "pkv_decode_step",
                     "pkv_paged_prefill", "pkv_copy_blocks", "pkv_store_kvcache_fp8",
                     "pkv_paged_decode_fp8", "pkv_decode_step_fp8", "pkv_mixed_step",
                     "pkv_get_device_errors",
                     "pkv_selftest_bounded_wait"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def _check(status: int, what: str):
    if status != 0:
        raise PkvError(status, what)


def _stream(t: torch.Tensor, stream=None):
    s = stream if stream is not None else torch.cuda.current_stream(t.device)
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, ndim=None, contiguous=False, on_gpu=True):
    """dtype, rank and (optionally) dense row-major layout, then the device (unless
    on_gpu is False: the caller checks every tensor's device after every layout).
    The kernels take a raw pointer and assume the layout, so a strided view would
    be misread."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got {t.dim()}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if on_gpu:
        _need_gpu((t, name))


def _need_gpu(*named):
    for t, name in named:
        if not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")


def _out_like(out, q: torch.Tensor) -> torch.Tensor:
    """The caller's output buffer (checked: bf16, contiguous, shaped like q, on q's
    device), or a new one."""
    if out is None:
        return torch.empty_like(q)
    _need(out, "out", torch.bfloat16, q.dim())
    if out.shape != q.shape or not out.is_contiguous() or out.device != q.device:
        raise ValueError("out must be a contiguous tensor shaped like q, on q's device")
    return out


def _ptr(t: torch.Tensor):
    return ctypes.c_void_p(t.data_ptr())


def version() -> int:
    return load().pkv_version()


def store_kvcache(key, value, k_cache, v_cache, slot_mapping, stream=None) -> None:
    """Write key/value [T, Hkv, D] (token rows may be strided) into the caches
    [NB, bs, Hkv, D] at slot_mapping [T] (int32; negative = skip)."""
    lib = load()
    for t, n in ((key, "key"), (value, "value")):
        _need(t, n, torch.bfloat16, 3)
        if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
            raise ValueError(f"{n} rows must be contiguous [Hkv, D] blocks")
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.bfloat16, 4)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    _need(slot_mapping, "slot_mapping", torch.int32, 1)
    nb, bs, hkv, d = k_cache.shape
    t = slot_mapping.shape[0]
    if v_cache.shape != k_cache.shape or key.shape != (t, hkv, d) or value.shape != (t, hkv, d):
        raise ValueError("shape mismatch between key/value/caches/slot_mapping")
    _check(lib.pkv_store_kvcache(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                                 _ptr(slot_mapping.contiguous()), t, hkv, d, bs, nb,
                                 key.stride(0), value.stride(0), PKV_BF16,
                                 _stream(k_cache, stream)), "pkv_store_kvcache")


def _need_fp8_cache(k_cache, v_cache, k_scales, v_scales):
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.uint8, 4)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache / v_cache shape mismatch")
    nb, bs, hkv, d = k_cache.shape
    for t, n in ((k_scales, "k_scales"), (v_scales, "v_scales")):
        _need(t, n, torch.float32, 2)
        if t.shape != (nb * bs, hkv) or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous [num_blocks * block_size, Hkv] tensor")
    return nb, bs, hkv, d


def store_kvcache_fp8(key, value, k_cache, v_cache, k_scales, v_scales, slot_mapping,
                      stream=None) -> None:
    """Quantize key/value [T, Hkv, 128] bf16 into the fp8 E4M3 caches [NB, bs, Hkv, 128]
    (uint8 codes) and their row scales [NB * bs, Hkv] float32 at slot_mapping [T]."""
    lib = load()
    for t, n in ((key, "key"), (value, "value")):
        _need(t, n, torch.bfloat16, 3)
        if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
            raise ValueError(f"{n} rows must be contiguous [Hkv, D] blocks")
    nb, bs, hkv, d = _need_fp8_cache(k_cache, v_cache, k_scales, v_scales)
    _need(slot_mapping, "slot_mapping", torch.int32, 1)
    t = slot_mapping.shape[0]
    if key.shape != (t, hkv, d) or value.shape != (t, hkv, d):
        raise ValueError("shape mismatch between key/value/caches/slot_mapping")
    _check(lib.pkv_store_kvcache_fp8(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                                     _ptr(k_scales), _ptr(v_scales),
                                     _ptr(slot_mapping.contiguous()), t, hkv, d, bs, nb,
                                     key.stride(0), value.stride(0), _stream(k_cache, stream)),
           "pkv_store_kvcache_fp8")


def paged_decode_fp8(q, k_cache, v_cache, k_scales, v_scales, block_tables, context_lens,
                     scale: float, max_context_len: int | None = None, out=None, workspace=None,
                     stream=None) -> torch.Tensor:
    """Decode attention over fp8 E4M3 caches with row scales; returns out [S, Hq, 128] bf16."""
    lib = load()
    _need(q, "q", torch.bfloat16, 3)
    nb, bs, hkv, d = _need_fp8_cache(k_cache, v_cache, k_scales, v_scales)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    if not (q.is_contiguous() and block_tables.is_contiguous() and context_lens.is_contiguous()):
        raise ValueError("decode tensors must be contiguous")
    s, hq, dq = q.shape
    if dq != d:
        raise ValueError("q / cache head_dim mismatch")
    if block_tables.shape[0] != s or context_lens.shape[0] != s:
        raise ValueError("metadata rows must equal the number of sequences")
    mb = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = mb * bs
    out = _out_like(out, q)
    need = decode_workspace_size(s, hq, hkv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(lib.pkv_paged_decode_fp8(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(k_scales), _ptr(v_scales), _ptr(block_tables), mb,
                                    _ptr(context_lens), s, int(max_context_len), hq, hkv, d, bs, nb,
                                    float(scale), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(),
                                    _stream(q, stream)), "pkv_paged_decode_fp8")
    return out


def decode_step_fp8(q, key_new, value_new, k_cache, v_cache, k_scales, v_scales, block_tables,
                    context_lens, scale: float, max_context_len: int | None = None, out=None,
                    workspace=None, stream=None) -> torch.Tensor:
    """One decode step over fp8 E4M3 caches: quantizes each sequence's newest K/V row
    (key_new / value_new [S, Hkv, 128] bf16, token rows may be strided) into logical
    position context_lens[i] - 1 (codes and row scale), then decodes; returns out
    [S, Hq, 128] bf16."""
    lib = load()
    _need(q, "q", torch.bfloat16, 3)
    for t, n in ((key_new, "key_new"), (value_new, "value_new")):
        _need(t, n, torch.bfloat16, 3)
        if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
            raise ValueError(f"{n} rows must be contiguous [Hkv, D] blocks")
    nb, bs, hkv, d = _need_fp8_cache(k_cache, v_cache, k_scales, v_scales)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    if not (q.is_contiguous() and block_tables.is_contiguous() and context_lens.is_contiguous()):
        raise ValueError("decode tensors must be contiguous")
    s, hq, dq = q.shape
    if dq != d:
        raise ValueError("q / cache head_dim mismatch")
    if key_new.shape != (s, hkv, d) or value_new.shape != (s, hkv, d):
        raise ValueError("key_new / value_new must be [S, Hkv, D]")
    if block_tables.shape[0] != s or context_lens.shape[0] != s:
        raise ValueError("metadata rows must equal the number of sequences")
    mb = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = mb * bs
    out = _out_like(out, q)
    need = decode_workspace_size(s, hq, hkv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(lib.pkv_decode_step_fp8(_ptr(out), _ptr(q), _ptr(key_new), _ptr(value_new),
                                   key_new.stride(0), value_new.stride(0), _ptr(k_cache),
                                   _ptr(v_cache), _ptr(k_scales), _ptr(v_scales),
                                   _ptr(block_tables), mb, _ptr(context_lens), s,
                                   int(max_context_len), hq, hkv, d, bs, nb, float(scale),
                                   _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _stream(q, stream)), "pkv_decode_step_fp8")
    return out


def mixed_workspace_size(num_decode_seqs: int, num_q_heads: int, num_kv_heads: int,
                         head_dim: int = 128) -> int:
    return int(load().pkv_mixed_workspace_size(num_decode_seqs, num_q_heads, num_kv_heads,
                                               head_dim))


def mixed_step(q, key, value, slot_mapping, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k,
               block_tables, num_decode_seqs: int, scale: float, max_seqlen_q: int,
               max_seqlen_k: int, out=None, workspace=None, stream=None) -> torch.Tensor:
    """One mixed round: sequences [0, num_decode_seqs) are decode requests with one
    query row each (rows 0..D-1), the rest prefill chunks; every query row's K/V
    (key / value [total_q, Hkv, D]) is stored at slot_mapping first. Returns out
    [total_q, Hq, D] bf16."""
    _need(q, "q", torch.bfloat16, 3, contiguous=True, on_gpu=False)
    for t, n in ((key, "key"), (value, "value")):
        _need(t, n, torch.bfloat16, 3, on_gpu=False)
        if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
            raise ValueError(f"{n} rows must be contiguous [Hkv, D] blocks")
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.bfloat16, 4, contiguous=True, on_gpu=False)
    for t, n in ((cu_seqlens_q, "cu_seqlens_q"), (cu_seqlens_k, "cu_seqlens_k"),
                 (slot_mapping, "slot_mapping")):
        _need(t, n, torch.int32, 1, contiguous=True, on_gpu=False)
    _need(block_tables, "block_tables", torch.int32, 2, contiguous=True, on_gpu=False)
    _need_gpu((q, "q"), (key, "key"), (value, "value"), (k_cache, "k_cache"),
              (v_cache, "v_cache"), (cu_seqlens_q, "cu_seqlens_q"), (cu_seqlens_k, "cu_seqlens_k"),
              (slot_mapping, "slot_mapping"), (block_tables, "block_tables"))
    lib = load()
    total_q, hq, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    s = cu_seqlens_q.shape[0] - 1
    if (cu_seqlens_k.shape[0] != s + 1 or block_tables.shape[0] != s
            or slot_mapping.shape[0] != total_q or key.shape != (total_q, hkv, d)
            or value.shape != (total_q, hkv, d)):
        raise ValueError("metadata shape mismatch")
    out = _out_like(out, q)
    need = mixed_workspace_size(num_decode_seqs, hq, hkv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(lib.pkv_mixed_step(_ptr(out), _ptr(q), _ptr(key), _ptr(value), _ptr(slot_mapping),
                              key.stride(0), value.stride(0), _ptr(k_cache), _ptr(v_cache),
                              _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(max_seqlen_q),
                              int(max_seqlen_k), _ptr(block_tables), block_tables.shape[1], s,
                              int(num_decode_seqs), total_q, hq, hkv, d, bs, nb, float(scale),
                              _ptr(workspace), workspace.numel() * workspace.element_size(),
                              PKV_BF16, _stream(q, stream)), "pkv_mixed_step")
    return out


def copy_blocks(k_cache, v_cache, src_block_ids, dst_block_ids, num_rows=None,
                stream=None) -> None:
    """Copy rows [0, num_rows[p]) (whole blocks when num_rows is None) of block
    src_block_ids[p] to block dst_block_ids[p] in both caches [NB, bs, Hkv, D]."""
    lib = load()
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.bfloat16, 4)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache / v_cache shape mismatch")
    _need(src_block_ids, "src_block_ids", torch.int32, 1)
    _need(dst_block_ids, "dst_block_ids", torch.int32, 1)
    n = src_block_ids.shape[0]
    if dst_block_ids.shape[0] != n:
        raise ValueError("src / dst length mismatch")
    rows_ptr = ctypes.c_void_p(0)
    if num_rows is not None:
        _need(num_rows, "num_rows", torch.int32, 1)
        if num_rows.shape[0] != n:
            raise ValueError("num_rows length mismatch")
        num_rows = num_rows.contiguous()
        rows_ptr = _ptr(num_rows)
    nb, bs, hkv, d = k_cache.shape
    src_block_ids, dst_block_ids = src_block_ids.contiguous(), dst_block_ids.contiguous()
    _check(lib.pkv_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(src_block_ids),
                               _ptr(dst_block_ids), rows_ptr, n, hkv, d, bs, nb, PKV_BF16,
                               _stream(k_cache, stream)), "pkv_copy_blocks")


def decode_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                          head_dim: int = 128) -> int:
    return int(load().pkv_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim))


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                 max_context_len: int | None = None, out=None, workspace=None,
                 stream=None) -> torch.Tensor:
    """Decode attention; returns out [S, Hq, D] bf16.

    ``max_context_len`` is the host-side upper bound of context_lens (defaults
    to the block-table capacity, max_blocks_per_seq * block_size)."""
    lib = load()
    _need(q, "q", torch.bfloat16, 3)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    if not (q.is_contiguous() and k_cache.is_contiguous() and v_cache.is_contiguous()
            and block_tables.is_contiguous() and context_lens.is_contiguous()):
        raise ValueError("decode tensors must be contiguous")
    s, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if d2 != d or v_cache.shape != k_cache.shape:
        raise ValueError("q / cache head_dim mismatch")
    if block_tables.shape[0] != s or context_lens.shape[0] != s:
        raise ValueError("metadata rows must equal the number of sequences")
    mb = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = mb * bs
    out = _out_like(out, q)
    need = decode_workspace_size(s, hq, hkv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(lib.pkv_paged_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                _ptr(block_tables), mb, _ptr(context_lens), s, int(max_context_len),
                                hq, hkv, d, bs, nb, float(scale), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), PKV_BF16,
                                _stream(q, stream)), "pkv_paged_decode")
    return out


def decode_step(q, key_new, value_new, k_cache, v_cache, block_tables, context_lens,
                scale: float, max_context_len: int | None = None, out=None, workspace=None,
                stream=None) -> torch.Tensor:
    """One decode step: writes each sequence's newest K/V row (key_new / value_new
    [S, Hkv, D], token rows may be strided) at its last logical position
    context_lens[i] - 1, then decodes; returns out [S, Hq, D] bf16."""
    lib = load()
    _need(q, "q", torch.bfloat16, 3)
    for t, n in ((key_new, "key_new"), (value_new, "value_new")):
        _need(t, n, torch.bfloat16, 3)
        if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
            raise ValueError(f"{n} rows must be contiguous [Hkv, D] blocks")
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    if not (q.is_contiguous() and k_cache.is_contiguous() and v_cache.is_contiguous()
            and block_tables.is_contiguous() and context_lens.is_contiguous()):
        raise ValueError("decode tensors must be contiguous")
    s, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if d2 != d or v_cache.shape != k_cache.shape:
        raise ValueError("q / cache head_dim mismatch")
    if key_new.shape != (s, hkv, d) or value_new.shape != (s, hkv, d):
        raise ValueError("key_new / value_new must be [S, Hkv, D]")
    if block_tables.shape[0] != s or context_lens.shape[0] != s:
        raise ValueError("metadata rows must equal the number of sequences")
    mb = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = mb * bs
    out = _out_like(out, q)
    need = decode_workspace_size(s, hq, hkv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(lib.pkv_decode_step(_ptr(out), _ptr(q), _ptr(key_new), _ptr(value_new),
                               key_new.stride(0), value_new.stride(0), _ptr(k_cache),
                               _ptr(v_cache), _ptr(block_tables), mb, _ptr(context_lens), s,
                               int(max_context_len), hq, hkv, d, bs, nb, float(scale),
                               _ptr(workspace), workspace.numel() * workspace.element_size(),
                               PKV_BF16, _stream(q, stream)), "pkv_decode_step")
    return out


def prefill_workspace_size(num_seqs: int, total_q: int, num_q_heads: int,
                           head_dim: int = 128) -> int:
    return int(load().pkv_prefill_workspace_size(num_seqs, total_q, num_q_heads, head_dim))


def paged_prefill(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_tables, scale: float,
                  max_seqlen_q: int, max_seqlen_k: int, causal: bool = True, out=None,
                  workspace=None, stream=None) -> torch.Tensor:
    """Varlen chunked-prefill attention; returns out [total_q, Hq, D] bf16."""
    named = ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (cu_seqlens_q, "cu_seqlens_q"),
             (cu_seqlens_k, "cu_seqlens_k"), (block_tables, "block_tables"))
    _need(q, "q", torch.bfloat16, 3, contiguous=True, on_gpu=False)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.bfloat16, 4, contiguous=True, on_gpu=False)
    for t, n in ((cu_seqlens_q, "cu_seqlens_q"), (cu_seqlens_k, "cu_seqlens_k")):
        _need(t, n, torch.int32, 1, contiguous=True, on_gpu=False)
    _need(block_tables, "block_tables", torch.int32, 2, contiguous=True, on_gpu=False)
    _need_gpu(*named)
    lib = load()
    total_q, hq, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    s = cu_seqlens_q.shape[0] - 1
    if cu_seqlens_k.shape[0] != s + 1 or block_tables.shape[0] != s:
        raise ValueError("metadata shape mismatch")
    out = _out_like(out, q)
    need = prefill_workspace_size(s, total_q, hq, d)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _ptr(workspace) if workspace is not None else ctypes.c_void_p(0)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.pkv_paged_prefill(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                 _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(max_seqlen_q),
                                 int(max_seqlen_k), _ptr(block_tables), block_tables.shape[1], s,
                                 total_q, hq, hkv, d, bs, nb, float(scale), 1 if causal else 0,
                                 ws_ptr, ws_bytes, PKV_BF16, _stream(q, stream)),
           "pkv_paged_prefill")
    return out


def selftest_bounded_wait(fail_step: int, stream=None) -> list:
    """Run the library's on-GPU failure-path check (see pkv.h); returns
    [step warp 0 left, step warp 1 left, timeout reported, steps completed]."""
    lib = load()
    res = torch.zeros(4, dtype=torch.int32, device="cuda")
    s = stream if stream is not None else torch.cuda.current_stream()
    _check(lib.pkv_selftest_bounded_wait(int(fail_step), _ptr(res), ctypes.c_void_p(s.cuda_stream)),
           "pkv_selftest_bounded_wait")
    return res.cpu().tolist()


def get_device_errors(stream=None) -> int:
    """Synchronise the stream, then return and clear the device error bits."""
    lib = load()
    bits = ctypes.c_uint32(0)
    s = stream if stream is not None else torch.cuda.current_stream()
    st = lib.pkv_get_device_errors(ctypes.c_void_p(s.cuda_stream), ctypes.byref(bits))
    if st not in (0, -6):
        raise PkvError(st, "pkv_get_device_errors")
    return int(bits.value)
