"""ctypes front end to the C oracle ``pkv_oracle.c`` (test infrastructure only).

All arrays are numpy: bf16 values travel as their raw 16-bit patterns
(``np.uint16``), indices as ``np.int32``, results come back as ``np.float64``.
The arithmetic lives in the C file; this module only marshals arguments and
builds the shared object with gcc when it is missing or stale.

Sources of each definition are cited in ``pkv_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB = os.path.join(_HERE, "libpkv_oracle.so")
_lock = threading.Lock()
_lib = None


class OracleError(RuntimeError):
    pass


_CODES = {-1: "bad argument", -2: "index out of range", -3: "out of memory"}


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle C source into a shared object (gcc, OpenMP)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall", "-Wextra",
               src, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def load_library(path: str):
    """Load an oracle shared object and declare its C signatures."""
    lib = ctypes.CDLL(path)
    i64, i32, vp, dbl = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_double
    lib.pkvo_store_kvcache.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64]
    lib.pkvo_paged_decode.argtypes = [vp, vp, vp, vp, vp, i64, vp, i64, i64, i64, i64,
                                      i64, i64, dbl, vp]
    lib.pkvo_paged_prefill.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64,
                                       i64, i64, i64, dbl, i32, vp]
    u8, f32 = ctypes.c_uint8, ctypes.c_float
    lib.pkvo_e4m3_value.argtypes = [u8]
    lib.pkvo_e4m3_value.restype = dbl
    lib.pkvo_e4m3_encode.argtypes = [f32]
    lib.pkvo_e4m3_encode.restype = u8
    lib.pkvo_quantize_row_fp8.argtypes = [vp, i64, vp, vp]
    lib.pkvo_quantize_row_fp8.restype = None
    lib.pkvo_store_kvcache_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64]
    lib.pkvo_paged_decode_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, vp, i64, i64, i64,
                                          i64, i64, i64, dbl, vp]
    for f in (lib.pkvo_store_kvcache, lib.pkvo_paged_decode, lib.pkvo_paged_prefill,
              lib.pkvo_store_kvcache_fp8, lib.pkvo_paged_decode_fp8):
        f.restype = ctypes.c_int
    lib.pkvo_max_threads.restype = ctypes.c_int
    lib.pkvo_set_threads.argtypes = [ctypes.c_int]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype).name}, got {a.dtype}")
    return a


def _check(rc: int):
    if rc != 0:
        raise OracleError(_CODES.get(rc, f"error {rc}"))


def max_threads() -> int:
    return _load().pkvo_max_threads()


def set_threads(n: int) -> None:
    _load().pkvo_set_threads(int(n))


def store_kvcache(key, value, k_cache, v_cache, slot_mapping, block_size: int, lib=None) -> None:
    """Scatter ``key``/``value`` [T, Hkv, D] into the caches [NB, bs, Hkv, D] in place."""
    key, value = _c(key, np.uint16), _c(value, np.uint16)
    slot_mapping = _c(slot_mapping, np.int32)
    if not (k_cache.flags.c_contiguous and v_cache.flags.c_contiguous):
        raise ValueError("caches must be C-contiguous")
    if k_cache.dtype != np.uint16 or v_cache.dtype != np.uint16:
        raise TypeError("caches must be uint16 (bf16 bits)")
    nb, bs, hkv, d = k_cache.shape
    if bs != block_size:
        raise ValueError("cache shape does not match block_size")
    t = slot_mapping.shape[0]
    if key.shape != (t, hkv, d) or value.shape != (t, hkv, d):
        raise ValueError("key/value shape mismatch")
    _check((lib or _load()).pkvo_store_kvcache(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                                      _ptr(slot_mapping), t, hkv, d, bs, nb))


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                 seq_mask=None, lib=None) -> np.ndarray:
    """Decode attention: ``q`` [S, Hq, D] -> out [S, Hq, D] float64.

    With ``seq_mask`` only the selected sequences are computed (the others are NaN).
    """
    q = _c(q, np.uint16)
    k_cache, v_cache = _c(k_cache, np.uint16), _c(v_cache, np.uint16)
    block_tables = _c(block_tables, np.int32)
    context_lens = _c(context_lens, np.int32)
    s, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if d2 != d or v_cache.shape != k_cache.shape:
        raise ValueError("cache shape mismatch")
    if block_tables.ndim != 2 or block_tables.shape[0] != s or context_lens.shape != (s,):
        raise ValueError("metadata shape mismatch")
    mask = None if seq_mask is None else _c(np.asarray(seq_mask, dtype=np.uint8), np.uint8)
    out = np.full((s, hq, d), np.nan, dtype=np.float64)
    _check((lib or _load()).pkvo_paged_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                     _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
                                     s, hq, hkv, d, bs, nb, float(scale), _ptr(mask)))
    return out


def paged_prefill(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_tables, scale: float,
                  causal: bool = True, row_mask=None, lib=None) -> np.ndarray:
    """Varlen prefill attention: ``q`` [total_q, Hq, D] -> out [total_q, Hq, D] float64.

    With ``row_mask`` only the selected query rows are computed (the others are NaN).
    """
    q = _c(q, np.uint16)
    k_cache, v_cache = _c(k_cache, np.uint16), _c(v_cache, np.uint16)
    cu_q, cu_k = _c(cu_seqlens_q, np.int32), _c(cu_seqlens_k, np.int32)
    block_tables = _c(block_tables, np.int32)
    total_q, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    s = cu_q.shape[0] - 1
    if d2 != d or v_cache.shape != k_cache.shape or cu_k.shape != cu_q.shape:
        raise ValueError("shape mismatch")
    if block_tables.ndim != 2 or block_tables.shape[0] != s or cu_q[-1] != total_q:
        raise ValueError("metadata shape mismatch")
    mask = None if row_mask is None else _c(np.asarray(row_mask, dtype=np.uint8), np.uint8)
    out = np.full((total_q, hq, d), np.nan, dtype=np.float64)
    _check((lib or _load()).pkvo_paged_prefill(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                      _ptr(cu_q), _ptr(cu_k), _ptr(block_tables),
                                      block_tables.shape[1], s, hq, hkv, d, bs, nb, float(scale),
                                      1 if causal else 0, _ptr(mask)))
    return out


# ------------------------------------------------------------------ fp8 KV --

def e4m3_value(code: int, lib=None) -> float:
    """Value of one OCP FP8 E4M3 code (NaN for S.1111.111)."""
    return float((lib or _load()).pkvo_e4m3_value(int(code) & 0xFF))


def e4m3_encode(x: float, lib=None) -> int:
    """Nearest finite E4M3 code of a float32 value, ties to even, saturating at 448."""
    return int((lib or _load()).pkvo_e4m3_encode(float(np.float32(x))))


def quantize_rows_fp8(x, lib=None):
    """Rows of bf16 bits [R, D] -> (codes [R, D] uint8, scales [R] float32)."""
    x = _c(x, np.uint16)
    r, d = x.shape
    codes = np.zeros((r, d), dtype=np.uint8)
    scales = np.zeros(r, dtype=np.float32)
    lib = lib or _load()
    for i in range(r):
        lib.pkvo_quantize_row_fp8(_ptr(x[i]), d, _ptr(codes[i]), _ptr(scales[i:i + 1]))
    return codes, scales


def store_kvcache_fp8(key, value, k_codes, v_codes, k_scales, v_scales, slot_mapping,
                      block_size: int, lib=None) -> None:
    """Quantize ``key``/``value`` [T, Hkv, D] (bf16 bits) into the fp8 caches
    [NB, bs, Hkv, D] uint8 and their scales [NB * bs, Hkv] float32, in place."""
    key, value = _c(key, np.uint16), _c(value, np.uint16)
    slot_mapping = _c(slot_mapping, np.int32)
    for a, dt in ((k_codes, np.uint8), (v_codes, np.uint8), (k_scales, np.float32),
                  (v_scales, np.float32)):
        if a.dtype != dt or not a.flags.c_contiguous:
            raise TypeError("fp8 caches must be C-contiguous uint8, scales float32")
    nb, bs, hkv, d = k_codes.shape
    if bs != block_size or k_scales.shape != (nb * bs, hkv) or v_scales.shape != k_scales.shape:
        raise ValueError("cache / scale shapes do not match")
    t = slot_mapping.shape[0]
    if key.shape != (t, hkv, d) or value.shape != (t, hkv, d):
        raise ValueError("key/value shape mismatch")
    _check((lib or _load()).pkvo_store_kvcache_fp8(
        _ptr(key), _ptr(value), _ptr(k_codes), _ptr(v_codes), _ptr(k_scales), _ptr(v_scales),
        _ptr(slot_mapping), t, hkv, d, bs, nb))


def paged_decode_fp8(q, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens,
                     scale: float, seq_mask=None, lib=None) -> np.ndarray:
    """Decode attention over the dequantized fp8 cache: ``q`` [S, Hq, D] bf16 bits ->
    out [S, Hq, D] float64 (NaN rows where seq_mask excludes a sequence)."""
    q = _c(q, np.uint16)
    k_codes, v_codes = _c(k_codes, np.uint8), _c(v_codes, np.uint8)
    k_scales, v_scales = _c(k_scales, np.float32), _c(v_scales, np.float32)
    block_tables = _c(block_tables, np.int32)
    context_lens = _c(context_lens, np.int32)
    s, hq, d = q.shape
    nb, bs, hkv, d2 = k_codes.shape
    if d2 != d or v_codes.shape != k_codes.shape or k_scales.shape != (nb * bs, hkv):
        raise ValueError("cache shape mismatch")
    if block_tables.ndim != 2 or block_tables.shape[0] != s or context_lens.shape != (s,):
        raise ValueError("metadata shape mismatch")
    mask = None if seq_mask is None else _c(np.asarray(seq_mask, dtype=np.uint8), np.uint8)
    out = np.full((s, hq, d), np.nan, dtype=np.float64)
    _check((lib or _load()).pkvo_paged_decode_fp8(
        _ptr(out), _ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scales), _ptr(v_scales),
        _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), s, hq, hkv, d, bs, nb,
        float(scale), _ptr(mask)))
    return out
