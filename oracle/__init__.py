"""CPU oracle for the paged FP8-KV decode path (TEST INFRASTRUCTURE ONLY).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` import this package.  The CUDA library and its Python
binding never do, and nothing here imports them: the two sides share only the
seeded input generators in ``workloads``.

The arithmetic lives in ``oracle.c`` (plain scalar C, fp64), compiled with gcc
into ``oracle/_build/liboracle.so`` on first use.  This module only marshals
NumPy arrays into it.  What each routine computes, with the passages it
follows, is written at the top of ``oracle.c``:

* ``e4m3_value`` / ``e4m3_encode``  -- the E4M3 format ("FP8量化与长上下文实测：
  Llama 3 70B部署优化指南", §1.1: range up to 448, smallest step 2^-9) with
  round-to-nearest-even and saturation at +-448.
* ``kv_append`` -- byte = E4M3(x / scale) written at page slot // P, row
  slot % P (division by the scale: same guide §3.1/§3.2; pages of P tokens
  behind a block table: 0539edu.com Llama 3 notes §2.2, §5.2).
* ``paged_decode`` -- fp64 softmax(q.K^T/sqrt(D)).V over the dequantised
  cache, reached through the block table, query head i reading KV head i // G.
* ``paged_prefill`` -- chunked prefill: the n queries of a sequence's chunk
  sit at positions L - n .. L - 1 and each attends causally to cached tokens
  0 .. its position (0539edu.com Llama 3 notes §2.2).
* ``kv_absmax_update`` / ``kv_scale_from_max`` -- the per-layer running
  maximum of |K| (or |V|) per kv head over prefill batches, and the scale
  max / 448 floored at 1e-12 (same guide §3.2 running max, §3.1 recipe).

Parity status of every function is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_*.py`` (no function here is unpinned).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (portable C11, no intrinsics, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.oracle_e4m3_value.restype = dbl
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode_array.restype = None
        lib.oracle_e4m3_encode_array.argtypes = [P, P, i64]
        lib.oracle_e4m3_encode_array_mt.restype = i32
        lib.oracle_e4m3_encode_array_mt.argtypes = [P, P, i64, i32]
        lib.oracle_e4m3_value_array.restype = None
        lib.oracle_e4m3_value_array.argtypes = [P, P, i64]
        lib.oracle_kv_append.restype = i64
        lib.oracle_kv_append.argtypes = [P, i32, i64, i32, i32, P, P, P, i64, i32]
        lib.oracle_paged_decode.restype = i32
        lib.oracle_paged_decode.argtypes = [P, P, P, P, P, P, i32, P, P, i32, i32, i32, i32,
                                            i32, i64, dbl, P, i64, P, P, i64, i32]
        lib.oracle_paged_prefill.restype = i32
        lib.oracle_paged_prefill.argtypes = [P, P, P, P, P, P, P, i32, P, P, i32, i32, i32, i32, i32, i64, dbl, P,
                                             i32]
        lib.oracle_kv_absmax_update.restype = None
        lib.oracle_kv_absmax_update.argtypes = [P, i32, i64, i32, i32, P]
        lib.oracle_kv_scale_from_max.restype = None
        lib.oracle_kv_scale_from_max.argtypes = [P, i32, P]
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return np.ascontiguousarray(a)


def e4m3_value(codes) -> np.ndarray:
    """fp64 value of every E4M3 code in `codes` (uint8); NaN codes give NaN."""
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().oracle_e4m3_value_array(_ptr(c), _ptr(out), c.size)
    return out


def e4m3_encode(y, threads: int = 1) -> np.ndarray:
    """E4M3 code of every fp32 value in `y` (RNE, saturate to +-448, NaN -> 0x7F)."""
    y = _c(y, np.float32)
    out = np.empty(y.shape, np.uint8)
    if threads > 1:
        _load().oracle_e4m3_encode_array_mt(_ptr(y), _ptr(out), y.size, int(threads))
    else:
        _load().oracle_e4m3_encode_array(_ptr(y), _ptr(out), y.size)
    return out


def kv_append(x, slots, scale, cache: np.ndarray) -> int:
    """Quantise `x` [T, Hkv, D] (fp32, or bf16 bits as uint16) into `cache`
    [num_pages, Hkv, P, D] (uint8, modified in place) at `slots` [T] (int64,
    negative = skip).  Returns how many slots fell outside the pool."""
    x = np.asarray(x)
    in_bf16 = 1 if x.dtype == np.uint16 else 0
    x = _c(x, np.uint16 if in_bf16 else np.float32)
    slots = _c(slots, np.int64)
    scale = _c(scale, np.float32)
    if not (cache.flags.c_contiguous and cache.dtype == np.uint8 and cache.ndim == 4):
        raise TypeError("cache must be a C-contiguous uint8 [num_pages, Hkv, P, D] array")
    T, H, D = x.shape
    NP, H2, P, D2 = cache.shape
    if H2 != H or D2 != D or slots.shape != (T,) or scale.shape != (H,):
        raise ValueError("shape mismatch")
    return int(_load().oracle_kv_append(_ptr(x), in_bf16, T, H, D, _ptr(slots), _ptr(scale),
                                        _ptr(cache), NP, P))


def paged_decode(q_bits, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens,
                 sm_scale: float | None = None, sel=None, threads: int = 1,
                 want_weights: bool = False, seq_page_sizes=None):
    """fp64 decode attention.

    q_bits: [B, Hq, D] bf16 bit patterns (uint16).  k_cache/v_cache: uint8
    [num_pages, Hkv, P, D].  k_scale/v_scale: fp32 [Hkv].  block_table: int32
    [B, max_pages].  seq_lens: int32 [B].  sel: optional int32 [n, 2] list of
    (b, q_head) rows to compute (default: all, in row-major order).
    seq_page_sizes: optional int32 [B], tokens per page of each sequence (a
    page of P_b tokens is P_b / P consecutive pool pages starting at its table
    entry; default P for every sequence).
    Returns out [n, D] (fp64), and the softmax weights [n, max(seq_lens)] if
    `want_weights`.
    """
    q_bits = _c(q_bits, np.uint16)
    k_cache = _c(k_cache, np.uint8)
    v_cache = _c(v_cache, np.uint8)
    k_scale = _c(k_scale, np.float32)
    v_scale = _c(v_scale, np.float32)
    block_table = _c(block_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    B, Hq, D = q_bits.shape
    NP, Hkv, P, D2 = k_cache.shape
    if v_cache.shape != k_cache.shape or D2 != D:
        raise ValueError("cache shape mismatch")
    if block_table.ndim != 2 or block_table.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("block_table / seq_lens shape mismatch")
    if seq_page_sizes is not None:
        seq_page_sizes = _c(seq_page_sizes, np.int32)
        if seq_page_sizes.shape != (B,):
            raise ValueError("seq_page_sizes shape mismatch")
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    if sel is None:
        bb, ii = np.meshgrid(np.arange(B), np.arange(Hq), indexing="ij")
        sel = np.stack([bb.ravel(), ii.ravel()], axis=1)
    sel = _c(np.asarray(sel, dtype=np.int32).reshape(-1, 2), np.int32)
    n = sel.shape[0]
    out = np.zeros((n, D), np.float64)
    w_stride = int(seq_lens.max()) if (want_weights and B > 0) else 0
    weights = np.zeros((n, max(w_stride, 1)), np.float64) if want_weights else None
    st = _load().oracle_paged_decode(
        _ptr(q_bits), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
        _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
        _ptr(seq_page_sizes) if seq_page_sizes is not None else None, B, Hq, Hkv, D, P, NP,
        float(sm_scale), _ptr(sel), n, _ptr(out),
        _ptr(weights) if want_weights else None, w_stride, int(threads))
    if st != 0:
        raise ValueError(f"oracle_paged_decode failed with status {st}")
    return (out, weights[:, :w_stride]) if want_weights else out


def kv_absmax_update(x, running_max: np.ndarray) -> None:
    """Fold the rows x [T, Hkv, D] (fp32, or bf16 bits as uint16) into the
    running per-head maximum of |x| (fp32 [Hkv], modified in place; NaN skipped)."""
    x = np.asarray(x)
    in_bf16 = 1 if x.dtype == np.uint16 else 0
    x = _c(x, np.uint16 if in_bf16 else np.float32)
    if not (running_max.flags.c_contiguous and running_max.dtype == np.float32):
        raise TypeError("running_max must be a C-contiguous float32 array")
    T, H, D = x.shape
    if running_max.shape != (H,):
        raise ValueError("shape mismatch")
    _load().oracle_kv_absmax_update(_ptr(x), in_bf16, T, H, D, _ptr(running_max))


def kv_scale_from_max(running_max) -> np.ndarray:
    """fp32 scale per head: max(running_max / 448, 1e-12)."""
    rm = _c(running_max, np.float32)
    out = np.empty_like(rm)
    _load().oracle_kv_scale_from_max(_ptr(rm), rm.size, _ptr(out))
    return out


def paged_prefill(q_bits, cu_q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens,
                  sm_scale: float | None = None, threads: int = 1, seq_page_sizes=None) -> np.ndarray:
    """fp64 chunked-prefill attention.  q_bits: [T, Hq, D] bf16 bit patterns,
    the chunks of all sequences back to back; cu_q: [B + 1] row offsets;
    seq_lens[b] includes the chunk; seq_page_sizes as in paged_decode.
    Returns out [T, Hq, D] (fp64)."""
    q_bits = _c(q_bits, np.uint16)
    cu_q = _c(cu_q, np.int32)
    k_cache = _c(k_cache, np.uint8)
    v_cache = _c(v_cache, np.uint8)
    k_scale = _c(k_scale, np.float32)
    v_scale = _c(v_scale, np.float32)
    block_table = _c(block_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    T, Hq, D = q_bits.shape
    NP, Hkv, P, D2 = k_cache.shape
    B = seq_lens.shape[0]
    if (v_cache.shape != k_cache.shape or D2 != D or cu_q.shape != (B + 1,) or block_table.shape[0] != B
            or cu_q[0] != 0 or cu_q[-1] != T):
        raise ValueError("shape mismatch")
    if seq_page_sizes is not None:
        seq_page_sizes = _c(seq_page_sizes, np.int32)
        if seq_page_sizes.shape != (B,):
            raise ValueError("seq_page_sizes shape mismatch")
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    out = np.zeros((T, Hq, D), np.float64)
    st = _load().oracle_paged_prefill(_ptr(q_bits), _ptr(cu_q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                      _ptr(v_scale), _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
                                      _ptr(seq_page_sizes) if seq_page_sizes is not None else None,
                                      B, Hq, Hkv, D, P, NP, float(sm_scale), _ptr(out), int(threads))
    if st != 0:
        raise ValueError(f"oracle_paged_prefill failed with status {st}")
    return out
