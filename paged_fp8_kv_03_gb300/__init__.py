"""Python binding of libpagedfp8 (paged FP8 KV cache + GQA decode, sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libpagedfp8.so``.  torch supplies device memory and the current
stream.  The entry points mirror the C ABI in ``include/pagedfp8.h``:

* ``pkv_kv_append_fp8``       -- quantise new K/V rows into their pages
* ``pkv_paged_gqa_decode``    -- grouped-query decode attention over the pages
* ``pkv_append_decode_fp8``    -- both in one launch (one whole decode step)
* ``pkv_kv_calibrate``         -- running |K|, |V| maxima per kv head and the scales
* ``pkv_decode_calibrate_split``, ``pkv_decode_set_split_weights``,
  ``pkv_decode_get_split_weights`` -- per-CTA weights of the decode split
* ``pkv_decode_workspace_size``, ``pkv_status_string``, ``pkv_version``

``kv_append_fp8`` / ``paged_gqa_decode`` are the same calls with the output
and workspace allocated by torch when not given.  There is no CPU fallback:
if the library is not built, loading raises.
"""
from __future__ import annotations

import contextlib
import ctypes
import math
import os
import threading

import torch

from . import build as _build

PKV_F32, PKV_BF16 = 0, 1
DEVERR_SLOT, DEVERR_PAGE, DEVERR_SEQLEN, DEVERR_TIMEOUT, DEVERR_PAGESIZE, DEVERR_INTERNAL = 1, 2, 4, 8, 16, 32
HEAD_DIM = 128
MAX_GROUP = 8
MAX_BATCH = 8192

_lib = None
_lock = threading.Lock()


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        msg = f"{what}: status {status} ({pkv_status_string(status)})"
        if status == 6:
            code, name = pkv_last_cuda_error()
            msg += f" [{name} ({code})]"
        super().__init__(msg)
        self.status = status


def lib_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libpagedfp8.so (built in-tree by build()); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build the CUDA library first "
                               "(python -m paged_fp8_kv_03_gb300.build)")
        lib = ctypes.CDLL(path)
        vp, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
        lib.pkv_kv_append_fp8.restype = i32
        lib.pkv_kv_append_fp8.argtypes = [vp, vp, i32, i64, i32, i32, vp, vp, vp, vp, vp, i64, i32, vp, vp]
        lib.pkv_decode_workspace_size.restype = sz
        lib.pkv_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
        lib.pkv_paged_gqa_decode.restype = i32
        lib.pkv_paged_gqa_decode.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, vp, i32, i32, i32, i32, i32,
                                             i64, f32, vp, i32, vp, sz, vp, i32, vp]
        lib.pkv_append_decode_fp8.restype = i32
        lib.pkv_append_decode_fp8.argtypes = [vp, vp, i32, i32, vp, vp, vp, vp, vp, vp, i32, vp, i32, vp, i32, i32,
                                              i32, i32, i32, i64, f32, vp, i32, vp, sz, vp, i32, vp]
        lib.pkv_kv_calibrate.restype = i32
        lib.pkv_kv_calibrate.argtypes = [vp, vp, i32, i64, i32, i32, vp, vp, vp, vp, vp]
        lib.pkv_paged_gqa_decode_noalloc.restype = i32
        lib.pkv_paged_gqa_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, vp, i32, i32, i32, i32,
                                                     i32, i64, f32, vp, i32, vp, i32, vp]
        lib.pkv_decode_noalloc_scratch_bytes.restype = sz
        lib.pkv_decode_noalloc_scratch_bytes.argtypes = []
        lib.pkv_prefill_workspace_size.restype = sz
        lib.pkv_prefill_workspace_size.argtypes = [i32, i32, i32, i64]
        lib.pkv_paged_prefill.restype = i32
        lib.pkv_paged_prefill.argtypes = [vp, vp, i32, i32, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i64, i32, i32,
                                          i32, i32, i64, ctypes.c_float, vp, i32, vp, sz, vp, vp]
        lib.pkv_read_device_error.restype = i32
        lib.pkv_read_device_error.argtypes = [vp, i32, ctypes.POINTER(ctypes.c_int32), vp]
        lib.pkv_decode_set_split_weights.restype = i32
        lib.pkv_decode_set_split_weights.argtypes = [vp, i32]
        lib.pkv_decode_get_split_weights.restype = i32
        lib.pkv_decode_get_split_weights.argtypes = [vp, i32, ctypes.POINTER(ctypes.c_int)]
        lib.pkv_decode_calibrate_split.restype = i32
        lib.pkv_decode_calibrate_split.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, vp, i32, i32, i32, i32, i32,
                                                   i64, f32, vp, i32, vp, sz, i32, i32, vp, i32,
                                                   ctypes.POINTER(ctypes.c_int), vp]
        lib.pkv_last_cuda_error.restype = i32
        lib.pkv_last_cuda_error.argtypes = [ctypes.POINTER(ctypes.c_char_p)]
        lib.pkv_test_withhold_load.restype = None
        lib.pkv_test_withhold_load.argtypes = [i32]
        lib.pkv_status_string.restype = ctypes.c_char_p
        lib.pkv_status_string.argtypes = [i32]
        lib.pkv_version.restype = i32
        lib.pkv_version.argtypes = []
        _lib = lib
        return lib


def pkv_read_device_error(device_error, clear: bool = False, stream=None) -> int:
    """The bits of a device error word (waits for the work enqueued on the
    stream); with clear=True the word is reset to 0 afterwards."""
    _need(device_error, "device_error", torch.int32)
    code = ctypes.c_int32(0)
    with _device_of(device_error):
        st = load().pkv_read_device_error(_ptr(device_error), 1 if clear else 0, ctypes.byref(code), _stream(stream))
    if st != 0:
        raise PkvError(st, "pkv_read_device_error")
    return int(code.value)


def pkv_decode_set_split_weights(weights, device=None) -> None:
    """Install per-CTA split weights (ints in [768, 1280]) for decode calls on
    `device` (default: the current one) whose grid has len(weights) CTAs;
    None or an empty sequence removes them (even split)."""
    w = [int(x) for x in (weights if weights is not None else [])]
    if any(x < 0 or x > 0xFFFF for x in w):
        raise PkvError(2, "pkv_decode_set_split_weights")
    buf = (ctypes.c_uint16 * max(1, len(w)))(*w)
    with _device_of_index(device):
        st = load().pkv_decode_set_split_weights(ctypes.addressof(buf), len(w))
    if st != 0:
        raise PkvError(st, "pkv_decode_set_split_weights")


def pkv_decode_get_split_weights(device=None) -> list:
    """The split weights installed for `device` (empty: even split)."""
    cap = 1024
    buf = (ctypes.c_uint16 * cap)()
    n = ctypes.c_int(0)
    with _device_of_index(device):
        st = load().pkv_decode_get_split_weights(ctypes.addressof(buf), cap, ctypes.byref(n))
    if st != 0:
        raise PkvError(st, "pkv_decode_get_split_weights")
    return list(buf[:n.value])


def pkv_decode_calibrate_split(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out, workspace,
                               sm_scale=None, max_ctas=0, rounds=6, stream=None, max_seq_len=0,
                               seq_page_sizes=None) -> list:
    """Measure and install split weights for decode calls shaped like this
    one (runs 4 * rounds decode calls on these inputs, writing out and
    workspace, and synchronises the stream).  Returns the weights."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.uint8, 4)
    _need(v_cache, "v_cache", torch.uint8, 4)
    _need(k_scale, "k_scale", torch.float32, 1)
    _need(v_scale, "v_scale", torch.float32, 1)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(out, "out", dim=3)
    _need(workspace, "workspace", torch.uint8)
    B, Hq, D = q.shape
    NP, Hkv, P, D2 = k_cache.shape
    if v_cache.shape != k_cache.shape or D2 != D or out.shape != q.shape:
        raise ValueError("q / cache / out shapes disagree")
    if block_table.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("block_table / seq_lens shapes disagree with q")
    _check_page_sizes(seq_page_sizes, B)
    _same_device(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out, workspace, seq_page_sizes)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    cap = 1024
    buf = (ctypes.c_uint16 * cap)()
    n = ctypes.c_int(0)
    with _device_of(q):
        st = load().pkv_decode_calibrate_split(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                               _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
                                               int(max_seq_len), _ptr(seq_page_sizes), B, Hq, Hkv, D, P, NP,
                                               float(sm_scale), _ptr(out), _act_code(out), _ptr(workspace),
                                               workspace.numel(), int(max_ctas), int(rounds),
                                               ctypes.addressof(buf), cap, ctypes.byref(n), _stream(stream))
    if st != 0:
        raise PkvError(st, "pkv_decode_calibrate_split")
    return list(buf[:n.value])


def pkv_test_withhold_load(index: int) -> None:
    """Test facility (failure-detection tests only): decode worker warp /
    prefill CTA `index` skips its first load so its bounded wait runs out;
    a negative index turns it off."""
    load().pkv_test_withhold_load(int(index))


def pkv_last_cuda_error():
    """(code, name) of the CUDA error behind this thread's last PKV_ERR_CUDA."""
    name = ctypes.c_char_p()
    code = load().pkv_last_cuda_error(ctypes.byref(name))
    return int(code), (name.value or b"").decode()


def pkv_status_string(status: int) -> str:
    return load().pkv_status_string(int(status)).decode()


def pkv_version() -> int:
    return int(load().pkv_version())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _device_of(t):
    """Runs a call with the tensors' device current: the library launches on
    the current device and takes the current stream of that device."""
    if t.device.index == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(t.device)


def _device_of_index(device):
    if device is None:
        return contextlib.nullcontext()
    return torch.cuda.device(device)


def _same_device(ref, *ts):
    for t in ts:
        if t is not None and t.device != ref.device:
            raise ValueError(f"all tensors must be on {ref.device}, got one on {t.device}")


def _check_page_sizes(seq_page_sizes, batch):
    if seq_page_sizes is not None:
        _need(seq_page_sizes, "seq_page_sizes", torch.int32, 1)
        if seq_page_sizes.shape[0] != batch:
            raise ValueError("seq_page_sizes must have one entry per sequence")


def _need(t, name, dtype=None, dim=None, cuda=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _act_code(t) -> int:
    if t.dtype == torch.float32:
        return PKV_F32
    if t.dtype == torch.bfloat16:
        return PKV_BF16
    raise TypeError(f"activations must be float32 or bfloat16, got {t.dtype}")


def pkv_kv_append_fp8(k_new, v_new, slot_mapping, k_scale, v_scale, k_cache, v_cache,
                      device_error=None, stream=None) -> None:
    """k_new/v_new [T, Hkv, 128] fp32|bf16; slot_mapping int64 [T]; scales fp32
    [Hkv]; caches uint8 [num_pages, Hkv, P, 128] (written in place)."""
    _need(k_new, "k_new", dim=3)
    _need(v_new, "v_new", dtype=k_new.dtype, dim=3)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    _need(k_scale, "k_scale", torch.float32, 1)
    _need(v_scale, "v_scale", torch.float32, 1)
    _need(k_cache, "k_cache", torch.uint8, 4)
    _need(v_cache, "v_cache", torch.uint8, 4)
    if device_error is not None:
        _need(device_error, "device_error", torch.int32)
    T, H, D = k_new.shape
    NP, H2, P, D2 = k_cache.shape
    if v_new.shape != k_new.shape or v_cache.shape != k_cache.shape or H2 != H or D2 != D:
        raise ValueError("k/v shapes disagree")
    if slot_mapping.shape[0] != T or k_scale.shape[0] != H or v_scale.shape[0] != H:
        raise ValueError("slot_mapping / scale shapes disagree")
    _same_device(k_new, v_new, slot_mapping, k_scale, v_scale, k_cache, v_cache, device_error)
    with _device_of(k_new):
        st = load().pkv_kv_append_fp8(_ptr(k_new), _ptr(v_new), _act_code(k_new), T, H, D, _ptr(slot_mapping),
                                      _ptr(k_scale), _ptr(v_scale), _ptr(k_cache), _ptr(v_cache), NP, P,
                                      _ptr(device_error), _stream(stream))
    if st != 0:
        raise PkvError(st, "pkv_kv_append_fp8")


def pkv_kv_calibrate(k_new, v_new, k_running_max, v_running_max, k_scale=None, v_scale=None,
                     stream=None) -> None:
    """Fold prefill rows k_new/v_new [T, Hkv, 128] (fp32|bf16) into the running
    per-head maxima (fp32 [Hkv], in place) and, if given, write the scales
    max(running_max / 448, 1e-12)."""
    _need(k_new, "k_new", dim=3)
    _need(v_new, "v_new", dtype=k_new.dtype, dim=3)
    for t, n in ((k_running_max, "k_running_max"), (v_running_max, "v_running_max")):
        _need(t, n, torch.float32, 1)
    if (k_scale is None) != (v_scale is None):
        raise ValueError("give both scales or neither")
    if k_scale is not None:
        _need(k_scale, "k_scale", torch.float32, 1)
        _need(v_scale, "v_scale", torch.float32, 1)
    T, H, D = k_new.shape
    if v_new.shape != k_new.shape or k_running_max.shape[0] != H or v_running_max.shape[0] != H:
        raise ValueError("shapes disagree")
    _same_device(k_new, v_new, k_running_max, v_running_max, k_scale, v_scale)
    with _device_of(k_new):
        st = load().pkv_kv_calibrate(_ptr(k_new), _ptr(v_new), _act_code(k_new), T, H, D, _ptr(k_running_max),
                                     _ptr(v_running_max), _ptr(k_scale), _ptr(v_scale), _stream(stream))
    if st != 0:
        raise PkvError(st, "pkv_kv_calibrate")


def pkv_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim=HEAD_DIM, max_seq_len=0, page_size=16,
                              max_ctas=0) -> int:
    """Workspace bytes of a decode call whose seq_lens are all <= max_seq_len."""
    return int(load().pkv_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, int(max_seq_len),
                                                page_size, max_ctas))


def pkv_paged_gqa_decode(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out, workspace,
                         sm_scale=None, device_error=None, max_ctas=0, stream=None, max_seq_len=0,
                         seq_page_sizes=None) -> None:
    """q bf16 [B, Hq, 128]; caches uint8 [num_pages, Hkv, P, 128]; scales fp32
    [Hkv]; block_table int32 [B, max_pages]; seq_lens int32 [B]; out
    [B, Hq, 128] bf16 or fp32; workspace uint8 (pkv_decode_workspace_size
    bytes for max_seq_len); seq_page_sizes int32 [B] or None (tokens per page
    of each sequence, a power-of-two multiple of P: runs of pool pages)."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.uint8, 4)
    _need(v_cache, "v_cache", torch.uint8, 4)
    _need(k_scale, "k_scale", torch.float32, 1)
    _need(v_scale, "v_scale", torch.float32, 1)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(out, "out", dim=3)
    _need(workspace, "workspace", torch.uint8)
    if device_error is not None:
        _need(device_error, "device_error", torch.int32)
    B, Hq, D = q.shape
    NP, Hkv, P, D2 = k_cache.shape
    if v_cache.shape != k_cache.shape or D2 != D or out.shape != q.shape:
        raise ValueError("q / cache / out shapes disagree")
    if block_table.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("block_table / seq_lens shapes disagree with q")
    _check_page_sizes(seq_page_sizes, B)
    _same_device(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out, workspace, device_error,
                 seq_page_sizes)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    with _device_of(q):
        st = load().pkv_paged_gqa_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                         _ptr(block_table), block_table.shape[1], _ptr(seq_lens), int(max_seq_len),
                                         _ptr(seq_page_sizes), B, Hq, Hkv, D, P, NP, float(sm_scale), _ptr(out),
                                         _act_code(out), _ptr(workspace), workspace.numel(), _ptr(device_error),
                                         int(max_ctas), _stream(stream))
    if st != 0:
        raise PkvError(st, "pkv_paged_gqa_decode")


def pkv_append_decode_fp8(k_new, v_new, q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out,
                          workspace, sm_scale=None, device_error=None, max_ctas=0, stream=None, max_seq_len=0,
                          seq_page_sizes=None) -> None:
    """One fused decode step: k_new/v_new [B, n_new, Hkv, 128] (fp32|bf16) are
    quantised into the cache at positions seq_lens[b] - n_new .. seq_lens[b] - 1
    (seq_lens counts them), then attention as pkv_paged_gqa_decode."""
    _need(k_new, "k_new", dim=4)
    _need(v_new, "v_new", dtype=k_new.dtype, dim=4)
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.uint8, 4)
    _need(v_cache, "v_cache", torch.uint8, 4)
    _need(k_scale, "k_scale", torch.float32, 1)
    _need(v_scale, "v_scale", torch.float32, 1)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(out, "out", dim=3)
    _need(workspace, "workspace", torch.uint8)
    if device_error is not None:
        _need(device_error, "device_error", torch.int32)
    B, Hq, D = q.shape
    NP, Hkv, P, D2 = k_cache.shape
    Bn, n_new, Hn, Dn = k_new.shape
    if v_cache.shape != k_cache.shape or D2 != D or out.shape != q.shape:
        raise ValueError("q / cache / out shapes disagree")
    if v_new.shape != k_new.shape or Bn != B or Hn != Hkv or Dn != D:
        raise ValueError("k_new / v_new must be [B, n_new, Hkv, head_dim]")
    if block_table.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("block_table / seq_lens shapes disagree with q")
    _check_page_sizes(seq_page_sizes, B)
    _same_device(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out, workspace, k_new, v_new,
                 device_error, seq_page_sizes)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    with _device_of(k_new):
        st = load().pkv_append_decode_fp8(_ptr(k_new), _ptr(v_new), _act_code(k_new), n_new, _ptr(q), _ptr(k_cache),
                                          _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_table),
                                          block_table.shape[1], _ptr(seq_lens), int(max_seq_len),
                                          _ptr(seq_page_sizes), B, Hq, Hkv, D, P, NP, float(sm_scale), _ptr(out),
                                          _act_code(out), _ptr(workspace), workspace.numel(), _ptr(device_error),
                                          int(max_ctas), _stream(stream))
    if st != 0:
        raise PkvError(st, "pkv_append_decode_fp8")


def append_decode_fp8(k_new, v_new, q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out=None,
                      out_dtype=torch.bfloat16, workspace=None, sm_scale=None, device_error=None, max_ctas=0,
                      stream=None, max_seq_len=0, seq_page_sizes=None) -> torch.Tensor:
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    max_seq_len = _default_max_len(block_table, k_cache, max_seq_len, seq_page_sizes)
    if workspace is None:
        workspace = decode_workspace(q.shape[0], q.shape[1], k_cache.shape[1], k_cache.shape[2], q.device,
                                     max_ctas, max_seq_len)
    pkv_append_decode_fp8(k_new, v_new, q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out,
                          workspace, sm_scale, device_error, max_ctas, stream, max_seq_len, seq_page_sizes)
    return out


def _default_max_len(block_table, k_cache, max_seq_len, seq_page_sizes):
    """The allocating forms bound seq_lens by the table's capacity at the pool
    page size unless told otherwise; with per-sequence page sizes the bound
    must be given."""
    if max_seq_len:
        return int(max_seq_len)
    if seq_page_sizes is not None:
        raise ValueError("give max_seq_len when seq_page_sizes is given")
    return int(block_table.shape[1] * k_cache.shape[2])


def pkv_paged_gqa_decode_noalloc(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out,
                                 sm_scale=None, device_error=None, max_ctas=0, stream=None, max_seq_len=0,
                                 seq_page_sizes=None) -> None:
    """pkv_paged_gqa_decode without a workspace, for callers that cannot
    allocate device memory: the split-K scratch is a fixed array inside the
    library (see pkv_decode_noalloc_scratch_bytes).  Calls that overlap on the
    GPU share that array and race; calls on one stream are safe."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.uint8, 4)
    _need(v_cache, "v_cache", torch.uint8, 4)
    _need(k_scale, "k_scale", torch.float32, 1)
    _need(v_scale, "v_scale", torch.float32, 1)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(out, "out", dim=3)
    if device_error is not None:
        _need(device_error, "device_error", torch.int32)
    B, Hq, D = q.shape
    NP, Hkv, P, D2 = k_cache.shape
    if v_cache.shape != k_cache.shape or D2 != D or out.shape != q.shape:
        raise ValueError("q / cache / out shapes disagree")
    if block_table.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("block_table / seq_lens shapes disagree with q")
    _check_page_sizes(seq_page_sizes, B)
    _same_device(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out, device_error, seq_page_sizes)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    with _device_of(q):
        st = load().pkv_paged_gqa_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                                 _ptr(v_scale), _ptr(block_table), block_table.shape[1],
                                                 _ptr(seq_lens), int(max_seq_len), _ptr(seq_page_sizes), B, Hq, Hkv,
                                                 D, P, NP, float(sm_scale), _ptr(out), _act_code(out),
                                                 _ptr(device_error), int(max_ctas), _stream(stream))
    if st != 0:
        raise PkvError(st, "pkv_paged_gqa_decode_noalloc")


def pkv_decode_noalloc_scratch_bytes() -> int:
    return int(load().pkv_decode_noalloc_scratch_bytes())


_ws_cache: dict = {}


def decode_workspace(batch, num_q_heads, num_kv_heads, page_size, device=None, max_ctas=0,
                     max_seq_len=0) -> torch.Tensor:
    """A workspace tensor for these sizes, cached per (device, stream, sizes).
    Calls that use it must not overlap on the GPU (same stream is fine)."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    stream = torch.cuda.current_stream(device).cuda_stream
    key = (device.index, stream, batch, num_q_heads, num_kv_heads, page_size, max_ctas, max_seq_len)
    ws = _ws_cache.get(key)
    if ws is None:
        with torch.cuda.device(device):
            n = pkv_decode_workspace_size(batch, num_q_heads, num_kv_heads, HEAD_DIM, max_seq_len, page_size,
                                          max_ctas)
        if n == 0:
            raise PkvError(4, "pkv_decode_workspace_size")
        ws = torch.empty(n, dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def kv_append_fp8(k_new, v_new, slot_mapping, k_scale, v_scale, k_cache, v_cache, device_error=None,
                  stream=None) -> None:
    pkv_kv_append_fp8(k_new, v_new, slot_mapping, k_scale, v_scale, k_cache, v_cache, device_error, stream)


def paged_gqa_decode(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out=None,
                     out_dtype=torch.bfloat16, workspace=None, sm_scale=None, device_error=None, max_ctas=0,
                     stream=None, max_seq_len=0, seq_page_sizes=None) -> torch.Tensor:
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    max_seq_len = _default_max_len(block_table, k_cache, max_seq_len, seq_page_sizes)
    if workspace is None:
        workspace = decode_workspace(q.shape[0], q.shape[1], k_cache.shape[1], k_cache.shape[2], q.device,
                                     max_ctas, max_seq_len)
    pkv_paged_gqa_decode(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out, workspace,
                         sm_scale, device_error, max_ctas, stream, max_seq_len, seq_page_sizes)
    return out


def pkv_prefill_workspace_size(batch, num_kv_heads, max_kv_len, max_total_kv=0) -> int:
    return int(load().pkv_prefill_workspace_size(int(batch), int(num_kv_heads), int(max_kv_len),
                                                 int(max_total_kv)))


def pkv_paged_prefill(q, cu_q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out, max_q_len,
                      max_kv_len, workspace, sm_scale=None, device_error=None, stream=None, max_total_kv=0,
                      seq_page_sizes=None) -> None:
    """q bf16 [total_q, Hq, 128] (the chunks of all sequences back to back);
    cu_q int32 [B + 1] row offsets; seq_lens int32 [B] (lengths including the
    chunk); caches, scales, block_table and seq_page_sizes as for decode; out
    [total_q, Hq, 128] bf16 or fp32; max_q_len / max_kv_len bounds of the
    chunk lengths and of seq_lens, max_total_kv (0 or) a bound of their sum;
    workspace uint8 (pkv_prefill_workspace_size bytes)."""
    _need(q, "q", torch.bfloat16, 3)
    _need(cu_q, "cu_q", torch.int32, 1)
    _need(k_cache, "k_cache", torch.uint8, 4)
    _need(v_cache, "v_cache", torch.uint8, 4)
    _need(k_scale, "k_scale", torch.float32, 1)
    _need(v_scale, "v_scale", torch.float32, 1)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(out, "out", dim=3)
    _need(workspace, "workspace", torch.uint8)
    if device_error is not None:
        _need(device_error, "device_error", torch.int32)
    T, Hq, D = q.shape
    NP, Hkv, P, D2 = k_cache.shape
    B = seq_lens.shape[0]
    if v_cache.shape != k_cache.shape or D2 != D or out.shape != q.shape:
        raise ValueError("q / cache / out shapes disagree")
    if block_table.shape[0] != B or cu_q.shape[0] != B + 1:
        raise ValueError("block_table / cu_q shapes disagree with seq_lens")
    _check_page_sizes(seq_page_sizes, B)
    _same_device(q, cu_q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out, workspace, device_error,
                 seq_page_sizes)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    with _device_of(q):
        st = load().pkv_paged_prefill(_ptr(q), _ptr(cu_q), T, int(max_q_len), _ptr(k_cache), _ptr(v_cache),
                                      _ptr(k_scale), _ptr(v_scale), _ptr(block_table), block_table.shape[1],
                                      _ptr(seq_lens), _ptr(seq_page_sizes), B, int(max_kv_len), int(max_total_kv),
                                      Hq, Hkv, D, P, NP, float(sm_scale), _ptr(out), _act_code(out),
                                      _ptr(workspace), workspace.numel(), _ptr(device_error), _stream(stream))
    if st != 0:
        raise PkvError(st, "pkv_paged_prefill")


def paged_prefill(q, cu_q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, max_q_len, out=None,
                  out_dtype=torch.bfloat16, max_kv_len=None, workspace=None, sm_scale=None, device_error=None,
                  stream=None, max_total_kv=0, seq_page_sizes=None) -> torch.Tensor:
    """Allocating convenience form: max_kv_len defaults to the block table's
    capacity (max_pages x page size; give it with seq_page_sizes), the
    workspace to a fresh buffer."""
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    if max_kv_len is None:
        if seq_page_sizes is not None:
            raise ValueError("give max_kv_len when seq_page_sizes is given")
        max_kv_len = block_table.shape[1] * k_cache.shape[2]
    if workspace is None:
        workspace = torch.empty(pkv_prefill_workspace_size(seq_lens.shape[0], k_cache.shape[1], max_kv_len,
                                                           max_total_kv), dtype=torch.uint8, device=q.device)
    pkv_paged_prefill(q, cu_q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out, max_q_len,
                      max_kv_len, workspace, sm_scale, device_error, stream, max_total_kv, seq_page_sizes)
    return out


__all__ = ["load", "lib_path", "pkv_kv_append_fp8", "pkv_paged_gqa_decode", "pkv_decode_workspace_size",
           "pkv_paged_gqa_decode_noalloc", "pkv_decode_noalloc_scratch_bytes", "pkv_append_decode_fp8",
           "append_decode_fp8", "pkv_kv_calibrate", "pkv_paged_prefill", "paged_prefill", "pkv_prefill_workspace_size",
           "pkv_status_string", "pkv_version", "pkv_read_device_error", "pkv_test_withhold_load", "kv_append_fp8",
           "paged_gqa_decode", "decode_workspace", "pkv_decode_set_split_weights", "pkv_decode_get_split_weights",
           "pkv_decode_calibrate_split",
           "PkvError", "PKV_F32", "PKV_BF16", "DEVERR_SLOT", "DEVERR_PAGE", "DEVERR_SEQLEN",
           "DEVERR_TIMEOUT", "DEVERR_PAGESIZE", "DEVERR_INTERNAL", "pkv_last_cuda_error"]
