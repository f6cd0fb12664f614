"""paged_kv_flash_cache_gb300 -- attention over a paged KV cache on NVIDIA GB300 (sm_103a).

A thin Python binding over the C ABI of libpkv (include/pkv.h). Every step of the
computation runs in the library's CUDA kernels; this module only checks tensor
shapes, dtypes and devices, allocates outputs / workspace with PyTorch when the
caller does not pass them, and forwards raw device pointers and the current CUDA
stream. There is no CPU fallback: if the library is missing every call raises.

Entry points (same names as the C ABI without the ``pkv_`` prefix):
  kv_cache_append, paged_attn_decode, paged_attn_decode_step, paged_attn_prefill, paged_attn_mixed,
  attn_combine, decode_workspace_size, decode_split_tokens, get_device_error.
Cache tensors have shape [num_blocks, 2, num_kv_heads, block_size, head_dim]
(K at index 0, V at index 1) in float16 or bfloat16, or hold FP8 E4M3 codes
(torch.float8_e4m3fn or uint8) with a float32 `scales` tensor
[num_blocks, 2, num_kv_heads, block_size], one scale per cached row; q, k_new and
v_new then stay float16 / bfloat16 (see pkv_kv_format in include/pkv.h).
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional

__all__ = [
    "PkvError", "library_path", "load_library", "kv_cache_append", "paged_attn_decode", "paged_attn_prefill",
    "attn_combine", "decode_workspace_size", "decode_split_tokens", "get_device_error", "STATUS",
    "paged_attn_decode_noalloc", "paged_attn_mixed", "selftest_wait_timeout", "paged_attn_decode_step",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_lib", "libpkv.so")
_lock = threading.Lock()
_lib = None

STATUS = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED", 3: "PKV_ERR_WORKSPACE",
          4: "PKV_ERR_CUDA", 5: "PKV_ERR_DEVICE_RANGE", 6: "PKV_ERR_TIMEOUT"}
F16, BF16, F32 = 0, 1, 2
KV_NATIVE, KV_FP8_E4M3 = 0, 1

# Every symbol include/pkv.h declares.
EXPORTS = ("pkv_kv_cache_append", "pkv_decode_workspace_size", "pkv_decode_split_tokens", "pkv_paged_attn_decode",
           "pkv_paged_attn_decode_step", "pkv_paged_attn_decode_noalloc", "pkv_paged_attn_prefill", "pkv_paged_attn_mixed", "pkv_attn_combine",
           "pkv_get_device_error", "pkv_selftest_wait_timeout", "pkv_status_string", "pkv_version")
DECODE_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024   # PKV_DECODE_NOALLOC_SCRATCH_BYTES in include/pkv.h


class PkvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (where, STATUS.get(status, "unknown"), status))


class _Cache(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("num_blocks", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
                ("block_size", ctypes.c_int), ("head_dim", ctypes.c_int), ("dtype", ctypes.c_int),
                ("format", ctypes.c_int), ("scales", ctypes.c_void_p)]


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libpkv.so (built in-tree by paged_kv_flash_cache_gb300.build). Raises if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError("libpkv.so is not built (%s); run `python -m paged_kv_flash_cache_gb300.build` or "
                               "__graft_entry__.build()" % _LIB_PATH)
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.pkv_kv_cache_append.argtypes = [_Cache, P, P, P, P, P, I, I, I, P]
        lib.pkv_kv_cache_append.restype = I
        lib.pkv_decode_workspace_size.argtypes = [I, I, I, I, I, I, I]
        lib.pkv_decode_workspace_size.restype = Z
        lib.pkv_decode_split_tokens.argtypes = [I, I, I, I, I, I, I]
        lib.pkv_decode_split_tokens.restype = I
        lib.pkv_paged_attn_decode.argtypes = [_Cache, P, I, P, P, I, I, F, I, P, Z, P, I, P, P]
        lib.pkv_paged_attn_decode.restype = I
        lib.pkv_paged_attn_decode_step.argtypes = [_Cache, P, I, P, P, I, I, F, I, P, Z, P, I, P, P, P, P]
        lib.pkv_paged_attn_decode_step.restype = I
        lib.pkv_paged_attn_decode_noalloc.argtypes = [_Cache, P, I, P, P, I, I, F, I, P, I, P, P]
        lib.pkv_paged_attn_decode_noalloc.restype = I
        lib.pkv_paged_attn_prefill.argtypes = [_Cache, P, I, P, P, P, I, I, I, I, F, I, P, I, P, P]
        lib.pkv_paged_attn_prefill.restype = I
        lib.pkv_paged_attn_mixed.argtypes = [_Cache, P, I, P, P, P, I, I, I, I, F, I, I, P, Z, P, I, P, P]
        lib.pkv_paged_attn_mixed.restype = I
        lib.pkv_attn_combine.argtypes = [P, P, I, I, I, P, I, P, P]
        lib.pkv_attn_combine.restype = I
        lib.pkv_selftest_wait_timeout.argtypes = [ctypes.c_uint, P]
        lib.pkv_selftest_wait_timeout.restype = I
        lib.pkv_get_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_int)]
        lib.pkv_get_device_error.restype = I
        lib.pkv_status_string.argtypes = [I]
        lib.pkv_status_string.restype = ctypes.c_char_p
        lib.pkv_version.argtypes = []
        lib.pkv_version.restype = I
        _lib = lib
        return lib


# ---------------------------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _dtype_code(dt) -> int:
    torch = _torch()
    if dt == torch.float16:
        return F16
    if dt == torch.bfloat16:
        return BF16
    if dt == torch.float32:
        return F32
    raise TypeError("unsupported dtype %s" % dt)


def _dev(t, name):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor (there is no CPU path)" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return ctypes.c_void_p(t.data_ptr())


def _i32(t, name):
    torch = _torch()
    if t.dtype != torch.int32:
        raise TypeError("%s must be int32" % name)
    return _dev(t, name)


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def is_fp8_cache(cache) -> bool:
    torch = _torch()
    return cache.dtype == torch.uint8 or cache.dtype == getattr(torch, "float8_e4m3fn", None)


def _cache_struct(cache, act_dtype, scales=None) -> _Cache:
    """The C view of `cache`; act_dtype is the type of q / k_new / v_new."""
    torch = _torch()
    if cache.dim() != 5 or cache.shape[1] != 2:
        raise ValueError("cache must be [num_blocks, 2, num_kv_heads, block_size, head_dim]")
    nb, _, hkv, bs, d = cache.shape
    if is_fp8_cache(cache):
        if scales is None or scales.dtype != torch.float32 or tuple(scales.shape) != (nb, 2, hkv, bs):
            raise ValueError("an FP8 cache needs float32 scales [num_blocks, 2, num_kv_heads, block_size]")
        return _Cache(_dev(cache, "cache"), nb, hkv, bs, d, _dtype_code(act_dtype), KV_FP8_E4M3,
                      _dev(scales, "scales"))
    if scales is not None:
        raise ValueError("scales are only for an FP8 cache")
    if act_dtype != cache.dtype:
        raise TypeError("q / k_new / v_new must have the cache dtype")
    return _Cache(_dev(cache, "cache"), nb, hkv, bs, d, _dtype_code(cache.dtype), KV_NATIVE, None)


def _check(status: int, where: str):
    if status != 0:
        raise PkvError(status, where)


# ---------------------------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------------------------

def kv_cache_append(cache, k_new, v_new, cu_new_lens, ctx_before, block_tables, stream=None, scales=None) -> None:
    """Scatter new tokens' K/V ([T_new, Hkv, D], packed by sequence) into their pages (an FP8
    cache: quantised, with their row scales written to `scales`)."""
    lib = load_library()
    if k_new.dtype != v_new.dtype or k_new.shape != v_new.shape:
        raise TypeError("k_new / v_new must match each other")
    c = _cache_struct(cache, k_new.dtype, scales)
    batch, mb = block_tables.shape
    _check(lib.pkv_kv_cache_append(c, _dev(k_new, "k_new"), _dev(v_new, "v_new"), _i32(cu_new_lens, "cu_new_lens"),
                                   _i32(ctx_before, "ctx_before"), _i32(block_tables, "block_tables"), batch, mb,
                                   int(k_new.shape[0]), _stream(stream)), "pkv_kv_cache_append")


def decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                          num_splits=0) -> int:
    return int(load_library().pkv_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, block_size,
                                                        max_blocks_per_seq, num_splits))


def decode_split_tokens(batch, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                        num_splits=0) -> int:
    return int(load_library().pkv_decode_split_tokens(batch, num_q_heads, num_kv_heads, head_dim, block_size,
                                                      max_blocks_per_seq, num_splits))


def paged_attn_decode(cache, q, block_tables, context_lens, scale: Optional[float] = None, num_splits: int = 0,
                      workspace=None, out=None, out_dtype=None, lse=None, stream=None, scales=None):
    """One query per sequence ([B, Hq, D]) against its paged context. Returns `out`."""
    torch = _torch()
    lib = load_library()
    c = _cache_struct(cache, q.dtype, scales)
    batch, hq, d = q.shape
    mb = block_tables.shape[1]
    if out is None:
        out = torch.empty((batch, hq, d), dtype=out_dtype or q.dtype, device=q.device)
    need = decode_workspace_size(batch, hq, cache.shape[2], d, cache.shape[3], mb, num_splits)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    scale = (1.0 / math.sqrt(d)) if scale is None else float(scale)
    _check(lib.pkv_paged_attn_decode(c, _dev(q, "q"), hq, _i32(block_tables, "block_tables"),
                                     _i32(context_lens, "context_lens"), batch, mb, scale, int(num_splits),
                                     _dev(workspace, "workspace"), ws_bytes, _dev(out, "out"),
                                     _dtype_code(out.dtype), _dev(lse, "lse"), _stream(stream)),
           "pkv_paged_attn_decode")
    return out


def paged_attn_decode_step(cache, q, block_tables, context_lens, k_new, v_new, scale: Optional[float] = None,
                           num_splits: int = 0, workspace=None, out=None, out_dtype=None, lse=None, stream=None,
                           scales=None):
    """One decode step: paged_attn_decode over context_lens[b] cached tokens, and the step's new
    token (k_new / v_new [B, Hkv, D]) written at position context_lens[b]. Returns `out`."""
    torch = _torch()
    lib = load_library()
    if k_new.dtype != q.dtype or v_new.dtype != q.dtype or k_new.shape != v_new.shape:
        raise TypeError("k_new / v_new must match each other and q's dtype")
    c = _cache_struct(cache, q.dtype, scales)
    batch, hq, d = q.shape
    if tuple(k_new.shape) != (batch, cache.shape[2], d):
        raise ValueError("k_new / v_new must be [batch, num_kv_heads, head_dim]")
    mb = block_tables.shape[1]
    if out is None:
        out = torch.empty((batch, hq, d), dtype=out_dtype or q.dtype, device=q.device)
    need = decode_workspace_size(batch, hq, cache.shape[2], d, cache.shape[3], mb, num_splits)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    scale = (1.0 / math.sqrt(d)) if scale is None else float(scale)
    _check(lib.pkv_paged_attn_decode_step(c, _dev(q, "q"), hq, _i32(block_tables, "block_tables"),
                                          _i32(context_lens, "context_lens"), batch, mb, scale, int(num_splits),
                                          _dev(workspace, "workspace"), ws_bytes, _dev(out, "out"),
                                          _dtype_code(out.dtype), _dev(lse, "lse"), _dev(k_new, "k_new"),
                                          _dev(v_new, "v_new"), _stream(stream)),
           "pkv_paged_attn_decode_step")
    return out


def paged_attn_decode_noalloc(cache, q, block_tables, context_lens, scale: Optional[float] = None,
                              num_splits: int = 0, out=None, out_dtype=None, lse=None, stream=None, scales=None):
    """paged_attn_decode without a workspace: for callers that cannot allocate device memory.
    The split partials go to a fixed array the library holds on each device (see
    include/pkv.h); sizes needing more than DECODE_NOALLOC_SCRATCH_BYTES raise PkvError
    (PKV_ERR_WORKSPACE). Calls sharing a device must not overlap on the GPU. Returns `out`
    (allocated here with PyTorch only when the caller passes none)."""
    torch = _torch()
    lib = load_library()
    c = _cache_struct(cache, q.dtype, scales)
    batch, hq, d = q.shape
    mb = block_tables.shape[1]
    if out is None:
        out = torch.empty((batch, hq, d), dtype=out_dtype or q.dtype, device=q.device)
    scale = (1.0 / math.sqrt(d)) if scale is None else float(scale)
    _check(lib.pkv_paged_attn_decode_noalloc(c, _dev(q, "q"), hq, _i32(block_tables, "block_tables"),
                                             _i32(context_lens, "context_lens"), batch, mb, scale, int(num_splits),
                                             _dev(out, "out"), _dtype_code(out.dtype), _dev(lse, "lse"),
                                             _stream(stream)), "pkv_paged_attn_decode_noalloc")
    return out


def paged_attn_prefill(cache, q, cu_q_lens, context_lens, block_tables, max_q_len: int,
                       scale: Optional[float] = None, causal: bool = True, out=None, out_dtype=None, lse=None,
                       stream=None, scales=None):
    """A chunk of queries per sequence ([sum q_len, Hq, D]) against its paged context
    (the chunk's own K/V already appended). Returns `out`. An FP8 cache (pass `scales`) needs
    head_dim 128; with head_dim 64 it raises PkvError (PKV_ERR_UNSUPPORTED)."""
    torch = _torch()
    lib = load_library()
    c = _cache_struct(cache, q.dtype, scales)
    total_q, hq, d = q.shape
    batch, mb = block_tables.shape
    if out is None:
        out = torch.empty((total_q, hq, d), dtype=out_dtype or q.dtype, device=q.device)
    scale = (1.0 / math.sqrt(d)) if scale is None else float(scale)
    _check(lib.pkv_paged_attn_prefill(c, _dev(q, "q"), hq, _i32(cu_q_lens, "cu_q_lens"),
                                      _i32(context_lens, "context_lens"), _i32(block_tables, "block_tables"), batch,
                                      mb, total_q, int(max_q_len), scale, 1 if causal else 0, _dev(out, "out"),
                                      _dtype_code(out.dtype), _dev(lse, "lse"), _stream(stream)),
           "pkv_paged_attn_prefill")
    return out


def paged_attn_mixed(cache, q, cu_q_lens, context_lens, block_tables, max_q_len: int,
                     scale: Optional[float] = None, causal: bool = True, num_splits: int = 0, workspace=None,
                     out=None, out_dtype=None, lse=None, stream=None, scales=None):
    """One call over a batch mixing decode rows (q_len 1) and prefill chunks (q_len > 1):
    q [sum q_len, Hq, D], rows by cu_q_lens. Returns `out`."""
    torch = _torch()
    lib = load_library()
    c = _cache_struct(cache, q.dtype, scales)
    total_q, hq, d = q.shape
    batch, mb = block_tables.shape
    if out is None:
        out = torch.empty((total_q, hq, d), dtype=out_dtype or q.dtype, device=q.device)
    need = decode_workspace_size(batch, hq, cache.shape[2], d, cache.shape[3], mb, num_splits)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    scale = (1.0 / math.sqrt(d)) if scale is None else float(scale)
    _check(lib.pkv_paged_attn_mixed(c, _dev(q, "q"), hq, _i32(cu_q_lens, "cu_q_lens"), _i32(context_lens, "context_lens"),
                                    _i32(block_tables, "block_tables"), batch, mb, total_q, int(max_q_len), scale,
                                    1 if causal else 0, int(num_splits), _dev(workspace, "workspace"), ws_bytes,
                                    _dev(out, "out"), _dtype_code(out.dtype), _dev(lse, "lse"), _stream(stream)),
           "pkv_paged_attn_mixed")
    return out


def attn_combine(partial_o, partial_lse, out=None, out_dtype=None, lse=None, stream=None):
    """Merge FP32 split partials [N, S, D] with their lse [N, S]. Returns `out` [N, D]."""
    torch = _torch()
    lib = load_library()
    n, s, d = partial_o.shape
    if out is None:
        out = torch.empty((n, d), dtype=out_dtype or torch.float32, device=partial_o.device)
    _check(lib.pkv_attn_combine(_dev(partial_o, "partial_o"), _dev(partial_lse, "partial_lse"), n, s, d,
                                _dev(out, "out"), _dtype_code(out.dtype), _dev(lse, "lse"), _stream(stream)),
           "pkv_attn_combine")
    return out


def selftest_wait_timeout(timeout_us: int = 20000, stream=None) -> None:
    """Launch one warp that waits on a barrier nothing completes, bounded by timeout_us; the
    device error word then holds PKV_ERR_TIMEOUT (read it with get_device_error)."""
    _check(load_library().pkv_selftest_wait_timeout(int(timeout_us), _stream(stream)), "pkv_selftest_wait_timeout")


def get_device_error(stream=None) -> int:
    """Synchronise the stream, then read and clear the device error word (0 = none)."""
    lib = load_library()
    code = ctypes.c_int(0)
    _check(lib.pkv_get_device_error(_stream(stream), ctypes.byref(code)), "pkv_get_device_error")
    return int(code.value)
