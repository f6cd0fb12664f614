"""CPU oracle for attention over a paged KV cache -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import this module. The library never calls it, and it shares no code
with the CUDA path: `oracle.c` is plain double-precision C compiled with gcc,
wrapped here with ctypes. Inputs are numpy arrays; fp16 / bf16 tensors are
passed as their raw 16-bit patterns (uint16) and converted exactly to double
inside the C code.

Functions and the passages they follow (page titles of the subject's web pages):
  * kv_cache_append -- the decode step appends the new token's K and V to the
    cache ("为什么Attention是O(n²)", prefill / decode section), at block
    block_table[i // block_size], offset i % block_size ("企业官网建设流程全解析",
    section 2.1), in the layout [num_blocks, 2, num_heads, block_size, head_dim]
    ("Flash Attention与Paged Attention如何共同优化大模型推理？", section 3).
  * paged_attention -- softmax(Q K^T / sqrt(d)) V ("为什么Attention是O(n²)",
    mathematics section) by a token walk through the block table and an explicit
    two-pass softmax; causal masking as the library call's `is_causal`
    ("Flash Attention与Paged Attention...", section 2), bottom-right aligned.
  * attn_combine -- log-sum-exp merge of split partial results; the rescale
    identity is the one of the online-softmax update in section 2 of the
    ipipp.com page (old terms scaled by exp(m_old - m_new)).
  * e4m3_encode / e4m3_decode, kv_cache_append_fp8, paged_attention_fp8 -- the
    FP8 cache: the "KV cache compression" the answer.freetools.me page names
    without a scheme, read as one FP32 scale per cached row (amax / 448) and OCP
    FP8 E4M3 codes (round to nearest even, saturating); attention over the
    exactly dequantised values.
Pins (tests/test_oracle_pins.py) tie every function to closed forms,
invariants and a library routine; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import NamedTuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

DTYPE_CODE = {"f16": 0, "bf16": 1}


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (no FP contraction, so x86 and Arm agree)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
               "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            L = ctypes.c_long
            D = ctypes.c_double
            lib.oracle_kv_cache_append.argtypes = [P, I, I, I, I, P, P, P, P, P, I, I]
            lib.oracle_kv_cache_append.restype = I
            lib.oracle_paged_attention.argtypes = [I, P, I, I, I, I, P, I, P, P, P, I, I, D, I, P, L, P, P, I]
            lib.oracle_paged_attention.restype = I
            lib.oracle_attn_combine.argtypes = [P, P, L, I, I, P, P]
            lib.oracle_attn_combine.restype = I
            lib.oracle_e4m3_encode.argtypes = [P, P, L]
            lib.oracle_e4m3_encode.restype = None
            lib.oracle_e4m3_decode.argtypes = [P, P, L]
            lib.oracle_e4m3_decode.restype = None
            lib.oracle_kv_cache_append_fp8.argtypes = [P, P, I, I, I, I, I, P, P, P, P, P, I, I]
            lib.oracle_kv_cache_append_fp8.restype = I
            lib.oracle_paged_attention_fp8.argtypes = [I, P, P, I, I, I, I, P, I, P, P, P, I, I, D, I, P, L, P, P, I]
            lib.oracle_paged_attention_fp8.restype = I
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    """fp16/bf16 torch tensor or uint16 ndarray -> contiguous uint16 ndarray of the same bits."""
    if isinstance(a, np.ndarray):
        assert a.dtype == np.uint16
        return np.ascontiguousarray(a)
    import torch
    assert a.dtype in (torch.float16, torch.bfloat16, torch.int16, torch.uint16)
    return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _i32(a) -> np.ndarray:
    if not isinstance(a, np.ndarray):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def kv_cache_append(cache_bits: np.ndarray, k_new, v_new, cu_new_lens, ctx_before, block_tables) -> int:
    """In-place append into `cache_bits` (uint16 [NB, 2, Hkv, bs, D]). Returns the C status."""
    assert cache_bits.dtype == np.uint16 and cache_bits.flags.c_contiguous and cache_bits.ndim == 5
    nb, two, hkv, bs, d = cache_bits.shape
    assert two == 2
    k = _u16(k_new)
    v = _u16(v_new)
    cu = _i32(cu_new_lens)
    cb = _i32(ctx_before)
    bt = _i32(block_tables)
    batch, mb = bt.shape
    assert k.shape == v.shape and k.size == int(cu[-1]) * hkv * d
    return _load().oracle_kv_cache_append(_ptr(cache_bits), nb, hkv, bs, d, _ptr(k), _ptr(v), _ptr(cu), _ptr(cb),
                                          _ptr(bt), batch, mb)


def paged_attention(dtype: str, cache_bits: np.ndarray, q, num_q_heads: int, cu_q_lens, context_lens,
                    block_tables, scale: float, causal: bool, rows=None, nthreads: int = 0):
    """Attention of the selected query rows (all by default) against the paged cache.

    Returns (out [n, Hq, D] float64, lse [n, Hq] float64). Raises on a bad page id."""
    nb, two, hkv, bs, d = cache_bits.shape
    qb = _u16(q)
    cu = _i32(cu_q_lens)
    cl = _i32(context_lens)
    bt = _i32(block_tables)
    batch, mb = bt.shape
    total_rows = int(cu[-1])
    sel = None
    if rows is not None:
        sel = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = int(sel.size)
    else:
        n = total_rows
    out = np.zeros((n, num_q_heads, d), dtype=np.float64)
    lse = np.zeros((n, num_q_heads), dtype=np.float64)
    if nthreads <= 0:
        nthreads = os.cpu_count() or 1
    rc = _load().oracle_paged_attention(DTYPE_CODE[dtype], _ptr(cache_bits), nb, hkv, bs, d, _ptr(qb),
                                        num_q_heads, _ptr(cu), _ptr(cl), _ptr(bt), batch, mb, float(scale),
                                        1 if causal else 0, _ptr(sel), n, _ptr(out), _ptr(lse), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_paged_attention: status %d (bad page id, table slot or row)" % rc)
    return out, lse


def attn_combine(partial_o: np.ndarray, partial_lse: np.ndarray):
    """Merge [N, S, D] partial outputs with [N, S] partial lse. Returns (out [N, D], lse [N])."""
    po = np.ascontiguousarray(partial_o, dtype=np.float64)
    pl = np.ascontiguousarray(partial_lse, dtype=np.float64)
    n, s, d = po.shape
    assert pl.shape == (n, s)
    out = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    _load().oracle_attn_combine(_ptr(po), _ptr(pl), n, s, d, _ptr(out), _ptr(lse))
    return out, lse


class Fp8Cache(NamedTuple):
    """An FP8 cache on the host: E4M3 codes uint8 [NB, 2, Hkv, bs, D], scales float32 [NB, 2, Hkv, bs]."""
    codes: np.ndarray
    scales: np.ndarray


def e4m3_encode(x) -> np.ndarray:
    """float32 values -> E4M3 codes (round to nearest even, saturating to +-448)."""
    xf = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.zeros(xf.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode(_ptr(xf), _ptr(out), int(xf.size))
    return out


def e4m3_decode(codes) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.zeros(c.shape, dtype=np.float64)
    _load().oracle_e4m3_decode(_ptr(c), _ptr(out), int(c.size))
    return out


def kv_cache_append_fp8(cache: Fp8Cache, dtype: str, k_new, v_new, cu_new_lens, ctx_before, block_tables) -> int:
    """In-place quantising append into an Fp8Cache (k_new / v_new in `dtype`). Returns the C status."""
    codes, scales = cache
    assert codes.dtype == np.uint8 and codes.flags.c_contiguous and codes.ndim == 5
    assert scales.dtype == np.float32 and scales.flags.c_contiguous and scales.shape == codes.shape[:4]
    nb, two, hkv, bs, d = codes.shape
    k = _u16(k_new)
    v = _u16(v_new)
    cu = _i32(cu_new_lens)
    cb = _i32(ctx_before)
    bt = _i32(block_tables)
    batch, mb = bt.shape
    assert k.shape == v.shape and k.size == int(cu[-1]) * hkv * d
    return _load().oracle_kv_cache_append_fp8(_ptr(codes), _ptr(scales), nb, hkv, bs, d, DTYPE_CODE[dtype], _ptr(k),
                                              _ptr(v), _ptr(cu), _ptr(cb), _ptr(bt), batch, mb)


def paged_attention_fp8(dtype: str, cache: Fp8Cache, q, num_q_heads: int, cu_q_lens, context_lens, block_tables,
                        scale: float, causal: bool, rows=None, nthreads: int = 0):
    """paged_attention over an FP8 cache (q in `dtype`). Returns (out, lse) as float64."""
    codes, scales = cache
    nb, two, hkv, bs, d = codes.shape
    qb = _u16(q)
    cu = _i32(cu_q_lens)
    cl = _i32(context_lens)
    bt = _i32(block_tables)
    batch, mb = bt.shape
    sel = None
    if rows is not None:
        sel = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = int(sel.size)
    else:
        n = int(cu[-1])
    out = np.zeros((n, num_q_heads, d), dtype=np.float64)
    lse = np.zeros((n, num_q_heads), dtype=np.float64)
    if nthreads <= 0:
        nthreads = os.cpu_count() or 1
    rc = _load().oracle_paged_attention_fp8(DTYPE_CODE[dtype], _ptr(np.ascontiguousarray(codes)),
                                            _ptr(np.ascontiguousarray(scales)), nb, hkv, bs, d, _ptr(qb),
                                            num_q_heads, _ptr(cu), _ptr(cl), _ptr(bt), batch, mb, float(scale),
                                            1 if causal else 0, _ptr(sel), n, _ptr(out), _ptr(lse), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_paged_attention_fp8: status %d (bad page id, table slot or row)" % rc)
    return out, lse


def empty_cache_bits(problem) -> np.ndarray:
    """The pool as uint16 bits (an Fp8Cache for an FP8 problem), starting from the problem's
    seeded noise (or zeros)."""
    shape = (problem.num_blocks, 2, problem.num_kv_heads, problem.block_size, problem.head_dim)
    if getattr(problem, "kv_format", "native") == "fp8":
        if problem.pool_init is None:
            return Fp8Cache(np.zeros(shape, dtype=np.uint8), np.zeros(shape[:4], dtype=np.float32))
        codes, scales = problem.pool_init
        return Fp8Cache(np.ascontiguousarray(codes.cpu().numpy().reshape(shape)).copy(),
                        np.ascontiguousarray(scales.cpu().numpy().reshape(shape[:4])).copy())
    if problem.pool_init is None:
        return np.zeros(shape, dtype=np.uint16)
    return _u16(problem.pool_init).reshape(shape).copy()


def build_cache(problem) -> np.ndarray:
    """Pool bits after appending every context token of `problem` (ctx_before = 0)."""
    import torch
    cache = empty_cache_bits(problem)
    if isinstance(cache, Fp8Cache):
        rc = kv_cache_append_fp8(cache, problem.dtype, problem.k_ctx, problem.v_ctx, problem.cu_ctx_lens,
                                 torch.zeros(problem.batch, dtype=torch.int32), problem.block_tables)
    else:
        rc = kv_cache_append(cache, problem.k_ctx, problem.v_ctx, problem.cu_ctx_lens,
                             torch.zeros(problem.batch, dtype=torch.int32), problem.block_tables)
    if rc != 0:
        raise ValueError("oracle append failed: %d" % rc)
    return cache


def attention_of(problem, cache_bits: np.ndarray, rows=None, nthreads: int = 0, q=None, cu_q_lens=None,
                 context_lens=None):
    """paged_attention with a problem's own tensors (optionally overriding q / lengths)."""
    if isinstance(cache_bits, Fp8Cache):
        return paged_attention_fp8(problem.dtype, cache_bits, problem.q if q is None else q, problem.num_q_heads,
                                   problem.cu_q_lens if cu_q_lens is None else cu_q_lens,
                                   problem.context_lens if context_lens is None else context_lens,
                                   problem.block_tables, problem.scale, problem.causal, rows=rows, nthreads=nthreads)
    return paged_attention(problem.dtype, cache_bits, problem.q if q is None else q, problem.num_q_heads,
                           problem.cu_q_lens if cu_q_lens is None else cu_q_lens,
                           problem.context_lens if context_lens is None else context_lens,
                           problem.block_tables, problem.scale, problem.causal, rows=rows, nthreads=nthreads)
