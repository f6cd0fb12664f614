"""The C-ABI library builds, loads without a GPU and exports every symbol include/pkv.h
declares; host-side validation rejects bad calls before anything is launched."""
import ctypes
import os
import re

import pytest

import paged_kv_flash_cache_gb300 as pkv
from paged_kv_flash_cache_gb300 import build as pkv_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pkv.h")


@pytest.fixture(scope="module")
def lib():
    pkv_build.build()
    return pkv.load_library()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_symbols() == sorted(pkv.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert lib.pkv_version() == 101
    assert lib.pkv_status_string(0) == b"PKV_OK"
    assert lib.pkv_status_string(3) == b"PKV_ERR_WORKSPACE"


def test_only_c_abi_symbols_are_exported(lib):
    """Internal C++ symbols stay hidden (-fvisibility=hidden); nm lists the dynamic exports."""
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", pkv.library_path()], capture_output=True, text=True).stdout
    ours = sorted({l.split()[-1] for l in out.splitlines() if " T " in l and l.split()[-1].startswith("pkv_")})
    assert ours == sorted(pkv.EXPORTS)


def _cache(ptr=16, nb=4, hkv=2, bs=16, d=128, dt=0, fmt=0, scales=None):
    return pkv._Cache(ctypes.c_void_p(ptr), nb, hkv, bs, d, dt, fmt, None if scales is None else ctypes.c_void_p(scales))


def test_host_validation_without_gpu(lib):
    P = ctypes.c_void_p
    good = P(4096)
    # null cache pointer
    assert lib.pkv_kv_cache_append(_cache(ptr=0), good, good, good, good, good, 1, 4, 3, None) == 1
    # misaligned cache pointer
    assert lib.pkv_kv_cache_append(_cache(ptr=4098), good, good, good, good, good, 1, 4, 3, None) == 1
    # unsupported head_dim / block_size / dtype
    assert lib.pkv_kv_cache_append(_cache(d=96), good, good, good, good, good, 1, 4, 3, None) == 2
    assert lib.pkv_kv_cache_append(_cache(bs=24), good, good, good, good, good, 1, 4, 3, None) == 2
    assert lib.pkv_kv_cache_append(_cache(bs=1024), good, good, good, good, good, 1, 4, 3, None) == 2
    assert lib.pkv_kv_cache_append(_cache(dt=2), good, good, good, good, good, 1, 4, 3, None) == 2
    # negative sizes
    assert lib.pkv_kv_cache_append(_cache(), good, good, good, good, good, -1, 4, 3, None) == 1
    # nothing to do is fine and launches nothing
    assert lib.pkv_kv_cache_append(_cache(), good, good, good, good, good, 1, 4, 0, None) == 0
    # decode: Hq not a multiple of Hkv, group unsupported over an FP8 cache, out dtype (a native
    # cache takes any group; nothing here reaches a launch)
    F = ctypes.c_float
    args = lambda hq, out_dt=0: (_cache(), good, hq, good, good, 2, 4, F(0.1), 0, good, 1 << 20, good, out_dt, None,
                                 None)
    fp8_args = lambda hq: (_cache(fmt=1, scales=4096), good, hq, good, good, 2, 4, F(0.1), 0, good, 1 << 20, good, 0,
                           None, None)
    assert lib.pkv_paged_attn_decode(*args(3)) == 1
    assert lib.pkv_paged_attn_decode(*fp8_args(6)) == 2      # group 3
    assert lib.pkv_paged_attn_decode(*fp8_args(20)) == 2     # group 10: not a multiple of 8
    # FP8 cache with head_dim 64: groups above 8 are not supported
    fp8_64 = (_cache(fmt=1, scales=4096, d=64), good, 32, good, good, 2, 4, F(0.1), 0, good, 1 << 20, good, 0, None,
              None)
    assert lib.pkv_paged_attn_decode(*fp8_64) == 2
    assert lib.pkv_paged_attn_decode(*args(2, out_dt=1)) == 2   # bf16 out for an fp16 cache
    # decode step: the new token's K and V are required (and 16-byte aligned) when batch > 0; a
    # step whose decode is refused is refused whole
    step = lambda hq, k, v: args(hq)[:-1] + (k, v, None)
    assert lib.pkv_paged_attn_decode_step(*step(2, None, good)) == 1
    assert lib.pkv_paged_attn_decode_step(*step(2, good, P(4100))) == 1
    assert lib.pkv_paged_attn_decode_step(*step(3, good, good)) == 1
    assert lib.pkv_paged_attn_decode_step(*(fp8_args(6)[:-1] + (good, good, None))) == 2
    # prefill: negative total_q
    assert lib.pkv_paged_attn_prefill(_cache(), good, 2, good, good, good, 1, 4, -1, 4, F(0.1), 1, good, 0, None,
                                      None) == 1
    # prefill grid (heads, sequences, 256-row blocks): more than 65535 sequences or row blocks
    assert lib.pkv_paged_attn_prefill(_cache(), good, 2, good, good, good, 65536, 4, 65536, 1, F(0.1), 1, good, 0,
                                      None, None) == 2
    assert lib.pkv_paged_attn_prefill(_cache(), good, 2, good, good, good, 1, 4, 1 << 25, 1 << 25, F(0.1), 1, good,
                                      0, None, None) == 2
    # head_dim 256 runs 128-row blocks: 65537 of them are too many
    assert lib.pkv_paged_attn_prefill(_cache(d=256), good, 2, good, good, good, 1, 4, (1 << 23) + 1, (1 << 23) + 1,
                                      F(0.1), 1, good, 0, None, None) == 2
    # combine: bad head_dim, bad split count
    assert lib.pkv_attn_combine(good, good, 4, 2, 96, good, 2, None, None) == 2
    assert lib.pkv_attn_combine(good, good, 4, 0, 128, good, 2, None, None) == 1


def test_fp8_cache_validation_without_gpu(lib):
    P = ctypes.c_void_p
    F = ctypes.c_float
    good = P(4096)
    # FP8 cache without scales, with misaligned scales, with an unknown format
    assert lib.pkv_kv_cache_append(_cache(fmt=1), good, good, good, good, good, 1, 4, 3, None) == 1
    assert lib.pkv_kv_cache_append(_cache(fmt=1, scales=4100), good, good, good, good, good, 1, 4, 3, None) == 1
    assert lib.pkv_kv_cache_append(_cache(fmt=7, scales=4096), good, good, good, good, good, 1, 4, 3, None) == 2
    # nothing to append: accepted, nothing launched
    assert lib.pkv_kv_cache_append(_cache(fmt=1, scales=4096), good, good, good, good, good, 1, 4, 0, None) == 0
    # prefill over an FP8 cache with an unsupported head_dim
    assert lib.pkv_paged_attn_prefill(_cache(fmt=1, scales=4096, d=96), good, 2, good, good, good, 1, 4, 8, 4,
                                      F(0.1), 1, good, 0, None, None) == 2
    # decode: the activation dtype must still be fp16 / bf16
    args = (_cache(fmt=1, scales=4096, dt=2), good, 2, good, good, 2, 4, F(0.1), 0, good, 1 << 20, good, 0, None, None)
    assert lib.pkv_paged_attn_decode(*args) == 2


def test_selftest_rejects_bad_limits_without_gpu(lib):
    assert lib.pkv_selftest_wait_timeout(0, None) == 1
    assert lib.pkv_selftest_wait_timeout(2000000, None) == 1


def test_workspace_sizing_with_explicit_splits(lib):
    # capacity 4 * 16 = 64 tokens in 1 split: no workspace
    assert pkv.decode_workspace_size(2, 4, 4, 128, 16, 4, num_splits=1) == 0
    # capacity 512 * 16 = 8192 tokens in 4 splits of 2048: B * Hq * 4 * (D + 1) floats, then a
    # 16-byte slot (the split size the split kernel took)
    assert pkv.decode_split_tokens(16, 32, 32, 128, 16, 512, num_splits=4) == 2048
    assert pkv.decode_workspace_size(16, 32, 32, 128, 16, 512, num_splits=4) == 16 * 32 * 4 * 129 * 4 + 16
    # the partials are padded to 16 bytes before the slot: 1 * 1 * 2 * 65 floats = 520 -> 528
    assert pkv.decode_split_tokens(1, 1, 1, 64, 16, 16, num_splits=2) == 128
    assert pkv.decode_workspace_size(1, 1, 1, 64, 16, 16, num_splits=2) == 528 + 16
    # split size is rounded up to 128 tokens (splits start at multiples of 128)
    assert pkv.decode_split_tokens(1, 8, 8, 64, 16, 10, num_splits=3) == 128


def test_automatic_split_size_without_gpu(lib):
    # The automatic split is the largest of 768, 512, 384, 256, 128 tokens at or below
    # B * Hkv * capacity / (8 * CTAs); with no device in this process the CTA count is 0, so the
    # rule gives its largest size. A context has at most 2048 splits: a 4M-token capacity needs
    # splits of at least 2048 tokens.
    if not hasattr(lib, "pkv_decode_split_tokens"):
        pytest.skip("library without the split query")
    import torch
    if torch.cuda.is_available():
        pytest.skip("the no-device rule; on a GPU the SM count enters")
    assert pkv.decode_split_tokens(16, 32, 32, 128, 16, 512) == 768
    assert pkv.decode_split_tokens(1, 1, 1, 128, 16, 1 << 18) == 2048
    # and the workspace follows the split: B * Hq * ceil(8192 / 768) * (D + 1) floats, then the slot
    assert pkv.decode_workspace_size(16, 32, 32, 128, 16, 512) == 16 * 32 * 11 * 129 * 4 + 16


def test_device_slot_from_eight_threads(lib):
    """The per-device state behind every entry point is set up by whichever call comes first;
    eight threads calling at once (ctypes releases the GIL during each call) must all see the
    same answers. Only calls that launch nothing are made while a device could be visible."""
    import threading

    import torch

    n_threads, n_calls = 8, 300
    start = threading.Barrier(n_threads)
    results = [None] * n_threads

    def worker(i):
        code = ctypes.c_int(-1)
        start.wait()
        seen = set()
        for _ in range(n_calls):
            seen.add(("ws", lib.pkv_decode_workspace_size(16, 32, 8, 128, 16, 512, 0)))
            seen.add(("split", lib.pkv_decode_split_tokens(16, 32, 8, 128, 16, 512, 0)))
            seen.add(("err", lib.pkv_get_device_error(None, ctypes.byref(code)), code.value))
        results[i] = seen

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(n_threads)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert all(r == results[0] for r in results), results
    assert len(results[0]) == 3, results[0]   # one answer per call kind, the same in every thread
    err = [x for x in results[0] if x[0] == "err"][0]
    if torch.cuda.is_available() or err[1] != 4:
        return
    # no usable device: entry points that would launch must fail with PKV_ERR_CUDA after their
    # argument checks, from every thread, and never cache the failed device lookup
    P, F = ctypes.c_void_p, ctypes.c_float
    good = P(4096)
    codes = [None] * n_threads

    def launcher(i):
        start.wait()
        codes[i] = {(lib.pkv_kv_cache_append(_cache(), good, good, good, good, good, 1, 4, 3, None),
                     lib.pkv_attn_combine(good, good, 4, 2, 128, good, 2, None, None),
                     lib.pkv_paged_attn_prefill(_cache(), good, 2, good, good, good, 1, 4, 8, 8, F(0.1), 1, good, 0,
                                                None, None))
                    for _ in range(50)}

    threads = [threading.Thread(target=launcher, args=(i,)) for i in range(n_threads)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert all(c == {(4, 4, 4)} for c in codes), codes
