"""pkv_paged_attn_decode_noalloc, the decode entry point for callers that cannot allocate device
memory (a plugin handed only its input and output buffers, or a runtime that keeps all device
memory in its own pool): called through the C ABI, it must give the same result as the regular
pkv_paged_attn_decode with a caller-provided workspace, on two calls in a row (the second one
runs on the scratch array the first one left behind), and must refuse sizes whose split partials
do not fit in its fixed array. This file is collected last on purpose."""
import ctypes
import math

import pytest
import torch

import paged_kv_flash_cache_gb300 as pkv
from paged_kv_flash_cache_gb300 import workloads as W
from tests.helpers import MAX_ABS, REL_L2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from paged_kv_flash_cache_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    return pkv.load_library()


def device_problem(p):
    shape = (p.num_blocks, 2, p.num_kv_heads, p.block_size, p.head_dim)
    cache = p.pool_init.reshape(shape).to("cuda")
    pkv.kv_cache_append(cache, p.k_ctx.cuda(), p.v_ctx.cuda(), p.cu_ctx_lens.cuda(),
                        torch.zeros(p.batch, dtype=torch.int32, device="cuda"), p.block_tables.cuda())
    return cache


def call_noalloc(lib, cache, q, bt, ctx, scale, num_splits, out, lse):
    c = pkv._cache_struct(cache, cache.dtype)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.pkv_paged_attn_decode_noalloc(c, ctypes.c_void_p(q.data_ptr()), q.shape[1],
                                             ctypes.c_void_p(bt.data_ptr()), ctypes.c_void_p(ctx.data_ptr()),
                                             q.shape[0], bt.shape[1], ctypes.c_float(scale), num_splits,
                                             ctypes.c_void_p(out.data_ptr()), pkv._dtype_code(out.dtype),
                                             ctypes.c_void_p(lse.data_ptr()), stream)


def assert_close(a, b, dtype):
    a64, b64 = a.double().cpu(), b.double().cpu()
    assert torch.isfinite(a64).all()
    assert (a64 - b64).abs().max().item() <= MAX_ABS[dtype]
    assert ((a64 - b64).norm() / b64.norm()).item() <= REL_L2


@pytest.mark.parametrize("dtype,hq,hkv,bs", [(W.F16, 8, 8, 16), (W.BF16, 16, 4, 32)])
def test_noalloc_matches_regular_decode_twice(lib, dtype, hq, hkv, bs):
    lens = [1, 700, 4096, 2049, 0, 64]
    pages = sum((L + bs - 1) // bs for L in lens)
    p = W.make_problem("na", batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim=128, block_size=bs,
                       context_lens=lens, q_lens=[1] * len(lens), dtype=dtype, causal=False, seed=77,
                       num_blocks=pages + 5, max_blocks_per_seq=4096 // bs)
    cache = device_problem(p)
    bt, ctx = p.block_tables.cuda(), p.context_lens.cuda()
    scale = 1.0 / math.sqrt(128)
    need = pkv.decode_workspace_size(p.batch, hq, hkv, 128, bs, bt.shape[1])
    assert 0 < need <= pkv.DECODE_NOALLOC_SCRATCH_BYTES
    ref_lse = torch.empty((p.batch, hq), dtype=torch.float32, device="cuda")
    for call in range(2):
        q = W.randn_t(torch.Generator().manual_seed(100 + call), (p.batch, hq, 128), dtype).cuda()
        ref = pkv.paged_attn_decode(cache, q, bt, ctx, scale=scale, lse=ref_lse)
        out = torch.full_like(ref, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        assert call_noalloc(lib, cache, q, bt, ctx, scale, 0, out, lse) == 0
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        assert_close(out, ref, dtype)
        finite = torch.isfinite(ref_lse)
        assert torch.equal(finite, torch.isfinite(lse))
        assert torch.allclose(lse[finite], ref_lse[finite], rtol=1e-5, atol=1e-5)


def test_noalloc_rejects_sizes_beyond_its_array(lib):
    # 64 sequences x 32 heads with a 32768-token capacity in 512-token splits needs
    # 64 * 32 * 64 * 129 * 4 bytes (~68 MB) of partials: more than the fixed array.
    need = pkv.decode_workspace_size(64, 32, 8, 128, 32, 1024, num_splits=64)
    assert need > pkv.DECODE_NOALLOC_SCRATCH_BYTES
    cache = torch.zeros((4, 2, 8, 32, 128), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((64, 32, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((64, 1024), dtype=torch.int32, device="cuda")
    ctx = torch.ones(64, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty((64, 32), dtype=torch.float32, device="cuda")
    assert call_noalloc(lib, cache, q, bt, ctx, 0.1, 64, out, lse) == 3      # PKV_ERR_WORKSPACE, nothing launched
