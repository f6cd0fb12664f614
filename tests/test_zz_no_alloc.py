"""pkv_paged_attn_decode_noalloc, the decode entry point for callers that cannot allocate device
memory (a plugin handed only its input and output buffers, or a runtime that keeps all device
memory in its own pool): called through the C ABI, it must give the same bits as the regular
pkv_paged_attn_decode with a caller-provided workspace, on two calls in a row (the second one
runs on the scratch array the first one left behind), and must refuse sizes whose split partials
do not fit in its fixed array. This file is collected last on purpose."""
import ctypes
import math

import pytest
import torch

import paged_kv_flash_cache_gb300 as pkv
from paged_kv_flash_cache_gb300 import workloads as W

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


@pytest.mark.parametrize("dtype,hq,hkv,bs", [(W.F16, 8, 8, 16), (W.BF16, 16, 4, 32)])
def test_noalloc_matches_regular_decode_twice(lib, dtype, hq, hkv, bs):
    """Both entry points run the same kernels with the same split choice, so their outputs must
    agree bit for bit. The two calls differ in batch and split count, so the second one runs on
    an array that the first one left holding partials in another layout: any read of a partial
    that the second call did not write itself would show."""
    lens = [1, 700, 4096, 2049, 0, 64]
    pages = sum((L + bs - 1) // bs for L in lens)
    p = W.make_problem("na", batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim=128, block_size=bs,
                       context_lens=lens, q_lens=[1] * len(lens), dtype=dtype, causal=False, seed=77,
                       num_blocks=pages + 5, max_blocks_per_seq=4096 // bs)
    cache = device_problem(p)
    bt_all, ctx_all = p.block_tables.cuda(), p.context_lens.cuda()
    scale = 1.0 / math.sqrt(128)
    for call, (batch, splits) in enumerate([(6, 7), (4, 0)]):
        bt, ctx = bt_all[:batch].contiguous(), ctx_all[:batch].contiguous()
        need = pkv.decode_workspace_size(batch, hq, hkv, 128, bs, bt.shape[1], num_splits=splits)
        assert 0 < need <= pkv.DECODE_NOALLOC_SCRATCH_BYTES
        q = W.randn_t(torch.Generator().manual_seed(100 + call), (batch, hq, 128), dtype).cuda()
        ref_lse = torch.empty((batch, hq), dtype=torch.float32, device="cuda")
        ref = pkv.paged_attn_decode(cache, q, bt, ctx, scale=scale, num_splits=splits, lse=ref_lse)
        out = torch.full_like(ref, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        assert call_noalloc(lib, cache, q, bt, ctx, scale, splits, out, lse) == 0
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        assert torch.isfinite(out).all()
        assert torch.equal(out, ref), "call %d: output differs from the regular decode" % call
        assert torch.equal(lse, ref_lse), "call %d: lse differs from the regular decode" % call


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
