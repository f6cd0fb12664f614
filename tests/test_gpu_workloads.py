"""GPU parity at the full sizes of the named decode workloads, in the launch configuration the
benchmark times (the library's own append, the default split choice, a caller-provided
workspace), against the CPU oracle: the 7B-like decode batch, the block-size sweep (identical
token data for every block size) and the mixed serving batch with its fragmented pool, plus the
multi-query batch. Every output row is checked; the oracle takes a few seconds per case. The
appends are compared with the oracle's cache bit for bit first, so that the attention check
reads the same bytes on both sides."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_flash_cache_gb300 as pkv
from paged_kv_flash_cache_gb300 import workloads as W
from tests.helpers import cache_bits, check_close, device_cache

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_flash_cache_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available()


def decode_like_the_benchmark(p, cache):
    """One decode call as the benchmark issues it: auto splits, workspace and output passed in."""
    bt, ctx, q = p.block_tables.cuda(), p.context_lens.cuda(), p.q.cuda()
    ws_bytes = pkv.decode_workspace_size(p.batch, p.num_q_heads, p.num_kv_heads, p.head_dim, p.block_size,
                                         bt.shape[1])
    ws = torch.empty(max(16, ws_bytes), dtype=torch.uint8, device="cuda")
    out = torch.empty((p.batch, p.num_q_heads, p.head_dim), dtype=q.dtype, device="cuda")
    lse = torch.empty((p.batch, p.num_q_heads), dtype=torch.float32, device="cuda")
    pkv.paged_attn_decode(cache, q, bt, ctx, scale=p.scale, workspace=ws, out=out, lse=lse)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    return out, lse


def check_workload(p, what):
    cache = device_cache(p)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    bits = cache_bits(cache)
    assert np.array_equal(bits, oracle.build_cache(p)), "%s: appended cache differs from the oracle's" % what
    out, lse = decode_like_the_benchmark(p, cache)
    ref, ref_lse = oracle.attention_of(p, bits)
    # the output is the only rounding to the input type on the decode path (the tensor-core P.V
    # of four or more query heads per KV head takes P as a rounded part plus its remainder)
    check_close(out, ref, p.dtype, roundings=1, what=what)
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-5)


def test_decode_7b_full_size_every_row():
    """16 sequences with contexts U[1024, 8192] (76k cached tokens), 32 heads x 128, fp16, bs 16,
    pages shuffled over a pool 1.2x the pages needed whose other pages hold seeded noise."""
    check_workload(W.decode_7b(), "7B decode")


def test_decode_7b_step_full_size_every_row():
    """The step the benchmark times: paged_attn_decode_step over the same 7B-like batch (attention
    over every context, the step's token appended at position context_lens[b] by the split kernel),
    with the benchmark's workspace and output: every output row against the oracle, and the whole
    pool bit for bit against the oracle's append of the step's tokens."""
    p = W.decode_7b()
    cache = device_cache(p)
    torch.cuda.synchronize()
    bits = cache_bits(cache)
    assert np.array_equal(bits, oracle.build_cache(p))
    step = W.append_step(p, seed=7)
    bt, ctx, q = step["block_tables"].cuda(), p.context_lens.cuda(), p.q.cuda()
    ws_bytes = pkv.decode_workspace_size(p.batch, p.num_q_heads, p.num_kv_heads, p.head_dim, p.block_size,
                                         bt.shape[1])
    ws = torch.empty(max(16, ws_bytes), dtype=torch.uint8, device="cuda")
    out = torch.empty((p.batch, p.num_q_heads, p.head_dim), dtype=q.dtype, device="cuda")
    lse = torch.empty((p.batch, p.num_q_heads), dtype=torch.float32, device="cuda")
    pkv.paged_attn_decode_step(cache, q, bt, ctx, step["k_new"].cuda(), step["v_new"].cuda(), scale=p.scale,
                               workspace=ws, out=out, lse=lse)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    ref, ref_lse = oracle.attention_of(p, bits)
    check_close(out, ref, p.dtype, roundings=1, what="7B decode step")
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-5)
    assert oracle.kv_cache_append(bits, step["k_new"], step["v_new"], step["cu_new_lens"], step["ctx_before"],
                                  step["block_tables"]) == 0
    assert np.array_equal(cache_bits(cache), bits), "7B decode step: cache differs from the oracle's append"


@pytest.mark.parametrize("bs", [8, 16, 32, 64, 128, 512])
def test_block_size_sweep_full_size_every_row(bs):
    """32 sequences x 4096 tokens, 32 heads x 128, fp16: the same token data through every page size."""
    kv = test_block_size_sweep_full_size_every_row.kv
    if kv is None:
        kv = test_block_size_sweep_full_size_every_row.kv = W.bs_sweep_kv()
    check_workload(W.bs_sweep(bs, kv_data=kv, pool_init="none"), "bs sweep %d" % bs)


test_block_size_sweep_full_size_every_row.kv = None


def test_mixed_serving_full_size_every_row():
    """64 sequences with lognormal contexts (median 2048, up to 32768), 32 query heads on 8 KV heads,
    bf16, bs 32, in a pool twice the pages needed, half of it freed and handed out again at random
    (the other pages hold seeded noise)."""
    check_workload(W.mixed_serving(), "mixed serving")


def test_mixed_serving_fp32_output_literal_bounds():
    """The mixed serving batch (32 query heads on 8 KV heads, bf16) with an FP32 output: nothing on
    the decode path is rounded to bf16, so every row must meet the stated bounds as written
    (max-abs 1e-2, relative L2 1e-3) against the oracle, with no allowance for roundings."""
    p = W.mixed_serving()
    cache = device_cache(p)
    torch.cuda.synchronize()
    bt, ctx, q = p.block_tables.cuda(), p.context_lens.cuda(), p.q.cuda()
    lse = torch.empty((p.batch, p.num_q_heads), dtype=torch.float32, device="cuda")
    out = pkv.paged_attn_decode(cache, q, bt, ctx, scale=p.scale, out_dtype=torch.float32, lse=lse)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    ref, ref_lse = oracle.attention_of(p, cache_bits(cache))
    info = check_close(out, ref, p.dtype, roundings=0, what="mixed serving fp32 out")
    assert info["max_abs"] <= 1e-2 and info["rel_l2"] <= 1e-3, info
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-5)


def test_mqa_batch_full_size_every_row():
    """128 sequences with contexts U[1024, 8192], 32 query heads on one KV head of 128, bf16, bs 16
    (one 32-head unit per split)."""
    gen = torch.Generator().manual_seed(1241)
    lens = torch.randint(1024, 8193, (128,), generator=gen).tolist()
    nb = sum((L + 15) // 16 for L in lens) + 64
    order = torch.randperm(nb, generator=gen).tolist()
    p = W.make_problem("mqa", batch=128, num_q_heads=32, num_kv_heads=1, head_dim=128, block_size=16,
                       context_lens=lens, q_lens=[1] * 128, dtype=W.BF16, causal=False, seed=1242, num_blocks=nb,
                       free_order=order, pool_init="cheap")
    check_workload(p, "MQA")
