"""GPU parity under prefix caching (pwwt.cn write-up on chunked attention, section 5.4): several
requests' block tables hold the same prompt pages. The prompt is appended once, each request's
own rows after it; appends are bit-exact and never touch the shared pages; prefill of the
uncached rows and decode over the aliased tables match the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_flash_cache_gb300 as pkv
from paged_kv_flash_cache_gb300 import workloads as W
from tests.helpers import cache_bits, check_close, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_flash_cache_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available()


def shared_cache(p):
    """Pool with the prompt appended once and every request's own rows after it."""
    shape = (p.num_blocks, 2, p.num_kv_heads, p.block_size, p.head_dim)
    cache = p.pool_init.reshape(shape).cuda()
    for args in (W.shared_append(p), W.private_append(p)):
        pkv.kv_cache_append(cache, to_dev(args["k_new"]), to_dev(args["v_new"]), to_dev(args["cu_new_lens"]),
                            to_dev(args["ctx_before"]), to_dev(args["block_tables"]))
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    return cache


def shared_rows(p, bits):
    return bits[np.array(p.meta["shared_blocks"])]


@pytest.mark.parametrize("bs", [8, 16, 128])
def test_prefix_append_bit_exact(bs):
    p = W.prefix_shared(batch=6, prefix=300, lo=1, hi=200, block_size=bs, heads=4, head_dim=128)
    cache = shared_cache(p)
    assert np.array_equal(cache_bits(cache), oracle.build_cache(p))


@pytest.mark.parametrize("heads,kv_heads,dtype", [(8, 8, W.F16), (16, 4, W.BF16)])
def test_prefix_decode_and_a_decode_step(heads, kv_heads, dtype):
    p = W.prefix_shared(batch=6, prefix=1000, lo=1, hi=700, block_size=16, heads=heads, kv_heads=kv_heads,
                        head_dim=128, dtype=dtype, seed=heads)
    cache = shared_cache(p)
    before = cache_bits(cache)
    lse = torch.empty((p.batch, heads), dtype=torch.float32, device="cuda")
    out = pkv.paged_attn_decode(cache, to_dev(p.q), to_dev(p.block_tables), to_dev(p.context_lens),
                                scale=p.scale, lse=lse)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    ref, ref_lse = oracle.attention_of(p, before)
    check_close(out, ref, dtype, roundings=1, what="prefix decode")
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-5)
    # one decode step's new tokens land in private pages only
    step = W.append_step(p, seed=3)
    shared = set(p.meta["shared_blocks"])
    for b, L in enumerate(p.context_lens.tolist()):
        assert int(step["block_tables"][b, L // p.block_size]) not in shared
    pkv.kv_cache_append(cache, to_dev(step["k_new"]), to_dev(step["v_new"]), to_dev(step["cu_new_lens"]),
                        to_dev(step["ctx_before"]), to_dev(step["block_tables"]))
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    after = cache_bits(cache)
    assert np.array_equal(shared_rows(p, after), shared_rows(p, before))
    ref_after = before.copy()
    assert oracle.kv_cache_append(ref_after, **step) == 0
    assert np.array_equal(after, ref_after)


@pytest.mark.parametrize("prefix,bs", [(512, 16), (777, 32)])
def test_prefix_prefill_of_the_uncached_rows(prefix, bs):
    """A prefix-cache hit computes attention only for the rows after the shared pages, causal over
    the whole context (shared prompt + the prompt's partial page + the request's own rows)."""
    p = W.prefix_shared(batch=4, prefix=prefix, lo=1, hi=600, block_size=bs, heads=8, head_dim=128,
                        dtype=W.BF16, prefill=True, seed=prefix)
    cache = shared_cache(p)
    lse = torch.empty((p.total_q, 8), dtype=torch.float32, device="cuda")
    out = pkv.paged_attn_prefill(cache, to_dev(p.q), to_dev(p.cu_q_lens), to_dev(p.context_lens),
                                 to_dev(p.block_tables), max_q_len=int(p.q_lens.max()), scale=p.scale,
                                 causal=True, lse=lse)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    ref, ref_lse = oracle.attention_of(p, cache_bits(cache))
    check_close(out, ref, W.BF16, roundings=2, what="prefix prefill")
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-4, atol=1e-4)
