"""Failure detection without faulting the GPU: every wait inside the kernels is bounded. The
self-test entry point makes one such wait run out (an mbarrier nothing completes, a 20 ms limit);
the host must read PKV_ERR_TIMEOUT from the device error word within the limit's order of time,
and the context must stay usable: a decode right after matches the oracle with no error."""
import time

import pytest
import torch

import oracle
import paged_kv_flash_cache_gb300 as pkv
from paged_kv_flash_cache_gb300 import workloads as W
from tests.helpers import cache_bits, check_close, device_cache, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_flash_cache_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available()


def test_bounded_wait_reports_timeout_and_the_context_stays_usable():
    assert pkv.get_device_error() == 0          # reads and clears the word
    t0 = time.time()
    pkv.selftest_wait_timeout(20000)
    assert pkv.get_device_error() == 6          # PKV_ERR_TIMEOUT
    assert time.time() - t0 < 5.0
    assert pkv.get_device_error() == 0          # cleared by the read
    p = W.make_problem("after", batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                       context_lens=[300, 77], q_lens=[1, 1], dtype=W.BF16, causal=False, seed=4, num_blocks=30)
    cache = device_cache(p)
    out = pkv.paged_attn_decode(cache, to_dev(p.q), to_dev(p.block_tables), to_dev(p.context_lens), scale=p.scale)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    ref, _ = oracle.attention_of(p, cache_bits(cache))
    check_close(out, ref, W.BF16, roundings=1, what="decode after a timeout")
