"""Eight host threads make the first library calls of a fresh process at the same moment, each
on its own CUDA stream: the per-device set-up behind the entry points (device attributes, the
error word's address, the kernels' shared-memory opt-in) is raced for real, since ctypes
releases the GIL during each call. Every thread must get the same bits as a later serial call."""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent("""
    import threading
    import torch
    import paged_kv_flash_cache_gb300 as pkv
    from paged_kv_flash_cache_gb300 import workloads as W

    torch.cuda.set_device(0)
    # the cache is filled by torch, so the first library call happens inside the threads
    gen = torch.Generator().manual_seed(11)
    lens = [700, 1, 3000, 129, 2048, 0]
    hq, hkv, d, bs = 16, 4, 128, 16
    mb = 3000 // bs + 1
    nb = len(lens) * mb
    cache = W.randn_t(gen, (nb, 2, hkv, bs, d), W.BF16).cuda()
    bt = torch.randperm(nb, generator=gen).to(torch.int32).reshape(len(lens), mb).cuda()
    ctx = torch.tensor(lens, dtype=torch.int32).cuda()
    q = W.randn_t(gen, (len(lens), hq, d), W.BF16).cuda()
    qp = W.randn_t(gen, (64, hq, d), W.BF16).cuda()
    cu = torch.tensor([0, 64], dtype=torch.int32).cuda()
    ctxp = torch.tensor([700], dtype=torch.int32).cuda()
    torch.cuda.synchronize()
    n = 8
    start = threading.Barrier(n)
    outs = [None] * n
    errs = [None] * n

    def work(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                start.wait()
                o_dec = pkv.paged_attn_decode(cache, q, bt, ctx, scale=0.088)
                o_pre = pkv.paged_attn_prefill(cache, qp, cu, ctxp, bt[:1].contiguous(), max_q_len=64, scale=0.088,
                                               causal=True)
            s.synchronize()
            outs[i] = (o_dec.cpu(), o_pre.cpu())
        except Exception as e:  # reported below
            errs[i] = repr(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(n)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert all(e is None for e in errs), errs
    assert pkv.get_device_error() == 0
    ref_d = pkv.paged_attn_decode(cache, q, bt, ctx, scale=0.088).cpu()
    ref_p = pkv.paged_attn_prefill(cache, qp, cu, ctxp, bt[:1].contiguous(), max_q_len=64, scale=0.088,
                                   causal=True).cpu()
    for i, (a, b) in enumerate(outs):
        assert torch.equal(a, ref_d), "thread %d: decode differs" % i
        assert torch.equal(b, ref_p), "thread %d: prefill differs" % i
    print("threads ok")
""")


def test_first_calls_from_eight_threads_fresh_process():
    from paged_kv_flash_cache_gb300 import build
    build.build()
    r = subprocess.run([sys.executable, "-c", SCRIPT], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "threads ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
