"""GPU parity of paged_attn_mixed: one call over a batch that mixes decode sequences (one query
row each) and prefill chunks, against the CPU oracle over the same rows, through the C ABI. The
decode rows run on the split-KV decode kernels, the chunks on the prefill kernel; each must leave
the other's rows alone (checked by pre-filling the output with a sentinel)."""
import numpy as np
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


def problem(*, lens, q_lens, hq, hkv, d=128, bs=16, dtype=W.BF16, seed=7, kv_format="native"):
    nb = sum((L + bs - 1) // bs for L in lens) + 6
    order = torch.randperm(nb, generator=torch.Generator().manual_seed(seed + 5)).tolist()
    return W.make_problem("mix", batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                          context_lens=lens, q_lens=q_lens, dtype=dtype, causal=True, seed=seed, num_blocks=nb,
                          free_order=order, kv_format=kv_format)


def run(p, cache, scales=None, num_splits=0):
    out = torch.full((p.total_q, p.num_q_heads, p.head_dim), float("nan"), dtype=p.q.dtype, device="cuda")
    lse = torch.full((p.total_q, p.num_q_heads), float("nan"), dtype=torch.float32, device="cuda")
    pkv.paged_attn_mixed(cache, to_dev(p.q), to_dev(p.cu_q_lens), to_dev(p.context_lens), to_dev(p.block_tables),
                         max_q_len=int(p.q_lens.max()), scale=p.scale, causal=True, num_splits=num_splits, out=out,
                         lse=lse, scales=scales)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    return out, lse


def check_rows(p, out, ref, chunk_roundings, what):
    """Decode rows (q_len 1) at the decode path's bound (the output is its one rounding to 16
    bits); chunk rows at the prefill path's (P and the output)."""
    cu, ql = p.cu_q_lens.tolist(), p.q_lens.tolist()
    dec = [cu[b] for b in range(p.batch) if ql[b] == 1]
    chunk = [r for b in range(p.batch) if ql[b] > 1 for r in range(cu[b], cu[b + 1])]
    for rows, k, kind in ((dec, 1, "decode rows"), (chunk, chunk_roundings, "chunk rows")):
        if rows:
            check_close(out[torch.as_tensor(rows, device=out.device)], ref[rows], p.dtype, roundings=k,
                        what="%s, %s" % (what, kind))


# decode rows (q_len 1), chunks (q_len > 1) and an empty sequence, interleaved
LENS = [3000, 700, 129, 2048, 1, 900, 5000, 64, 333]
QLENS = [1, 300, 1, 512, 1, 0, 1, 64, 1]


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (16, 4), (32, 1)])
@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
def test_mixed_batch_matches_oracle(hq, hkv, dtype):
    p = problem(lens=LENS, q_lens=QLENS, hq=hq, hkv=hkv, dtype=dtype, seed=hq + hkv)
    cache = device_cache(p)
    out, lse = run(p, cache)
    ref, ref_lse = oracle.attention_of(p, cache_bits(cache))
    # every row written (no sentinel left), then parity
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    check_rows(p, out, ref, 2, "mixed hq=%d hkv=%d %s" % (hq, hkv, dtype))
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-4, atol=1e-4)


def test_mixed_batch_with_forced_splits_and_all_decode_or_all_chunks():
    # every sequence a decode row; every sequence a chunk (the 1-token context stays one row)
    for q_lens in ([1] * len(LENS), [min(L, max(2, q)) for L, q in zip(LENS, QLENS)]):
        p = problem(lens=LENS, q_lens=q_lens, hq=8, hkv=2, dtype=W.BF16, seed=sum(q_lens))
        cache = device_cache(p)
        out, lse = run(p, cache, num_splits=5)
        ref, ref_lse = oracle.attention_of(p, cache_bits(cache))
        check_rows(p, out, ref, 2, "mixed q_lens=%s" % q_lens[:3])
        np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-4, atol=1e-4)


def test_mixed_batch_fp8_cache():
    p = problem(lens=LENS, q_lens=QLENS, hq=16, hkv=4, dtype=W.BF16, seed=3, kv_format="fp8")
    codes, scales = p.pool_init
    codes, scales = codes.cuda().contiguous(), scales.cuda().contiguous()
    pkv.kv_cache_append(codes, to_dev(p.k_ctx), to_dev(p.v_ctx), to_dev(p.cu_ctx_lens),
                        torch.zeros(p.batch, dtype=torch.int32, device="cuda"), to_dev(p.block_tables),
                        scales=scales)
    out, lse = run(p, codes, scales=scales)
    ref, ref_lse = oracle.attention_of(p, oracle.Fp8Cache(codes.cpu().numpy(), scales.cpu().numpy()))
    assert torch.isfinite(out).all()
    check_rows(p, out, ref, 2, "mixed fp8")
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-4, atol=1e-4)
