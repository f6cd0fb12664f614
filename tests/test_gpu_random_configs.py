"""GPU parity on seeded random configurations: head_dim, page size, head grouping, dtype, output
type, split count, context and chunk lengths (0, 1, page multiples and ragged values mixed), for
the decode, prefill and mixed calls over 16-bit and FP8 caches. Each configuration is drawn from
its index alone, so a failure names a reproducible case; every output is checked against the
oracle (prefill: every row of small chunks, else the first, last and 12 seeded rows of each)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_flash_cache_gb300 as pkv
from paged_kv_flash_cache_gb300 import workloads as W
from tests.helpers import cache_bits, check_close, device_cache, to_dev

pytestmark = pytest.mark.gpu

BLOCK_SIZES = [8, 16, 32, 64, 128, 256, 512]
# (Hq, Hkv): MHA, GQA groups 2..32, MQA, and groups taken as several tensor-core units
GROUPS_DECODE = [(4, 4), (8, 4), (16, 4), (32, 8), (16, 2), (32, 2), (16, 1), (32, 1), (64, 2), (48, 1), (24, 3)]
GROUPS_FP8_D64 = [(4, 4), (8, 4), (16, 4), (8, 1)]  # the CUDA-core FP8 kernel: groups 1, 2, 4, 8
GROUPS_PREFILL = [(4, 4), (8, 2), (6, 3), (12, 4), (16, 1), (9, 3)]


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_flash_cache_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available()


# head_dim 256 on a native cache only (an FP8 cache with head_dim 256 is refused)
HEAD_DIMS = {"native": [64, 128, 256], "fp8": [64, 128]}


def draw_lengths(rng, n, hi, bs):
    out = []
    for _ in range(n):
        kind = rng.integers(0, 5)
        if kind == 0:
            out.append(int(rng.integers(0, 2)))                     # empty or one token
        elif kind == 1:
            out.append(int(bs * rng.integers(1, max(2, hi // bs))))  # a page multiple
        else:
            out.append(int(rng.integers(2, hi)))
    return out


def make(rng, *, lens, q_lens, hq, hkv, d, bs, dtype, causal, kv_format, seed):
    nb = sum((L + bs - 1) // bs for L in lens) + int(rng.integers(0, 9))
    order = torch.randperm(max(nb, 1), generator=torch.Generator().manual_seed(seed)).tolist()
    return W.make_problem("rand", batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                          context_lens=lens, q_lens=q_lens, dtype=dtype, causal=causal, seed=seed,
                          num_blocks=max(nb, 1), free_order=order, kv_format=kv_format)


def on_device(p):
    """(cache, scales, oracle's view of the cache) with the context appended by the library."""
    if p.kv_format == "native":
        cache = device_cache(p)
        torch.cuda.synchronize()
        return cache, None, cache_bits(cache)
    codes, scales = p.pool_init
    codes, scales = codes.cuda().contiguous(), scales.cuda().contiguous()
    if p.k_ctx.shape[0]:
        pkv.kv_cache_append(codes, to_dev(p.k_ctx), to_dev(p.v_ctx), to_dev(p.cu_ctx_lens),
                            torch.zeros(p.batch, dtype=torch.int32, device="cuda"), to_dev(p.block_tables),
                            scales=scales)
    torch.cuda.synchronize()
    return codes, scales, oracle.Fp8Cache(codes.cpu().numpy().copy(), scales.cpu().numpy().copy())


def compare(p, out, lse, host, roundings, what, rows=None):
    assert pkv.get_device_error() == 0, what
    ref, ref_lse = oracle.attention_of(p, host, rows=rows)
    sel = None if rows is None else torch.as_tensor(rows, device=out.device)
    got = out if sel is None else out[sel]
    check_close(got, ref, p.dtype, roundings=roundings, what=what)
    got_lse = (lse if sel is None else lse[sel]).cpu().numpy()
    assert np.array_equal(np.isneginf(got_lse), np.isneginf(ref_lse)), what
    fin = np.isfinite(ref_lse)
    np.testing.assert_allclose(got_lse[fin], ref_lse[fin], rtol=1e-4, atol=1e-4, err_msg=what)


def sample_rows(p, rng, full_below=64):
    cu = p.cu_q_lens.tolist()
    rows = []
    for b in range(p.batch):
        n = cu[b + 1] - cu[b]
        if n <= full_below:
            rows += list(range(cu[b], cu[b + 1]))
        else:
            rows += [cu[b], cu[b + 1] - 1] + [cu[b] + int(x) for x in rng.choice(np.arange(1, n - 1), 12, replace=False)]
    return rows


@pytest.mark.parametrize("fmt", ["native", "fp8"])
@pytest.mark.parametrize("i", range(16))
def test_random_decode(fmt, i):
    rng = np.random.default_rng(1000 + i + (500 if fmt == "fp8" else 0))
    d = int(rng.choice(HEAD_DIMS[fmt]))
    bs = int(rng.choice(BLOCK_SIZES))
    if fmt == "native":
        # any group 1..48 (uneven ones included) over 1, 2, 3, 4 or 8 KV heads
        hkv = int(rng.choice([1, 2, 3, 4, 8]))
        hq = hkv * int(rng.integers(1, 49 if hkv <= 2 else 17))
    else:
        groups = GROUPS_FP8_D64 if d == 64 else GROUPS_DECODE
        hq, hkv = groups[int(rng.integers(0, len(groups)))]
    dtype = W.F16 if rng.integers(0, 2) else W.BF16
    lens = draw_lengths(rng, int(rng.integers(1, 7)), 2500, bs)
    splits = int(rng.choice([0, 0, 1, 3, 7]))
    fp32 = bool(rng.integers(0, 4) == 0)
    what = "decode %s d=%d bs=%d %d/%d %s splits=%d fp32=%s lens=%s" % (fmt, d, bs, hq, hkv, dtype, splits, fp32, lens)
    p = make(rng, lens=lens, q_lens=[1] * len(lens), hq=hq, hkv=hkv, d=d, bs=bs, dtype=dtype, causal=False,
             kv_format=fmt, seed=2000 + i)
    cache, scales, host = on_device(p)
    lse = torch.empty((p.batch, hq), dtype=torch.float32, device="cuda")
    out = pkv.paged_attn_decode(cache, to_dev(p.q), to_dev(p.block_tables), to_dev(p.context_lens), scale=p.scale,
                                num_splits=splits, out_dtype=torch.float32 if fp32 else None, lse=lse, scales=scales)
    torch.cuda.synchronize()
    # roundings to 16 bits on the decode path: the output, unless FP32 (tensor-core P.V takes P as
    # a rounded part plus its remainder)
    compare(p, out, lse, host, 0 if fp32 else 1, what)


@pytest.mark.parametrize("fmt", ["native", "fp8"])
@pytest.mark.parametrize("i", range(8))
def test_random_prefill(fmt, i):
    rng = np.random.default_rng(3000 + i + (500 if fmt == "fp8" else 0))
    d = int(rng.choice(HEAD_DIMS[fmt]))
    bs = int(rng.choice(BLOCK_SIZES))
    hq, hkv = GROUPS_PREFILL[int(rng.integers(0, len(GROUPS_PREFILL)))]
    dtype = W.F16 if rng.integers(0, 2) else W.BF16
    n = int(rng.integers(1, 4))
    lens = [int(rng.integers(1, 1300)) for _ in range(n)]
    q_lens = [int(min(L, rng.choice([1, L, rng.integers(1, 300)]))) for L in lens]
    causal = bool(rng.integers(0, 3) > 0)
    fp32 = bool(rng.integers(0, 4) == 0)
    what = "prefill %s d=%d bs=%d %d/%d %s causal=%s fp32=%s lens=%s q=%s" % (fmt, d, bs, hq, hkv, dtype, causal,
                                                                               fp32, lens, q_lens)
    p = make(rng, lens=lens, q_lens=q_lens, hq=hq, hkv=hkv, d=d, bs=bs, dtype=dtype, causal=causal, kv_format=fmt,
             seed=4000 + i)
    cache, scales, host = on_device(p)
    lse = torch.empty((p.total_q, hq), dtype=torch.float32, device="cuda")
    out = pkv.paged_attn_prefill(cache, to_dev(p.q), to_dev(p.cu_q_lens), to_dev(p.context_lens),
                                 to_dev(p.block_tables), max_q_len=max(q_lens), scale=p.scale, causal=causal,
                                 out_dtype=torch.float32 if fp32 else None, lse=lse, scales=scales)
    torch.cuda.synchronize()
    # roundings: output (unless FP32) and P (over an FP8 cache P times the V row scale / W)
    r = (0 if fp32 else 1) + 1
    compare(p, out, lse, host, r, what, rows=sample_rows(p, rng))


@pytest.mark.parametrize("i", range(6))
def test_random_mixed(i):
    rng = np.random.default_rng(5000 + i)
    fmt = "fp8" if i % 3 == 2 else "native"
    d = int(rng.choice(HEAD_DIMS[fmt]))
    bs = int(rng.choice(BLOCK_SIZES))
    hq, hkv = [(8, 8), (8, 4), (16, 4), (32, 1), (16, 2)][int(rng.integers(0, 5))]
    dtype = W.F16 if rng.integers(0, 2) else W.BF16
    n = int(rng.integers(2, 8))
    lens = [int(rng.integers(1, 1500)) for _ in range(n)]
    q_lens = [int(min(L, rng.choice([1, 1, 0, rng.integers(2, 200)]))) for L in lens]
    if all(q == 0 for q in q_lens):
        q_lens[0] = 1
    splits = int(rng.choice([0, 0, 2, 5]))
    what = "mixed %s d=%d bs=%d %d/%d %s splits=%d lens=%s q=%s" % (fmt, d, bs, hq, hkv, dtype, splits, lens, q_lens)
    p = make(rng, lens=lens, q_lens=q_lens, hq=hq, hkv=hkv, d=d, bs=bs, dtype=dtype, causal=True, kv_format=fmt,
             seed=6000 + i)
    cache, scales, host = on_device(p)
    out = torch.full((p.total_q, hq, d), float("nan"), dtype=p.q.dtype, device="cuda")
    lse = torch.full((p.total_q, hq), float("nan"), dtype=torch.float32, device="cuda")
    pkv.paged_attn_mixed(cache, to_dev(p.q), to_dev(p.cu_q_lens), to_dev(p.context_lens), to_dev(p.block_tables),
                         max_q_len=max(q_lens), scale=p.scale, causal=True, num_splits=splits, out=out, lse=lse,
                         scales=scales)
    torch.cuda.synchronize()
    assert not torch.isnan(out).any() and not torch.isnan(lse).any(), what
    # decode rows at the decode bound (the output); chunk rows at the prefill bound (output, P)
    rows = sample_rows(p, rng)
    single = {p.cu_q_lens[b].item() for b in range(p.batch) if p.q_lens[b].item() == 1}
    dec = [r for r in rows if r in single]
    chunk = [r for r in rows if r not in single]
    if dec:
        compare(p, out, lse, host, 1, what + " (decode rows)", rows=dec)
    if chunk:
        compare(p, out, lse, host, 2, what + " (chunk rows)", rows=chunk)


@pytest.mark.parametrize("hq,hkv,fmt", [(4, 4, "native"), (8, 2, "native"), (12, 2, "native"), (8, 8, "fp8")])
def test_decode_batches_above_2048(hq, hkv, fmt):
    """Batches of more than 2048 sequences run in slices (the unit tables of a launch live in
    shared memory): 4100 short contexts (0..300 tokens, one of them empty) through the MHA, the
    mma.sync group, the tcgen05 and the FP8 kernels, with forced splits, every row checked."""
    rng = np.random.default_rng(77 + hq)
    lens = [int(x) for x in rng.integers(0, 301, 4100)]
    lens[5] = 0
    p = make(rng, lens=lens, q_lens=[1] * len(lens), hq=hq, hkv=hkv, d=64, bs=16, dtype=W.BF16, causal=False,
             kv_format=fmt, seed=91 + hq)
    cache, scales, host = on_device(p)
    lse = torch.empty((p.batch, hq), dtype=torch.float32, device="cuda")
    out = pkv.paged_attn_decode(cache, to_dev(p.q), to_dev(p.block_tables), to_dev(p.context_lens), scale=p.scale,
                                num_splits=3, lse=lse, scales=scales)
    torch.cuda.synchronize()
    compare(p, out, lse, host, 1, "batch 4100 %d/%d %s" % (hq, hkv, fmt))


@pytest.mark.parametrize("hq,hkv,fmt", [(8, 1, "native"), (32, 1, "native"), (8, 1, "fp8"), (2, 2, "fp8")])
def test_decode_large_batch_head_dim_128(hq, hkv, fmt):
    """2100 sequences at head_dim 128: with 8-head units the unit tables of a 2048-sequence slice
    leave no room for two CTAs an SM in the group kernels' shared memory, so those launches run one
    CTA an SM; the MQA unit and the FP8 MHA unit keep two."""
    rng = np.random.default_rng(99 + hq)
    lens = [int(x) for x in rng.integers(0, 200, 2100)]
    p = make(rng, lens=lens, q_lens=[1] * len(lens), hq=hq, hkv=hkv, d=128, bs=16, dtype=W.BF16, causal=False,
             kv_format=fmt, seed=93 + hq)
    cache, scales, host = on_device(p)
    lse = torch.empty((p.batch, hq), dtype=torch.float32, device="cuda")
    out = pkv.paged_attn_decode(cache, to_dev(p.q), to_dev(p.block_tables), to_dev(p.context_lens), scale=p.scale,
                                num_splits=3, lse=lse, scales=scales)
    torch.cuda.synchronize()
    compare(p, out, lse, host, 1, "batch 2100 d=128 %d/%d %s" % (hq, hkv, fmt))


def test_mixed_call_batch_above_2048():
    """A mixed call of 2500 sequences (decode rows and short chunks): the decode rows run in
    slices, their rows found through cu_q_lens."""
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(1, 200, 2500)]
    q_lens = [1 if rng.integers(0, 4) else int(min(L, rng.integers(2, 20))) for L in lens]
    p = make(rng, lens=lens, q_lens=q_lens, hq=6, hkv=2, d=64, bs=16, dtype=W.F16, causal=True, kv_format="native",
             seed=17)
    cache, scales, host = on_device(p)
    out = torch.full((p.total_q, 6, 64), float("nan"), dtype=p.q.dtype, device="cuda")
    lse = torch.full((p.total_q, 6), float("nan"), dtype=torch.float32, device="cuda")
    pkv.paged_attn_mixed(cache, to_dev(p.q), to_dev(p.cu_q_lens), to_dev(p.context_lens), to_dev(p.block_tables),
                         max_q_len=max(q_lens), scale=p.scale, causal=True, num_splits=2, out=out, lse=lse)
    torch.cuda.synchronize()
    assert not torch.isnan(out).any()
    single = {p.cu_q_lens[b].item() for b in range(p.batch) if q_lens[b] == 1}
    rows = list(range(p.total_q))
    compare(p, out, lse, host, 1, "mixed 2500 decode rows", rows=[r for r in rows if r in single])
    compare(p, out, lse, host, 2, "mixed 2500 chunk rows", rows=[r for r in rows if r not in single])
