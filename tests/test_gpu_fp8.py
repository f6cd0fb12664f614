"""GPU parity for the FP8 cache (E4M3 codes with one FP32 scale per cached row) through the C ABI:
the quantising append is bit-exact against the oracle (codes and scales, every pool element), and
decode over the FP8 cache matches the oracle's attention over the exactly dequantised values
within the stated tolerances, for every head grouping, block sizes 8..512, splits and FP32 output."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_flash_cache_gb300 as pkv
from paged_kv_flash_cache_gb300 import workloads as W
from tests.helpers import check_close, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_flash_cache_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available()


def problem(*, lens, hq=8, hkv=8, d=128, bs=16, dtype=W.BF16, seed=5, extra=7, mb=None, kv_data=None):
    nb = sum((L + bs - 1) // bs for L in lens) + extra
    order = torch.randperm(nb, generator=torch.Generator().manual_seed(seed + 9)).tolist()
    return W.make_problem("f", batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                          context_lens=lens, q_lens=[1] * len(lens), dtype=dtype, causal=False, seed=seed,
                          num_blocks=nb, free_order=order, max_blocks_per_seq=mb, kv_format="fp8", kv_data=kv_data)


def device_fp8(p):
    """Pool noise on the device, then every context token appended by the library."""
    codes, scales = p.pool_init
    codes, scales = codes.cuda().contiguous(), scales.cuda().contiguous()
    pkv.kv_cache_append(codes, to_dev(p.k_ctx), to_dev(p.v_ctx), to_dev(p.cu_ctx_lens),
                        torch.zeros(p.batch, dtype=torch.int32, device="cuda"), to_dev(p.block_tables),
                        scales=scales)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    return codes, scales


def roundings(p, fp32_out=False):
    """Roundings to 16 bits on the decode path: the output, unless FP32. The tensor-core path
    (head_dim 128) takes P into the P.V product as an f16 part plus its f16 remainder, and the
    CUDA-core path (head_dim 64) keeps P in FP32."""
    return 0 if fp32_out else 1


def host(codes, scales):
    return oracle.Fp8Cache(codes.cpu().numpy().copy(), scales.cpu().numpy().copy())


def decode(p, codes, scales, num_splits=0, out_dtype=None):
    lse = torch.empty((p.batch, p.num_q_heads), dtype=torch.float32, device="cuda")
    out = pkv.paged_attn_decode(codes, to_dev(p.q), to_dev(p.block_tables), to_dev(p.context_lens), scale=p.scale,
                                num_splits=num_splits, out_dtype=out_dtype, lse=lse, scales=scales)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    return out, lse


@pytest.mark.parametrize("bs", [8, 16, 128])
@pytest.mark.parametrize("d,dtype", [(128, W.BF16), (64, W.F16)])
def test_fp8_append_bit_exact(bs, d, dtype):
    p = problem(lens=[1, 37, 100, 513], bs=bs, d=d, dtype=dtype, hq=4, hkv=4)
    codes, scales = device_fp8(p)
    ref = oracle.build_cache(p)
    got = host(codes, scales)
    assert np.array_equal(got.codes, ref.codes)
    assert np.array_equal(got.scales.view(np.uint32), ref.scales.view(np.uint32))


def test_fp8_append_special_rows():
    """Zero rows, rows of +-0, huge and tiny magnitudes, ties of the scaled values."""
    d, hkv = 128, 3
    k = torch.randn(6, hkv, d, generator=torch.Generator().manual_seed(1))
    k[0] = 0.0
    k[1] = -0.0
    k[2, 0] = 60000.0
    k[3] = k[3] * 1e-6
    k[4, 1, :8] = torch.tensor([448.0, 1.0625, 1.1875, -3.0, 2.0 ** -10, 0.0, -0.0, 7.0])
    k = k.to(torch.float16)
    v = torch.flip(k, dims=[0]).contiguous()
    p = problem(lens=[6], hq=hkv, hkv=hkv, d=d, bs=8, dtype=W.F16, kv_data=(k, v))
    codes, scales = device_fp8(p)
    ref = oracle.build_cache(p)
    got = host(codes, scales)
    assert np.array_equal(got.codes, ref.codes)
    assert np.array_equal(got.scales.view(np.uint32), ref.scales.view(np.uint32))


LENS = [1, 63, 64, 65, 1000, 3001, 17, 4096]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bs", [8, 16, 32, 64, 128, 512])
def test_fp8_decode_block_sizes(bs, d):
    p = problem(lens=LENS, bs=bs, hq=4, hkv=4, d=d, dtype=W.F16, seed=bs)
    codes, scales = device_fp8(p)
    out, lse = decode(p, codes, scales)
    ref, ref_lse = oracle.attention_of(p, host(codes, scales))
    check_close(out, ref, W.F16, roundings=roundings(p), what="fp8 bs=%d d=%d" % (bs, d))
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (16, 4), (32, 4)])
@pytest.mark.parametrize("d", [64, 128])
def test_fp8_decode_groupings(dtype, hq, hkv, d):
    p = problem(lens=[5, 700, 129, 2000], hq=hq, hkv=hkv, d=d, dtype=dtype, bs=32, seed=hq + hkv + d)
    codes, scales = device_fp8(p)
    out, lse = decode(p, codes, scales)
    ref, ref_lse = oracle.attention_of(p, host(codes, scales))
    check_close(out, ref, dtype, roundings=roundings(p), what="fp8 %s hq=%d hkv=%d d=%d" % (dtype, hq, hkv, d))
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("num_splits", [1, 3, 64])
def test_fp8_decode_splits_fp32_output(num_splits):
    """FP32 output: only P is rounded to 16 bits (f16) on the way."""
    p = problem(lens=[3000, 64, 1, 2500], hq=8, hkv=2, bs=16, dtype=W.BF16, mb=256)
    codes, scales = device_fp8(p)
    out, lse = decode(p, codes, scales, num_splits=num_splits, out_dtype=torch.float32)
    ref, ref_lse = oracle.attention_of(p, host(codes, scales))
    check_close(out, ref, W.BF16, roundings=roundings(p, fp32_out=True), what="fp8 splits=%d fp32 out" % num_splits)
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("bs", [128, 512])
def test_fp8_decode_seven_splits_in_large_pages(bs):
    """7 requested splits over a 3072-token capacity: splits are rounded up to a multiple of 128
    tokens (512 here, 6 splits), and inside 128- and 512-token pages a split's tiles start at
    offsets 0 and 128..384 of a page."""
    p = problem(lens=[3000, 700, 129], hq=8, hkv=8, bs=bs, dtype=W.BF16, mb=3072 // bs)
    assert pkv.decode_split_tokens(3, 8, 8, 128, bs, 3072 // bs, num_splits=7) == 512
    codes, scales = device_fp8(p)
    out, lse = decode(p, codes, scales, num_splits=7)
    ref, ref_lse = oracle.attention_of(p, host(codes, scales))
    check_close(out, ref, W.BF16, roundings=roundings(p), what="fp8 bs=%d 7 splits" % bs)
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("hq,hkv", [(32, 1), (64, 4)])
def test_fp8_decode_mqa_and_wide_groups(hq, hkv):
    p = problem(lens=[5, 700, 129, 2000], hq=hq, hkv=hkv, d=128, dtype=W.BF16, bs=16, seed=hq)
    codes, scales = device_fp8(p)
    out, lse = decode(p, codes, scales)
    ref, ref_lse = oracle.attention_of(p, host(codes, scales))
    check_close(out, ref, W.BF16, roundings=roundings(p), what="fp8 hq=%d hkv=%d" % (hq, hkv))
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-5)


def test_fp8_decode_step_append_then_decode():
    """A decode step: one new token per sequence quantised into its page, then attention over it."""
    p = problem(lens=[100, 31, 512, 7], hq=8, hkv=2, bs=16, dtype=W.BF16, extra=12, mb=40)
    codes, scales = device_fp8(p)
    step = W.append_step(p, seed=4)
    pkv.kv_cache_append(codes, to_dev(step["k_new"]), to_dev(step["v_new"]), to_dev(step["cu_new_lens"]),
                        to_dev(step["ctx_before"]), to_dev(step["block_tables"]), scales=scales)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    ref_cache = oracle.build_cache(p)
    assert oracle.kv_cache_append_fp8(ref_cache, p.dtype, **step) == 0
    got = host(codes, scales)
    assert np.array_equal(got.codes, ref_cache.codes) and np.array_equal(got.scales, ref_cache.scales)
    lens = p.context_lens + 1
    out = pkv.paged_attn_decode(codes, to_dev(p.q), to_dev(step["block_tables"]), to_dev(lens), scale=p.scale,
                                scales=scales)
    torch.cuda.synchronize()
    ref, _ = oracle.paged_attention_fp8(p.dtype, got, p.q, p.num_q_heads, p.cu_q_lens, lens, step["block_tables"],
                                        p.scale, False)
    check_close(out, ref, W.BF16, roundings=roundings(p), what="fp8 decode step")


def prefill_problem(*, lens, q_lens, hq=8, hkv=8, d=128, bs=16, dtype=W.BF16, causal=True, seed=11, extra=5):
    nb = sum((L + bs - 1) // bs for L in lens) + extra
    order = torch.randperm(nb, generator=torch.Generator().manual_seed(seed + 3)).tolist()
    return W.make_problem("fp", batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                          context_lens=lens, q_lens=q_lens, dtype=dtype, causal=causal, seed=seed,
                          num_blocks=nb, free_order=order, kv_format="fp8")


def run_prefill_fp8(p, codes, scales, out_dtype=None):
    lse = torch.empty((p.total_q, p.num_q_heads), dtype=torch.float32, device="cuda")
    out = pkv.paged_attn_prefill(codes, to_dev(p.q), to_dev(p.cu_q_lens), to_dev(p.context_lens),
                                 to_dev(p.block_tables), max_q_len=int(p.q_lens.max()), scale=p.scale,
                                 causal=p.causal, out_dtype=out_dtype, lse=lse, scales=scales)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    return out, lse


# Roundings on the FP8 prefill path: the output and P' = P * (V row scale / W) in f16. The codes
# enter the products exactly, and the row scales only in FP32.
PREFILL_ROUNDINGS = 2


@pytest.mark.parametrize("bs", [8, 16, 128, 512])
def test_fp8_prefill_block_sizes(bs):
    p = prefill_problem(lens=[300, 129, 700], q_lens=[300, 1, 257], bs=bs, hq=4, hkv=4, seed=bs)
    codes, scales = device_fp8(p)
    out, lse = run_prefill_fp8(p, codes, scales)
    ref, ref_lse = oracle.attention_of(p, host(codes, scales))
    check_close(out, ref, p.dtype, roundings=PREFILL_ROUNDINGS, what="fp8 prefill bs=%d" % bs)
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-4, atol=1e-4)


@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 4), (32, 1)])
def test_fp8_prefill_dtypes_gqa_causality(dtype, causal, hq, hkv):
    p = prefill_problem(lens=[520, 77, 1000], q_lens=[200, 77, 384], hq=hq, hkv=hkv, dtype=dtype, causal=causal,
                        seed=hq * 7 + hkv)
    codes, scales = device_fp8(p)
    out, lse = run_prefill_fp8(p, codes, scales)
    ref, ref_lse = oracle.attention_of(p, host(codes, scales))
    check_close(out, ref, dtype, roundings=PREFILL_ROUNDINGS,
                what="fp8 prefill %s causal=%s hq=%d hkv=%d" % (dtype, causal, hq, hkv))
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-4, atol=1e-4)


def test_fp8_prefill_fp32_output():
    p = prefill_problem(lens=[640, 333], q_lens=[512, 333], hq=4, hkv=4, dtype=W.BF16, bs=32, seed=3)
    codes, scales = device_fp8(p)
    out, lse = run_prefill_fp8(p, codes, scales, out_dtype=torch.float32)
    ref, _ = oracle.attention_of(p, host(codes, scales))
    check_close(out, ref, W.BF16, roundings=PREFILL_ROUNDINGS - 1, what="fp8 prefill fp32 out")


def test_fp8_prefill_chunks_match_decode():
    """The last row of a causal chunk over the FP8 cache and a decode of that row's query over the
    same context compute the same attention."""
    p = prefill_problem(lens=[900, 300], q_lens=[128, 300], hq=8, hkv=2, dtype=W.BF16, seed=21)
    codes, scales = device_fp8(p)
    out, _ = run_prefill_fp8(p, codes, scales, out_dtype=torch.float32)
    last = (p.cu_q_lens[1:] - 1).long()
    qd = p.q[last].contiguous()
    dec = pkv.paged_attn_decode(codes, to_dev(qd), to_dev(p.block_tables), to_dev(p.context_lens), scale=p.scale,
                                out_dtype=torch.float32, scales=scales)
    torch.cuda.synchronize()
    np.testing.assert_allclose(out[last.cuda()].cpu().numpy(), dec.cpu().numpy(), atol=2e-2, rtol=0)


@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
@pytest.mark.parametrize("bs", [8, 16, 128])
def test_fp8_prefill_head_dim_64(dtype, bs):
    """head_dim 64: the codes (64-byte rows) land in buffers of their own and are converted into
    the f16 tile; causal chunks, a one-token context, GQA, ragged lengths and page sizes."""
    p = prefill_problem(lens=[40, 1, 700, 300], q_lens=[8, 1, 300, 300], hq=8, hkv=2, d=64, bs=bs, dtype=dtype,
                        seed=bs + 1)
    codes, scales = device_fp8(p)
    out, lse = run_prefill_fp8(p, codes, scales)
    ref, ref_lse = oracle.attention_of(p, host(codes, scales))
    check_close(out, ref, dtype, roundings=PREFILL_ROUNDINGS, what="fp8 prefill d=64 %s bs=%d" % (dtype, bs))
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-4, atol=1e-4)


def test_fp8_decode_full_7b_size_sampled():
    """The 7B-like decode batch (16 x 1k-8k contexts, 32 heads x 128) on an FP8 cache, in the
    launch configuration the benchmark times; every row against the oracle."""
    p = W.decode_7b(pool_init="none", device="cuda", kv_format="fp8")
    shape = (p.num_blocks, 2, 32, 16, 128)
    codes = torch.zeros(shape, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(shape[:4], dtype=torch.float32, device="cuda")
    pkv.kv_cache_append(codes, p.k_ctx, p.v_ctx, p.cu_ctx_lens.cuda(),
                        torch.zeros(p.batch, dtype=torch.int32, device="cuda"), p.block_tables.cuda(), scales=scales)
    out = pkv.paged_attn_decode(codes, p.q, p.block_tables.cuda(), p.context_lens.cuda(), scale=p.scale,
                                scales=scales)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    p.q = p.q.cpu()
    ref, _ = oracle.attention_of(p, host(codes, scales))
    check_close(out, ref, W.F16, roundings=roundings(p), what="fp8 7B decode")


@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
def test_fp8_prefill_tiny_zero_and_growing_v_scales(dtype):
    """V rows whose magnitudes rise from 2^-20 to 2^4 along each sequence (some rows all zero):
    row scales far below f16's normal range, and a largest V scale that keeps growing from key
    tile to key tile, so the factor W the kernel keeps on O grows several times mid-sequence
    (each time O is rescaled by a power of two). Decode over the same cache is checked too."""
    lens, q_lens = [900, 1300, 257], [300, 1300, 257]
    gen = torch.Generator().manual_seed(41)
    tot = sum(lens)
    k = W.randn_t(gen, (tot, 4, 128), dtype)
    v = W.randn_t(gen, (tot, 4, 128), dtype).float()
    mag = torch.cat([torch.exp2(torch.linspace(-20.0, 4.0, L)) for L in lens])
    v = v * mag[:, None, None]
    v[torch.arange(0, tot, 97)] = 0.0                     # all-zero rows: scale 0
    v = v.to(W.TORCH_DTYPE[dtype])
    p = prefill_problem(lens=lens, q_lens=q_lens, hq=8, hkv=4, dtype=dtype, seed=43)
    p = W.make_problem("fp", batch=3, num_q_heads=8, num_kv_heads=4, head_dim=128, block_size=16,
                       context_lens=lens, q_lens=q_lens, dtype=dtype, causal=True, seed=43,
                       num_blocks=p.num_blocks, kv_format="fp8", kv_data=(k, v))
    codes, scales = device_fp8(p)
    out, lse = run_prefill_fp8(p, codes, scales)
    ref, ref_lse = oracle.attention_of(p, host(codes, scales))
    check_close(out, ref, dtype, roundings=PREFILL_ROUNDINGS, what="fp8 prefill growing scales %s" % dtype)
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-4, atol=1e-4)
    # decode of one query per sequence over the same cache
    qd = W.randn_t(gen, (3, 8, 128), dtype)
    dec = pkv.paged_attn_decode(codes, to_dev(qd), to_dev(p.block_tables), to_dev(p.context_lens), scale=p.scale,
                                scales=scales)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    ref_d, _ = oracle.attention_of(p, host(codes, scales), q=qd, cu_q_lens=W.cu_lens([1, 1, 1]))
    check_close(dec, ref_d, dtype, roundings=roundings(p), what="fp8 decode growing scales %s" % dtype)


@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 128), (32, 4, 128), (16, 2, 64)])
def test_fp8_decode_workspace_contents_and_repeated_calls(hq, hkv, d):
    """Over an FP8 cache too: a workspace of random bytes, an output full of NaN and three calls on
    the same workspace give the same bits, within the oracle's bounds."""
    p = problem(lens=[0, 700, 1, 2500, 129, 2048], hq=hq, hkv=hkv, d=d, dtype=W.BF16, bs=16, mb=160, seed=hq + d)
    codes, scales = device_fp8(p)
    q, bt, ctx = to_dev(p.q), to_dev(p.block_tables), to_dev(p.context_lens)
    need = pkv.decode_workspace_size(p.batch, hq, hkv, d, 16, bt.shape[1], 7)
    gen = torch.Generator(device="cuda").manual_seed(12)
    ws = torch.randint(0, 256, (need,), dtype=torch.uint8, device="cuda", generator=gen)
    runs = []
    for _ in range(3):
        out = torch.full((p.batch, hq, d), float("nan"), dtype=q.dtype, device="cuda")
        lse = torch.full((p.batch, hq), float("nan"), dtype=torch.float32, device="cuda")
        pkv.paged_attn_decode(codes, q, bt, ctx, scale=p.scale, num_splits=7, workspace=ws, out=out, lse=lse,
                              scales=scales)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        runs.append((out.cpu(), lse.cpu()))
    for o, l in runs[1:]:
        assert torch.equal(o, runs[0][0]) and torch.equal(l, runs[0][1])
    ref, ref_lse = oracle.attention_of(p, host(codes, scales))
    check_close(runs[0][0], ref, W.BF16, roundings=roundings(p), what="fp8 hq=%d hkv=%d d=%d" % (hq, hkv, d))
    np.testing.assert_allclose(runs[0][1].numpy(), ref_lse, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("hq,hkv,d", [(8, 2, 128), (4, 4, 64)])
def test_fp8_decode_step_is_decode_then_append(hq, hkv, d):
    """paged_attn_decode_step over an FP8 cache: the decode's output bits, and the oracle's
    quantising append of the step's token (the append kernel runs after the decode)."""
    p = problem(lens=[100, 31, 512, 7, 0], hq=hq, hkv=hkv, d=d, bs=16, dtype=W.BF16, extra=12, mb=40)
    codes, scales = device_fp8(p)
    step = W.append_step(p, seed=6)
    q, bt, ctx = to_dev(p.q), to_dev(step["block_tables"]), to_dev(p.context_lens)
    ref_out = pkv.paged_attn_decode(codes, q, bt, ctx, scale=p.scale, scales=scales)
    torch.cuda.synchronize()
    ref_cache = host(codes, scales)
    assert oracle.kv_cache_append_fp8(ref_cache, p.dtype, **step) == 0
    out = pkv.paged_attn_decode_step(codes, q, bt, ctx, to_dev(step["k_new"]), to_dev(step["v_new"]), scale=p.scale,
                                     scales=scales)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    assert torch.equal(out, ref_out)
    got = host(codes, scales)
    assert np.array_equal(got.codes, ref_cache.codes) and np.array_equal(got.scales, ref_cache.scales)
