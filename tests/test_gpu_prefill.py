"""GPU parity of paged_attn_prefill (tcgen05 tensor-core kernel) against the CPU oracle through
the C ABI: causal (bottom-right aligned) and non-causal chunks, ragged query / context lengths,
block sizes 8..512, GQA, fp16 / bf16, FP32 output, and the long-prefill workload at full size on
sampled rows."""
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


def problem(*, lens, q_lens, hq=8, hkv=8, d=128, bs=16, dtype=W.BF16, causal=True, seed=11, extra=5):
    pages = sum((L + bs - 1) // bs for L in lens)
    nb = pages + extra
    order = torch.randperm(nb, generator=torch.Generator().manual_seed(seed + 3)).tolist()
    return W.make_problem("p", batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                          context_lens=lens, q_lens=q_lens, dtype=dtype, causal=causal, seed=seed,
                          num_blocks=nb, free_order=order)


def run_prefill(p, cache, out_dtype=None):
    lse = torch.empty((p.total_q, p.num_q_heads), dtype=torch.float32, device="cuda")
    out = pkv.paged_attn_prefill(cache, to_dev(p.q), to_dev(p.cu_q_lens), to_dev(p.context_lens),
                                 to_dev(p.block_tables), max_q_len=int(p.q_lens.max()), scale=p.scale,
                                 causal=p.causal, out_dtype=out_dtype, lse=lse)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    return out, lse


def check(p, cache, out, lse, roundings, what, rows=None):
    ref, ref_lse = oracle.attention_of(p, cache_bits(cache), rows=rows)
    got = out if rows is None else out[torch.as_tensor(rows, device=out.device)]
    info = check_close(got, ref, p.dtype, roundings=roundings, what=what)
    gl = (lse if rows is None else lse[torch.as_tensor(rows, device=lse.device)]).cpu().numpy()
    np.testing.assert_allclose(gl, ref_lse, rtol=1e-4, atol=1e-4)
    return info


def test_tiny_prefill_chunk_all_elements():
    _, pre = W.tiny()
    cache = device_cache(pre)
    out, lse = run_prefill(pre, cache)
    check(pre, cache, out, lse, roundings=2, what="tiny prefill")


@pytest.mark.parametrize("bs", [8, 16, 32, 64, 128, 256, 512])
def test_prefill_block_sizes(bs):
    p = problem(lens=[300, 129, 700], q_lens=[300, 1, 257], bs=bs, hq=4, hkv=4, seed=bs)
    cache = device_cache(p)
    out, lse = run_prefill(p, cache)
    check(p, cache, out, lse, roundings=2, what="bs=%d" % bs)


@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 128), (16, 4, 128), (8, 2, 64)])
def test_prefill_dtypes_gqa_causality(dtype, causal, hq, hkv, d):
    p = problem(lens=[520, 77, 1000], q_lens=[200, 77, 384], hq=hq, hkv=hkv, d=d, dtype=dtype, causal=causal,
                bs=16, seed=hq * 7 + d)
    cache = device_cache(p)
    out, lse = run_prefill(p, cache)
    check(p, cache, out, lse, roundings=2, what="%s causal=%s hq=%d hkv=%d d=%d" % (dtype, causal, hq, hkv, d))


def test_prefill_inputs_written_by_the_previous_kernel():
    """Query offsets, lengths, block table and q produced by device kernels queued just before
    the prefill call, with no synchronisation in between (the kernel starts early under
    programmatic launch and must still see them)."""
    p = problem(lens=[520, 77, 1000], q_lens=[200, 77, 384], hq=8, hkv=8, bs=16, seed=21)
    cache = device_cache(p)
    ref, _ = oracle.attention_of(p, cache_bits(cache))
    srcs = [to_dev(t) for t in (p.cu_q_lens, p.context_lens, p.block_tables, p.q)]
    dsts = [torch.empty_like(t) for t in srcs]
    busy = torch.empty(1 << 26, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    for _ in range(3):
        for t in dsts:
            t.fill_(1)
        busy.fill_(1.0)
        for src, dst in zip(srcs, dsts):
            torch.add(src, 0, out=dst)
        cu, ctx, bt, q = dsts
        out = pkv.paged_attn_prefill(cache, q, cu, ctx, bt, max_q_len=int(p.q_lens.max()), scale=p.scale,
                                     causal=True)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        check_close(out, ref, p.dtype, roundings=2, what="prefill inputs from kernels")


def test_prefill_mqa():
    p = problem(lens=[520, 77], q_lens=[200, 77], hq=32, hkv=1, d=128, dtype=W.BF16, causal=True, bs=16, seed=31)
    cache = device_cache(p)
    out, lse = run_prefill(p, cache)
    check(p, cache, out, lse, roundings=2, what="prefill mqa")


def test_prefill_fp32_output_single_rounding():
    p = problem(lens=[640, 333], q_lens=[512, 333], hq=4, hkv=4, dtype=W.BF16, bs=32, seed=3)
    cache = device_cache(p)
    out, lse = run_prefill(p, cache, out_dtype=torch.float32)
    # the only rounding to bf16 left on the path is P before the P.V contraction
    check(p, cache, out, lse, roundings=1, what="fp32 out")


def test_prefill_first_row_is_v0_and_q_len_one_is_decode():
    """Row 0 of a full causal prefill sees only key 0: its output is V_0 exactly (weight 1).
    A q_len-1 chunk equals the decode kernel's answer for the same context."""
    p = problem(lens=[256], q_lens=[256], hq=4, hkv=4, dtype=W.F16, bs=16, seed=9)
    cache = device_cache(p)
    out, _ = run_prefill(p, cache, out_dtype=torch.float32)
    v0 = p.v_ctx[0].to(torch.float32)
    assert torch.equal(out[0].cpu(), v0)
    d = problem(lens=[1000], q_lens=[1], hq=8, hkv=2, dtype=W.BF16, bs=16, seed=10)
    cache_d = device_cache(d)
    out_p, _ = run_prefill(d, cache_d, out_dtype=torch.float32)
    out_d = pkv.paged_attn_decode(cache_d, to_dev(d.q), to_dev(d.block_tables), to_dev(d.context_lens),
                                  scale=d.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    # both within their bounds of the oracle; the prefill rounds P to bf16, the decode nothing
    ref, _ = oracle.attention_of(d, cache_bits(cache_d))
    check_close(out_p, ref, "bf16", roundings=1, what="q_len 1 prefill")
    check_close(out_d, ref, "bf16", roundings=0, what="decode")


def test_prefill_bad_lengths_flag_error():
    p = problem(lens=[100], q_lens=[50], hq=4, hkv=4)
    cache = device_cache(p)
    bad = torch.tensor([40], dtype=torch.int32)        # q_len > context: invalid, flagged, no output
    pkv.paged_attn_prefill(cache, to_dev(p.q), to_dev(p.cu_q_lens), to_dev(bad), to_dev(p.block_tables),
                           max_q_len=50, scale=p.scale)
    assert pkv.get_device_error() == 5
    bt = p.block_tables.clone()
    bt[0, 2] = 10 ** 6                                # page id out of range: read as page 0, flagged
    pkv.paged_attn_prefill(cache, to_dev(p.q), to_dev(p.cu_q_lens), to_dev(p.context_lens), to_dev(bt),
                           max_q_len=50, scale=p.scale)
    assert pkv.get_device_error() == 5
    assert pkv.get_device_error() == 0


def long_prefill_rows(seed=5):
    """Rows checked at full size: every row of the first chunk (the 512 x 512 causal triangle,
    all boundary tiles) and of the last (the deepest rescale chains, 8k keys), plus a seeded
    1/64 of the rows of every other chunk (its first, its last and 6 more), for all 4 sequences;
    each row with all 32 heads."""
    gen = np.random.default_rng(seed)
    sel = []
    for b in range(4):
        for c in range(16):
            base = b * 8192 + c * 512
            if c in (0, 15):
                sel += list(range(base, base + 512))
            else:
                sel += [base, base + 511] + list(base + gen.choice(np.arange(1, 511), 6, replace=False))
    return sel


def run_long_prefill(p, cache, scales=None):
    """The 16 chunk calls exactly as the benchmark runs them: append the chunk, then attend."""
    bt = p.block_tables.cuda()
    outs = torch.empty_like(p.q)
    for c in range(16):
        v = W.prefill_chunk_view(p, c)
        rows = v["rows"].cuda()
        pkv.kv_cache_append(cache, p.k_ctx[rows].contiguous(), p.v_ctx[rows].contiguous(), v["cu_q_lens"].cuda(),
                            v["ctx_before"].cuda(), bt, scales=scales)
        outs[rows] = pkv.paged_attn_prefill(cache, p.q[rows].contiguous(), v["cu_q_lens"].cuda(),
                                            v["context_lens"].cuda(), bt, max_q_len=512, scale=p.scale,
                                            scales=scales)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    return outs


@pytest.mark.slow
def test_long_prefill_full_size():
    """4 x 8192 bf16, bs 16, 16 causal chunks of 512, as the benchmark runs it. The appended cache
    is compared bit for bit with the oracle's; then every row of chunks 0 and 15 and 1/64 of the
    others (35 328 rows x 32 heads) against the oracle, which takes about 10 s on 16 cores."""
    p = W.prefill_long(device="cuda")
    shape = (p.num_blocks, 2, p.num_kv_heads, p.block_size, p.head_dim)
    cache = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    outs = run_long_prefill(p, cache)
    bits = cache_bits(cache)
    assert np.array_equal(bits, oracle.build_cache(p))          # the appends, bit-exact
    sel = long_prefill_rows()
    ref, _ = oracle.paged_attention(p.dtype, bits, p.q, 32, p.cu_q_lens, p.context_lens, p.block_tables, p.scale,
                                    True, rows=sel)
    check_close(outs[torch.as_tensor(sel, device="cuda")], ref, "bf16", roundings=2, what="long prefill")


@pytest.mark.slow
def test_long_prefill_full_size_fp8_cache():
    """The same 4 x 8192 pass over an FP8 cache (the quantising append, then the FP8 prefill),
    the same rows checked: codes and scales bit for bit, then attention over the exactly
    dequantised cache within the FP8 prefill's bound."""
    from tests.test_gpu_fp8 import PREFILL_ROUNDINGS
    p = W.prefill_long(device="cuda", kv_format="fp8")
    shape = (p.num_blocks, 2, p.num_kv_heads, p.block_size, p.head_dim)
    codes = torch.zeros(shape, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(shape[:4], dtype=torch.float32, device="cuda")
    outs = run_long_prefill(p, codes, scales)
    host = oracle.Fp8Cache(codes.cpu().numpy(), scales.cpu().numpy())
    want = oracle.build_cache(p)
    assert np.array_equal(host.codes, want.codes) and np.array_equal(host.scales, want.scales)
    sel = long_prefill_rows()
    ref, _ = oracle.attention_of(p, host, rows=sel)
    check_close(outs[torch.as_tensor(sel, device="cuda")], ref, "bf16", roundings=PREFILL_ROUNDINGS,
                what="long prefill fp8")


# ------------------------------------------------------------------------------------------------
# head_dim 256 (prefill_wide.cu: one 128-row query tile a CTA, 64-key tiles)
# ------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (6, 1)])
def test_prefill_head_dim_256(dtype, causal, hq, hkv):
    p = problem(lens=[520, 77, 1000, 64], q_lens=[200, 77, 384, 1], hq=hq, hkv=hkv, d=256, dtype=dtype,
                causal=causal, bs=16, seed=hq * 5 + hkv)
    cache = device_cache(p)
    out, lse = run_prefill(p, cache)
    check(p, cache, out, lse, roundings=2, what="d=256 %s causal=%s hq=%d hkv=%d" % (dtype, causal, hq, hkv))


@pytest.mark.parametrize("bs", [8, 64, 256])
def test_prefill_head_dim_256_block_sizes_fp32_output(bs):
    """Block sizes below, at and above the 64-key tile; FP32 output leaves P's rounding alone."""
    p = problem(lens=[300, 129, 700], q_lens=[300, 2, 257], bs=bs, hq=4, hkv=2, d=256, seed=bs + 256)
    cache = device_cache(p)
    out, lse = run_prefill(p, cache, out_dtype=torch.float32)
    check(p, cache, out, lse, roundings=1, what="d=256 bs=%d fp32 out" % bs)


def test_prefill_head_dim_256_first_row_is_v0():
    p = problem(lens=[130], q_lens=[130], hq=2, hkv=2, d=256, dtype=W.F16, bs=16, seed=19)
    cache = device_cache(p)
    out, _ = run_prefill(p, cache, out_dtype=torch.float32)
    assert torch.equal(out[0].cpu(), p.v_ctx[0].to(torch.float32))


def test_mixed_call_head_dim_256():
    """Decode rows and prefill chunks in one call at head_dim 256: the tcgen05 decode for the single
    rows, the wide prefill kernel for the chunks."""
    lens, q_lens = [700, 1, 300, 1500, 90], [1, 1, 200, 1, 90]
    p = problem(lens=lens, q_lens=q_lens, hq=8, hkv=2, d=256, dtype=W.BF16, bs=16, seed=77)
    cache = device_cache(p)
    lse = torch.empty((p.total_q, p.num_q_heads), dtype=torch.float32, device="cuda")
    out = pkv.paged_attn_mixed(cache, to_dev(p.q), to_dev(p.cu_q_lens), to_dev(p.context_lens),
                               to_dev(p.block_tables), max_q_len=int(p.q_lens.max()), scale=p.scale, causal=True,
                               lse=lse)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    ref, ref_lse = oracle.attention_of(p, cache_bits(cache))
    check_close(out, ref, p.dtype, roundings=2, what="mixed d=256")
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-4, atol=1e-4)
