"""GPU parity: kv_cache_append (bit-exact) and paged_attn_decode (within the stated tolerances)
against the CPU oracle, through the C ABI."""
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


def problem(*, lens, hq=8, hkv=8, d=128, bs=16, dtype=W.F16, seed=5, extra=7, mb=None):
    pages = sum((L + bs - 1) // bs for L in lens)
    nb = pages + extra
    order = torch.randperm(nb, generator=torch.Generator().manual_seed(seed + 9)).tolist()
    return W.make_problem("t", batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                          context_lens=lens, q_lens=[1] * len(lens), dtype=dtype, causal=False, seed=seed,
                          num_blocks=nb, free_order=order, max_blocks_per_seq=mb)


def run_decode(p, cache, num_splits=0, out_dtype=None, with_lse=True):
    q = to_dev(p.q)
    lse = torch.empty((p.batch, p.num_q_heads), dtype=torch.float32, device="cuda") if with_lse else None
    out = pkv.paged_attn_decode(cache, q, to_dev(p.block_tables), to_dev(p.context_lens), scale=p.scale,
                                num_splits=num_splits, out_dtype=out_dtype, lse=lse)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    return out, lse


# ------------------------------------------------------------------------------------------------
# append
# ------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("bs", [8, 16, 64, 512])
@pytest.mark.parametrize("d,dtype", [(128, W.F16), (64, W.BF16)])
def test_append_bit_exact(bs, d, dtype):
    p = problem(lens=[1, 37, 100, 513], bs=bs, d=d, dtype=dtype, hq=4, hkv=4)
    dev = device_cache(p)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    ref = oracle.build_cache(p)
    assert np.array_equal(cache_bits(dev), ref)       # every pool element, untouched pages included


def test_append_two_steps_and_decode_step_tokens():
    """Context then a chunk (ctx_before > 0), then one decode-step token per sequence."""
    dec, pre = W.tiny()
    cu = pre.cu_ctx_lens.tolist()
    first = [37, 100]
    rows1 = torch.cat([torch.arange(cu[0], cu[0] + 37), torch.arange(cu[1], cu[1] + 100)])
    rows2 = torch.cat([torch.arange(cu[0] + 37, cu[1]), torch.arange(cu[1] + 100, cu[2])])
    dev = pre.pool_init.to("cuda")
    ref = oracle.empty_cache_bits(pre)
    bt = to_dev(pre.block_tables)
    for rows, lens, before in ((rows1, first, [0, 0]), (rows2, [48, 48], first)):
        k, v = pre.k_ctx[rows], pre.v_ctx[rows]
        pkv.kv_cache_append(dev, to_dev(k), to_dev(v), to_dev(W.cu_lens(lens)),
                            to_dev(torch.tensor(before, dtype=torch.int32)), bt)
        oracle.kv_cache_append(ref, k, v, W.cu_lens(lens), torch.tensor(before, dtype=torch.int32),
                               pre.block_tables)
    torch.cuda.synchronize()
    assert np.array_equal(cache_bits(dev), ref)
    step = W.append_step(dec, seed=3)
    pkv.kv_cache_append(dev, to_dev(step["k_new"]), to_dev(step["v_new"]), to_dev(step["cu_new_lens"]),
                        to_dev(step["ctx_before"]), to_dev(step["block_tables"]))
    oracle.kv_cache_append(ref, step["k_new"], step["v_new"], step["cu_new_lens"], step["ctx_before"],
                           step["block_tables"])
    torch.cuda.synchronize()
    assert np.array_equal(cache_bits(dev), ref)
    assert pkv.get_device_error() == 0


def test_append_bad_page_is_flagged_not_faulted():
    p = problem(lens=[40, 20], bs=16, hq=2, hkv=2)
    bt = p.block_tables.clone()
    bt[0, 1] = p.num_blocks + 5          # out of range: tokens 16..31 of sequence 0 must be skipped
    dev = p.pool_init.to("cuda")
    pkv.kv_cache_append(dev, to_dev(p.k_ctx), to_dev(p.v_ctx), to_dev(p.cu_ctx_lens),
                        torch.zeros(2, dtype=torch.int32, device="cuda"), to_dev(bt))
    assert pkv.get_device_error() == 5
    assert pkv.get_device_error() == 0     # the word is cleared by the read
    ref = oracle.empty_cache_bits(p)
    assert oracle.kv_cache_append(ref, p.k_ctx, p.v_ctx, p.cu_ctx_lens, torch.zeros(2, dtype=torch.int32), bt) == -1
    assert np.array_equal(cache_bits(dev), ref)


# ------------------------------------------------------------------------------------------------
# decode
# ------------------------------------------------------------------------------------------------

def test_tiny_decode_all_elements():
    dec, _ = W.tiny()
    cache = device_cache(dec)
    out, lse = run_decode(dec, cache)
    ref, ref_lse = oracle.attention_of(dec, cache_bits(cache))
    check_close(out, ref, "f16", roundings=1, what="tiny decode")
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-5)


LENS = [1, 63, 64, 65, 1000, 3001, 17, 4096]


@pytest.mark.parametrize("bs", [8, 16, 32, 64, 128, 512])
def test_decode_block_sizes(bs):
    p = problem(lens=LENS, bs=bs, hq=4, hkv=4)
    cache = device_cache(p)
    out, lse = run_decode(p, cache)
    ref, ref_lse = oracle.attention_of(p, cache_bits(cache))
    check_close(out, ref, "f16", roundings=1, what="bs=%d" % bs)
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (16, 4), (16, 2)])
@pytest.mark.parametrize("d", [64, 128])
def test_decode_gqa_dtypes(dtype, hq, hkv, d):
    p = problem(lens=[5, 700, 129, 2000], hq=hq, hkv=hkv, d=d, dtype=dtype, bs=32, seed=hq + hkv + d)
    cache = device_cache(p)
    out, lse = run_decode(p, cache)
    ref, ref_lse = oracle.attention_of(p, cache_bits(cache))
    check_close(out, ref, dtype, roundings=1, what="%s hq=%d hkv=%d d=%d" % (dtype, hq, hkv, d))
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("num_splits", [1, 2, 3, 7, 64])
def test_decode_explicit_splits_and_fp32_output(num_splits):
    p = problem(lens=[3000, 64, 1, 2500], hq=8, hkv=2, bs=16, dtype=W.BF16, mb=256)
    cache = device_cache(p)
    out, lse = run_decode(p, cache, num_splits=num_splits, out_dtype=torch.float32)
    ref, ref_lse = oracle.attention_of(p, cache_bits(cache))
    # FP32 output: nothing on the path is rounded to bf16 (P enters the 4-head group's tensor-core
    # P.V as a bf16 part plus its bf16 remainder) -> the literal bounds
    check_close(out, ref, "bf16", roundings=0, what="splits=%d fp32 out" % num_splits)
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-5)


def test_decode_fp32_output_literal_bounds_mha():
    """MHA decode keeps P in FP32: with an FP32 output nothing is rounded to bf16 -> literal bounds."""
    p = problem(lens=[3000, 64, 1, 2500], hq=4, hkv=4, bs=16, dtype=W.BF16, mb=256)
    cache = device_cache(p)
    out, lse = run_decode(p, cache, num_splits=3, out_dtype=torch.float32)
    ref, ref_lse = oracle.attention_of(p, cache_bits(cache))
    check_close(out, ref, "bf16", roundings=0, what="mha fp32 out")
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-5)


def test_decode_special_cases():
    """Empty context -> 0 / -inf; one token -> V exactly; identical keys -> mean(V)."""
    L = 300
    gen = torch.Generator().manual_seed(4)
    krow = torch.randn(1, 4, 128, generator=gen).to(torch.float16)
    k = torch.cat([torch.randn(1, 4, 128, generator=gen).to(torch.float16), krow.expand(L, 4, 128)])
    v = torch.randn(1 + L, 4, 128, generator=gen).to(torch.float16)
    p = problem(lens=[0, 1, L], hq=4, hkv=4, bs=16)
    p2 = W.make_problem("s", batch=3, num_q_heads=4, num_kv_heads=4, head_dim=128, block_size=16,
                        context_lens=[0, 1, L], q_lens=[1, 1, 1], dtype=W.F16, causal=False, seed=5,
                        num_blocks=p.num_blocks, free_order=list(range(p.num_blocks)), kv_data=(k, v))
    cache = device_cache(p2)
    out, lse = run_decode(p2, cache, out_dtype=torch.float32)
    o = out.cpu()
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0].cpu()))
    assert torch.equal(o[1], v[0].to(torch.float32))                       # bit-exact V
    mean_v = v[1:].to(torch.float64).mean(0)
    assert torch.allclose(o[2].to(torch.float64), mean_v, atol=1e-5, rtol=0)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 4)])
def test_decode_inputs_written_by_the_previous_kernel(hq, hkv):
    """Lengths, block table and q produced by device kernels queued just before the decode call
    (no synchronisation in between), after a kernel that left other values there: the decode
    kernels start early under programmatic launch, so they must still see the final inputs."""
    p = problem(lens=[700, 1, 2049, 130], hq=hq, hkv=hkv, bs=16, dtype=W.F16, seed=hq)
    cache = device_cache(p)
    ref, _ = oracle.attention_of(p, cache_bits(cache))
    lens_true, bt_true, q_true = to_dev(p.context_lens), to_dev(p.block_tables), to_dev(p.q)
    lens, bt, q = torch.empty_like(lens_true), torch.empty_like(bt_true), torch.empty_like(q_true)
    busy = torch.empty(1 << 26, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    for _ in range(3):
        lens.fill_(3)
        bt.fill_(0)
        q.fill_(0.5)
        busy.fill_(1.0)                                   # a long kernel ahead of the writers
        torch.add(lens_true, 0, out=lens)
        torch.add(bt_true, 0, out=bt)
        torch.mul(q_true, 1, out=q)
        out = pkv.paged_attn_decode(cache, q, bt, lens, scale=p.scale)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        check_close(out, ref, "f16", roundings=1, what="inputs from kernels hq=%d" % hq)


@pytest.mark.parametrize("hq,hkv", [(2, 2), (8, 2)])
def test_decode_large_batch_many_equal_lengths(hq, hkv):
    """Hundreds of sequences, most sharing a handful of lengths: every CTA numbers the work
    units from the lengths on its own, so the numbering must not depend on thread timing."""
    gen = torch.Generator().manual_seed(17)
    choices = torch.tensor([0, 1, 64, 65, 300, 1000, 1500])
    lens = choices[torch.randint(0, len(choices), (600,), generator=gen)].tolist()
    p = problem(lens=lens, hq=hq, hkv=hkv, d=64, bs=16, dtype=W.BF16, seed=hq, mb=128)
    cache = device_cache(p)
    ref, ref_lse = oracle.attention_of(p, cache_bits(cache))
    for splits in (0, 5):
        out, lse = run_decode(p, cache, num_splits=splits)
        check_close(out, ref, W.BF16, roundings=1, what="batch 600 splits=%d" % splits)
        np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
@pytest.mark.parametrize("hq,hkv,d", [(32, 1, 128), (16, 1, 64), (64, 4, 128), (24, 1, 128), (64, 1, 128),
                                     (32, 1, 64)])
def test_decode_mqa_and_wide_groups(dtype, hq, hkv, d):
    """One KV head for many query heads (MQA) and groups above 8: the tensor-core kernel takes
    the query heads of a KV head in units of 32 (head_dim 128), 16 or 8, all units reading that
    KV head's pages (64 heads: two units of 32; 24: three of 8; head_dim 64 at 32: two of 16)."""
    p = problem(lens=[5, 700, 129, 2000], hq=hq, hkv=hkv, d=d, dtype=dtype, bs=32, seed=hq * 3 + d)
    cache = device_cache(p)
    out, lse = run_decode(p, cache)
    ref, ref_lse = oracle.attention_of(p, cache_bits(cache))
    check_close(out, ref, dtype, roundings=1, what="%s hq=%d hkv=%d d=%d" % (dtype, hq, hkv, d))
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-5)


def test_decode_bad_page_flags_error():
    p = problem(lens=[200, 50], hq=4, hkv=4, bs=16)
    cache = device_cache(p)
    bt = p.block_tables.clone()
    bt[0, 3] = -7
    pkv.paged_attn_decode(cache, to_dev(p.q), to_dev(bt), to_dev(p.context_lens), scale=p.scale)
    assert pkv.get_device_error() == 5
    lens = p.context_lens.clone()
    lens[1] = 10 ** 6                      # beyond the table's capacity: clamped and flagged
    pkv.paged_attn_decode(cache, to_dev(p.q), to_dev(p.block_tables), to_dev(lens), scale=p.scale)
    assert pkv.get_device_error() == 5
    assert pkv.get_device_error() == 0


@pytest.mark.parametrize("d", [64, 128, 256])
def test_attn_combine_entry_point(d):
    rng = np.random.default_rng(3)
    po = rng.standard_normal((37, 5, d))
    pl = rng.standard_normal((37, 5)) * 3
    pl[0, :] = -np.inf
    pl[1, 2:] = -np.inf
    ref, ref_lse = oracle.attn_combine(po, pl)
    lse = torch.empty(37, dtype=torch.float32, device="cuda")
    out = pkv.attn_combine(torch.tensor(po, dtype=torch.float32, device="cuda"),
                           torch.tensor(pl, dtype=torch.float32, device="cuda"), lse=lse)
    torch.cuda.synchronize()
    np.testing.assert_allclose(out.cpu().numpy(), ref, rtol=2e-6, atol=2e-6)
    got_lse = lse.cpu().numpy()
    assert np.isneginf(got_lse[0]) and np.all(out[0].cpu().numpy() == 0)
    np.testing.assert_allclose(got_lse[1:], ref_lse[1:], rtol=1e-6, atol=1e-6)


# ------------------------------------------------------------------------------------------------
# head_dim 256 (every grouping runs on the tcgen05 decode kernel, with 64-token key tiles)
# ------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("bs", [16, 64])
def test_append_bit_exact_head_dim_256(bs):
    p = problem(lens=[1, 37, 300, 513], bs=bs, d=256, dtype=W.BF16, hq=2, hkv=2)
    dev = device_cache(p)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    assert np.array_equal(cache_bits(dev), oracle.build_cache(p))


@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
@pytest.mark.parametrize("hq,hkv", [(2, 2), (4, 2), (6, 2), (8, 2), (16, 2), (32, 1)])
def test_decode_head_dim_256(dtype, hq, hkv):
    p = problem(lens=[5, 700, 129, 2000, 1], hq=hq, hkv=hkv, d=256, dtype=dtype, bs=32, seed=hq + 256)
    cache = device_cache(p)
    out, lse = run_decode(p, cache)
    ref, ref_lse = oracle.attention_of(p, cache_bits(cache))
    check_close(out, ref, dtype, roundings=1, what="d=256 %s hq=%d hkv=%d" % (dtype, hq, hkv))
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("num_splits", [1, 3, 7])
def test_decode_head_dim_256_splits_fp32_output(num_splits):
    """head_dim 256 with forced splits and an FP32 output: the stated bounds as written."""
    p = problem(lens=[3000, 64, 1, 2500], hq=8, hkv=8, d=256, bs=16, dtype=W.BF16, mb=256, seed=9)
    cache = device_cache(p)
    out, lse = run_decode(p, cache, num_splits=num_splits, out_dtype=torch.float32)
    ref, ref_lse = oracle.attention_of(p, cache_bits(cache))
    check_close(out, ref, "bf16", roundings=0, what="d=256 splits=%d fp32 out" % num_splits)
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("hq,hkv,d,dtype", [(8, 8, 128, W.F16), (4, 2, 64, W.BF16), (16, 4, 128, W.BF16),
                                            (16, 2, 64, W.F16), (24, 1, 128, W.BF16)])
@pytest.mark.parametrize("num_splits", [0, 7])
def test_decode_workspace_contents_and_repeated_calls(hq, hkv, d, dtype, num_splits):
    """The workspace needs no initialisation and a call leaves nothing in it that the next call
    depends on: a workspace full of random bytes, an output full of NaN (the rows of the empty
    context must be written) and three calls on the same workspace give the same bits, within the
    oracle's bounds, on every split-kernel path (CUDA cores, mma.sync groups, tcgen05)."""
    p = problem(lens=[0, 700, 1, 2500, 129, 2048], hq=hq, hkv=hkv, d=d, dtype=dtype, bs=16, mb=160,
                seed=hq + 3 * hkv + d)
    cache = device_cache(p)
    q, bt, ctx = to_dev(p.q), to_dev(p.block_tables), to_dev(p.context_lens)
    need = pkv.decode_workspace_size(p.batch, hq, hkv, d, 16, bt.shape[1], num_splits)
    assert need > 0
    gen = torch.Generator(device="cuda").manual_seed(11)
    ws = torch.randint(0, 256, (need,), dtype=torch.uint8, device="cuda", generator=gen)
    ws[: need // 3].fill_(255)
    runs = []
    for _ in range(3):
        out = torch.full((p.batch, hq, d), float("nan"), dtype=q.dtype, device="cuda")
        lse = torch.full((p.batch, hq), float("nan"), dtype=torch.float32, device="cuda")
        pkv.paged_attn_decode(cache, q, bt, ctx, scale=p.scale, num_splits=num_splits, workspace=ws, out=out, lse=lse)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        runs.append((out.cpu(), lse.cpu()))
    for o, l in runs[1:]:
        assert torch.equal(o, runs[0][0]) and torch.equal(l, runs[0][1])
    ref, ref_lse = oracle.attention_of(p, cache_bits(cache))
    check_close(runs[0][0], ref, dtype, roundings=1, what="hq=%d hkv=%d d=%d splits=%d" % (hq, hkv, d, num_splits))
    np.testing.assert_allclose(runs[0][1].numpy(), ref_lse, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("hq,hkv,d,dtype", [(8, 8, 128, W.F16), (4, 2, 64, W.BF16), (16, 4, 128, W.BF16),
                                            (16, 2, 64, W.F16), (24, 1, 128, W.BF16), (4, 2, 256, W.BF16)])
@pytest.mark.parametrize("bs", [16, 64])
def test_decode_step_is_decode_then_append(hq, hkv, d, dtype, bs):
    """paged_attn_decode_step: the same output and lse bits as paged_attn_decode over the context,
    and the cache of the oracle's append of the step's token at position context_lens[b] (the
    append written by the split kernel's merge warps for groups of 1, 2, 4, 8 at head_dim 64/128;
    by the append kernel after the tcgen05 decode for 24 heads on one KV head and head_dim 256)."""
    p = problem(lens=[0, 700, 1, 2500, 129, 2047, 64], hq=hq, hkv=hkv, d=d, dtype=dtype, bs=bs, mb=2560 // bs,
                seed=hq + hkv + d + bs, extra=9)
    step = W.append_step(p, seed=5)
    cache = device_cache(p)
    q, bt, ctx = to_dev(p.q), to_dev(step["block_tables"]), to_dev(p.context_lens)
    ref_lse = torch.empty((p.batch, hq), dtype=torch.float32, device="cuda")
    ref_out = pkv.paged_attn_decode(cache, q, bt, ctx, scale=p.scale, num_splits=3, lse=ref_lse)
    torch.cuda.synchronize()
    ref_bits = cache_bits(cache)
    assert oracle.kv_cache_append(ref_bits, step["k_new"], step["v_new"], step["cu_new_lens"], step["ctx_before"],
                                  step["block_tables"]) == 0
    lse = torch.full((p.batch, hq), float("nan"), dtype=torch.float32, device="cuda")
    out = pkv.paged_attn_decode_step(cache, q, bt, ctx, to_dev(step["k_new"]), to_dev(step["v_new"]), scale=p.scale,
                                     num_splits=3, lse=lse)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    assert np.array_equal(cache_bits(cache), ref_bits)


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2)])
def test_decode_step_full_table_is_flagged_and_skipped(hq, hkv):
    """A sequence whose table is full (context_lens[b] = capacity) has no position for the step's
    token: that token is skipped and PKV_ERR_DEVICE_RANGE raised; the others are appended and the
    attention is that of the whole contexts."""
    bs, mb = 16, 8
    p = problem(lens=[bs * mb, 40, bs * mb - 1], hq=hq, hkv=hkv, d=128, dtype=W.F16, bs=bs, mb=mb, extra=4)
    cache = device_cache(p)
    bt, ctx, q = to_dev(p.block_tables), to_dev(p.context_lens), to_dev(p.q)
    gen = torch.Generator().manual_seed(8)
    k_new = torch.randn(p.batch, hkv, 128, generator=gen).to(torch.float16)
    v_new = torch.randn(p.batch, hkv, 128, generator=gen).to(torch.float16)
    ref_out = pkv.paged_attn_decode(cache, q, bt, ctx, scale=p.scale)
    torch.cuda.synchronize()
    ref_bits = cache_bits(cache)
    assert oracle.kv_cache_append(ref_bits, k_new, v_new, W.cu_lens([1] * p.batch), p.context_lens,
                                  p.block_tables) == -1
    out = pkv.paged_attn_decode_step(cache, q, bt, ctx, to_dev(k_new), to_dev(v_new), scale=p.scale)
    assert pkv.get_device_error() == 5
    assert torch.equal(out, ref_out)
    assert np.array_equal(cache_bits(cache), ref_bits)


def _chosen_split(ws, need):
    # the split kernel leaves the split size it took in the workspace's last 16-byte slot
    return int(ws[need - 16:need - 12].view(torch.int32).item())


def _model_split(lens, c0, cap, unit_heads, grid):
    """The device's choice restated: the host split c0 or 1.5, 2, 3, 4 times it (rounded up to 128,
    at most the capacity rounded up), whichever minimises ceil(units / grid) * (split + 150)."""
    top = (cap + 127) // 128 * 128
    best = None
    for k, m in enumerate((2, 3, 4, 6, 8)):
        c = min((c0 * m // 2 + 127) // 128 * 128, top)
        units = sum((L - 1) // c + 1 for L in lens if L > 0) * unit_heads
        key = (-(-units // grid) * (min(c, cap) + 150), k)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


@pytest.mark.parametrize("batch,lo,hi,seed", [(128, 1024, 8192, 1241), (64, 2048, 16384, 3), (256, 512, 4096, 4)])
def test_decode_split_chosen_on_device(batch, lo, hi, seed):
    """Multi-query decode (32 query heads on one KV head, the tcgen05 path with two CTAs an SM)
    with an automatic split: the split kernel picks the split size from the lengths. The choice
    matches the model restated here, and the result is bit for bit the decode with that split
    requested explicitly."""
    gen = torch.Generator().manual_seed(seed)
    lens = torch.randint(lo, hi + 1, (batch,), generator=gen).tolist()
    bs = 16
    nb = sum((L + bs - 1) // bs for L in lens)
    p = W.make_problem("m", batch=batch, num_q_heads=32, num_kv_heads=1, head_dim=128, block_size=bs,
                       context_lens=lens, q_lens=[1] * batch, dtype=W.BF16, causal=False, seed=seed + 1,
                       num_blocks=nb, free_order=torch.randperm(nb, generator=gen).tolist())
    cache = device_cache(p)
    q, bt, ctx = to_dev(p.q), to_dev(p.block_tables), to_dev(p.context_lens)
    mb = bt.shape[1]
    cap = mb * bs
    need = pkv.decode_workspace_size(batch, 32, 1, 128, bs, mb)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    lse = torch.empty((batch, 32), dtype=torch.float32, device="cuda")
    out = pkv.paged_attn_decode(cache, q, bt, ctx, scale=p.scale, workspace=ws, lse=lse)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    chosen = _chosen_split(ws, need)
    c0 = pkv.decode_split_tokens(batch, 32, 1, 128, bs, mb)
    grid = 2 * torch.cuda.get_device_properties(0).multi_processor_count
    assert chosen == _model_split(lens, c0, cap, 1, grid), (chosen, c0)
    assert chosen >= c0 and chosen % 128 == 0
    # the same split requested (a split count whose split size is the chosen one, where one exists)
    ns = next((n for n in range(1, 2049) if pkv.decode_split_tokens(batch, 32, 1, 128, bs, mb, n) == chosen), None)
    if ns is not None:
        lse2 = torch.empty_like(lse)
        out2 = pkv.paged_attn_decode(cache, q, bt, ctx, scale=p.scale, num_splits=ns, lse=lse2)
        torch.cuda.synchronize()
        assert torch.equal(out, out2) and torch.equal(lse, lse2)
    ref, ref_lse = oracle.attention_of(p, cache_bits(cache))
    check_close(out, ref, W.BF16, roundings=1, what="split chosen on the device (%d tokens)" % chosen)
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("hq,hkv", [(2, 2), (8, 2)])
def test_decode_step_batch_slices(hq, hkv):
    """A decode step over more sequences than one launch's unit tables hold (the call runs in
    slices): every slice's split kernel appends its own sequences' new rows."""
    gen = torch.Generator().manual_seed(21)
    lens = torch.randint(0, 70, (2500,), generator=gen).tolist()
    p = problem(lens=lens, hq=hq, hkv=hkv, d=64, dtype=W.F16, bs=16, mb=8, seed=22, extra=2600)
    step = W.append_step(p, seed=23)
    cache = device_cache(p)
    q, bt, ctx = to_dev(p.q), to_dev(step["block_tables"]), to_dev(p.context_lens)
    ref_out = pkv.paged_attn_decode(cache, q, bt, ctx, scale=p.scale)
    torch.cuda.synchronize()
    ref_bits = cache_bits(cache)
    assert oracle.kv_cache_append(ref_bits, step["k_new"], step["v_new"], step["cu_new_lens"], step["ctx_before"],
                                  step["block_tables"]) == 0
    out = pkv.paged_attn_decode_step(cache, q, bt, ctx, to_dev(step["k_new"]), to_dev(step["v_new"]), scale=p.scale)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    assert torch.equal(out, ref_out)
    assert np.array_equal(cache_bits(cache), ref_bits)
