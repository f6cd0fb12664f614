"""Pins for the CPU oracle: each test ties it to something other than itself --
a library routine, a closed form, an invariant, or the online-softmax algorithm
printed on the ipipp.com page ("Flash Attention与Paged Attention如何共同优化大模型推理？",
section 2) -- so that a dropped term, a wrong sign or index, or a transposed
operand in the oracle fails at least one of them."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from paged_kv_flash_cache_gb300 import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def small_problem(*, seed=7, lens=(5, 33, 70), hq=4, hkv=4, d=32, bs=16, dtype=W.F16, causal=False,
                  q_lens=None, extra_blocks=3, free_order=None, kv_data=None):
    q_lens = q_lens or [1] * len(lens)
    pages = sum((L + bs - 1) // bs for L in lens)
    nb = pages + extra_blocks
    if free_order is None:
        free_order = torch.randperm(nb, generator=torch.Generator().manual_seed(seed + 100)).tolist()
    return W.make_problem("t", batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                          context_lens=list(lens), q_lens=list(q_lens), dtype=dtype, causal=causal, seed=seed,
                          num_blocks=nb, free_order=free_order, kv_data=kv_data)


def contiguous_kv(p, b):
    """Sequence b's K and V as [Hkv, L, D] float64, straight from the generator (no pages)."""
    cu = p.cu_ctx_lens.tolist()
    k = p.k_ctx[cu[b]:cu[b + 1]].to(torch.float64).permute(1, 0, 2)
    v = p.v_ctx[cu[b]:cu[b + 1]].to(torch.float64).permute(1, 0, 2)
    return k, v


def sdpa_reference(p, b):
    """torch's scaled_dot_product_attention in float64 for sequence b (KV heads replicated per group)."""
    k, v = contiguous_kv(p, b)
    g = p.num_q_heads // p.num_kv_heads
    k = k.repeat_interleave(g, dim=0)[None]
    v = v.repeat_interleave(g, dim=0)[None]
    cq = p.cu_q_lens.tolist()
    q = p.q[cq[b]:cq[b + 1]].to(torch.float64).permute(1, 0, 2)[None]
    L = int(p.context_lens[b])
    ql = int(p.q_lens[b])
    mask = None
    if p.causal:
        pos = torch.arange(L - ql, L)[:, None]
        mask = torch.arange(L)[None, :] <= pos
        mask = mask[None, None]
    out = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=p.scale)
    return out[0].permute(1, 0, 2).numpy()


# ----------------------------------------------------------------------------------------------
# append
# ----------------------------------------------------------------------------------------------

def test_append_contiguous_special_case():
    """bs = max length with one page per sequence and an identity table is a contiguous cache:
    page b, K half, head h, row i must equal token i of sequence b."""
    lens = [9, 30, 17]
    bs = 32
    p = W.make_problem("c", batch=3, num_q_heads=2, num_kv_heads=2, head_dim=16, block_size=bs, context_lens=lens,
                       q_lens=[1, 1, 1], dtype=W.F16, causal=False, seed=3, num_blocks=3, free_order=[2, 1, 0])
    assert p.block_tables[:, 0].tolist() == [0, 1, 2]
    cache = oracle.build_cache(p)
    c = torch.from_numpy(cache.view(np.int16)).view(torch.float16)
    for b in range(3):
        k, v = contiguous_kv(p, b)
        L = lens[b]
        assert torch.equal(c[b, 0, :, :L, :].to(torch.float64), k)
        assert torch.equal(c[b, 1, :, :L, :].to(torch.float64), v)


def test_append_touches_only_its_rows_and_is_permutation_covariant():
    lens = [5, 33, 70]
    p = small_problem(lens=lens, free_order=list(range(14)), extra_blocks=5)
    sentinel = np.full((p.num_blocks, 2, 4, 16, 32), 0x7E00, dtype=np.uint16)   # fp16 NaN pattern, never in data
    c_ident = sentinel.copy()
    assert oracle.kv_cache_append(c_ident, p.k_ctx, p.v_ctx, p.cu_ctx_lens, torch.zeros(3, dtype=torch.int32),
                                  p.block_tables) == 0
    written = int((c_ident != 0x7E00).sum())
    # every (token, head, element) of K and V lands somewhere (random N(0,1) data is never that NaN)
    assert written == sum(lens) * 4 * 32 * 2
    # relabel physical pages by a permutation: pool pages move, content per logical page does not
    perm = torch.randperm(p.num_blocks, generator=torch.Generator().manual_seed(5))
    bt2 = p.block_tables.clone()
    m = bt2 >= 0
    bt2[m] = perm[bt2[m].long()].to(torch.int32)
    c_perm = sentinel.copy()
    assert oracle.kv_cache_append(c_perm, p.k_ctx, p.v_ctx, p.cu_ctx_lens, torch.zeros(3, dtype=torch.int32), bt2) == 0
    assert np.array_equal(c_perm[perm.numpy()], c_ident)


def test_append_in_two_steps_equals_one():
    """Appending a context then a chunk (ctx_before > 0) equals appending everything at once."""
    p = small_problem(lens=[20, 45], extra_blocks=0)
    one = oracle.empty_cache_bits(p)
    oracle.kv_cache_append(one, p.k_ctx, p.v_ctx, p.cu_ctx_lens, torch.zeros(2, dtype=torch.int32), p.block_tables)
    two = oracle.empty_cache_bits(p)
    first = [7, 30]
    cu = p.cu_ctx_lens.tolist()
    rows1 = torch.cat([torch.arange(cu[0], cu[0] + 7), torch.arange(cu[1], cu[1] + 30)])
    rows2 = torch.cat([torch.arange(cu[0] + 7, cu[1]), torch.arange(cu[1] + 30, cu[2])])
    oracle.kv_cache_append(two, p.k_ctx[rows1], p.v_ctx[rows1], W.cu_lens(first), torch.zeros(2, dtype=torch.int32),
                           p.block_tables)
    oracle.kv_cache_append(two, p.k_ctx[rows2], p.v_ctx[rows2], W.cu_lens([13, 15]),
                           torch.tensor(first, dtype=torch.int32), p.block_tables)
    assert np.array_equal(one, two)


def test_append_rejects_bad_page():
    p = small_problem(lens=[20])
    bt = p.block_tables.clone()
    bt[0, 1] = p.num_blocks            # out of range page id
    c = oracle.empty_cache_bits(p)
    before = c.copy()
    rc = oracle.kv_cache_append(c, p.k_ctx, p.v_ctx, p.cu_ctx_lens, torch.zeros(1, dtype=torch.int32), bt)
    assert rc == -1
    # tokens 16..19 (page slot 1) were skipped, tokens 0..15 written
    assert not np.array_equal(c, before)


# ----------------------------------------------------------------------------------------------
# attention: definition pins
# ----------------------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (4, 1)])
def test_decode_matches_library_sdpa(dtype, hq, hkv):
    p = small_problem(dtype=dtype, hq=hq, hkv=hkv, lens=(1, 16, 17, 70))
    cache = oracle.build_cache(p)
    out, lse = oracle.attention_of(p, cache)
    for b in range(p.batch):
        ref = sdpa_reference(p, b)
        np.testing.assert_allclose(out[b:b + 1], ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("q_lens,lens", [((48, 48), (85, 148)), ((20, 1), (20, 9)), ((7, 3), (50, 3))])
def test_causal_prefill_matches_library_sdpa(q_lens, lens):
    p = small_problem(lens=lens, q_lens=q_lens, causal=True, hq=4, hkv=2)
    cache = oracle.build_cache(p)
    out, _ = oracle.attention_of(p, cache)
    cq = p.cu_q_lens.tolist()
    for b in range(p.batch):
        ref = sdpa_reference(p, b)
        np.testing.assert_allclose(out[cq[b]:cq[b + 1]], ref, rtol=1e-12, atol=1e-13)


def test_full_causal_is_library_is_causal():
    """q_len = L: bottom-right and top-left alignment coincide with the library's is_causal=True."""
    L = 40
    p = small_problem(lens=(L,), q_lens=(L,), causal=True)
    cache = oracle.build_cache(p)
    out, _ = oracle.attention_of(p, cache)
    k, v = contiguous_kv(p, 0)
    q = p.q.to(torch.float64).permute(1, 0, 2)[None]
    ref = F.scaled_dot_product_attention(q, k[None], v[None], is_causal=True, scale=p.scale)[0].permute(1, 0, 2)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_lse_matches_logsumexp():
    p = small_problem(lens=(3, 50))
    cache = oracle.build_cache(p)
    _, lse = oracle.attention_of(p, cache)
    for b in range(p.batch):
        k, _ = contiguous_kv(p, b)
        q = p.q[b].to(torch.float64)                       # [Hq, D]
        s = torch.einsum("hd,hld->hl", q, k) * p.scale
        np.testing.assert_allclose(lse[b], torch.logsumexp(s, dim=1).numpy(), rtol=1e-13)


# ----------------------------------------------------------------------------------------------
# attention: closed forms and special cases
# ----------------------------------------------------------------------------------------------

def test_one_token_context_returns_v_exactly():
    p = small_problem(lens=(1, 1), dtype=W.BF16)
    cache = oracle.build_cache(p)
    out, lse = oracle.attention_of(p, cache)
    for b in range(2):
        v = p.v_ctx[b].to(torch.float64).numpy()            # [Hkv, D]
        assert np.array_equal(out[b], v)
        s = (p.q[b].to(torch.float64) * p.k_ctx[b].to(torch.float64)).sum(-1) * p.scale
        np.testing.assert_allclose(lse[b], s.numpy(), rtol=1e-14)


def test_identical_keys_give_mean_of_v():
    L = 37
    gen = torch.Generator().manual_seed(11)
    krow = torch.randn(1, 2, 16, generator=gen).to(torch.float16)
    k = krow.expand(L, 2, 16).contiguous()
    v = torch.randn(L, 2, 16, generator=gen).to(torch.float16)
    p = small_problem(lens=(L,), hq=2, hkv=2, d=16, kv_data=(k, v))
    cache = oracle.build_cache(p)
    out, lse = oracle.attention_of(p, cache)
    np.testing.assert_allclose(out[0], v.to(torch.float64).mean(0).numpy(), rtol=1e-13, atol=1e-15)
    s = (p.q[0].to(torch.float64) * krow[0].to(torch.float64)).sum(-1) * p.scale
    np.testing.assert_allclose(lse[0], (s + math.log(L)).numpy(), rtol=1e-13)


def test_empty_context():
    p = small_problem(lens=(0, 5), extra_blocks=1)
    cache = oracle.build_cache(p)
    out, lse = oracle.attention_of(p, cache)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


def test_linearity_in_v():
    """o(2V) = 2 o(V) and o(V + 1) = o(V) + 1: V is built from multiples of 1/64 so both edits are
    exact in fp16."""
    L = 60
    gen = torch.Generator().manual_seed(12)
    k = torch.randn(L, 2, 16, generator=gen).to(torch.float16)
    v = (torch.randint(-128, 128, (L, 2, 16), generator=gen).to(torch.float32) / 64).to(torch.float16)
    base = small_problem(lens=(L,), hq=2, hkv=2, d=16, kv_data=(k, v), seed=3)
    o0, _ = oracle.attention_of(base, oracle.build_cache(base))
    dbl = small_problem(lens=(L,), hq=2, hkv=2, d=16, kv_data=(k, v * 2), seed=3)
    o2, _ = oracle.attention_of(dbl, oracle.build_cache(dbl))
    sh = small_problem(lens=(L,), hq=2, hkv=2, d=16, kv_data=(k, v + 1), seed=3)
    o1, _ = oracle.attention_of(sh, oracle.build_cache(sh))
    np.testing.assert_allclose(o2, 2 * o0, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(o1, o0 + 1, rtol=1e-13, atol=1e-13)


def test_scores_use_scale_and_the_right_operands():
    """Swapping the roles of K and V changes the answer; scale -> 0 gives mean(V)."""
    p = small_problem(lens=(25,), hq=2, hkv=2, d=16)
    cache = oracle.build_cache(p)
    out0, _ = oracle.paged_attention(p.dtype, cache, p.q, 2, p.cu_q_lens, p.context_lens, p.block_tables, 0.0, False)
    _, v = contiguous_kv(p, 0)
    np.testing.assert_allclose(out0[0], v.mean(1).numpy(), rtol=1e-13, atol=1e-15)
    swapped = cache.copy()
    swapped[:, 0], swapped[:, 1] = cache[:, 1], cache[:, 0]
    a, _ = oracle.attention_of(p, cache)
    b, _ = oracle.attention_of(p, swapped)
    assert np.abs(a - b).max() > 1e-3


# ----------------------------------------------------------------------------------------------
# attention: invariants of the paging
# ----------------------------------------------------------------------------------------------

def test_invariant_under_page_permutation_bit_identical():
    p = small_problem(lens=(5, 33, 70), hq=8, hkv=2)
    cache = oracle.build_cache(p)
    out, lse = oracle.attention_of(p, cache)
    for s in range(3):
        order = torch.randperm(p.num_blocks, generator=torch.Generator().manual_seed(50 + s)).tolist()
        p2 = small_problem(lens=(5, 33, 70), hq=8, hkv=2, free_order=order)
        assert not torch.equal(p2.block_tables, p.block_tables)
        out2, lse2 = oracle.attention_of(p2, oracle.build_cache(p2))
        assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


@pytest.mark.parametrize("causal", [False, True])
def test_invariant_under_block_size_bit_identical(causal):
    lens = (70, 129)
    q_lens = (9, 4) if causal else (1, 1)
    ref = None
    for bs in (8, 16, 32, 64, 128, 512):
        p = small_problem(lens=lens, q_lens=q_lens, causal=causal, bs=bs, hq=4, hkv=4)
        out, lse = oracle.attention_of(p, oracle.build_cache(p))
        if ref is None:
            ref = (out, lse)
        else:
            assert np.array_equal(out, ref[0]) and np.array_equal(lse, ref[1]), bs


def test_gqa_equals_mha_with_replicated_kv():
    gqa = small_problem(lens=(40, 9), hq=8, hkv=2, seed=21)
    out_g, lse_g = oracle.attention_of(gqa, oracle.build_cache(gqa))
    k = gqa.k_ctx.repeat_interleave(4, dim=1)
    v = gqa.v_ctx.repeat_interleave(4, dim=1)
    mha = small_problem(lens=(40, 9), hq=8, hkv=8, seed=21, kv_data=(k, v))
    mha.q = gqa.q
    out_m, lse_m = oracle.attention_of(mha, oracle.build_cache(mha))
    assert np.array_equal(out_g, out_m) and np.array_equal(lse_g, lse_m)


def test_causal_row_equals_decode_of_its_prefix():
    """Bottom-right alignment: row r of a q_len chunk over L keys is a decode over L - q_len + r + 1 keys."""
    L, ql = 77, 12
    p = small_problem(lens=(L,), q_lens=(ql,), causal=True)
    cache = oracle.build_cache(p)
    out, lse = oracle.attention_of(p, cache)
    for r in range(ql):
        od, ld = oracle.paged_attention(p.dtype, cache, p.q[r:r + 1], p.num_q_heads, W.cu_lens([1]),
                                        torch.tensor([L - ql + r + 1], dtype=torch.int32), p.block_tables,
                                        p.scale, False)
        assert np.array_equal(od[0], out[r]) and np.array_equal(ld[0], lse[r])


def test_row_selection_matches_full_run():
    p = small_problem(lens=(30, 60), q_lens=(10, 20), causal=True)
    cache = oracle.build_cache(p)
    full, lse = oracle.attention_of(p, cache, nthreads=3)
    rows = [0, 9, 10, 29, 17]
    part, lse_p = oracle.attention_of(p, cache, rows=rows, nthreads=1)
    assert np.array_equal(full[rows], part) and np.array_equal(lse[rows], lse_p)


def test_bad_page_id_raises():
    p = small_problem(lens=(20,))
    cache = oracle.build_cache(p)
    bt = p.block_tables.clone()
    bt[0, 1] = -1
    with pytest.raises(ValueError):
        oracle.paged_attention(p.dtype, cache, p.q, p.num_q_heads, p.cu_q_lens, p.context_lens, bt, p.scale, False)


# ----------------------------------------------------------------------------------------------
# the pages' online-softmax recurrence equals the two-pass oracle
# ----------------------------------------------------------------------------------------------

def online_softmax_attention(q, k, v, scale, tile):
    """The tiled recurrence of the ipipp.com page, section 2, restated in float64 numpy:
    running max m and sum l; each tile rescales the old sum and output by exp(m_old - m_new)."""
    n = q.shape[0]
    o = np.zeros_like(q)
    m = np.full(n, -np.inf)
    l = np.zeros(n)
    for start in range(0, k.shape[0], tile):
        kj, vj = k[start:start + tile], v[start:start + tile]
        s = q @ kj.T * scale
        m_new = np.maximum(m, s.max(axis=1))
        p = np.exp(s - m_new[:, None])
        alpha = np.exp(m - m_new)
        l = alpha * l + p.sum(axis=1)
        o = o * alpha[:, None] + p @ vj
        m = m_new
    return o / l[:, None], m + np.log(l)


@pytest.mark.parametrize("tile", [1, 3, 16, 128, 1000])
def test_online_recurrence_equals_two_pass(tile):
    p = small_problem(lens=(300,), hq=2, hkv=2, d=64, seed=31)
    out, lse = oracle.attention_of(p, oracle.build_cache(p))
    k, v = contiguous_kv(p, 0)
    q = p.q[0].to(torch.float64).numpy()
    for h in range(2):
        o_on, lse_on = online_softmax_attention(q[h:h + 1], k[h].numpy(), v[h].numpy(), p.scale, tile)
        np.testing.assert_allclose(o_on[0], out[0, h], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(lse_on[0], lse[0, h], rtol=1e-13)


# ----------------------------------------------------------------------------------------------
# split-KV merge
# ----------------------------------------------------------------------------------------------

def split_partials(p, cache, bounds):
    """Partial (O_s, lse_s) of one sequence for key ranges starting on page boundaries, each
    computed by the oracle over a shifted block table."""
    bs = p.block_size
    outs, lses = [], []
    for a, b in bounds:
        assert a % bs == 0
        bt = torch.full_like(p.block_tables[:1], -1)
        tail = p.block_tables[0, a // bs:]
        bt[0, :tail.numel()] = tail
        o, l = oracle.paged_attention(p.dtype, cache, p.q[:1], p.num_q_heads, W.cu_lens([1]),
                                      torch.tensor([b - a], dtype=torch.int32), bt, p.scale, False)
        outs.append(o[0])
        lses.append(l[0])
    return np.stack(outs, 1), np.stack(lses, 1)        # [Hq, S, D], [Hq, S]


@pytest.mark.parametrize("bounds", [[(0, 64), (64, 200)], [(0, 16), (16, 32), (32, 48), (48, 200)],
                                    [(0, 200)], [(0, 96), (96, 96), (96, 200)]])
def test_combine_of_splits_equals_unsplit(bounds):
    p = small_problem(lens=(200,), hq=4, hkv=4, seed=41)
    cache = oracle.build_cache(p)
    full, lse = oracle.attention_of(p, cache)
    po, pl = split_partials(p, cache, bounds)
    out, lse_m = oracle.attn_combine(po, pl)
    np.testing.assert_allclose(out, full[0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse_m, lse[0], rtol=1e-13)


def test_combine_all_empty_and_weightless_splits():
    po = np.random.default_rng(0).standard_normal((3, 4, 8))
    pl = np.full((3, 4), -np.inf)
    pl[1, 2] = 0.5
    out, lse = oracle.attn_combine(po, pl)
    assert np.all(out[0] == 0) and np.isneginf(lse[0])
    assert np.array_equal(out[1], po[1, 2]) and lse[1] == 0.5


# ----------------------------------------------------------------------------------------------
# the pages' allocator (ipipp.com page, section 3)
# ----------------------------------------------------------------------------------------------

def test_allocator_pops_from_the_end_and_rounds_up():
    a = W.BlockAllocator(8, 16)
    assert a.allocate(33) == [7, 6, 5]           # ceil(33/16) = 3 blocks from the end of the free list
    assert a.allocate(16) == [4]
    assert a.allocate(0) == []
    a.release([6, 7])
    assert a.free == [0, 1, 2, 3, 6, 7]
    with pytest.raises(W.OutOfBlocks):
        a.allocate(16 * 7)


def test_mixed_serving_pool_is_fragmented_and_disjoint():
    p = W.mixed_serving(pool_init="none", kv_data="skip")
    used = p.block_tables[p.block_tables >= 0]
    assert used.unique().numel() == used.numel()           # no page shared by two sequences
    assert p.num_blocks == 2 * used.numel()
    lens = p.context_lens.tolist()
    assert min(lens) >= 16 and max(lens) <= 32768
    # fragmented: consecutive logical pages are rarely consecutive physical pages
    bt = p.block_tables
    m = (bt[:, 1:] >= 0) & (bt[:, :-1] >= 0)
    adj = ((bt[:, 1:] - bt[:, :-1]).abs() == 1) & m
    assert adj.sum().item() < 0.05 * m.sum().item()


# ----------------------------------------------------------------------------------------------
# prefix caching: reference-counted pages shared by several block tables (pwwt.cn write-up on
# chunked attention, section 5.4)
# ----------------------------------------------------------------------------------------------

def test_allocator_reference_counts():
    a = W.BlockAllocator(6, 16)
    pre = a.allocate(32)                          # [5, 4], one reference each
    t1 = a.share(pre) + a.allocate(10)
    t2 = a.share(pre) + a.allocate(20)
    assert t1[:2] == t2[:2] == pre and a.refs[5] == a.refs[4] == 3
    a.release(t1)                                 # private page freed, shared pages still held
    assert a.free == [0, t1[2]] and a.refs[5] == 2
    a.release(pre)
    a.release(t2)                                 # last holder: pages return in release order
    assert sorted(a.free) == list(range(6)) and a.free[-4:] == t2 and a.refs == [0] * 6
    with pytest.raises(ValueError):
        a.release([3])                            # not held
    with pytest.raises(ValueError):
        a.share([3])                              # free blocks cannot be shared
    b = a.allocate(16)
    with pytest.raises(ValueError):
        a.release(b + b)                          # released twice in one call, held once
    assert a.refs[b[0]] == 1                      # a rejected release changes nothing


def test_prefix_workload_tables_share_exactly_the_prompt_pages():
    p = W.prefix_shared(batch=5, prefix=100, lo=3, hi=60, block_size=16, heads=2, head_dim=32, pool_init="none")
    s = p.meta["shared_tokens"]
    assert s == 96
    shared = p.meta["shared_blocks"]
    bt = p.block_tables
    for b in range(p.batch):
        assert bt[b, :6].tolist() == shared
    private = [x for x in bt[:, 6:].flatten().tolist() if x >= 0]
    assert len(set(private)) == len(private) and not set(private) & set(shared)
    refs = p.meta["allocator"].refs
    assert all(refs[x] == p.batch + 1 for x in shared) and all(refs[x] == 1 for x in private)
    # the prompt's rows are identical in every request's context
    cu = p.cu_ctx_lens.tolist()
    for b in range(1, p.batch):
        assert torch.equal(p.k_ctx[cu[b]:cu[b] + 100], p.k_ctx[:100])
        assert torch.equal(p.v_ctx[cu[b]:cu[b] + 100], p.v_ctx[:100])


def test_prefix_appends_once_equal_every_context_appended():
    """Writing the shared pages once plus each request's own rows gives the pool that appending
    every request's whole context gives (the shared pages then receive identical rows)."""
    p = W.prefix_shared(batch=4, prefix=70, lo=1, hi=50, block_size=16, heads=2, head_dim=32)
    whole = oracle.build_cache(p)
    cache = oracle.empty_cache_bits(p)
    for args in (W.shared_append(p), W.private_append(p)):
        assert oracle.kv_cache_append(cache, **args) == 0
    assert np.array_equal(cache, whole)


@pytest.mark.parametrize("prefill", [False, True])
def test_shared_pages_equal_private_copies_bit_identical(prefill):
    """Attention over tables that alias the prompt's pages equals attention over tables that give
    every request its own copy of them (the oracle reads a page by id; aliasing is invisible)."""
    p = W.prefix_shared(batch=3, prefix=50, lo=1, hi=40, block_size=8, heads=4, kv_heads=2, head_dim=32,
                        prefill=prefill)
    got, got_lse = oracle.attention_of(p, oracle.build_cache(p))
    lens = p.context_lens.tolist()
    copy = W.make_problem("unshared", batch=p.batch, num_q_heads=4, num_kv_heads=2, head_dim=32, block_size=8,
                          context_lens=lens, q_lens=p.q_lens.tolist(), dtype=p.dtype, causal=p.causal, seed=3,
                          kv_data=(p.k_ctx, p.v_ctx))
    ref, ref_lse = oracle.attention_of(copy, oracle.build_cache(copy), q=p.q)
    assert copy.block_tables.unique().numel() > p.block_tables.unique().numel()
    assert np.array_equal(got, ref) and np.array_equal(got_lse, ref_lse)
