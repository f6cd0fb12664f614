"""Pins for the oracle's FP8 cache (E4M3 codes with one FP32 scale per cached row).

The format and the conversion are tied to torch's float8_e4m3fn (a library routine) and to the
format's closed forms; the quantising append to its definition (scale = amax / 448, codes of
x * (448 / amax)); the attention over an FP8 cache to a brute-force softmax over values
dequantised by torch, written out here in numpy."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_flash_cache_gb300 import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


@pytest.fixture(scope="module", autouse=True)
def built():
    oracle.build()


def torch_decode(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_encode(x: np.ndarray) -> np.ndarray:
    """torch's float32 -> float8_e4m3fn conversion (round to nearest even; used in range only)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def test_decode_every_code_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    got, ref = oracle.e4m3_decode(codes), torch_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.isnan(got).sum() == 2                          # S.1111.111 only
    ok = ~np.isnan(got)
    assert np.array_equal(got[ok], ref[ok])
    # closed forms: largest finite, smallest normal, smallest subnormal, one
    assert got[0x7E] == 448.0 and got[0x08] == 2.0 ** -6 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0
    assert got[0x80] == 0.0 and np.signbit(got[0x80])


def test_encode_matches_torch_in_range_including_ties():
    finite = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))     # 0 .. 448, increasing
    mids = (finite[:-1] + finite[1:]) / 2                             # exact ties (exact in float32)
    rng = np.random.default_rng(5)
    rand = np.exp(rng.uniform(np.log(2.0 ** -12), np.log(447.0), 20000))
    x = np.concatenate([finite, mids, rand, finite * (1 + 2.0 ** -20), finite * (1 - 2.0 ** -20)])
    x = x[(x <= 448.0)].astype(np.float32)
    x = np.concatenate([x, -x])
    assert np.array_equal(oracle.e4m3_encode(x), torch_encode(x))


def test_encode_ties_go_to_even_and_saturates():
    # 1 + 1/16 lies halfway between 1 (code 0x38, even) and 1.125 (0x39): even wins
    assert oracle.e4m3_encode(np.float32([1.0625]))[0] == 0x38
    assert oracle.e4m3_encode(np.float32([1.1875]))[0] == 0x3A      # between 0x39 and 0x3A (even)
    big = np.float32([448.0, 449.0, 463.9, 464.0, 1000.0, 3.0e38])
    assert np.all(oracle.e4m3_encode(big) == 0x7E)
    assert np.all(oracle.e4m3_encode(-big) == 0xFE)
    # subnormals: 2^-10 is the tie between 0 and 2^-9 -> 0 (even); 3 * 2^-10 -> 2 * 2^-9
    assert list(oracle.e4m3_encode(np.float32([2.0 ** -10, 3 * 2.0 ** -10]))) == [0x00, 0x02]
    assert oracle.e4m3_encode(np.float32([-0.0]))[0] == 0x80


def small_fp8(seed=3, lens=(5, 40, 100), hq=4, hkv=2, d=64, bs=16, dtype=W.BF16, q_lens=None, causal=False,
              kv_data=None):
    q_lens = q_lens or [1] * len(lens)
    nb = sum((L + bs - 1) // bs for L in lens) + 4
    return W.make_problem("f", batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                          context_lens=list(lens), q_lens=list(q_lens), dtype=dtype, causal=causal, seed=seed,
                          num_blocks=nb, kv_format="fp8", kv_data=kv_data)


def rows_of(p, cache, b, kv):
    """Sequence b's K (kv=0) or V rows as (codes [L, Hkv, D], scales [L, Hkv]) through its table."""
    L = int(p.context_lens[b])
    codes = np.zeros((L, p.num_kv_heads, p.head_dim), dtype=np.uint8)
    scales = np.zeros((L, p.num_kv_heads), dtype=np.float32)
    for i in range(L):
        pb = int(p.block_tables[b, i // p.block_size])
        codes[i] = cache.codes[pb, kv, :, i % p.block_size]
        scales[i] = cache.scales[pb, kv, :, i % p.block_size]
    return codes, scales


def test_append_follows_the_definition():
    p = small_fp8()
    cache = oracle.build_cache(p)
    cu = p.cu_ctx_lens.tolist()
    for b in range(p.batch):
        for kv, src in ((0, p.k_ctx), (1, p.v_ctx)):
            x = src[cu[b]:cu[b + 1]].to(torch.float32).numpy()            # exact
            codes, scales = rows_of(p, cache, b, kv)
            amax = np.abs(x).max(axis=2).astype(np.float32)
            assert np.array_equal(scales, np.where(amax > 0, amax / np.float32(448.0), 0).astype(np.float32))
            inv = np.where(amax > 0, np.float32(448.0) / np.maximum(amax, np.float32(1e-30)), 0).astype(np.float32)
            want = torch_encode((x * inv[..., None]).astype(np.float32))
            assert np.array_equal(codes, want)
            # the largest element of every row is the largest code (448, or just below it)
            assert np.all(np.abs(torch_decode(codes)).max(axis=2) >= 416.0)


def test_append_zero_row_and_exact_rows():
    """An all-zero row stores scale 0 and zero codes; a row of E4M3 values whose largest magnitude
    is 448 has scale 1 and comes back exactly; scaling a row by 2^k scales only its scale."""
    d = 64
    e4 = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    rng = np.random.default_rng(2)
    row = rng.choice(e4, size=(d,)) * rng.choice([-1.0, 1.0], size=(d,))
    row[7] = 448.0
    k = torch.zeros((3, 1, d), dtype=torch.float32)
    k[1, 0] = torch.from_numpy(row)
    k[2, 0] = torch.from_numpy(row * 2.0 ** -5)
    k = k.to(torch.bfloat16)                                 # E4M3 values are exact in bf16
    p = small_fp8(lens=(3,), hq=1, hkv=1, d=d, kv_data=(k, k.clone()))
    cache = oracle.build_cache(p)
    codes, scales = rows_of(p, cache, 0, 0)
    assert scales[0, 0] == 0 and not codes[0].any()
    assert scales[1, 0] == 1.0 and np.array_equal(torch_decode(codes[1, 0]), row)
    assert scales[2, 0] == 2.0 ** -5 and np.array_equal(codes[2, 0], codes[1, 0])


def test_append_roundtrip_error_bound():
    """|x - decode(code) * scale| <= half an E4M3 step at the scaled magnitude (2^-4 relative in the
    normal range, 2^-10 * scale absolute below it)."""
    p = small_fp8(lens=(300,), hq=2, hkv=2, d=128)
    cache = oracle.build_cache(p)
    codes, scales = rows_of(p, cache, 0, 1)
    x = p.v_ctx.to(torch.float64).numpy()
    xh = torch_decode(codes) * scales[..., None].astype(np.float64)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * scales[..., None]) * (1 + 1e-6)
    assert np.all(np.abs(x - xh) <= bound)


@pytest.mark.parametrize("causal,q_lens", [(False, None), (True, (3, 17, 40))])
def test_attention_over_fp8_is_softmax_of_dequantised(causal, q_lens):
    lens = (5, 40, 100)
    p = small_fp8(lens=lens, causal=causal, q_lens=q_lens, hq=4, hkv=2)
    cache = oracle.build_cache(p)
    got, got_lse = oracle.attention_of(p, cache)
    cq = p.cu_q_lens.tolist()
    g = p.num_q_heads // p.num_kv_heads
    for b, L in enumerate(lens):
        kc, ks = rows_of(p, cache, b, 0)
        vc, vs = rows_of(p, cache, b, 1)
        K = torch_decode(kc) * ks[..., None].astype(np.float64)
        V = torch_decode(vc) * vs[..., None].astype(np.float64)
        ql = cq[b + 1] - cq[b]
        for r in range(ql):
            kmax = L - ql + r + 1 if causal else L
            for h in range(p.num_q_heads):
                q = p.q[cq[b] + r, h].to(torch.float64).numpy()
                s = p.scale * (K[:kmax, h // g] @ q)
                w = np.exp(s - s.max())
                o = (w[:, None] * V[:kmax, h // g]).sum(0) / w.sum()
                np.testing.assert_allclose(got[cq[b] + r, h], o, rtol=1e-12, atol=1e-13)
                np.testing.assert_allclose(got_lse[cq[b] + r, h], s.max() + np.log(w.sum()), rtol=1e-12)


def test_fp8_attention_close_to_unquantised():
    """The quantisation error of the method itself (not a parity bound): attention over the FP8
    cache stays within a few percent of attention over the 16-bit cache."""
    lens = (64, 500)
    p8 = small_fp8(lens=lens, hq=4, hkv=4, d=128, seed=9)
    p16 = W.make_problem("n", batch=2, num_q_heads=4, num_kv_heads=4, head_dim=128, block_size=16,
                         context_lens=list(lens), q_lens=[1, 1], dtype=W.BF16, causal=False, seed=9,
                         num_blocks=p8.num_blocks, kv_data=(p8.k_ctx, p8.v_ctx))
    o8, _ = oracle.attention_of(p8, oracle.build_cache(p8), q=p8.q)
    o16, _ = oracle.attention_of(p16, oracle.build_cache(p16), q=p8.q)
    rel = np.linalg.norm(o8 - o16) / np.linalg.norm(o16)
    assert rel < 0.06, rel
