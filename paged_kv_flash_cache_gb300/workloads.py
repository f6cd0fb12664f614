"""Seeded synthetic inputs for paged KV-cache attention, and the host-side block
allocator that builds block tables.

This module draws random numbers and decides which physical pages each sequence
owns. It holds none of the attention arithmetic and none of the cache
addressing: tensors here are the *inputs* of `kv_cache_append`,
`paged_attn_decode` and `paged_attn_prefill`, given to the CUDA path and to the
CPU oracle alike.

Sources (page titles from the subject's web pages):
  * "Flash Attention与Paged Attention如何共同优化大模型推理？" (ipipp.com), section 3:
    the `PagedKVCache` allocator -- a free list initialised to every block id,
    `allocate(num_tokens)` takes ceil(num_tokens / block_size) blocks popped
    from the END of the free list and fails when too few are free,
    `release(blocks)` appends them back; cache shape
    [num_blocks, 2, num_heads, block_size, head_dim].
  * "企业官网建设流程全解析" (cf-1.com), section 2.1: block table maps logical block
    i // block_size to a physical block.
  * pwwt.cn write-up on chunked attention (a 7B model 70x slower), section 5.4: prefix
    caching -- requests sharing a prompt reuse its cached K/V pages.
Values follow the workloads of the pages' 7B-like cases (32 heads x head_dim
128, contexts of 4k-8k tokens, batch 16, block sizes 8-512): Q/K/V ~ N(0, 1)
cast to fp16 or bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import torch

F16 = "f16"
BF16 = "bf16"
TORCH_DTYPE = {F16: torch.float16, BF16: torch.bfloat16}


class OutOfBlocks(RuntimeError):
    """Raised when the pool has fewer free blocks than a request needs."""


class BlockAllocator:
    """Free-list page allocator (ipipp.com page, section 3, `PagedKVCache`), with a reference
    count per block so that several block tables can hold the same pages (prefix caching,
    pwwt.cn write-up on chunked attention, section 5.4: requests that open with the same prompt
    reuse its cached K/V instead of recomputing it).

    `free` starts as ``list(range(num_blocks))`` unless an explicit order is given (a seeded
    permutation spreads a sequence's pages over the pool). `allocate` hands out blocks with one
    reference each; `share` adds a reference to blocks already handed out; `release` drops one
    reference per listed block and returns a block to the free list when its count reaches 0.
    """

    def __init__(self, num_blocks: int, block_size: int,
                 free_order: Optional[Sequence[int]] = None):
        if num_blocks < 0 or block_size <= 0:
            raise ValueError("num_blocks >= 0 and block_size > 0 required")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free: List[int] = list(range(num_blocks)) if free_order is None else [int(x) for x in free_order]
        if sorted(self.free) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of range(num_blocks)")
        self.refs: List[int] = [0] * num_blocks

    def blocks_needed(self, num_tokens: int) -> int:
        return (num_tokens + self.block_size - 1) // self.block_size

    def allocate(self, num_tokens: int) -> List[int]:
        needed = self.blocks_needed(num_tokens)
        if len(self.free) < needed:
            raise OutOfBlocks("not enough free KV cache blocks: need %d, have %d" % (needed, len(self.free)))
        out = [self.free.pop() for _ in range(needed)]
        for b in out:
            self.refs[b] = 1
        return out

    def _counts(self, blocks: Sequence[int]) -> dict:
        counts: dict = {}
        for b in blocks:
            b = int(b)
            if not 0 <= b < self.num_blocks:
                raise ValueError("block %d is outside the pool" % b)
            counts[b] = counts.get(b, 0) + 1
        return counts

    def share(self, blocks: Sequence[int]) -> List[int]:
        """One more reference to each of `blocks` (all must be allocated); returns them, for the
        new owner's block table."""
        counts = self._counts(blocks)
        for b in counts:
            if self.refs[b] == 0:
                raise ValueError("block %d is free: only allocated blocks can be shared" % b)
        for b, n in counts.items():
            self.refs[b] += n
        return [int(b) for b in blocks]

    def release(self, blocks: Sequence[int]) -> None:
        counts = self._counts(blocks)
        for b, n in counts.items():
            if self.refs[b] < n:
                raise ValueError("block %d released more often than it is held" % b)
        for b in blocks:
            b = int(b)
            self.refs[b] -= 1
            if self.refs[b] == 0:
                self.free.append(b)


def block_table_tensor(tables: Sequence[Sequence[int]], max_blocks_per_seq: int) -> torch.Tensor:
    """Pack per-sequence page lists into an int32 [B, MB] table; unused slots hold -1."""
    bt = torch.full((len(tables), max_blocks_per_seq), -1, dtype=torch.int32)
    for b, t in enumerate(tables):
        if len(t) > max_blocks_per_seq:
            raise ValueError("sequence %d needs %d blocks > max_blocks_per_seq %d" % (b, len(t), max_blocks_per_seq))
        if len(t):
            bt[b, :len(t)] = torch.tensor(list(t), dtype=torch.int32)
    return bt


def cu_lens(lens: Sequence[int]) -> torch.Tensor:
    """Exclusive prefix sums [0, l0, l0+l1, ...] as int32."""
    out = torch.zeros(len(lens) + 1, dtype=torch.int32)
    if len(lens):
        out[1:] = torch.cumsum(torch.tensor(list(lens), dtype=torch.int64), 0).to(torch.int32)
    return out


def randn_t(gen: torch.Generator, shape, dtype: str) -> torch.Tensor:
    """N(0, 1) draws in fp32 on the generator's device, rounded to fp16 / bf16."""
    return torch.randn(shape, generator=gen, dtype=torch.float32, device=gen.device).to(TORCH_DTYPE[dtype])


def data_generator(seed: int, device="cpu") -> torch.Generator:
    """Generator for token data. Large workloads draw on the GPU (a CPU draw of a few GB takes
    minutes); each problem instance is then self-consistent: the oracle reads the same tensors
    after a copy to the host."""
    return torch.Generator(device=device).manual_seed(seed)


@dataclass
class PagedProblem:
    """One batch of paged-attention inputs (all tensors on the CPU).

    k_ctx / v_ctx hold every context token packed as [sum(L_b), Hkv, D] in
    sequence order; they are appended into the pool by `kv_cache_append` with
    ctx_before = 0. q holds [sum(q_len_b), Hq, D]; decode has q_len_b = 1.
    `pool_init` is the pool's content before any append (seeded noise, so a
    wrong page read changes the result); for an FP8 cache it is the pair
    (codes uint8 [NB, 2, Hkv, bs, D], scales float32 [NB, 2, Hkv, bs]).
    """
    name: str
    dtype: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    context_lens: torch.Tensor          # [B] int32, tokens in cache incl. any prefill chunk
    q_lens: torch.Tensor                # [B] int32
    block_tables: torch.Tensor          # [B, MB] int32, -1 padded
    k_ctx: torch.Tensor                 # [sum L, Hkv, D]
    v_ctx: torch.Tensor
    q: torch.Tensor                     # [sum q_len, Hq, D]
    pool_init: Optional[torch.Tensor]   # [NB, 2, Hkv, bs, D] or None (left uninitialised)
    causal: bool
    scale: float
    meta: dict = field(default_factory=dict)
    kv_format: str = "native"           # "fp8": the cache holds E4M3 codes + per-row FP32 scales

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def cu_ctx_lens(self) -> torch.Tensor:
        return cu_lens(self.context_lens.tolist())

    @property
    def cu_q_lens(self) -> torch.Tensor:
        return cu_lens(self.q_lens.tolist())

    @property
    def total_q(self) -> int:
        return int(self.q_lens.sum())

    def kv_bytes_read(self) -> int:
        """Bytes of K and V one decode pass reads: each cached token once per KV head."""
        return int(self.context_lens.to(torch.int64).sum()) * self.num_kv_heads * self.head_dim * 2 * 2

    def causal_flops(self) -> int:
        """4*D FLOPs per (query row, Q head, key it sees) -- QK^T and PV, masked keys excluded."""
        total = 0
        for L, ql in zip(self.context_lens.tolist(), self.q_lens.tolist()):
            if self.causal:
                first = L - ql + 1
                seen = ql * first + ql * (ql - 1) // 2
            else:
                seen = ql * L
            total += seen
        return 4 * self.head_dim * self.num_q_heads * total


def _pool_noise(gen: torch.Generator, nb: int, hkv: int, bs: int, d: int, dtype: str, cheap: bool) -> torch.Tensor:
    if not cheap:
        return randn_t(gen, (nb, 2, hkv, bs, d), dtype)
    # One seeded page repeated: same noise role, O(page) random draws.
    page = randn_t(gen, (1, 2, hkv, bs, d), dtype)
    return page.expand(nb, 2, hkv, bs, d).clone()


def _pool_noise_fp8(gen: torch.Generator, nb: int, hkv: int, bs: int, d: int, cheap: bool):
    """Noise for an FP8 pool: random E4M3 codes (the two NaN codes replaced by 0) and scales."""
    n = 1 if cheap else nb
    codes = torch.randint(0, 256, (n, 2, hkv, bs, d), generator=gen, dtype=torch.int32, device=gen.device)
    codes = torch.where((codes & 0x7F) == 0x7F, torch.zeros_like(codes), codes).to(torch.uint8)
    scales = (torch.rand((n, 2, hkv, bs), generator=gen, device=gen.device) * 0.05 + 1e-3).to(torch.float32)
    if cheap:
        codes = codes.expand(nb, 2, hkv, bs, d).clone()
        scales = scales.expand(nb, 2, hkv, bs).clone()
    return codes, scales


def make_problem(name: str, *, batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                 block_size: int, context_lens: Sequence[int], q_lens: Sequence[int], dtype: str,
                 causal: bool, seed: int, num_blocks: Optional[int] = None,
                 free_order: Optional[Sequence[int]] = None, tables: Optional[List[List[int]]] = None,
                 max_blocks_per_seq: Optional[int] = None, pool_init: str = "noise",
                 kv_data=None, scale: Optional[float] = None, device="cpu", kv_format: str = "native") -> PagedProblem:
    gen = torch.Generator().manual_seed(seed)
    dgen = data_generator(seed, device)
    context_lens = [int(x) for x in context_lens]
    q_lens = [int(x) for x in q_lens]
    if tables is None:
        pages = [(L + block_size - 1) // block_size for L in context_lens]
        if num_blocks is None:
            num_blocks = sum(pages)
        if free_order is None:
            free_order = torch.randperm(num_blocks, generator=gen).tolist()
        alloc = BlockAllocator(num_blocks, block_size, free_order)
        tables = [alloc.allocate(L) for L in context_lens]
    mb = max_blocks_per_seq or max(1, max(len(t) for t in tables))
    bt = block_table_tensor(tables, mb)
    total = sum(context_lens)
    if isinstance(kv_data, str) and kv_data == "skip":
        # tables / lengths only (no token data): for tests of the pool structure
        k_ctx = v_ctx = torch.empty((0, num_kv_heads, head_dim), dtype=TORCH_DTYPE[dtype])
    elif kv_data is not None:
        k_ctx, v_ctx = kv_data
    else:
        k_ctx = randn_t(dgen, (total, num_kv_heads, head_dim), dtype)
        v_ctx = randn_t(dgen, (total, num_kv_heads, head_dim), dtype)
    q = randn_t(dgen, (sum(q_lens), num_q_heads, head_dim), dtype)
    if kv_format not in ("native", "fp8"):
        raise ValueError("kv_format must be 'native' or 'fp8'")
    if pool_init == "none":
        pool = None
    elif kv_format == "fp8":
        pool = _pool_noise_fp8(dgen, num_blocks, num_kv_heads, block_size, head_dim, pool_init == "cheap")
    else:
        pool = _pool_noise(dgen, num_blocks, num_kv_heads, block_size, head_dim, dtype, pool_init == "cheap")
    return PagedProblem(
        name=name, dtype=dtype, batch=batch, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
        head_dim=head_dim, block_size=block_size, num_blocks=num_blocks,
        context_lens=torch.tensor(context_lens, dtype=torch.int32),
        q_lens=torch.tensor(q_lens, dtype=torch.int32), block_tables=bt, k_ctx=k_ctx, v_ctx=v_ctx,
        q=q, pool_init=pool, causal=causal,
        scale=(1.0 / math.sqrt(head_dim)) if scale is None else float(scale), kv_format=kv_format)


# --------------------------------------------------------------------------------------
# The five workloads (sizes from the pages' 7B-like cases; see the module docstring).
# --------------------------------------------------------------------------------------

def tiny(seed: int = 1235, chunk: int = 48):
    """The tiny case: batch 2, 4 heads, head_dim 64, block_size 16, fp16, cached contexts of 37 and
    100 tokens in a 32-block pool handed out in a seeded random order; then one causal prefill
    chunk of `chunk` tokens per sequence (positions 37..84 and 100..147) over the same cache.

    Returns (decode, prefill): both share block tables, pool noise and token data; the decode
    problem sees the first 37 / 100 tokens, the prefill problem all 85 / 148 with the last
    `chunk` of each as its queries' own keys."""
    gen = torch.Generator().manual_seed(seed)
    order = torch.randperm(32, generator=gen).tolist()
    full = [37 + chunk, 100 + chunk]
    pre = make_problem("tiny_prefill", batch=2, num_q_heads=4, num_kv_heads=4, head_dim=64,
                       block_size=16, context_lens=full, q_lens=[chunk, chunk], dtype=F16,
                       causal=True, seed=seed + 2, num_blocks=32, free_order=order)
    rows = torch.cat([torch.arange(0, 37), torch.arange(full[0], full[0] + 100)])
    qgen = torch.Generator().manual_seed(seed + 3)
    dec = PagedProblem(name="tiny_decode", dtype=F16, batch=2, num_q_heads=4, num_kv_heads=4, head_dim=64,
                       block_size=16, num_blocks=32, context_lens=torch.tensor([37, 100], dtype=torch.int32),
                       q_lens=torch.tensor([1, 1], dtype=torch.int32), block_tables=pre.block_tables.clone(),
                       k_ctx=pre.k_ctx[rows].contiguous(), v_ctx=pre.v_ctx[rows].contiguous(),
                       q=randn_t(qgen, (2, 4, 64), F16), pool_init=pre.pool_init, causal=False,
                       scale=pre.scale)
    return dec, pre


def decode_7b(seed: int = 1236, batch: int = 16, lo: int = 1024, hi: int = 8192, pool_init: str = "cheap",
              block_size: int = 16, dtype: str = F16, device="cpu", kv_format: str = "native") -> PagedProblem:
    """7B-like decode: 32 heads x 128, contexts uniform in [lo, hi], pool 1.2x the pages needed,
    pages handed out in a seeded random order (kv_format "fp8": the same tokens into an FP8 cache)."""
    gen = torch.Generator().manual_seed(seed)
    lens = torch.randint(lo, hi + 1, (batch,), generator=gen).tolist()
    pages = sum((L + block_size - 1) // block_size for L in lens)
    nb = int(math.ceil(1.2 * pages))
    order = torch.randperm(nb, generator=gen).tolist()
    return make_problem("decode_7b", batch=batch, num_q_heads=32, num_kv_heads=32, head_dim=128,
                        block_size=block_size, context_lens=lens, q_lens=[1] * batch, dtype=dtype,
                        causal=False, seed=seed + 1, num_blocks=nb, free_order=order, pool_init=pool_init,
                        max_blocks_per_seq=(hi + block_size - 1) // block_size, device=device, kv_format=kv_format)


def prefill_long(seed: int = 1237, batch: int = 4, seq: int = 8192, chunk: int = 512, heads: int = 32,
                 head_dim: int = 128, block_size: int = 16, dtype: str = BF16, device="cpu",
                 kv_format: str = "native") -> PagedProblem:
    """Long causal prefill: `batch` sequences of `seq` tokens in bf16, pages of 16 tokens
    spread by a seeded permutation over a pool of exactly the pages needed. The whole
    sequence is described once; `prefill_chunks` cuts it into `chunk`-token query calls
    (kv_format "fp8": the same tokens into an FP8 cache)."""
    gen = torch.Generator().manual_seed(seed)
    pages = batch * ((seq + block_size - 1) // block_size)
    order = torch.randperm(pages, generator=gen).tolist()
    p = make_problem("prefill_long", batch=batch, num_q_heads=heads, num_kv_heads=heads, head_dim=head_dim,
                     block_size=block_size, context_lens=[seq] * batch, q_lens=[seq] * batch, dtype=dtype,
                     causal=True, seed=seed + 1, num_blocks=pages, free_order=order, pool_init="none", device=device,
                     kv_format=kv_format)
    p.meta["chunk"] = chunk
    return p


def prefill_chunk_view(p: PagedProblem, c: int) -> dict:
    """Chunk c of a long prefill: queries at absolute positions [c*chunk, (c+1)*chunk) of every
    sequence attend to keys 0 .. (c+1)*chunk-1. Returns the per-call tensors."""
    chunk = p.meta["chunk"]
    seq = int(p.context_lens[0])
    assert all(int(x) == seq for x in p.context_lens.tolist())
    lo, hi = c * chunk, min((c + 1) * chunk, seq)
    rows = []
    for b in range(p.batch):
        rows.append(torch.arange(b * seq + lo, b * seq + hi))
    rows = torch.cat(rows)
    ql = hi - lo
    return dict(rows=rows, q=p.q[rows].contiguous(), q_lens=torch.full((p.batch,), ql, dtype=torch.int32),
                cu_q_lens=cu_lens([ql] * p.batch), context_lens=torch.full((p.batch,), hi, dtype=torch.int32),
                new_rows=rows, ctx_before=torch.full((p.batch,), lo, dtype=torch.int32))


def bs_sweep(block_size: int, seed: int = 1238, batch: int = 32, ctx: int = 4096,
             kv_data: Optional[tuple] = None, pool_init: str = "cheap", device="cpu") -> PagedProblem:
    """Block-size sweep: `batch` x `ctx` tokens, 32 heads x 128, fp16; the same K/V token data for
    every block size (pass kv_data from `bs_sweep_kv`); pool = exactly the pages needed, permuted."""
    gen = torch.Generator().manual_seed(seed * 1000 + block_size)
    pages = batch * ((ctx + block_size - 1) // block_size)
    order = torch.randperm(pages, generator=gen).tolist()
    return make_problem("bs_sweep_%d" % block_size, batch=batch, num_q_heads=32, num_kv_heads=32, head_dim=128,
                        block_size=block_size, context_lens=[ctx] * batch, q_lens=[1] * batch, dtype=F16,
                        causal=False, seed=seed, num_blocks=pages, free_order=order, kv_data=kv_data,
                        pool_init=pool_init, device=device)


def bs_sweep_kv(seed: int = 1238, batch: int = 32, ctx: int = 4096, device="cpu") -> tuple:
    gen = data_generator(seed + 7, device)
    k = randn_t(gen, (batch * ctx, 32, 128), F16)
    v = randn_t(gen, (batch * ctx, 32, 128), F16)
    return k, v


def mixed_lens(seed: int, batch: int = 64, median: float = 2048.0, sigma: float = 1.0,
               lo: int = 16, hi: int = 32768) -> List[int]:
    gen = torch.Generator().manual_seed(seed)
    z = torch.randn(batch, generator=gen, dtype=torch.float64)
    lens = torch.exp(math.log(median) + sigma * z).round().clamp(lo, hi).to(torch.int64)
    return lens.tolist()


def mixed_serving(seed: int = 1239, batch: int = 64, block_size: int = 32, pool_init: str = "cheap",
                  kv_data=None, device="cpu") -> PagedProblem:
    """Mixed serving batch: lognormal contexts (median 2048, sigma 1, clipped to [16, 32768]),
    32 Q heads sharing 8 KV heads, head_dim 128, bf16, block_size 32, fragmented pool.

    Fragmentation: the pool holds twice the pages needed; filler requests take every block,
    a seeded random half of them is released (in shuffled order), and the real sequences --
    visited in a shuffled order -- are allocated from what was freed."""
    gen = torch.Generator().manual_seed(seed)
    lens = mixed_lens(seed + 11, batch)
    need = [(L + block_size - 1) // block_size for L in lens]
    nb = 2 * sum(need)
    alloc = BlockAllocator(nb, block_size)
    filler = []
    while alloc.free:
        n = min(len(alloc.free), int(torch.randint(1, 64, (1,), generator=gen)))
        filler.extend(alloc.allocate(n * block_size))
    perm = torch.randperm(len(filler), generator=gen).tolist()
    alloc.release([filler[i] for i in perm[: nb // 2]])
    order = torch.randperm(batch, generator=gen).tolist()
    tables: List[List[int]] = [[] for _ in range(batch)]
    for b in order:
        tables[b] = alloc.allocate(lens[b])
    mb = (32768 + block_size - 1) // block_size
    return make_problem("mixed_serving", batch=batch, num_q_heads=32, num_kv_heads=8, head_dim=128,
                        block_size=block_size, context_lens=lens, q_lens=[1] * batch, dtype=BF16,
                        causal=False, seed=seed + 1, num_blocks=nb, tables=tables, max_blocks_per_seq=mb,
                        pool_init=pool_init, kv_data=kv_data, device=device)


def prefix_shared(seed: int = 1240, batch: int = 16, prefix: int = 4096, lo: int = 256, hi: int = 2048,
                  block_size: int = 16, heads: int = 32, kv_heads: Optional[int] = None, head_dim: int = 128,
                  dtype: str = F16, prefill: bool = False, pool_init: str = "cheap", device="cpu") -> PagedProblem:
    """Prefix caching (pwwt.cn write-up on chunked attention, section 5.4): `batch` requests open
    with the same `prefix`-token prompt, then carry their own tokens (uniform in [lo, hi]).

    The pages filled by the prompt alone (prefix // block_size of them) are allocated once and
    shared, through the allocator's reference counts, by every request's block table; the
    prompt's partial last page (if any) and each request's own tokens go to private pages, since
    a request writes into them; the prompt's pages keep one reference of their own (the prefix
    cache's) besides one per request. The pool holds the shared pages, the private pages and 10%
    spare, handed out in a seeded random order. k_ctx / v_ctx hold every request's whole context
    (the prompt rows identical across requests). With `prefill`, each request's queries are its
    tokens after the shared pages (the part a prefix-cache hit still has to compute, causal);
    otherwise one decode query per request. `shared_append` and `private_append` split the
    context's append into the prompt's shared pages (once) and each request's own rows."""
    kv_heads = heads if kv_heads is None else kv_heads
    gen = torch.Generator().manual_seed(seed)
    own = torch.randint(lo, hi + 1, (batch,), generator=gen).tolist()
    lens = [prefix + n for n in own]
    n_shared = prefix // block_size
    shared_tokens = n_shared * block_size
    private = [(L + block_size - 1) // block_size - n_shared for L in lens]
    nb = int(math.ceil(1.1 * (n_shared + sum(private))))
    order = torch.randperm(nb, generator=gen).tolist()
    alloc = BlockAllocator(nb, block_size, order)
    shared = alloc.allocate(shared_tokens)
    tables = [alloc.share(shared) + alloc.allocate(L - shared_tokens) for L in lens]
    dgen = data_generator(seed + 5, device)
    k_pre = randn_t(dgen, (prefix, kv_heads, head_dim), dtype)
    v_pre = randn_t(dgen, (prefix, kv_heads, head_dim), dtype)
    k_parts, v_parts = [], []
    for n in own:
        k_parts += [k_pre, randn_t(dgen, (n, kv_heads, head_dim), dtype)]
        v_parts += [v_pre, randn_t(dgen, (n, kv_heads, head_dim), dtype)]
    q_lens = [L - shared_tokens for L in lens] if prefill else [1] * batch
    mb = max(len(t) for t in tables)
    p = make_problem("prefix_shared", batch=batch, num_q_heads=heads, num_kv_heads=kv_heads, head_dim=head_dim,
                     block_size=block_size, context_lens=lens, q_lens=q_lens, dtype=dtype, causal=prefill,
                     seed=seed + 1, num_blocks=nb, tables=tables, max_blocks_per_seq=mb, pool_init=pool_init,
                     kv_data=(torch.cat(k_parts), torch.cat(v_parts)), device=device)
    p.meta.update(prefix=prefix, shared_tokens=shared_tokens, shared_blocks=shared, allocator=alloc)
    return p


def shared_append(p: PagedProblem) -> dict:
    """Append arguments that write the shared prompt pages once (request 0's first rows)."""
    s = p.meta["shared_tokens"]
    return dict(k_new=p.k_ctx[:s], v_new=p.v_ctx[:s], cu_new_lens=cu_lens([s]),
                ctx_before=torch.zeros(1, dtype=torch.int32), block_tables=p.block_tables[:1].clone())


def private_append(p: PagedProblem) -> dict:
    """Append arguments that write every request's rows after the shared pages."""
    s = p.meta["shared_tokens"]
    rows, start = [], 0
    for L in p.context_lens.tolist():
        rows.append(torch.arange(start + s, start + L))
        start += L
    rows = torch.cat(rows)
    return dict(k_new=p.k_ctx[rows].contiguous(), v_new=p.v_ctx[rows].contiguous(),
                cu_new_lens=cu_lens([L - s for L in p.context_lens.tolist()]),
                ctx_before=torch.full((p.batch,), s, dtype=torch.int32), block_tables=p.block_tables.clone())


def append_step(p: PagedProblem, seed: int = 99) -> dict:
    """One decode step's new tokens: one token per sequence at position context_lens[b]
    (its page is allocated from the pool's unused blocks when the last page is full)."""
    gen = torch.Generator().manual_seed(seed)
    used = set(int(x) for x in p.block_tables.flatten().tolist() if x >= 0)
    spare = [i for i in range(p.num_blocks) if i not in used]
    bt = p.block_tables.clone()
    for b, L in enumerate(p.context_lens.tolist()):
        if L % p.block_size == 0:
            if not spare:
                raise OutOfBlocks("no spare block for sequence %d's new token" % b)
            slot = L // p.block_size
            if slot >= bt.shape[1]:
                raise ValueError("sequence %d is at max_blocks_per_seq" % b)
            bt[b, slot] = spare.pop()
    k = randn_t(gen, (p.batch, p.num_kv_heads, p.head_dim), p.dtype)
    v = randn_t(gen, (p.batch, p.num_kv_heads, p.head_dim), p.dtype)
    return dict(k_new=k, v_new=v, cu_new_lens=cu_lens([1] * p.batch), ctx_before=p.context_lens.clone(),
                block_tables=bt)
