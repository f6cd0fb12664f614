// decode_tc.cu -- paged_attn_decode for a unit of many query heads of one KV head (grouped-query
// and multi-query attention) with the unit's two products on the 5th-generation tensor cores.
//
// Same computation as decode.cu: for each sequence and query head, softmax(q.K^T * scale) V over
// the cached tokens read through the block table ("企业官网建设流程全解析", section 2.1; layout of
// "Flash Attention与Paged Attention如何共同优化大模型推理？", section 3), with the running max /
// running sum of that page's section 2, split over key/value blocks and merged by log-sum-exp.
// Under grouped-query attention ("为什么Attention是O(n²)", GQA section) the Gu query heads a unit
// serves (a KV head's group, or an equal share of it) form a Gu x D matrix Q_u, and every key tile
// meets it in two dense products: S = Q_u K^T (heads x tokens) and O += P V. Here they are
// tcgen05.mma instructions with M = 128 rows: the unit's heads, rows past Gu being padding that
// is computed and never read (a decode step is bound by the K/V bytes, and the 5th-generation
// tensor cores have the throughput to spare; with mma.sync the same products bounded the call).
//
// Kernel structure (persistent, 6 warps a CTA; one CTA per SM, or two for units of at most 64
// heads at head_dim up to 128, see TcLayout):
//   * units (sequence, unit head, split) are numbered from the context lengths and dealt
//     round-robin, as in decode.cu; splits start at multiples of 128 tokens;
//   * warp 4 streams each unit's q (one TMA box per 64-column half: Gu rows, 128-byte swizzle,
//     into one of the q buffers) and then its key tiles (128 tokens; 64 at head_dim 256 or with two
//     CTAs an SM) into a ring of 2..6 slots, a slot holding a tile's K and then its V: one lane per
//     page issues the page's K boxes and then its V boxes (one 2-D box per 64-column half, as
//     prefill.cu), with an evict-first L2 policy (each line is read once);
//   * warp 5 owns the CTA's TMEM (S_0, S_1 of one key tile's columns, then one or two O buffers of
//     D columns) and one thread issues the MMAs: S_{t%2} = Q K_t^T for tile t, then O += P_t V_t
//     once the softmax has written P_t over S_{t%2}, in the order QK(0), QK(1), PV(0), QK(2),
//     PV(1), ... so that the softmax of tile t + 1 overlaps the P V of tile t;
//   * warps 0..3: the softmax of the unit's heads (M = 128 products: TMEM lanes 32w .. 32w + 31,
//     one row per thread; M = 64: lanes 0-15 of each quarter, a row's columns split between
//     threads t and t + 16; warps with no head rows idle): running max / sum with a lazy rescale
//     (the max moves only when a score exceeds it by more than 2^8), P written to TMEM as its part
//     rounded to the input type plus the rounded remainder, the two P V products accumulating both
//     in FP32, so P is not a rounding to the input type; the unit's epilogue reads O (with two O
//     buffers, while the next unit's products run) and writes the output of a single-split
//     context, or the split's partial and lse for the merge kernel.
#include <cuda.h>

#include "decode_common.cuh"
#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "tcgen05.cuh"
#include "warp_mma.cuh"

namespace pkv {
namespace {

constexpr int kRingMax = 6;   // key tiles (K and V) in flight
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 6 * 32;
constexpr float kRescale = 8.0f;  // lazy rescale threshold (log2 units)
constexpr uint32_t kColS = 0;     // S_0 [0, BN), S_1 [BN, 2 BN)

// Shared memory: the q buffers, then the ring of key tiles (K then V), the barriers and the unit
// tables. A q buffer holds only the unit's Gu rows (rounded up to 8) per 64-column half: the QK
// MMA reads 128 rows of A, and its reads past row Gu run on into the next half, buffer or ring
// tile (always inside the CTA's shared memory, the ring coming after the q buffers) and only
// produce TMEM rows that no one reads.
// kCtas = CTAs per SM: 1 (the SM's 512 TMEM columns and ~227 KB of shared memory), or 2 (each CTA
// 256 columns and half the shared memory: 64-token key tiles, one O buffer, one q buffer; two
// independent pipelines per SM, for units of at most 64 heads at head_dim up to 128).
template <int D, int kCtas>
struct TcLayout {
    static_assert(kCtas == 1 || (kCtas == 2 && D <= 128), "two CTAs an SM: S_0, S_1 and O in 256 columns");
    // tokens per key tile: 128, or 64 at head_dim 256 or two CTAs an SM (a K or V tile <= 32 KB)
    static constexpr int kBN = (D > 128 || kCtas == 2) ? 64 : 128;
    // O buffers in TMEM: two (a unit's epilogue overlaps the next unit), else one
    static constexpr int kNumO = (D > 128 || kCtas == 2) ? 1 : 2;
    static constexpr uint32_t kTmemCols = kCtas == 2 ? 256 : 512;
    // O_0 [kColO, kColO + D), O_1 [kColO + 128, ...) (one O buffer: O_0 only)
    static constexpr uint32_t kColO = kCtas == 2 ? 128 : 256;
    static constexpr int kQBufs = kCtas == 2 ? 1 : 2;
    static constexpr int kHalves = D / 64;                      // 128-byte swizzle atoms along D
    static constexpr uint32_t kTileHalf = kBN * 128;            // kBN rows x 128 bytes
    static constexpr uint32_t kTileBytes = kHalves * kTileHalf;  // a K or V tile
    static constexpr uint32_t kSlotBytes = 2 * kTileBytes;       // a ring slot: K, then V
    static constexpr uint32_t kBarBytes = 512;
    // bytes between the 64-column halves of a q buffer (a multiple of 1024)
    __host__ __device__ static uint32_t q_half(int gu) { return (uint32_t)((gu + 7) / 8) * 8u * 128u; }
    __host__ __device__ static uint32_t q_bytes(int gu) { return kHalves * q_half(gu); }
    __host__ __device__ static size_t ring_off(int gu) { return kQBufs * (size_t)q_bytes(gu); }
    __host__ __device__ static size_t bar_off(int gu, int ring) { return ring_off(gu) + (size_t)ring * kSlotBytes; }
    __host__ __device__ static size_t ints_off(int gu, int ring) { return bar_off(gu, ring) + kBarBytes; }
    __host__ __device__ static size_t smem_bytes(int gu, int batch, int s_max, int ring) {
        return ints_off(gu, ring) + unit_table_ints(batch, s_max) * 4 + 1024;  // + 1024-byte alignment slack
    }
    // the most ring slots (2 .. kRingMax) that fit in max_smem; 0 if not even 2 do
    static int ring_for(int gu, int batch, int s_max, size_t max_smem) {
        for (int r = kRingMax; r >= 2; --r)
            if (smem_bytes(gu, batch, s_max, r) <= max_smem) return r;
        return 0;
    }
};

// TMEM accesses of a softmax thread's columns. M = 128: thread = lane = row, 32x32b. M = 64: the
// .16x32bx2 shape, threads t and t + 16 sharing row t % 16 of the quarter, the second at OFF
// columns further on.
template <int kM, int OFF>
__device__ __forceinline__ void ld_cols32(uint32_t taddr, float (&v)[32]) {
    if constexpr (kM == 64) tc::tmem_ld16x2_32<OFF>(taddr, v);
    else tc::tmem_ld32(taddr, v);
}
template <int kM, int OFF>
__device__ __forceinline__ void st_cols32(uint32_t taddr, const float (&v)[32]) {
    if constexpr (kM == 64) tc::tmem_st16x2_32<OFF>(taddr, v);
    else tc::tmem_st32(taddr, v);
}
template <int kM, int OFF>
__device__ __forceinline__ void st_cols16(uint32_t taddr, const uint32_t (&v)[16]) {
    if constexpr (kM == 64) tc::tmem_st16x2_16<OFF>(taddr, v);
    else tc::tmem_st16(taddr, v);
}

template <int D, bool BF16, int kM, int kCtas>
__global__ void __launch_bounds__(kThreads, kCtas)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                     DecodeArgs a) {
    using L = TcLayout<D, kCtas>;
    constexpr int kBN = L::kBN;
    const int ring = a.stages;
    const int hu = a.cache.num_kv_heads * a.head_groups;  // unit heads
    const int gu = a.num_q_heads / hu;                    // query heads per unit (<= 128)
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment: the 128-byte swizzle pattern is a function of address bits 4-9.
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t *sQ = smem;  // q[kQBufs]
    uint8_t *sRing = smem + L::ring_off(gu);
    const uint32_t q_half = L::q_half(gu), q_bytes = L::q_bytes(gu);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::bar_off(gu, ring));
    uint64_t *kv_full = bars;                // [kRingMax] a key tile's K and V have landed
    uint64_t *kv_empty = bars + kRingMax;    // [kRingMax] its MMAs are done
    uint64_t *q_full = bars + 2 * kRingMax;  // [kQBufs] a unit's q has landed in q buffer i
    uint64_t *q_empty = q_full + 2;          // [kQBufs] the unit's QK MMAs are done with q buffer i
    uint64_t *s_full = q_empty + 2;          // [2] S_i computed
    uint64_t *p_full = s_full + 2;           // [2] P written over S_i (and O rescaled)
    uint64_t *o_done = p_full + 2;           // [2] the P V of the last tile t with t % 2 == i is done
    uint64_t *o_empty = o_done + 2;          // [kNumO] the epilogue has read O_i
    uint64_t *drain = o_empty + 2;           // every MMA issued has completed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const UnitTable ut = unit_table(reinterpret_cast<int *>(smem + L::ints_off(gu, ring)), a.batch, a.s_max);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_sm = kM == 64 ? (gu + 15) >> 4 : (gu + 31) >> 5;  // softmax warps with head rows

    if (threadIdx.x == 0) {
        for (int i = 0; i < ring; ++i) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&kv_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], n_sm);
            mbar_init(&o_done[i], 1);
            mbar_init(&o_empty[i], n_sm);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tc::tmem_alloc(tmem_slot, L::kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    pdl_wait();  // lengths, tables, q and the cache may come from the previous kernel
    const int num_units = decode_scan_units<kThreads>(a, ut);  // ends with __syncthreads
    const int chunk = ut.misc[0];  // the launch's split size
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp) {
        // ===================================== producer warp =====================================
        const int bs = a.cache.block_size, lbs = a.cache.log2_block_size;
        const int box_rows = bs < kBN ? bs : kBN;
        const uint64_t pol = l2_policy_evict_first();  // each K / V line is read once
        if (lane == 0) {
            tc::prefetch_tensormap(&tm_q);
            tc::prefetch_tensormap(&tm_kv);
        }
        uint32_t item = 0;  // key tiles issued
        uint32_t qn = 0;    // units whose q was issued
        bool ok = true;
        UnitCursor c = {};
        PageWindow win = {};
        if ((int)blockIdx.x < num_units) {
            c = unit_of(blockIdx.x, ut, a.s_max, hu, chunk);
            win = unit_pages(a, c, lane);
        }
        for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
            // the next unit's cursor and page ids, loading while this unit's copies go out
            UnitCursor cn = c;
            PageWindow wn = win;
            if (u + (int)gridDim.x < num_units) {
                cn = unit_of(u + gridDim.x, ut, a.s_max, hu, chunk);
                wn = unit_pages(a, cn, lane);
            }
            // q of the unit: rows qrow * Hq + unit head * Gu .. + Gu - 1, one box per 64 columns
            const uint32_t qb = qn % L::kQBufs;
            if (!(ok = mbar_wait(&q_empty[qb], ((qn / L::kQBufs) & 1u) ^ 1u, abort_flag, a.err))) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(&q_full[qb], (uint32_t)gu * D * 2u);
                const int row0 = ut.qrow[c.b] * a.num_q_heads + c.kvh * gu;
#pragma unroll
                for (int hf = 0; hf < L::kHalves; ++hf)
                    tc::tma_load_2d(sQ + qb * q_bytes + hf * q_half, &tm_q, hf * 64, row0, &q_full[qb]);
            }
            ++qn;
            const int *bt = a.block_tables + (size_t)c.b * a.max_blocks_per_seq;
            const int unit_last_page = (c.t1 - 1) >> lbs;
            const int kvr = c.kvh / a.head_groups;  // the unit's KV head
            for (int ts = c.t0; ok && ts < c.t1; ts += kBN) {
                const int n = min(kBN, c.t1 - ts);
                const int npages = bs < kBN ? (n + bs - 1) / bs : 1;  // <= 16 (block size >= 8)
                const int off = bs < kBN ? 0 : (ts & (bs - 1));     // tiles start at multiples of 128
                const int page0 = ts >> lbs;
                if (page0 + npages - 1 >= win.first + win.count)  // units of more than 64 pages
                    win = load_pages(bt, page0, unit_last_page - page0 + 1, lane);
                int pb = window_page(win, page0 + lane);
                if (lane < npages && (pb < 0 || pb >= a.cache.num_blocks)) {
                    set_error(a.err, kErrDeviceRange);
                    pb = 0;
                }
                // one slot per key tile: each lane loads its page's K rows, then its V rows (the same
                // page's lines, back to back)
                const uint32_t slot = item % (uint32_t)ring, ph = (item / (uint32_t)ring) & 1u;
                if (!(ok = mbar_wait(&kv_empty[slot], ph ^ 1u, abort_flag, a.err))) break;
                if (lane == 0)
                    mbar_arrive_expect_tx(&kv_full[slot], 2u * npages * box_rows * 128u * L::kHalves);
                __syncwarp();
                if (lane < npages) {
#pragma unroll
                    for (int kv = 0; kv < 2; ++kv) {
                        const int row = ((pb * 2 + kv) * a.cache.num_kv_heads + kvr) * bs + off;
                        uint8_t *dst = sRing + slot * L::kSlotBytes + kv * L::kTileBytes + (uint32_t)lane * box_rows * 128u;
#pragma unroll
                        for (int hf = 0; hf < L::kHalves; ++hf)
                            tc::tma_load_2d_hint(dst + hf * L::kTileHalf, &tm_kv, hf * 64, row, &kv_full[slot], pol);
                    }
                }
                ++item;
            }
            c = cn;
            win = wn;
        }
        if (!ok) {
            // let the copies in flight land before the CTA exits (bounded)
            volatile int no_abort = 0;
            const uint32_t first = item > (uint32_t)ring ? item - (uint32_t)ring : 0u;
            for (uint32_t i = first; i < item; ++i)
                mbar_wait(&kv_full[i % ring], (i / ring) & 1u, &no_abort, nullptr);
            const uint32_t qfirst = qn > (uint32_t)L::kQBufs ? qn - L::kQBufs : 0u;
            for (uint32_t i = qfirst; i < qn; ++i)
                mbar_wait(&q_full[i % L::kQBufs], (i / L::kQBufs) & 1u, &no_abort, nullptr);
        }
    } else if (warp == kMmaWarp) {
        // ====================================== MMA issuer ======================================
        if (lane == 0) {
            const uint32_t id_qk = tc::idesc_f16(BF16, kM, kBN, false);
            const uint32_t sP = (uint32_t)kBN / 2;  // TMEM columns of one P part (kBN 16-bit values, 2 a column)
            const uint32_t id_pv = tc::idesc_f16(BF16, kM, D, true);
            const uint32_t aQ = smem_addr(sQ), aRing = smem_addr(sRing);
            uint32_t T = 0, U = 0;  // key tiles and units consumed
            bool ok = true;
            auto kv_wait = [&](uint32_t i) {
                return mbar_wait(&kv_full[i % ring], (i / ring) & 1u, abort_flag, a.err);
            };
            // O_ob (+)= P_t V_t: P's rounded part (columns 0-63 of S_{t%2}), then its remainder
            // (columns 64-127); V is [tokens x D], D contiguous: MN-major B, 8-token groups 1024 B
            // apart, 64-column halves kTileHalf apart; 16 tokens = 8 TMEM columns of P
            auto pv = [&](uint32_t t, uint32_t tO, bool first, uint32_t u_of_t) -> bool {
                if (!mbar_wait(&p_full[t & 1u], (t >> 1) & 1u, abort_flag, a.err)) return false;
                // the unit's first P V overwrites its O buffer: the epilogue of the unit that had
                // it before (kNumO units back) must have read it
                if (first && !mbar_wait(&o_empty[u_of_t % L::kNumO], ((u_of_t / L::kNumO) & 1u) ^ 1u, abort_flag, a.err))
                    return false;
                tc::fence_after_sync();
                const uint32_t tP = tmem + kColS + (uint32_t)kBN * (t & 1u);
                const uint32_t aV = aRing + (t % ring) * L::kSlotBytes + L::kTileBytes;
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk)
                        tc::mma_f16_ts(tO, tP + sP * part + 8u * kk,
                                       tc::smem_desc(aV + (uint32_t)kk * 2048u, L::kTileHalf, 1024), id_pv,
                                       (first && part == 0 && kk == 0) ? 0u : 1u);
                tc::mma_commit(&o_done[t & 1u]);
                tc::mma_commit(&kv_empty[t % ring]);  // the slot's K and V are both done
                return true;
            };
            // the tile whose P V is still to be issued: after the next tile's QK, also across units
            bool pending = false, pend_first = false;
            uint32_t pend_t = 0, pend_o = 0, pend_u = 0;
            for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x, ++U) {
                const UnitCursor c = unit_of(u, ut, a.s_max, hu, chunk);
                const int ntiles = (c.t1 - c.t0 + kBN - 1) / kBN;
                const uint32_t qb = U % L::kQBufs, ob = U % L::kNumO;
                if (!(ok = mbar_wait(&q_full[qb], (U / L::kQBufs) & 1u, abort_flag, a.err))) break;
                tc::fence_after_sync();
                const uint32_t aQu = aQ + qb * q_bytes, tO = tmem + L::kColO + 128u * ob;
                for (int k = 0; k < ntiles; ++k, ++T) {
                    // S_{T%2} = Q K_k^T
                    if (!(ok = kv_wait(T))) break;
                    tc::fence_after_sync();
                    const uint32_t aK = aRing + (T % ring) * L::kSlotBytes;
                    const uint32_t tS = tmem + kColS + (uint32_t)kBN * (T & 1u);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t oq = (uint32_t)(kk >> 2) * q_half + (uint32_t)(kk & 3) * 32u;
                        const uint32_t ok_ = (uint32_t)(kk >> 2) * L::kTileHalf + (uint32_t)(kk & 3) * 32u;
                        tc::mma_f16_ss(tS, tc::smem_desc(aQu + oq, 16, 1024), tc::smem_desc(aK + ok_, 16, 1024), id_qk,
                                       kk > 0 ? 1u : 0u);
                    }
                    tc::mma_commit(&s_full[T & 1u]);
                    if (k == ntiles - 1) tc::mma_commit(&q_empty[qb]);  // every QK of the unit issued
                    // the previous tile's P V (its softmax overlapped this QK)
                    if (pending && !(ok = pv(pend_t, pend_o, pend_first, pend_u))) break;
                    pending = true;
                    pend_t = T;
                    pend_o = tO;
                    pend_first = (k == 0);
                    pend_u = U;
                }
            }
            if (ok && pending) ok = pv(pend_t, pend_o, pend_first, pend_u);
            tc::mma_commit(drain);
            volatile int no_abort = 0;
            mbar_wait(drain, 0, &no_abort, a.err);
        }
        __syncwarp();
    } else if (warp < n_sm) {
        // ================================ softmax + epilogue warps ================================
        // M = 128: thread = TMEM lane = row 32 w + lane, with all kBN columns of S and D of O. M = 64:
        // rows 16 w .. 16 w + 15 in lanes 0-15 of the warp's quarter; threads t and t + 16 share row
        // 16 w + t % 16, thread t / 16 = h taking S columns (tokens) [h kBN / 2, (h + 1) kBN / 2) and O
        // columns [h D / 2, (h + 1) D / 2): the row max and sum are combined by one shuffle.
        constexpr int kSplit = kM == 64 ? 2 : 1;
        constexpr int kCols = kBN / kSplit;  // S columns of this thread
        constexpr int kDCols = D / kSplit;   // O columns of this thread
        const int half = kM == 64 ? lane >> 4 : 0;
        const int r = kM == 64 ? warp * 16 + (lane & 15) : warp * 32 + lane;  // head r of the unit
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const float c2 = a.scale * kLog2e;
        uint32_t T = 0, U = 0;
        bool ok = true;
        // a finished unit whose epilogue is still to run
        struct Done {
            UnitCursor c;
            uint32_t U, t_last;
            float m, l;
        };
        bool have_prev = false;
        Done prev = {};
        // O / l of unit d once its last P V is done: the output of a single-split context, or the
        // split's partial and lse; then O_{d.U % 2} is free for the unit after next
        auto epilogue = [&](const Done &d) -> bool {
            if (!mbar_wait(&o_done[d.t_last & 1u], (d.t_last >> 1) & 1u, abort_flag, a.err)) return false;
            tc::fence_after_sync();
            const uint32_t tOd = tmem + L::kColO + 128u * (d.U % L::kNumO) + lane_base;
            const int splits = (ut.lens[d.c.b] + chunk - 1) / chunk;
            const bool row_ok = r < gu;
            float lt = d.l;
            if constexpr (kM == 64) lt += __shfl_xor_sync(0xffffffffu, lt, 16);  // the row's two halves
            const float inv = lt > 0.f ? 1.f / lt : 0.f;
            const float lse_v = lt > 0.f ? (d.m + __log2f(lt)) * kLn2 : -INFINITY;
            const size_t h = (size_t)d.c.kvh * gu + r;  // query head
            const size_t orow = (size_t)ut.qrow[d.c.b] * a.num_q_heads + h;
            const size_t prow = (size_t)d.c.b * a.num_q_heads + h;
#pragma unroll
            for (int cc = 0; cc < kDCols / 32; ++cc) {
                float o[32];
                ld_cols32<kM, kDCols>(tOd + cc * 32, o);
                tc::tmem_wait_ld();
                if (row_ok) {
                    const int col = half * kDCols + cc * 32;
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        const float x[4] = {o[4 * v] * inv, o[4 * v + 1] * inv, o[4 * v + 2] * inv,
                                            o[4 * v + 3] * inv};
                        if (splits == 1) store_out_vec<4>(a.out, orow * D + col + 4 * v, x, a.out_dtype);
                        else store_out_vec<4>(a.part_o, (prow * a.s_max + d.c.split) * D + col + 4 * v, x, 2);
                    }
                }
            }
            if (row_ok && half == 0) {
                if (splits == 1) {
                    if (a.lse) a.lse[orow] = lse_v;
                } else {
                    a.part_lse[prow * a.s_max + d.c.split] = lse_v;
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_empty[d.U % L::kNumO]);
            return true;
        };
        for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x, ++U) {
            const UnitCursor c = unit_of(u, ut, a.s_max, hu, chunk);
            const int ntiles = (c.t1 - c.t0 + kBN - 1) / kBN;
            const uint32_t tO = tmem + L::kColO + 128u * (U % L::kNumO) + lane_base;
            float m = -INFINITY, l = 0.f;
            for (int k = 0; k < ntiles; ++k, ++T) {
                const int n_valid = min(kBN, c.t1 - (c.t0 + k * kBN));
                if (!(ok = mbar_wait(&s_full[T & 1u], (T >> 1) & 1u, abort_flag, a.err))) break;
                tc::fence_after_sync();
                const uint32_t tS = tmem + kColS + (uint32_t)kBN * (T & 1u) + lane_base;
                float s[kCols];  // tokens half * kCols + i of the tile
#pragma unroll
                for (int cc = 0; cc < kCols / 32; ++cc)
                    ld_cols32<kM, kCols>(tS + cc * 32, *reinterpret_cast<float(*)[32]>(&s[cc * 32]));
                tc::tmem_wait_ld();
                const int nv = n_valid - half * kCols;  // visible tokens among this thread's columns
                if (nv < kCols) {
#pragma unroll
                    for (int i = 0; i < kCols; ++i) s[i] = (i < nv) ? s[i] : -INFINITY;
                }
                // row max as 8 independent chains
                float m8[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) m8[q] = fmax3(s[q], s[q + 8], s[q + 16]);
#pragma unroll
                for (int i = 24; i < kCols; i += 16)
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        m8[q] = fmax3(m8[q], s[i + q], (i + 8 + q < kCols) ? s[i + 8 + q] : -INFINITY);
                float mx = fmaxf(fmax3(m8[0], m8[1], m8[2]), fmax3(fmax3(m8[3], m8[4], m8[5]), m8[6], m8[7]));
                if constexpr (kM == 64) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float m_new = fmaxf(m, mx * c2);
                const bool grow = m_new > m + kRescale;  // false when m_new = -inf
                const float alpha = grow ? ex2f(m - m_new) : 1.f;  // 0 when m = -inf
                if (grow) {
                    m = m_new;
                    l *= alpha;
                }
                // every row has a visible key (n_valid >= 1), so m is finite here
                const float2 cc2 = make_float2(c2, c2), nm2 = make_float2(-m, -m);
                uint32_t ph[kCols / 2], pl[kCols / 2];  // P's rounded part and remainder, pairs of tokens
                float2 l4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                make_float2(0.f, 0.f)};
#pragma unroll
                for (int q = 0; q < kCols / 2; ++q) {
                    const float2 xq = ffma2(make_float2(s[2 * q], s[2 * q + 1]), cc2, nm2);
                    const float2 e = make_float2(ex2f(xq.x), ex2f(xq.y));  // ex2(-inf) = 0
                    l4[q & 3] = fadd2(l4[q & 3], e);
                    split_pair<BF16>(e.x, e.y, ph[q], pl[q]);
                }
                const float2 lsum = fadd2(fadd2(l4[0], l4[1]), fadd2(l4[2], l4[3]));
                l += lsum.x + lsum.y;
                // O is rescaled only after the previous tile's P V is done (its S was computed
                // before this tile's QK, so that tile's o_done phase is the only one pending)
                if (k > 0 && __any_sync(0xffffffffu, grow)) {
                    if (!(ok = mbar_wait(&o_done[(T - 1) & 1u], ((T - 1) >> 1) & 1u, abort_flag, a.err))) break;
                    tc::fence_after_sync();
#pragma unroll
                    for (int cc = 0; cc < kDCols / 32; ++cc) {
                        float o[32];
                        ld_cols32<kM, kDCols>(tO + cc * 32, o);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= alpha;
                        st_cols32<kM, kDCols>(tO + cc * 32, o);
                    }
                }
                // tokens at or beyond the unit's end may hold unwritten cache bytes (or the next
                // split's): warp 0 zeroes those V rows so that 0 * garbage cannot reach O
                if (n_valid < kBN && warp == 0) {
                    if (!(ok = mbar_wait(&kv_full[T % ring], (T / ring) & 1u, abort_flag, a.err))) break;
                    uint8_t *sV = sRing + (T % ring) * L::kSlotBytes + L::kTileBytes;
                    for (int row = n_valid + lane; row < kBN; row += 32)
#pragma unroll
                        for (int hf = 0; hf < L::kHalves; ++hf)
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                *reinterpret_cast<uint4 *>(sV + hf * L::kTileHalf + (uint32_t)row * 128u + q * 16) =
                                    make_uint4(0, 0, 0, 0);
                    tc::fence_proxy_async_smem();
                }
#pragma unroll
                for (int cc = 0; cc < kCols / 32; ++cc) {
                    st_cols16<kM, kCols / 2>(tS + cc * 16, *reinterpret_cast<uint32_t(*)[16]>(&ph[cc * 16]));
                    st_cols16<kM, kCols / 2>(tS + kBN / 2 + cc * 16, *reinterpret_cast<uint32_t(*)[16]>(&pl[cc * 16]));
                }
                tc::tmem_wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[T & 1u]);
                if (k == 0 && have_prev) {
                    have_prev = false;
                    if (!(ok = epilogue(prev))) break;
                }
            }
            if (!ok) break;
            // this unit's epilogue runs after the next unit's first tile (or at the end): its last
            // P V is issued after that tile's QK, so by then it is done and nothing waits on it
            have_prev = true;
            prev = {c, U, T - 1, m, l};
        }
        if (ok && have_prev) ok = epilogue(prev);
    }
    tc::fence_before_sync();
    __syncthreads();
    pdl_launch_dependents();
    if (warp == kMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, L::kTmemCols);
    }
}

template <int D, bool BF16, int kM, int kCtas>
cudaError_t launch_tc_t(const DecodeArgs &a, int grid, cudaStream_t s) {
    using L = TcLayout<D, kCtas>;
    constexpr int kBN = L::kBN;
    const int gu = a.num_q_heads / (a.cache.num_kv_heads * a.head_groups);
    if (gu < 1 || gu > kM) return cudaErrorInvalidValue;
    CUtensorMap tm_q, tm_kv;
    cudaError_t e = encode_rows_map(a.q, BF16 ? 1 : 0, (long long)a.q_rows * a.num_q_heads, D, 64, gu, &tm_q);
    if (e != cudaSuccess) return e;
    e = encode_cache_map(a.cache, a.cache.block_size < kBN ? a.cache.block_size : kBN, &tm_kv);
    if (e != cudaSuccess) return e;
    const DeviceInfo &info = device_info();
    // shared memory a CTA may take: what the SM gives one CTA, or with two CTAs an SM half of the
    // SM's total (one CTA's maximum plus its 1 KB reserve) less the reserve
    const size_t cta_smem = kCtas == 1 ? (size_t)info.max_smem : ((size_t)info.max_smem + 1024) / 2 - 1024;
    DecodeArgs args = a;
    int ctas = kCtas;
    args.stages = L::ring_for(gu, a.batch, a.s_max, cta_smem);
    if (args.stages == 0 && kCtas > 1) {  // large unit tables: one CTA an SM, with all its shared memory
        ctas = 1;
        args.stages = L::ring_for(gu, a.batch, a.s_max, (size_t)info.max_smem);
    }
    if (args.stages == 0) return cudaErrorInvalidValue;  // tables of this batch and split count do not fit
    auto kern = decode_tc_kernel<D, BF16, kM, kCtas>;
    static DeviceFlags configured;
    if (!configured.test(info.device)) {
        e = set_smem_attributes(kern, info.max_smem);
        if (e != cudaSuccess) return e;
        configured.set(info.device);
    }
    return launch_pdl(kern, dim3(grid * ctas), dim3(kThreads), L::smem_bytes(gu, a.batch, a.s_max, args.stages), s,
                      tm_q, tm_kv, args);
}

template <int D, int kM, int kCtas>
cudaError_t launch_tc_d(const DecodeArgs &a, bool bf16, int grid, cudaStream_t s) {
    return bf16 ? launch_tc_t<D, true, kM, kCtas>(a, grid, s) : launch_tc_t<D, false, kM, kCtas>(a, grid, s);
}

}  // namespace

cudaError_t launch_decode_tc(const DecodeArgs &a, int grid, cudaStream_t s) {
    if (a.batch == 0) return cudaSuccess;
    if (a.chunk % 128 != 0) return cudaErrorInvalidValue;  // splits start at multiples of 128 tokens
    const bool bf16 = a.cache.dtype == 1;
    // units of at most 64 query heads: M = 64 products (half the tensor time of M = 128, and their
    // rows spread over twice the softmax warps)
    const bool m64 = a.num_q_heads / (a.cache.num_kv_heads * a.head_groups) <= 64;
    // units of at most 64 heads at head_dim up to 128 run two CTAs an SM: two independent
    // pipelines, each with 64-token key tiles in half the SM's TMEM and shared memory
    switch (a.cache.head_dim) {
        case 256: return m64 ? launch_tc_d<256, 64, 1>(a, bf16, grid, s) : launch_tc_d<256, 128, 1>(a, bf16, grid, s);
        case 128: return m64 ? launch_tc_d<128, 64, 2>(a, bf16, grid, s) : launch_tc_d<128, 128, 1>(a, bf16, grid, s);
        case 64: return m64 ? launch_tc_d<64, 64, 2>(a, bf16, grid, s) : launch_tc_d<64, 128, 1>(a, bf16, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv
