// decode_gqa.cu -- paged_attn_decode for grouped-query attention with units of four or eight
// query heads per KV head, the group's q.K^T and P.V contractions on tensor cores (mma.sync; the
// kernel is written for units of up to 32 heads, and the library routes other groups to the
// tcgen05 kernel of decode_tc.cu).
//
// Same computation as decode.cu: for each sequence and query head, softmax(q.K^T * scale) V over
// the cached tokens read through the block table ("企业官网建设流程全解析", section 2.1; layout of
// "Flash Attention与Paged Attention如何共同优化大模型推理？", section 3), with the running max /
// running sum of that page's section 2, split over key/value blocks and merged by log-sum-exp.
// Under grouped-query attention ("为什么Attention是O(n²)", GQA section) the G query heads of a KV
// head form a G x D matrix, so every K and V tile meets a dense product: S^T = K_tile Q_g^T
// (tokens x heads) and O^T += V_tile^T P^T. On CUDA cores each K/V element would cost G FMAs plus
// conversions and cross-lane sums; here one mma.sync m16n8k16 covers 16 tokens x 8 head slots x
// 16 dims.
//
// Kernel structure (persistent, two CTAs per SM, each with half the SM's shared memory: two
// independent pipelines whose waits overlap; 6 warps a CTA, 10 for units of 16 or 32 query heads):
//   * units (sequence, KV head, split) are numbered from the context lengths and dealt
//     round-robin to the CTAs, as in decode.cu;
//   * the producer warp streams each unit's 64-token tiles with TMA: the page ids of a unit are
//     read one unit ahead, and each lane issues its page slice's boxes (K rows then V rows, 64
//     columns, 128-byte swizzle, through a 5-D tensor map over the cache; evict-first in L2, since
//     each line is read once), into a ring of as many stages (up to 6) as the shared memory left
//     by the merge buffers, the two q buffers and the unit tables holds; each unit's q goes to one
//     of two q buffers with barriers of their own (units can be shorter than the ring);
//   * warps 0-3 each own 16 tokens of a tile (units of 16 or 32 query heads: warps 0-7, two per 16
//     tokens, each with half the unit's 8-head n-tiles, so that each dependent chain is half as
//     long and every scheduler has two of them): ldmatrix from the swizzled tile gives the A fragments
//     of K (row) and of V (transposed); q, held as B fragments for the whole unit, has the group's
//     heads in the N slots (padding slots are zero); the scores stay in the accumulator fragments:
//     column max by shuffles, lazy rescale (threshold 2^8), exp2, and P, as a part rounded to the
//     input type plus its rounded remainder, moved into B-fragment layout with movmatrix; O^T
//     accumulates both parts' products in FP32 registers; at the end of a unit each warp leaves
//     its rows in a shared-memory merge buffer (two taking turns; one for 16- and 32-head units)
//     and goes on with the next unit;
//   * the last warp merges the four token slices' rows and writes the output (single split) or
//     the split partials.
#include <cuda.h>

#include "decode_common.cuh"
#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "tcgen05.cuh"
#include "warp_mma.cuh"

namespace pkv {
namespace {

constexpr int kWarps = 4;                         // token slices of a tile, 16 tokens each
constexpr int kTile = 64;                         // tokens per stage
constexpr int kStagesMax = 6;
constexpr int kCtasPerSm = 2;  // resident CTAs per SM (100 / 139 registers a thread for 4 / 8 heads)
constexpr float kRescale = 8.0f;                  // lazy rescale threshold (log2 units)

// Shared memory: the merge buffers, the barriers and unit ids (fixed sizes), then from the
// next 1024-byte boundary the ring of stages, then the unit tables (sized by batch and splits).
template <int D, int G>
struct GqaLayout {
    static constexpr int kHalves = D / 64;                          // 128-byte swizzle atoms along D
    static constexpr uint32_t kHalfBytes = kTile * 128;             // 64 rows x 128 bytes
    static constexpr uint32_t kKBytes = kHalves * kHalfBytes;       // one K (or V) tile
    // per 64-column half: page slices of br rows, each its br K rows then its br V rows
    static constexpr uint32_t kHalfRegion = 2 * kHalfBytes;
    static constexpr uint32_t kQBytes = G * D * 2;
    static constexpr uint32_t kStageBytes = 2 * kKBytes;  // K and V of a tile (q has its own buffers)
    static constexpr uint32_t kMergeFloats = kWarps * G * kMergeRow<D>;  // one merge buffer
    // 16 or 32 heads: one merge buffer (the consumers wait for the merge of the previous unit),
    // which leaves room for another stage; fewer heads: two, taking turns
    static constexpr int kMergeBufs = G >= 16 ? 1 : 2;
    // q of two units, taking turns (a unit's q is read at its first tile)
    static constexpr uint32_t kQOffset = kMergeBufs * kMergeFloats * 4;
    // barriers: full / empty per stage slot, merge full / empty per merge buffer, q full / empty
    // per q buffer; then the abort flag (padded to 16 bytes), the unit of each stage slot and the
    // unit of each merge buffer
    static constexpr uint32_t kBarOffset = kQOffset + 2 * kQBytes;
    static constexpr uint32_t kFixedBytes = kBarOffset + (2 * kStagesMax + 8) * 8 + 16 + (kStagesMax + 2) * 4;
    static constexpr uint32_t kStagesOffset = (kFixedBytes + 1023) / 1024 * 1024;
    __host__ __device__ static size_t ints_offset(int stages) { return kStagesOffset + (size_t)stages * kStageBytes; }
    __host__ __device__ static size_t smem_bytes(int batch, int s_max, int stages) {
        return ints_offset(stages) + unit_table_ints(batch, s_max) * 4 + 1024;  // + 1024-byte alignment slack
    }
    // the most stages (2 .. kStagesMax) that fit in max_smem; 0 if not even 2 do
    static int stages_for(int batch, int s_max, size_t max_smem) {
        for (int st = kStagesMax; st >= 2; --st)
            if (smem_bytes(batch, s_max, st) <= max_smem) return st;
        return 0;
    }
};

// Warp roles: kHS consumer warps per token slice, each with NT / kHS of the unit's n-tiles of 8
// head slots; then the producer and the merge warp.
template <int G>
struct GqaWarps {
    static constexpr int kHS = G >= 16 ? 2 : 1;
    static constexpr int kConsumers = kWarps * kHS;
    static constexpr int kProducer = kConsumers;
    static constexpr int kMerge = kConsumers + 1;
    static constexpr int kThreads = (kConsumers + 2) * 32;
};

// Shared-memory address of token row t, 16-byte chunk cc (0..7) of a 64-column half in the
// 128-byte-swizzled layout TMA writes (chunk position cc ^ (t & 7)).
__device__ __forceinline__ uint32_t swz(uint32_t half_base, int t, int cc) {
    return half_base + (uint32_t)t * 128u + ((uint32_t)(cc ^ (t & 7)) << 4);
}

template <int D, int G, bool BF16>
__global__ void __launch_bounds__(GqaWarps<G>::kThreads, kCtasPerSm)
    decode_gqa_kernel(const __grid_constant__ CUtensorMap tm_kv, DecodeArgs a) {
    using L = GqaLayout<D, G>;
    using W = GqaWarps<G>;
    const int nst = a.stages;  // stages of the ring: 2 .. kStagesMax, chosen at launch
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    float *merge = reinterpret_cast<float *>(base);  // [kMergeBufs][kWarps][G][kMergeRow<D>]
    uint64_t *full = reinterpret_cast<uint64_t *>(base + L::kBarOffset);
    uint64_t *empty = full + kStagesMax;
    uint64_t *mfull = empty + kStagesMax;  // [2] the consumer warps' rows of a unit are in buffer i
    uint64_t *mempty = mfull + 2;          // [2] the merge warp has read buffer i
    uint64_t *qfull = mempty + 2;          // [2] q of a unit has landed in q buffer i
    uint64_t *qempty = qfull + 2;          // [2] the consumer warps have read q buffer i
    uint8_t *qbuf = base + L::kQOffset;    // [2][G][D]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(qempty + 2);
    int *stage_unit = reinterpret_cast<int *>(qempty + 2) + 4;
    int *merge_unit = stage_unit + kStagesMax;  // [2] unit of each merge buffer, -1: end
    uint8_t *smem = base + L::kStagesOffset;    // stage i at i * kStageBytes
    const UnitTable ut = unit_table(reinterpret_cast<int *>(base + L::ints_offset(nst)), a.batch, a.s_max);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hkv = a.cache.num_kv_heads, bs = a.cache.block_size;
    const int hu = hkv * a.head_groups;  // unit heads (KV heads, or groups of query heads)
    const int br = bs < kTile ? bs : kTile;  // rows per page slice (tiles start at multiples of 64)

    if (tid == 0) {
        for (int i = 0; i < nst; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], W::kConsumers);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&mfull[i], W::kConsumers);
            mbar_init(&mempty[i], 1);
            mbar_init(&qfull[i], 1);
            mbar_init(&qempty[i], W::kConsumers);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    pdl_wait();  // lengths, tables, q and the cache may come from the previous kernel
    const int num_units = decode_scan_units<W::kThreads>(a, ut);
    const int chunk = ut.misc[0];  // the launch's split size

    if (warp == W::kProducer) {
        // ===================================== producer warp =====================================
        const uint64_t pol = l2_policy_evict_first();
        const uint16_t *qg = static_cast<const uint16_t *>(a.q);
        if (lane == 0) tc::prefetch_tensormap(&tm_kv);
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_mask = 0, issued_parity = 0;
        int qb = 0;                      // q buffer of the next unit
        uint32_t qphase = 0;
        uint32_t q_issued = 0, q_parity = 0;  // q copies issued per buffer (for the abort drain)
        UnitCursor c = {};
        PageWindow win = {};
        if ((int)blockIdx.x < num_units) {
            c = unit_of(blockIdx.x, ut, a.s_max, hu, chunk);
            win = unit_pages(a, c, lane);
        }
        // on a wait that gave up: let every copy in flight land before the warp exits (bounded)
        auto drain = [&]() {
            volatile int no_abort = 0;
            for (int i = 0; i < nst; ++i)
                if (issued_mask & (1u << i)) mbar_wait(&full[i], (issued_parity >> i) & 1u, &no_abort, nullptr);
            for (int i = 0; i < 2; ++i)
                if (q_issued & (1u << i)) mbar_wait(&qfull[i], (q_parity >> i) & 1u, &no_abort, nullptr);
        };
        for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
            // the next unit's cursor and page ids, loading while this unit's copies go out
            UnitCursor cn = c;
            PageWindow wn = win;
            if (u + (int)gridDim.x < num_units) {
                cn = unit_of(u + gridDim.x, ut, a.s_max, hu, chunk);
                wn = unit_pages(a, cn, lane);
            }
            const int *bt = a.block_tables + (size_t)c.b * a.max_blocks_per_seq;
            const int unit_last_page = (c.t1 - 1) >> a.cache.log2_block_size;
            // the unit's q into q buffer qb, once the consumers have read the unit two back from it
            if (!mbar_wait(&qempty[qb], qphase ^ 1u, abort_flag, a.err)) {
                drain();
                return;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(&qfull[qb], L::kQBytes);
                const uint16_t *qsrc = qg + ((size_t)ut.qrow[c.b] * a.num_q_heads + (size_t)c.kvh * G) * D;
                bulk_g2s(qbuf + qb * L::kQBytes, qsrc, L::kQBytes, &qfull[qb], pol);
            }
            q_issued |= 1u << qb;
            q_parity = (q_parity & ~(1u << qb)) | (qphase << qb);
            if (++qb == 2) {
                qb = 0;
                qphase ^= 1u;
            }
            for (int ts = c.t0; ts < c.t1; ts += kTile) {
                const int n = min(kTile, c.t1 - ts);
                const int nslices = (n + br - 1) / br;  // <= 8
                const int page0 = ts >> a.cache.log2_block_size;
                const int page_last = (ts + n - 1) >> a.cache.log2_block_size;
                if (page_last >= win.first + win.count)  // units of more than 64 pages
                    win = load_pages(bt, page0, unit_last_page - page0 + 1, lane);
                const int tok0 = ts + lane * br;  // this lane's slice
                const int off = tok0 & (bs - 1);
                int pb = window_page(win, tok0 >> a.cache.log2_block_size);
                if (lane < nslices) {
                    if (pb < 0 || pb >= a.cache.num_blocks) {
                        set_error(a.err, kErrDeviceRange);
                        pb = 0;
                    }
                }
                if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.err)) {
                    drain();
                    return;
                }
                uint8_t *st = smem + (size_t)stage * L::kStageBytes;
                if (lane == 0) {
                    stage_unit[stage] = u;
                    mbar_arrive_expect_tx(&full[stage], (uint32_t)nslices * br * 128u * L::kHalves * 2u);
                }
                __syncwarp();
                if (lane < nslices) {
                    // one box per 64-column half: the slice's K rows, then its V rows
                    const int kvr = c.kvh / a.head_groups;
                    const uint32_t dst = (uint32_t)lane * 2u * br * 128u;
#pragma unroll
                    for (int hf = 0; hf < L::kHalves; ++hf)
                        tc::tma_load_5d_hint(st + hf * L::kHalfRegion + dst, &tm_kv, hf * 64, off, kvr, 0, pb,
                                             &full[stage], pol);
                }
                issued_mask |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == nst) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            c = cn;
            win = wn;
        }
        if (mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.err) && lane == 0) {
            stage_unit[stage] = -1;
            mbar_arrive(&full[stage]);
        }
        return;
    }

    if (warp == W::kMerge) {
        // ====================================== merge warp ======================================
        merge_warp_loop<D, G, kWarps, L::kMergeBufs>(a, ut, merge, L::kMergeFloats, mfull, mempty, merge_unit, abort_flag,
                                                    lane);
        pdl_launch_dependents();
        return;
    }

    // ===================================== consumer warps =====================================
    // The group's heads fill n-tiles of 8 head slots (padding slots zero); this warp holds NT of
    // them, from n-tile nt0, for the 16 tokens of its slice.
    constexpr int kKSteps = D / 16;         // k-steps of q.K^T, m-tiles of O^T
    constexpr int NT = (G + 7) / 8 / W::kHS;
    static_assert(NT * W::kHS * 8 >= G, "n-tiles must cover the group");
    const int slice = warp % kWarps, nt0 = (warp / kWarps) * NT;
    const int gid = lane >> 2, tig = lane & 3;
    const int g_lo = 2 * tig;               // this lane's two head slots of each n-tile
    const float sl = a.scale * kLog2e;
    uint32_t bq[kKSteps][NT][2];            // q as B fragments (n = head slot, k = dims)
    int stage = 0;
    uint32_t phase = 0;
    int mbuf = 0;  // merge buffer of the next unit
    uint32_t mphase = 0;
    int qb = 0;    // q buffer of the next unit
    uint32_t qphase = 0;
    for (;;) {
        if (!mbar_wait(&full[stage], phase, abort_flag, a.err)) return;
        const int u = stage_unit[stage];
        if (u < 0) break;
        const UnitCursor c = unit_of(u, ut, a.s_max, hu, chunk);
        {
            // the unit's q as B fragments, then q buffer qb is free for the unit after next
            if (!mbar_wait(&qfull[qb], qphase, abort_flag, a.err)) return;
            const uint16_t *sq = reinterpret_cast<const uint16_t *>(qbuf + qb * L::kQBytes);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int hs = (nt0 + nt) * 8 + gid;  // head slot
#pragma unroll
                for (int kk = 0; kk < kKSteps; ++kk) {
                    if (hs < G) {
                        bq[kk][nt][0] = *reinterpret_cast<const uint32_t *>(sq + hs * D + kk * 16 + 2 * tig);
                        bq[kk][nt][1] = *reinterpret_cast<const uint32_t *>(sq + hs * D + kk * 16 + 8 + 2 * tig);
                    } else {
                        bq[kk][nt][0] = bq[kk][nt][1] = 0u;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&qempty[qb]);
            if (++qb == 2) {
                qb = 0;
                qphase ^= 1u;
            }
        }
        float m[NT][2], l[NT][2];
        float o[kKSteps][NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            m[nt][0] = m[nt][1] = -INFINITY;
            l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
            for (int mt = 0; mt < kKSteps; ++mt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
        }
        for (int ts = c.t0; ts < c.t1; ts += kTile) {
            const int n = min(kTile, c.t1 - ts);
            if (ts != c.t0 && !mbar_wait(&full[stage], phase, abort_flag, a.err)) return;
            uint8_t *st = smem + (size_t)stage * L::kStageBytes;
            const uint32_t aK = smem_addr(st), aV = aK + br * 128u;  // + slice row tp: K; + tp: V
            const int t0w = slice * 16;     // this warp's tokens in the tile
            if (t0w + 16 > n) {
                // tokens at or beyond the context end may hold unwritten cache bytes (or stale
                // tile data): zero this warp's V rows there so that 0 * garbage cannot reach O
                for (int t = t0w + (lane >> 3); t < t0w + 16; t += 4) {
                    if (t < n) continue;
                    const int tp = t + (t & -br);  // tile row t in the slice layout
#pragma unroll
                    for (int hf = 0; hf < L::kHalves; ++hf)
                        *reinterpret_cast<uint4 *>(st + hf * L::kHalfRegion + (tp + br) * 128 + (lane & 7) * 16) =
                            make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }
            // ---- S^T = K_w q^T: 16 tokens x 8 head slots per n-tile (one K fragment for all) ----
            float s[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
            {
                const int mi = lane >> 3;
                const int t = t0w + (lane & 7) + 8 * (mi & 1);
                const int tp = t + (t & -br);  // slice j starts at row 2 * j * br of its half
#pragma unroll
                for (int kk = 0; kk < kKSteps; ++kk) {
                    uint32_t af[4];
                    const int cc = 2 * (kk & 3) + (mi >> 1);
                    ldsm_x4(swz(aK + (kk >> 2) * L::kHalfRegion, tp, cc), af);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma16816<BF16>(s[nt], af, bq[kk][nt][0], bq[kk][nt][1]);
                }
            }
            const bool v0 = t0w + gid < n, v1 = t0w + gid + 8 < n;
            uint32_t pb[NT][2], pr[NT][2];  // P in the input type, and its remainders
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                s[nt][0] = v0 ? s[nt][0] : -INFINITY;
                s[nt][1] = v0 ? s[nt][1] : -INFINITY;
                s[nt][2] = v1 ? s[nt][2] : -INFINITY;
                s[nt][3] = v1 ? s[nt][3] : -INFINITY;
                // column max over the 16 tokens (lanes with the same tig)
                float mx0 = fmaxf(s[nt][0], s[nt][2]), mx1 = fmaxf(s[nt][1], s[nt][3]);
#pragma unroll
                for (int ofs = 4; ofs < 32; ofs <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, ofs));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, ofs));
                }
                mx0 *= sl;
                mx1 *= sl;
                // lazy rescale: a head's running max moves only when a score exceeds it by > 2^8
                if (mx0 > m[nt][0] + kRescale) {
                    const float al = ex2f(m[nt][0] - mx0);  // 0 when m = -inf
                    l[nt][0] *= al;
#pragma unroll
                    for (int mt = 0; mt < kKSteps; ++mt) {
                        o[mt][nt][0] *= al;
                        o[mt][nt][2] *= al;
                    }
                    m[nt][0] = mx0;
                }
                if (mx1 > m[nt][1] + kRescale) {
                    const float al = ex2f(m[nt][1] - mx1);
                    l[nt][1] *= al;
#pragma unroll
                    for (int mt = 0; mt < kKSteps; ++mt) {
                        o[mt][nt][1] *= al;
                        o[mt][nt][3] *= al;
                    }
                    m[nt][1] = mx1;
                }
                const float p0 = v0 ? ex2f(fmaf(s[nt][0], sl, -m[nt][0])) : 0.f;
                const float p1 = v0 ? ex2f(fmaf(s[nt][1], sl, -m[nt][1])) : 0.f;
                const float p2 = v1 ? ex2f(fmaf(s[nt][2], sl, -m[nt][0])) : 0.f;
                const float p3 = v1 ? ex2f(fmaf(s[nt][3], sl, -m[nt][1])) : 0.f;
                l[nt][0] += p0 + p2;
                l[nt][1] += p1 + p3;
                // P^T (tokens x head slots) in accumulator layout -> P as B fragments (k = tokens).
                // P goes in as a rounded part and a remainder, each its own MMA into the same FP32
                // accumulator, so P.V sees P almost unrounded: the only rounding to the input type
                // on the decode path stays the output's
                uint32_t h01, r01, h23, r23;
                split_pair<BF16>(p0, p1, h01, r01);
                split_pair<BF16>(p2, p3, h23, r23);
                pb[nt][0] = movmatrix_t(h01);
                pb[nt][1] = movmatrix_t(h23);
                pr[nt][0] = movmatrix_t(r01);
                pr[nt][1] = movmatrix_t(r23);
            }
            // ---- O^T += V_w^T P^T: D x 8 head slots per n-tile (one V fragment for all) ----
            {
                const int mi = lane >> 3;
                const int t = t0w + (lane & 7) + 8 * (mi >> 1);
                const int tp = t + (t & -br);
#pragma unroll
                for (int mt = 0; mt < kKSteps; ++mt) {
                    uint32_t af[4];
                    const int cc = 2 * (mt & 3) + (mi & 1);
                    ldsm_x4_t(swz(aV + (mt >> 2) * L::kHalfRegion, tp, cc), af);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        mma16816<BF16>(o[mt][nt], af, pr[nt][0], pr[nt][1]);
                        mma16816<BF16>(o[mt][nt], af, pb[nt][0], pb[nt][1]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == nst) {
                stage = 0;
                phase ^= 1u;
            }
        }
        // ---- merge: sum l over the lanes of each head slot, then across the warps ----
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int ofs = 4; ofs < 32; ofs <<= 1) {
                l[nt][0] += __shfl_xor_sync(0xffffffffu, l[nt][0], ofs);
                l[nt][1] += __shfl_xor_sync(0xffffffffu, l[nt][1], ofs);
            }
        // ---- hand this warp's rows to the merge warp ----
        if (!mbar_wait(&mempty[mbuf], mphase ^ 1u, abort_flag, a.err)) return;
        float *rows = merge + (size_t)mbuf * L::kMergeFloats;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int g = (nt0 + nt) * 8 + g_lo + j;
                if (g < G) {
                    float *row = rows + ((size_t)slice * G + g) * kMergeRow<D>;
#pragma unroll
                    for (int mt = 0; mt < kKSteps; ++mt) {
                        row[mt * 16 + gid] = o[mt][nt][j];
                        row[mt * 16 + gid + 8] = o[mt][nt][j + 2];
                    }
                    if (gid == 0) {
                        row[D] = m[nt][j];
                        row[D + 1] = l[nt][j];
                    }
                }
            }
        if (warp == 0 && lane == 0) merge_unit[mbuf] = u;
        __syncwarp();
        if (lane == 0) mbar_arrive(&mfull[mbuf]);
        if (++mbuf == L::kMergeBufs) {
            mbuf = 0;
            mphase ^= 1u;
        }
    }
    // end marker for the merge warp
    if (mbar_wait(&mempty[mbuf], mphase ^ 1u, abort_flag, a.err)) {
        if (warp == 0 && lane == 0) merge_unit[mbuf] = -1;
        __syncwarp();
        if (lane == 0) mbar_arrive(&mfull[mbuf]);
    }
    pdl_launch_dependents();
}

template <int D, int G, bool BF16>
cudaError_t launch_gqa_t(const DecodeArgs &a, int grid, cudaStream_t s) {
    using L = GqaLayout<D, G>;
    CUtensorMap tm;
    const int box_rows = a.cache.block_size < kTile ? a.cache.block_size : kTile;
    cudaError_t e = encode_kv5_map(a.cache, box_rows, &tm);
    if (e != cudaSuccess) return e;
    const DeviceInfo &info = device_info();
    DecodeArgs args = a;
    // each of the SM's kCtasPerSm CTAs takes its share of the SM's shared memory (one CTA's maximum
    // plus its 1 KB reserve), less the reserve
    const size_t cta_smem = ((size_t)info.max_smem + 1024) / kCtasPerSm - 1024;
    int ctas = kCtasPerSm;
    args.stages = L::stages_for(a.batch, a.s_max, cta_smem);
    if (args.stages == 0) {  // large unit tables: one CTA an SM, with the SM's whole shared memory
        ctas = 1;
        args.stages = L::stages_for(a.batch, a.s_max, (size_t)info.max_smem);
    }
    if (args.stages == 0) return cudaErrorInvalidValue;  // tables of this batch and split count do not fit
    auto kern = decode_gqa_kernel<D, G, BF16>;
    static DeviceFlags configured;
    if (!configured.test(info.device)) {
        e = set_smem_attributes(kern, info.max_smem);
        if (e != cudaSuccess) return e;
        configured.set(info.device);
    }
    return launch_pdl(kern, dim3(grid * ctas), dim3(GqaWarps<G>::kThreads), L::smem_bytes(a.batch, a.s_max, args.stages), s,
                      tm, args);
}

}  // namespace

cudaError_t launch_decode_gqa(const DecodeArgs &a, int grid, cudaStream_t s) {
    if (a.batch == 0) return cudaSuccess;
    const int group = a.num_q_heads / (a.cache.num_kv_heads * a.head_groups);  // query heads per unit
    const bool bf16 = a.cache.dtype == 1;
    // units of 4 or 8 query heads; other groups run on the tcgen05 kernel (decode_tc.cu), which
    // measured faster from 16 heads a unit on (MQA: 0.077 against 0.092 ms), slower below
    if (a.cache.head_dim == 128) {
        if (group == 4) return bf16 ? launch_gqa_t<128, 4, true>(a, grid, s) : launch_gqa_t<128, 4, false>(a, grid, s);
        if (group == 8) return bf16 ? launch_gqa_t<128, 8, true>(a, grid, s) : launch_gqa_t<128, 8, false>(a, grid, s);
    } else {
        if (group == 4) return bf16 ? launch_gqa_t<64, 4, true>(a, grid, s) : launch_gqa_t<64, 4, false>(a, grid, s);
        if (group == 8) return bf16 ? launch_gqa_t<64, 8, true>(a, grid, s) : launch_gqa_t<64, 8, false>(a, grid, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace pkv
