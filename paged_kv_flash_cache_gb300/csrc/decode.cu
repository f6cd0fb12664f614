// decode.cu -- paged_attn_decode (split-KV, online softmax) and the split merge.
//
// What it computes: for each sequence b and query head h, softmax(q.K^T * scale) V over the
// sequence's cached tokens ("为什么Attention是O(n²)", mathematics section), reading K/V
// through the block table ("企业官网建设流程全解析", section 2.1; cache layout of
// "Flash Attention与Paged Attention如何共同优化大模型推理？", section 3) with the running-max /
// running-sum update of that page's section 2: new max m', old sum and output scaled by
// exp(m - m'), final division by the sum.  Contexts are cut into splits of `chunk` tokens so a
// small batch still fills every SM (parallelism over key/value blocks, "从一次压测翻车说起",
// sections 3.3 and 5.3); split results are merged by their log-sum-exp instead of atomics.
//
// Kernel structure (persistent, two CTAs per SM: two independent pipelines of two stages each
// keep the same bytes in flight as one of four, and each covers the other's waits):
//   * work unit = (sequence, KV head, split); units are numbered in a prologue from the
//     context lengths (decode_common.cuh: split-major, all KV heads of a sequence together)
//     and dealt round-robin to the CTAs;
//   * warp 8 (producer) streams each unit's tokens in 64-token tiles into a ring of
//     shared-memory stages, completion on an mbarrier; page ids are read one unit ahead. A
//     16-bit cache comes by TMA, one box per page slice of min(block_size, 64) tokens holding
//     the slice's K rows and then its V rows (the cache viewed as [NB][2][Hkv][bs][D]); an FP8
//     cache by bulk copies, one per page slice of K, of V and of their row scales. Every read
//     carries an L2 evict-first policy: the stream is read once, and without the hint it
//     pushed the lines still in use out of L2;
//   * warps 0-7 (consumers) each take 8 tokens of a tile: lanes split D into 16-byte
//     chunks, q.k partial sums are reduced with xor shuffles, and every lane keeps running
//     (m, l, acc) for the query heads of its KV head, so each K/V byte is read from HBM once
//     per KV head;
//   * at the end of a unit each consumer warp merges its token slots by shuffles and leaves
//     its (m, l, acc) rows in one of two shared-memory merge buffers; warp 9 (merger) combines
//     the eight warps' rows while the consumers go on with the next unit. A single-split
//     context gets its final output there, otherwise the split's normalised output and lse go
//     to the workspace for the merge kernel.
#include <type_traits>

#include "decode_common.cuh"
#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "tcgen05.cuh"

namespace pkv {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kMergeWarp = kConsumerWarps + 1;
constexpr int kDecodeThreads = (kConsumerWarps + 2) * 32;
constexpr int kMaxBatch = 2048;  // unit tables (lengths, order, split offsets) kept in shared memory
constexpr float kRescaleLog2 = 8.0f;  // lazy rescale threshold (log2 units)

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int D, int G, bool FP8>
struct DecodeLayout {
    // resident CTAs per SM: two for a 16-bit cache (~75 KB of shared memory and 72 registers a
    // thread each), with two stages each; one with four stages over an FP8 cache, whose 4- and
    // 8-head units need more registers than two CTAs leave
    static constexpr int kCtasPerSm = FP8 ? 1 : 2;
    static constexpr int kStages = FP8 ? 4 : 2;
    static constexpr int kTile = kDecodeTile;
    static constexpr int kKB = FP8 ? 1 : 2;                        // bytes per cached element
    static constexpr int kTokPerWarp = kTile / kConsumerWarps;      // 8
    static constexpr int kLanesPerTok = D / 8;                      // 16 (D=128) or 8 (D=64)
    static constexpr int kTokPerStep = 32 / kLanesPerTok;           // 2 or 4
    static constexpr int kSteps = kTokPerWarp / kTokPerStep;        // 4 or 2
    static constexpr int kStepsPerBatch = (kSteps * G <= 16) ? kSteps : (16 / G);  // bounds registers
    static constexpr size_t kKBytes = (size_t)kTile * D * kKB;
    static constexpr size_t kQBytes = (size_t)G * D * 2;
    static constexpr size_t kSOffset = 2 * kKBytes + kQBytes;  // FP8: K row scales [kTile], V row scales [kTile]
    static constexpr size_t kStageBytes = ((kSOffset + (FP8 ? 2 * kTile * 4 : 0)) + 127) / 128 * 128;
    static constexpr size_t kMergeFloats = (size_t)kConsumerWarps * G * kMergeRow<D>;
    static constexpr size_t kBarOffset = kStages * kStageBytes;
    // barriers: full / empty per stage, merge full / empty per merge buffer; then the abort flag
    // (padded to 16 bytes), the unit of each stage and the unit of each merge buffer
    static constexpr size_t kMergeOffset = kBarOffset + (2 * kStages + 4) * 8 + 64;
    // grouped heads (G > 1): a batch of kGqaSteps steps gives each lane of a token group one
    // (token, head) score after a reduce-scatter, i.e. kGqaSteps * G <= kLanesPerTok values
    static constexpr int kGqaSteps = (kSteps * G <= kLanesPerTok) ? kSteps : (kLanesPerTok / G);
    static constexpr int kGqaN = kGqaSteps * G;
    static constexpr size_t kPOffset = kMergeOffset + 2 * kMergeFloats * 4;  // per-warp p broadcast buffer
    static constexpr size_t kPFloats = (size_t)kConsumerWarps * kTokPerStep * kGqaN;
    static constexpr size_t kIntsOffset = kPOffset + kPFloats * 4;
    static size_t smem_bytes(int batch, int s_max) { return kIntsOffset + unit_table_ints(batch, s_max) * 4; }
};

// This lane's 8 elements (chunk chk) of row t of a stage's K or V tile, as fp32 pairs.
template <typename Tag, int D, bool FP8>
__device__ __forceinline__ void load_row8(const uint8_t *tile, int t, int chk, float2 (&f)[4]) {
    if constexpr (FP8) {
        unpack_e4m3x8(*reinterpret_cast<const uint2 *>(tile + (size_t)t * D + chk * 8), f);
    } else {
        unpack8x2(*reinterpret_cast<const uint4 *>(tile + ((size_t)t * D + chk * 8) * 2), f, Tag());
    }
}

// Scale of row t of a tile (FP8 cache), 1 for a native cache.
template <bool FP8>
__device__ __forceinline__ float row_scale(const float *scales, int t) {
    if constexpr (FP8) return scales[t];
    else return 1.f;
}

// Tile row of token t. A native cache arrives by one TMA box per page slice of br = min(bs, 64)
// tokens holding the slice's K rows and then its V rows, so slice j starts at row 2 j br; an
// FP8 cache arrives by bulk copies, all K rows first and the V rows from row kTile on.
template <bool FP8>
__device__ __forceinline__ int k_row(int t, int br) {
    if constexpr (FP8) return t;
    else return t + (t & -br);
}
template <bool FP8>
__device__ __forceinline__ int v_row(int t, int br, int tile) {
    if constexpr (FP8) return t + tile;
    else return t + (t & -br) + br;
}

template <typename Tag, int D, int G, bool FP8>
__global__ void __launch_bounds__(kDecodeThreads, DecodeLayout<D, G, FP8>::kCtasPerSm)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_kv, DecodeArgs a) {
    using L = DecodeLayout<D, G, FP8>;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kBarOffset);
    uint64_t *empty = full + L::kStages;
    uint64_t *mfull = empty + L::kStages;   // [2] the consumer warps' rows of a unit are in buffer i
    uint64_t *mempty = mfull + 2;        // [2] the merger has read buffer i
    volatile int *abort_flag = reinterpret_cast<volatile int *>(mempty + 2);
    int *stage_unit = reinterpret_cast<int *>(mempty + 2) + 4;  // [L::kStages] unit of each filled stage, -1: end
    int *merge_unit = stage_unit + L::kStages;                     // [2] unit of each merge buffer, -1: end
    float *merge = reinterpret_cast<float *>(smem + L::kMergeOffset);  // [2][kConsumerWarps][G][kMergeRow<D>]
    const UnitTable ut = unit_table(reinterpret_cast<int *>(smem + L::kIntsOffset), a.batch, a.s_max);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hkv = a.cache.num_kv_heads, bs = a.cache.block_size;

    if (tid == 0) {
        for (int i = 0; i < L::kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&mfull[i], kConsumerWarps);
            mbar_init(&mempty[i], 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    // Everything below may read memory the previous kernel on the stream wrote (lengths, tables,
    // q, the cache), so only the barrier set-up above overlaps that kernel's tail.
    pdl_wait();
    // ---- prologue: clamp lengths, units per sequence, exclusive scan (all threads) ----
    const int num_units = decode_scan_units<kDecodeThreads>(a, ut);
    const int chunk = ut.misc[0];  // the launch's split size

    if (warp == kProducerWarp) {
        // ================================ producer warp ================================
        const uint64_t pol = l2_policy_evict_first();
        const uint8_t *cache = static_cast<const uint8_t *>(a.cache.ptr);
        const uint16_t *qg = static_cast<const uint16_t *>(a.q);
        const size_t head_bytes = (size_t)bs * D * L::kKB;
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_mask = 0;  // stages with copies issued (bit i), for the abort drain
        uint32_t issued_parity = 0;
        UnitCursor c = {};
        PageWindow win = {};
        if ((int)blockIdx.x < num_units) {
            c = unit_of(blockIdx.x, ut, a.s_max, hkv, chunk);
            win = unit_pages(a, c, lane);
        }
        for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
            // the next unit's cursor and page ids, loading while this unit's copies go out
            UnitCursor cn = c;
            PageWindow wn = win;
            if (u + (int)gridDim.x < num_units) {
                cn = unit_of(u + gridDim.x, ut, a.s_max, hkv, chunk);
                wn = unit_pages(a, cn, lane);
            }
            const int *bt = a.block_tables + (size_t)c.b * a.max_blocks_per_seq;
            const int unit_last_page = (c.t1 - 1) >> a.cache.log2_block_size;
            for (int ts = c.t0; ts < c.t1; ts += L::kTile) {
                const int n = min(L::kTile, c.t1 - ts);
                const int first_page = ts >> a.cache.log2_block_size;
                const int last_page = (ts + n - 1) >> a.cache.log2_block_size;
                const int npages = last_page - first_page + 1;  // <= 64/bs, or 1
                if (last_page >= win.first + win.count)         // units of more than 64 pages
                    win = load_pages(bt, first_page, unit_last_page - first_page + 1, lane);
                // page id of this lane's slice
                int pb = window_page(win, first_page + lane);
                if (lane < npages) {
                    if (pb < 0 || pb >= a.cache.num_blocks) {
                        set_error(a.err, kErrDeviceRange);
                        pb = 0;
                    }
                }
                if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.err)) {
                    // Stop issuing; let copies already in flight land before the CTA exits
                    // (each wait is bounded again).
                    for (int i = 0; i < L::kStages; ++i) {
                        if (issued_mask & (1u << i)) {
                            volatile int no_abort = 0;
                            mbar_wait(&full[i], (issued_parity >> i) & 1u, &no_abort, nullptr);
                        }
                    }
                    return;
                }
                uint8_t *st = smem + (size_t)stage * L::kStageBytes;
                const bool first_tile = (ts == c.t0);
                if (lane == 0) {
                    stage_unit[stage] = u;
                    // native: whole page slices (rows past the context come too; the consumers
                    // mask their scores and skip their V rows); FP8: the valid rows
                    uint32_t bytes = (FP8 ? (uint32_t)n : (uint32_t)npages * (uint32_t)(bs < L::kTile ? bs : L::kTile)) *
                                         D * L::kKB * 2 +
                                     (first_tile ? (uint32_t)L::kQBytes : 0u);
                    if constexpr (FP8) {
                        // row scales, each page slice's copy rounded up to 4 rows (16 bytes)
                        for (int lp = first_page; lp <= last_page; ++lp) {
                            const int m = min(ts + n, (lp + 1) * bs) - max(ts, lp * bs);
                            bytes += 2u * (uint32_t)((m + 3) & ~3) * 4u;
                        }
                    }
                    mbar_arrive_expect_tx(&full[stage], bytes);
                }
                __syncwarp();
                if constexpr (!FP8) {
                    if (lane < npages) {
                        // one box: the slice's K rows, then its V rows (page pb, head c.kvh, rows off..)
                        const int lp = first_page + lane;
                        const int off = max(ts, lp * bs) - lp * bs;
                        const int br = bs < L::kTile ? bs : L::kTile;
                        tc::tma_load_5d_hint(st + (size_t)lane * 2 * br * D * L::kKB, &tm_kv, 0, off, c.kvh, 0, pb,
                                             &full[stage], pol);
                    }
                } else if (lane < npages) {
                    const int lp = first_page + lane;
                    const int tok_lo = max(ts, lp * bs);
                    const int tok_hi = min(ts + n, (lp + 1) * bs);
                    const int off = tok_lo - lp * bs;
                    const uint32_t bytes = (uint32_t)(tok_hi - tok_lo) * D * L::kKB;
                    const size_t kbase = (((size_t)pb * 2) * hkv + c.kvh) * head_bytes + (size_t)off * D * L::kKB;
                    const size_t vbase = kbase + (size_t)hkv * head_bytes;
                    uint8_t *dk = st + (size_t)(tok_lo - ts) * D * L::kKB;
                    bulk_g2s(dk, cache + kbase, bytes, &full[stage], pol);
                    bulk_g2s(dk + L::kKBytes, cache + vbase, bytes, &full[stage], pol);
                    {
                        // off and tok_lo - ts are multiples of 4 rows, and a page holds a multiple
                        // of 4 rows, so the rounded-up copy stays inside the page's scale row
                        const float *ksrc = a.cache.scales + (((size_t)pb * 2) * hkv + c.kvh) * bs + off;
                        const uint32_t sbytes = (uint32_t)((tok_hi - tok_lo + 3) & ~3) * 4u;
                        uint8_t *ds = st + L::kSOffset + (size_t)(tok_lo - ts) * 4;
                        bulk_g2s(ds, ksrc, sbytes, &full[stage], pol);
                        bulk_g2s(ds + L::kTile * 4, ksrc + (size_t)hkv * bs, sbytes, &full[stage], pol);
                    }
                }
                if (first_tile && lane == 0) {
                    const uint16_t *qsrc = qg + ((size_t)ut.qrow[c.b] * a.num_q_heads + (size_t)c.kvh * G) * D;
                    bulk_g2s(st + 2 * L::kKBytes, qsrc, (uint32_t)L::kQBytes, &full[stage], pol);
                }
                issued_mask |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == L::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            c = cn;
            win = wn;
        }
        // end marker: one more stage carrying unit id -1
        if (mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.err) && lane == 0) {
            stage_unit[stage] = -1;
            mbar_arrive(&full[stage]);
        }
        return;
    }

    if (warp == kMergeWarp) {
        // ================================= merge warp =================================
        merge_warp_loop<D, G, kConsumerWarps>(a, ut, merge, L::kMergeFloats, mfull, mempty, merge_unit, abort_flag,
                                              lane);
        pdl_launch_dependents();
        return;
    }

    // ================================ consumer warps ================================
    const int br = bs < L::kTile ? bs : L::kTile;  // rows per page slice (native cache)
    const int slot = lane / L::kLanesPerTok;   // token slot within a step
    const int chk = lane % L::kLanesPerTok;    // this lane's 8-element chunk of D
    const float qscale = a.scale * kLog2e;     // scores in log2 units
    float2 qf[G][4];                           // q chunk, scaled, as fp32 pairs
    // grouped heads: after the reduce-scatter, lane (within its token group) owns value k_own =
    // step * G + head; `shift` drops the low lane bits that only replicate it
    constexpr int kLog2N = L::kGqaN >= 16 ? 4 : L::kGqaN >= 8 ? 3 : L::kGqaN >= 4 ? 2 : L::kGqaN >= 2 ? 1 : 0;
    constexpr int kLog2R = L::kLanesPerTok == 16 ? 4 : 3;
    constexpr int shift = kLog2R - kLog2N;
    const int group_base = lane & ~(L::kLanesPerTok - 1);
    const int k_own = (lane & (L::kLanesPerTok - 1)) >> shift;
    const int g_own = k_own % G;
    float *pbuf = reinterpret_cast<float *>(smem + L::kPOffset) + ((size_t)warp * L::kTokPerStep + slot) * L::kGqaN;
    (void)group_base; (void)g_own; (void)pbuf;
    int stage = 0;
    uint32_t phase = 0;
    int mbuf = 0;           // merge buffer of the next unit
    uint32_t mphase = 0;
    for (;;) {
        // the unit of the next stage (or the end marker) is known once that stage is full
        if (!mbar_wait(&full[stage], phase, abort_flag, a.err)) return;
        const int u = stage_unit[stage];
        if (u < 0) break;
        const UnitCursor c = unit_of(u, ut, a.s_max, hkv, chunk);
        float l_own = 0.f;                     // grouped heads: this lane's share of its head's sum
        (void)l_own;
        float m[G], l[G];
        float2 acc[G][4];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            m[g] = -INFINITY;
            l[g] = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[g][j] = make_float2(0.f, 0.f);
        }
        for (int ts = c.t0; ts < c.t1; ts += L::kTile) {
            const int n = min(L::kTile, c.t1 - ts);
            if (ts != c.t0 && !mbar_wait(&full[stage], phase, abort_flag, a.err)) return;
            const uint8_t *st = smem + (size_t)stage * L::kStageBytes;
            if (ts == c.t0) {
                const float2 qs2 = make_float2(qscale, qscale);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const uint4 raw = *reinterpret_cast<const uint4 *>(st + 2 * L::kKBytes + ((size_t)g * D + chk * 8) * 2);
                    unpack8x2(raw, qf[g], Tag());
#pragma unroll
                    for (int j = 0; j < 4; ++j) qf[g][j] = fmul2(qf[g][j], qs2);
                }
            }
            if constexpr (G == 1) {
            const float *ksc = reinterpret_cast<const float *>(st + L::kSOffset);  // FP8 row scales
            const float *vsc = ksc + L::kTile;
            (void)ksc; (void)vsc;
#pragma unroll
            for (int b0 = 0; b0 < L::kSteps; b0 += L::kStepsPerBatch) {
                float s[L::kStepsPerBatch][G];
                bool valid[L::kStepsPerBatch];
#pragma unroll
                for (int i = 0; i < L::kStepsPerBatch; ++i) {
                    const int t = warp * L::kTokPerWarp + (b0 + i) * L::kTokPerStep + slot;
                    valid[i] = t < n;
                    float2 kf[4];
                    load_row8<Tag, D, FP8>(st, k_row<FP8>(t, br), chk, kf);
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        float2 pp = fmul2(qf[g][0], kf[0]);
#pragma unroll
                        for (int j = 1; j < 4; ++j) pp = ffma2(qf[g][j], kf[j], pp);
                        float part = pp.x + pp.y;
#pragma unroll
                        for (int o = L::kLanesPerTok / 2; o > 0; o >>= 1)
                            part += __shfl_xor_sync(0xffffffffu, part, o);
                        s[i][g] = valid[i] ? part * row_scale<FP8>(ksc, t) : -INFINITY;
                    }
                }
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float mt = s[0][g];
#pragma unroll
                    for (int i = 1; i < L::kStepsPerBatch; ++i) mt = fmaxf(mt, s[i][g]);
                    // Lazy rescale: the running max moves only when a score exceeds it by more
                    // than 2^8; until then exp2(s - m) <= 256 and the final acc / l is unchanged.
                    if (mt > m[g] + kRescaleLog2) {
                        const float alpha = ex2_approx(m[g] - mt);  // 0 when m[g] = -inf
                        l[g] *= alpha;
                        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                        for (int j = 0; j < 4; ++j) acc[g][j] = fmul2(acc[g][j], a2);
                        m[g] = mt;
                    }
#pragma unroll
                    for (int i = 0; i < L::kStepsPerBatch; ++i) {
                        s[i][g] = valid[i] ? ex2_approx(s[i][g] - m[g]) : 0.f;
                        l[g] += s[i][g];
                    }
                }
#pragma unroll
                for (int i = 0; i < L::kStepsPerBatch; ++i) {
                    if (!valid[i]) continue;
                    const int t = warp * L::kTokPerWarp + (b0 + i) * L::kTokPerStep + slot;
                    float2 vf[4];
                    load_row8<Tag, D, FP8>(st, v_row<FP8>(t, br, L::kTile), chk, vf);
                    const float vs = row_scale<FP8>(vsc, t);
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float pv = s[i][g] * vs;
                        const float2 p2 = make_float2(pv, pv);
#pragma unroll
                        for (int j = 0; j < 4; ++j) acc[g][j] = ffma2(p2, vf[j], acc[g][j]);
                    }
                }
            }
            } else {
            const float *ksc = reinterpret_cast<const float *>(st + L::kSOffset);  // FP8 row scales
            const float *vsc = ksc + L::kTile;
            (void)ksc; (void)vsc;
#pragma unroll
            for (int b0 = 0; b0 < L::kSteps; b0 += L::kGqaSteps) {
                constexpr int S = L::kGqaSteps, N = L::kGqaN, R = L::kLanesPerTok;
                // q.k partial sums for S tokens x G heads, value k = i * G + g
                float v[N];
#pragma unroll
                for (int i = 0; i < S; ++i) {
                    const int t = warp * L::kTokPerWarp + (b0 + i) * L::kTokPerStep + slot;
                    float2 kf[4];
                    load_row8<Tag, D, FP8>(st, k_row<FP8>(t, br), chk, kf);
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        float2 pp = fmul2(qf[g][0], kf[0]);
#pragma unroll
                        for (int j = 1; j < 4; ++j) pp = ffma2(qf[g][j], kf[j], pp);
                        v[i * G + g] = pp.x + pp.y;
                    }
                }
                // reduce-scatter over the R lanes of the token group: each level halves the values a
                // lane keeps (upper or lower half by its lane bit) and adds the partner's other half;
                // once one value is left the remaining levels all-reduce it
#pragma unroll
                for (int lev = 0; (R >> (lev + 1)) >= 1; ++lev) {
                    const int o = R >> (lev + 1);
                    const int cnt = N >> lev;
                    if (cnt > 1) {
                        const int half = cnt >> 1;
                        const bool hi = (lane & o) != 0;
#pragma unroll
                        for (int q = 0; q < half; ++q) {
                            const float send = hi ? v[q] : v[q + half];
                            const float keep = hi ? v[q + half] : v[q];
                            v[q] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                        }
                    } else {
                        v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
                    }
                }
                const int tok_own = warp * L::kTokPerWarp + (b0 + k_own / G) * L::kTokPerStep + slot;
                const float s_own = (tok_own < n) ? v[0] * row_scale<FP8>(ksc, tok_own) : -INFINITY;
                // batch max of this lane's head over the S steps (the first log2(S) lane bits)
                float mb = s_own;
#pragma unroll
                for (int o = R >> 1; o > (R >> 1) / S; o >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
                float m_own = m[0];
#pragma unroll
                for (int g = 1; g < G; ++g) m_own = (g_own == g) ? m[g] : m_own;
                if (__any_sync(0xffffffffu, mb > m_own + kRescaleLog2)) {
                    // lazy rescale: every lane learns each head's batch max from a lane that owns it
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float Mg = __shfl_sync(0xffffffffu, mb, group_base | (g << shift));
                        if (Mg > m[g] + kRescaleLog2) {
                            const float alpha = ex2_approx(m[g] - Mg);  // 0 when m[g] = -inf
                            const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                            for (int j = 0; j < 4; ++j) acc[g][j] = fmul2(acc[g][j], a2);
                            if (g == g_own) l_own *= alpha;
                            m[g] = Mg;
                        }
                    }
#pragma unroll
                    for (int g = 0; g < G; ++g) m_own = (g_own == g) ? m[g] : m_own;
                }
                const float p_own = (s_own == -INFINITY) ? 0.f : ex2_approx(s_own - m_own);
                l_own += p_own;
                // broadcast the N probabilities of this token group through shared memory
                pbuf[k_own] = p_own;
                __syncwarp();
#pragma unroll
                for (int i = 0; i < S; ++i) {
                    const int t = warp * L::kTokPerWarp + (b0 + i) * L::kTokPerStep + slot;
                    if (t >= n) continue;
                    float2 vf[4];
                    load_row8<Tag, D, FP8>(st, v_row<FP8>(t, br, L::kTile), chk, vf);
                    const float vs = row_scale<FP8>(vsc, t);
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float pg = pbuf[i * G + g] * vs;
                        const float2 p2 = make_float2(pg, pg);
#pragma unroll
                        for (int j = 0; j < 4; ++j) acc[g][j] = ffma2(p2, vf[j], acc[g][j]);
                    }
                }
                __syncwarp();
            }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == L::kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if constexpr (G > 1) {
            // l[g] = sum of l_own over the lanes owning head g (all bits but the head bits),
            // divided by the replication of each value, then handed to every lane
            constexpr int R = L::kLanesPerTok, S = L::kGqaSteps;
            float lt = l_own;
#pragma unroll
            for (int o = R >> 1; o >= 1; o >>= 1) {
                const bool head_bit = (o <= (R >> 1) / S) && (o > ((R >> 1) / S) / G);
                if (!head_bit) lt += __shfl_xor_sync(0xffffffffu, lt, o);
            }
            lt *= 1.f / (float)(1 << shift);
#pragma unroll
            for (int g = 0; g < G; ++g) l[g] = __shfl_sync(0xffffffffu, lt, group_base | (g << shift));
        }
        // ---- merge the token slots of this warp (lanes with the same chunk) ----
#pragma unroll
        for (int o = L::kLanesPerTok; o < 32; o <<= 1) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float mo = __shfl_xor_sync(0xffffffffu, m[g], o);
                const float lo = __shfl_xor_sync(0xffffffffu, l[g], o);
                const float mn = fmaxf(m[g], mo);
                const float wa = (m[g] == -INFINITY) ? 0.f : exp2f(m[g] - mn);
                const float wb = (mo == -INFINITY) ? 0.f : exp2f(mo - mn);
                l[g] = l[g] * wa + lo * wb;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float ax = __shfl_xor_sync(0xffffffffu, acc[g][j].x, o);
                    const float ay = __shfl_xor_sync(0xffffffffu, acc[g][j].y, o);
                    acc[g][j].x = acc[g][j].x * wa + ax * wb;
                    acc[g][j].y = acc[g][j].y * wa + ay * wb;
                }
                m[g] = mn;
            }
        }
        // ---- hand this warp's rows to the merge warp ----
        if (!mbar_wait(&mempty[mbuf], mphase ^ 1u, abort_flag, a.err)) return;
        float *rows = merge + (size_t)mbuf * L::kMergeFloats;
        if (slot == 0) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float *row = rows + ((size_t)warp * G + g) * kMergeRow<D>;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    row[chk * 8 + 2 * j] = acc[g][j].x;
                    row[chk * 8 + 2 * j + 1] = acc[g][j].y;
                }
                if (chk == 0) {
                    row[D] = m[g];
                    row[D + 1] = l[g];
                }
            }
        }
        if (warp == 0 && lane == 0) merge_unit[mbuf] = u;
        __syncwarp();
        if (lane == 0) mbar_arrive(&mfull[mbuf]);
        if (++mbuf == 2) {
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

// V (2, 4 or 8) consecutive floats from a 16-byte (V = 2: 8-byte) aligned address, as vector loads.
template <int V>
__device__ __forceinline__ void load_vec(const float *src, float (&x)[V]) {
    if constexpr (V == 8) {
        const float4 v = *reinterpret_cast<const float4 *>(src), w = *reinterpret_cast<const float4 *>(src + 4);
        x[0] = v.x;
        x[1] = v.y;
        x[2] = v.z;
        x[3] = v.w;
        x[4] = w.x;
        x[5] = w.y;
        x[6] = w.z;
        x[7] = w.w;
    } else if constexpr (V == 4) {
        const float4 v = *reinterpret_cast<const float4 *>(src);
        x[0] = v.x;
        x[1] = v.y;
        x[2] = v.z;
        x[3] = v.w;
    } else {
        const float2 v = *reinterpret_cast<const float2 *>(src);
        x[0] = v.x;
        x[1] = v.y;
    }
}

// ---- split merge: one warp per output row --------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) combine_kernel(CombineArgs a) {
    constexpr int kPer = D / 32;  // elements per lane
    // Launched as a programmatic dependent of the split kernel: everything above the wait may
    // run while the split kernel drains; the wait returns once its writes are visible.
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    int S = a.num_splits;
    bool done_by_split = false;
    size_t out_row = (size_t)row;
    int len = 0;
    if (row < a.n_rows && a.context_lens) {
        const int b = row / a.rows_per_seq;
        len = __ldg(a.context_lens + b);
        len = len < 0 ? 0 : len;
        if (a.cu_q_lens) {  // mixed batch: rows of prefill chunks are not this kernel's
            const int q0 = __ldg(a.cu_q_lens + b);
            if (__ldg(a.cu_q_lens + b + 1) - q0 != 1) done_by_split = true;
            out_row = (size_t)q0 * a.rows_per_seq + (row - b * a.rows_per_seq);
        }
        if (!a.chunk_dev) {
            S = len > 0 ? (len - 1) / a.chunk + 1 : 0;
            if (S > a.num_splits) S = a.num_splits;
            done_by_split = done_by_split || (S == 1);  // (or finished by the split kernel)
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (row >= a.n_rows || done_by_split) return;
    if (a.chunk_dev && a.context_lens) {
        // the split size the split kernel chose (written by it; visible after the wait)
        const int chunk = *a.chunk_dev;
        S = len > 0 ? (len - 1) / chunk + 1 : 0;
        if (S > a.num_splits) S = a.num_splits;
        if (S == 1) return;  // finished by the split kernel
    }
    const float *pl = a.part_lse + (size_t)row * a.num_splits;
    const float *po = a.part_o + (size_t)row * a.num_splits * D + kPer * lane;
    float M = -INFINITY;
    for (int s = lane; s < S; s += 32) M = fmaxf(M, pl[s]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float o_acc[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) o_acc[j] = 0.f;
    float wsum = 0.f;
    if (M != -INFINITY) {
        // 32 splits at a time: lane s holds split s's weight; each lane reads its kPer consecutive
        // dims of a partial row as one vector, eight splits' loads in flight before their sums
        for (int s0 = 0; s0 < S; s0 += 32) {
            const int s_l = s0 + lane;
            const float ls = s_l < S ? pl[s_l] : -INFINITY;
            const float w_l = ls == -INFINITY ? 0.f : exp2f((ls - M) * kLog2e);
            wsum += w_l;
            const int n = min(32, S - s0);
            int k = 0;
            for (; k + 8 <= n; k += 8) {
                float x[8][kPer];
#pragma unroll
                for (int i = 0; i < 8; ++i) load_vec<kPer>(po + (size_t)(s0 + k + i) * D, x[i]);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float w = __shfl_sync(0xffffffffu, w_l, k + i);
#pragma unroll
                    for (int j = 0; j < kPer; ++j) o_acc[j] = fmaf(w, x[i][j], o_acc[j]);
                }
            }
            for (; k < n; ++k) {
                float x[kPer];
                load_vec<kPer>(po + (size_t)(s0 + k) * D, x);
                const float w = __shfl_sync(0xffffffffu, w_l, k);
#pragma unroll
                for (int j = 0; j < kPer; ++j) o_acc[j] = fmaf(w, x[j], o_acc[j]);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
    for (int j = 0; j < kPer; ++j) o_acc[j] *= inv;
    store_out_vec<kPer>(a.out, out_row * D + lane * kPer, o_acc, a.out_dtype);
    if (lane == 0 && a.lse) a.lse[out_row] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
}

template <typename Tag, int D, int G, bool FP8>
cudaError_t launch_decode_t(const DecodeArgs &a, int grid, cudaStream_t s) {
    const size_t smem = DecodeLayout<D, G, FP8>::smem_bytes(a.batch, a.s_max);
    auto kern = decode_split_kernel<Tag, D, G, FP8>;
    // opt in to the largest size this kernel can ask for, once per device
    static DeviceFlags configured;
    const int dev = device_info().device;
    if (dev < 64 && !configured.test(dev)) {
        const int max_smem = (int)DecodeLayout<D, G, FP8>::smem_bytes(kMaxBatch, kDecodeMaxSplits);
        cudaError_t e = set_smem_attributes(kern, max_smem);
        if (e != cudaSuccess) return e;
        configured.set(dev);
    } else if (dev >= 64) {
        cudaError_t e = set_smem_attributes(kern, (int)smem);
        if (e != cudaSuccess) return e;
    }
    CUtensorMap tm = {};  // native cache: K and V rows of a page slice per box; FP8: unused
    if constexpr (!FP8) {
        const int br = a.cache.block_size < kDecodeTile ? a.cache.block_size : kDecodeTile;
        const cudaError_t e = encode_kv5_rows_map(a.cache, br, &tm);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(kern, dim3(grid * DecodeLayout<D, G, FP8>::kCtasPerSm), dim3(kDecodeThreads), smem, s, tm, a);
}

template <typename Tag, int D>
cudaError_t dispatch_group(const DecodeArgs &a, int grid, cudaStream_t s) {
    if (a.cache.fp8) {
        switch (a.num_q_heads / a.cache.num_kv_heads) {
            case 1: return launch_decode_t<Tag, D, 1, true>(a, grid, s);
            case 2: return launch_decode_t<Tag, D, 2, true>(a, grid, s);
            case 4: return launch_decode_t<Tag, D, 4, true>(a, grid, s);
            case 8: return launch_decode_t<Tag, D, 8, true>(a, grid, s);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (a.num_q_heads / a.cache.num_kv_heads) {
        case 1: return launch_decode_t<Tag, D, 1, false>(a, grid, s);
        case 2: return launch_decode_t<Tag, D, 2, false>(a, grid, s);
        default: return cudaErrorInvalidValue;  // four or more heads per KV head: decode_gqa.cu
    }
}

}  // namespace

int decode_max_batch() { return kMaxBatch; }

int decode_ctas_per_sm(int head_dim, int group, int dtype) {
    (void)head_dim; (void)group; (void)dtype;
    // the split-size rule counts one CTA per SM for every decode kernel; this kernel launches
    // DecodeLayout::kCtasPerSm CTAs per SM over the same units
    return 1;
}

cudaError_t launch_decode(const DecodeArgs &a, int grid, cudaStream_t s) {
    if (a.batch == 0) return cudaSuccess;
    if (a.cache.dtype == 1) {
        return a.cache.head_dim == 128 ? dispatch_group<BF16Tag, 128>(a, grid, s) : dispatch_group<BF16Tag, 64>(a, grid, s);
    }
    return a.cache.head_dim == 128 ? dispatch_group<F16Tag, 128>(a, grid, s) : dispatch_group<F16Tag, 64>(a, grid, s);
}

cudaError_t launch_combine(const CombineArgs &a, cudaStream_t s) {
    if (a.n_rows == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((a.n_rows + 7) / 8);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    // programmatic dependent launch: may start while the preceding kernel on `s` finishes
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (a.head_dim == 256) return cudaLaunchKernelEx(&cfg, combine_kernel<256>, a);
    if (a.head_dim == 128) return cudaLaunchKernelEx(&cfg, combine_kernel<128>, a);
    return cudaLaunchKernelEx(&cfg, combine_kernel<64>, a);
}

}  // namespace pkv
