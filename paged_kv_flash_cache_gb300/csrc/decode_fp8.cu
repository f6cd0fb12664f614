// decode_fp8.cu -- paged_attn_decode over an FP8 (E4M3) cache, head_dim 128, any head grouping
// up to 8 query heads per KV head, with both contractions on tensor cores.
//
// Same computation as decode.cu: for each sequence and query head, softmax(q.K^T * scale) V over
// the cached tokens read through the block table ("企业官网建设流程全解析", section 2.1; layout of
// "Flash Attention与Paged Attention如何共同优化大模型推理？", section 3), with the running max /
// running sum of that page's section 2, split over key/value blocks and merged by log-sum-exp.
// Cached element = decode(code) * row scale (the FP8 reading of the KV-cache compression that
// "为什么Attention是O(n²)" names).
//
// Why tensor cores even for one query head per KV head: a byte of FP8 cache is half a token-dim
// of a 16-bit one, so at the same HBM rate the kernel must get through twice the tokens, and the
// CUDA-core loop (about 36 warp instructions per token and KV head, plus the code conversions)
// cannot keep up. Here 16 tokens x 8 head slots x 16 dims are one mma.sync m16n8k16 in f16: E4M3
// codes convert exactly to f16 (cvt.rn.f16x2.e4m3x2), q is converted to f16 once per unit, the K
// row scales multiply the fp32 scores, and the V row scales enter the probabilities relative to
// the largest scale of each 16-token block, whose product is then added to O times that scale.
//
// Operand layouts. The tile rows are tokens of 128 one-byte codes (one 128-byte swizzle atom,
// written by TMA). ldmatrix (.b16) hands lane (gid, tig) the four codes of dims 4*tig .. 4*tig+3
// of a 16-dim chunk: the k slots of the A fragment are taken as the permutation
// {2tig, 2tig+1, 2tig+8, 2tig+9} -> {4tig, 4tig+1, 4tig+2, 4tig+3}, and q's B fragment is built
// with the same permutation, so the dot products are unchanged. For P.V, ldmatrix.trans hands a
// lane codes (token 2tig, dims 2gid and 2gid+1) and (token 2tig+1, same dims); one byte permute
// regroups them per dim, so M slot gid of a 16-dim chunk holds dim 2gid and slot gid+8 dim 2gid+1.
//
// Kernel structure (persistent, two CTAs per SM, 6 warps each): as decode_gqa.cu -- warp 4
// streams each unit's 64-token tiles into a ring of 4 stages (3 for groups of 4 or 8 heads),
// warps 0-3 take 16 tokens each, warp 5 merges the warps' rows and writes the output or the split
// partials. A tile arrives as page slices of
// br = min(block_size, 64) tokens; one TMA box per slice holds its K and V code rows (a 5-D view
// of the cache [NB][2][Hkv][bs][D]) and one its K and V row scales, so a page costs two copies.
// Two CTAs per SM give every scheduler two consumer warps from two independent pipelines: the
// consumers' dependent ldmatrix / cvt / mma chains are the bound, and one CTA with 8 consumer
// warps and 128-token tiles (129 registers a thread, too many for two such CTAs) left them exposed
// at every unit boundary and stage hand-off (0.151 ms against 0.122 ms for the 7B-like batch).
#include <cuda.h>

#include "decode_common.cuh"
#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "tcgen05.cuh"
#include "warp_mma.cuh"

namespace pkv {
namespace {

constexpr int kD = 128;
constexpr int kWarps = 4;  // consumer warps, 16 tokens each
constexpr int kProducerWarp = kWarps;
constexpr int kMergeWarp = kWarps + 1;
constexpr int kThreads = (kWarps + 2) * 32;
constexpr int kTile = 64;  // tokens per stage (16 KB of K and V codes)
constexpr int kCtasPerSm = 2;
constexpr int kMaxBatch8 = 2048;
constexpr float kRescale = 8.0f;  // lazy rescale threshold (log2 units)
constexpr int kChunks = kD / 16;  // 16-dim chunks: k-steps of q.K^T, m-tiles of O^T

template <int G>
struct Fp8Layout {
    static constexpr int kStages8 = G >= 4 ? 3 : 4;  // the merge buffers of 8 heads take a stage's room
    // codes: per page slice of br = min(bs, 64) tokens, br K rows then br V rows (128 bytes each);
    // scales: per slice br K scales then br V scales, at a pitch of max(128, 8 * br) bytes
    static constexpr uint32_t kCodeBytes = 2 * kTile * kD;
    static constexpr uint32_t kQBytes = G * kD * 2;
    static constexpr uint32_t kQOffset = kCodeBytes;
    static constexpr uint32_t kSOffset = kQOffset + kQBytes;
    static constexpr uint32_t kSBytes = 1024;  // 8 slices x 128 bytes (br = 8), or kTile x 8 bytes
    static constexpr uint32_t kStageBytes = (kSOffset + kSBytes + 1023) / 1024 * 1024;
    static constexpr uint32_t kBarOffset = kStages8 * kStageBytes;
    // barriers: full / empty per stage, merge full / empty per merge buffer; then the abort flag
    // (padded to 16 bytes), the unit of each stage and the unit of each merge buffer
    static constexpr uint32_t kMergeOffset = kBarOffset + (2 * kStages8 + 4) * 8 + 64;
    static constexpr uint32_t kMergeFloats = kWarps * G * kMergeRow<kD>;  // one of two merge buffers
    static constexpr uint32_t kIntsOffset = kMergeOffset + 2 * kMergeFloats * 4;
    static size_t smem_bytes(int batch, int s_max) {
        return kIntsOffset + unit_table_ints(batch, s_max) * 4 + 1024;  // + 1024-byte alignment slack
    }
};

// Two E4M3 codes (low byte first) to an f16x2 register, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((unsigned short)(two_codes & 0xffffu)));
    return r;
}

// Shared-memory address of row t, 16-byte chunk cc of a tile of 128-byte rows in the 128-byte
// swizzled layout TMA writes (chunk position cc ^ (t & 7)).
__device__ __forceinline__ uint32_t swz(uint32_t tile, int t, int cc) {
    return tile + (uint32_t)t * 128u + ((uint32_t)(cc ^ (t & 7)) << 4);
}

// Four 16-bit q values (q_dtype) to two f16x2 registers.
template <bool BF16>
__device__ __forceinline__ void q4_to_f16(uint2 raw, uint32_t &lo, uint32_t &hi) {
    if (BF16) {
        const float f0 = __uint_as_float(raw.x << 16), f1 = __uint_as_float(raw.x & 0xffff0000u);
        const float f2 = __uint_as_float(raw.y << 16), f3 = __uint_as_float(raw.y & 0xffff0000u);
        lo = pack_pair<false>(f0, f1);
        hi = pack_pair<false>(f2, f3);
    } else {
        lo = raw.x;
        hi = raw.y;
    }
}

template <int G, bool BF16>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    decode_fp8_kernel(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_scales,
                      DecodeArgs a) {
    using L = Fp8Layout<G>;
    constexpr int kStages8 = L::kStages8;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kBarOffset);
    uint64_t *empty = full + kStages8;
    uint64_t *mfull = empty + kStages8;  // [2] the consumer warps' rows of a unit are in buffer i
    uint64_t *mempty = mfull + 2;        // [2] the merge warp has read buffer i
    volatile int *abort_flag = reinterpret_cast<volatile int *>(mempty + 2);
    int *stage_unit = reinterpret_cast<int *>(mempty + 2) + 4;
    int *merge_unit = stage_unit + kStages8;  // [2] unit of each merge buffer, -1: end
    float *merge = reinterpret_cast<float *>(smem + L::kMergeOffset);  // [2][kWarps][G][kMergeRow<kD>]
    const UnitTable ut = unit_table(reinterpret_cast<int *>(smem + L::kIntsOffset), a.batch, a.s_max);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hkv = a.cache.num_kv_heads, bs = a.cache.block_size;
    const int hu = hkv * a.head_groups;  // unit heads (KV heads, or groups of 8 query heads)
    // a tile is copied in slices of br = min(bs, 64) rows: tiles start at multiples of 64 tokens,
    // so every slice lies inside one page whatever the page size
    const int br = bs < 64 ? bs : 64;
    const int spitch = br * 8 > 128 ? br * 8 : 128;  // bytes per slice in the scale region

    if (tid == 0) {
        for (int i = 0; i < kStages8; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&mfull[i], kWarps);
            mbar_init(&mempty[i], 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    pdl_wait();  // lengths, tables, q and the cache may come from the previous kernel
    const int num_units = decode_scan_units<kThreads>(a, ut);
    const int chunk = ut.misc[0];  // the launch's split size

    if (warp == kProducerWarp) {
        // ===================================== producer warp =====================================
        const uint64_t pol = l2_policy_evict_first();
        const uint16_t *qg = static_cast<const uint16_t *>(a.q);
        if (lane == 0) {
            tc::prefetch_tensormap(&tm_codes);
            tc::prefetch_tensormap(&tm_scales);
        }
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_mask = 0, issued_parity = 0;
        UnitCursor c = {};
        PageWindow win = {};
        if ((int)blockIdx.x < num_units) {
            c = unit_of(blockIdx.x, ut, a.s_max, hu, chunk);
            win = unit_pages(a, c, lane);
        }
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
                    for (int i = 0; i < kStages8; ++i)
                        if (issued_mask & (1u << i)) {
                            volatile int no_abort = 0;
                            mbar_wait(&full[i], (issued_parity >> i) & 1u, &no_abort, nullptr);
                        }
                    return;
                }
                uint8_t *st = smem + (size_t)stage * L::kStageBytes;
                const bool first_tile = (ts == c.t0);
                if (lane == 0) {
                    stage_unit[stage] = u;
                    // codes of K and V (whole slices) and their row scales (same rows)
                    const uint32_t bytes = (uint32_t)nslices * br * (2u * kD + 8u) + (first_tile ? L::kQBytes : 0u);
                    mbar_arrive_expect_tx(&full[stage], bytes);
                }
                __syncwarp();
                if (lane < nslices) {
                    // one box: the slice's K rows then its V rows (page pb, head c.kvh, rows off..)
                    const int kvr = c.kvh / a.head_groups;  // the KV head of this unit
                    tc::tma_load_5d_hint(st + (size_t)lane * 2 * br * kD, &tm_codes, 0, off, kvr, 0, pb, &full[stage],
                                         pol);
                    tc::tma_load_4d_hint(st + L::kSOffset + (size_t)lane * spitch, &tm_scales, off, kvr, 0, pb,
                                         &full[stage], pol);
                }
                if (first_tile && lane == 0) {
                    const uint16_t *qsrc = qg + ((size_t)ut.qrow[c.b] * a.num_q_heads + (size_t)c.kvh * G) * kD;
                    bulk_g2s(st + L::kQOffset, qsrc, L::kQBytes, &full[stage], pol);
                }
                issued_mask |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == kStages8) {
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

    if (warp == kMergeWarp) {
        // ====================================== merge warp ======================================
        merge_warp_loop<kD, G, kWarps>(a, ut, merge, L::kMergeFloats, mfull, mempty, merge_unit, abort_flag, lane);
        pdl_launch_dependents();
        return;
    }

    // ===================================== consumer warps =====================================
    const int gid = lane >> 2, tig = lane & 3;
    const int g_lo = 2 * tig;  // this lane's two head slots (columns of S^T / O^T)
    const float sl = a.scale * kLog2e;
    uint32_t bq[kChunks][2];   // q as f16 B fragments, k slots permuted as the K codes
    int stage = 0;
    uint32_t phase = 0;
    int mbuf = 0;  // merge buffer of the next unit
    uint32_t mphase = 0;
    for (;;) {
        if (!mbar_wait(&full[stage], phase, abort_flag, a.err)) return;
        const int u = stage_unit[stage];
        if (u < 0) break;
        const UnitCursor c = unit_of(u, ut, a.s_max, hu, chunk);
        float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
        float o[kChunks][4];
#pragma unroll
        for (int mt = 0; mt < kChunks; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        for (int ts = c.t0; ts < c.t1; ts += kTile) {
            const int n = min(kTile, c.t1 - ts);
            if (ts != c.t0 && !mbar_wait(&full[stage], phase, abort_flag, a.err)) return;
            uint8_t *st = smem + (size_t)stage * L::kStageBytes;
            const uint32_t aK = smem_addr(st), aV = aK + br * 128u;  // row tp of K; row tp of V
            const uint8_t *sc = st + L::kSOffset;
            if (ts == c.t0) {
                const uint16_t *sq = reinterpret_cast<const uint16_t *>(st + L::kQOffset);
#pragma unroll
                for (int kk = 0; kk < kChunks; ++kk) {
                    if (gid < G) {
                        const uint2 raw = *reinterpret_cast<const uint2 *>(sq + gid * kD + kk * 16 + 4 * tig);
                        q4_to_f16<BF16>(raw, bq[kk][0], bq[kk][1]);
                    } else {
                        bq[kk][0] = bq[kk][1] = 0u;
                    }
                }
            }
            const int t0w = warp * 16;  // this warp's tokens in the tile
            if (t0w + 16 > n) {
                // rows at or beyond the context end may hold unwritten bytes (NaN codes among
                // them): zero this warp's V code rows there so that 0 * NaN cannot reach O
                for (int t = t0w + (lane >> 3); t < t0w + 16; t += 4) {
                    if (t < n) continue;
                    const int tp = t + (t & -br);  // tile row t in the slice layout
                    *reinterpret_cast<uint4 *>(st + (tp + br) * 128 + (lane & 7) * 16) = make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }
            // ---- S^T = K_w q^T: 16 tokens x 8 head slots, two 16-dim chunks per ldmatrix ----
            float s[4] = {0.f, 0.f, 0.f, 0.f};
            {
                const int mi = lane >> 3;
                const int t = t0w + (lane & 7) + 8 * (mi & 1);
                const int tp = t + (t & -br);  // row of tile token t: slice j starts at row 2 * j * br
#pragma unroll
                for (int cp = 0; cp < kChunks; cp += 2) {
                    uint32_t r[4];
                    ldsm_x4(swz(aK, tp, cp + (mi >> 1)), r);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t af[4] = {e4m3x2_to_f16x2(r[2 * h]), e4m3x2_to_f16x2(r[2 * h + 1]),
                                                e4m3x2_to_f16x2(r[2 * h] >> 16), e4m3x2_to_f16x2(r[2 * h + 1] >> 16)};
                        mma16816<false>(s, af, bq[cp + h][0], bq[cp + h][1]);
                    }
                }
            }
            const bool v0 = t0w + gid < n, v1 = t0w + gid + 8 < n;
            // scales of tokens ta = t0w + gid and tb = ta + 8: slice j at j * spitch, K then V
            const int ta = t0w + gid, tb = ta + 8;
            const float *sa = reinterpret_cast<const float *>(sc + (ta / br) * spitch) + (ta & (br - 1));
            const float *sb = reinterpret_cast<const float *>(sc + (tb / br) * spitch) + (tb & (br - 1));
            const float k0 = sa[0], k1 = sb[0];
            s[0] = v0 ? s[0] * k0 : -INFINITY;
            s[1] = v0 ? s[1] * k0 : -INFINITY;
            s[2] = v1 ? s[2] * k1 : -INFINITY;
            s[3] = v1 ? s[3] * k1 : -INFINITY;
            // column max over the 16 tokens (lanes with the same tig)
            float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
            for (int ofs = 4; ofs < 32; ofs <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, ofs));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, ofs));
            }
            mx0 *= sl;
            mx1 *= sl;
            // lazy rescale: the running max of a head moves only when a score exceeds it by > 2^8
            if (mx0 > m[0] + kRescale) {
                const float al = ex2f(m[0] - mx0);  // 0 when m = -inf
                l[0] *= al;
#pragma unroll
                for (int mt = 0; mt < kChunks; ++mt) {
                    o[mt][0] *= al;
                    o[mt][2] *= al;
                }
                m[0] = mx0;
            }
            if (mx1 > m[1] + kRescale) {
                const float al = ex2f(m[1] - mx1);
                l[1] *= al;
#pragma unroll
                for (int mt = 0; mt < kChunks; ++mt) {
                    o[mt][1] *= al;
                    o[mt][3] *= al;
                }
                m[1] = mx1;
            }
            const float p0 = v0 ? ex2f(fmaf(s[0], sl, -m[0])) : 0.f;
            const float p1 = v0 ? ex2f(fmaf(s[1], sl, -m[1])) : 0.f;
            const float p2 = v1 ? ex2f(fmaf(s[2], sl, -m[0])) : 0.f;
            const float p3 = v1 ? ex2f(fmaf(s[3], sl, -m[1])) : 0.f;
            l[0] += p0 + p2;
            l[1] += p1 + p3;
            // V row scales: P carries w_t / w_max of this warp's 16 tokens (at most 1, so P keeps
            // f16 precision however small the scales are) and the block's product is added to O
            // times w_max; rows beyond the context have p = 0 and take no part in w_max
            const float w0 = v0 ? sa[br] : 0.f, w1 = v1 ? sb[br] : 0.f;
            float wmax = fmaxf(w0, w1);
#pragma unroll
            for (int ofs = 4; ofs < 32; ofs <<= 1) wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, ofs));
            const float rw = wmax > 0.f ? 1.f / wmax : 0.f;
            const float r0 = w0 * rw, r1 = w1 * rw;
            // P^T (tokens x head slots) in accumulator layout -> P as B fragments (k = tokens), as
            // an f16 part and its f16 remainder, each its own MMA into the same FP32 accumulator:
            // P.V sees P almost unrounded, so the output's is the only 16-bit rounding on the path
            uint32_t h01, e01, h23, e23;
            split_pair<false>(p0 * r0, p1 * r0, h01, e01);
            split_pair<false>(p2 * r1, p3 * r1, h23, e23);
            const uint32_t pb0 = movmatrix_t(h01), pb1 = movmatrix_t(h23);
            const uint32_t pe0 = movmatrix_t(e01), pe1 = movmatrix_t(e23);
            // ---- O^T += w_max V_w^T P^T: 128 dims (permuted within each 16-dim chunk) x 8 slots ----
            float ot[kChunks][4];
#pragma unroll
            for (int mt = 0; mt < kChunks; ++mt) ot[mt][0] = ot[mt][1] = ot[mt][2] = ot[mt][3] = 0.f;
            {
                const int mi = lane >> 3;
                const int t = t0w + (lane & 7) + 8 * (mi & 1);
                const int tp = t + (t & -br);
#pragma unroll
                for (int cp = 0; cp < kChunks; cp += 2) {
                    uint32_t r[4];
                    ldsm_x4_t(swz(aV, tp, cp + (mi >> 1)), r);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        // r[2h]: tokens 2tig, 2tig+1 (rows 0-7) of dims 2gid, 2gid+1; r[2h+1]: rows 8-15
                        const uint32_t lo = __byte_perm(r[2 * h], 0, 0x3120);      // [d0: t0, t1][d1: t0, t1]
                        const uint32_t hi = __byte_perm(r[2 * h + 1], 0, 0x3120);
                        const uint32_t af[4] = {e4m3x2_to_f16x2(lo), e4m3x2_to_f16x2(lo >> 16), e4m3x2_to_f16x2(hi),
                                                e4m3x2_to_f16x2(hi >> 16)};
                        mma16816<false>(ot[cp + h], af, pe0, pe1);
                        mma16816<false>(ot[cp + h], af, pb0, pb1);
                    }
                }
            }
#pragma unroll
            for (int mt = 0; mt < kChunks; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i) o[mt][i] = fmaf(ot[mt][i], wmax, o[mt][i]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == kStages8) {
                stage = 0;
                phase ^= 1u;
            }
        }
        // ---- l summed over the lanes of each head slot; rows to the merge warp ----
#pragma unroll
        for (int ofs = 4; ofs < 32; ofs <<= 1) {
            l[0] += __shfl_xor_sync(0xffffffffu, l[0], ofs);
            l[1] += __shfl_xor_sync(0xffffffffu, l[1], ofs);
        }
        if (!mbar_wait(&mempty[mbuf], mphase ^ 1u, abort_flag, a.err)) return;
        float *rows = merge + (size_t)mbuf * L::kMergeFloats;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int g = g_lo + j;
            if (g < G) {
                float *row = rows + ((size_t)warp * G + g) * kMergeRow<kD>;
#pragma unroll
                for (int mt = 0; mt < kChunks; ++mt) {
                    row[mt * 16 + 2 * gid] = o[mt][j];          // M slot gid: dim 2gid of the chunk
                    row[mt * 16 + 2 * gid + 1] = o[mt][j + 2];  // M slot gid + 8: dim 2gid + 1
                }
                if (gid == 0) {
                    row[kD] = m[j];
                    row[kD + 1] = l[j];
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

template <int G, bool BF16>
cudaError_t launch_fp8_t(const DecodeArgs &a, int grid, cudaStream_t s) {
    CUtensorMap tm, tm_s;
    const int box_rows = a.cache.block_size < 64 ? a.cache.block_size : 64;
    cudaError_t e = encode_fp8_maps(a.cache, box_rows, &tm, &tm_s);
    if (e != cudaSuccess) return e;
    auto kern = decode_fp8_kernel<G, BF16>;
    static DeviceFlags configured;
    const int dev = device_info().device;
    if (!configured.test(dev)) {
        e = set_smem_attributes(kern, (int)Fp8Layout<G>::smem_bytes(kMaxBatch8, kDecodeMaxSplits));
        if (e != cudaSuccess) return e;
        configured.set(dev);
    }
    // two CTAs an SM when both fit in its shared memory (one CTA's maximum plus its 1 KB reserve,
    // each less the reserve); a batch with large unit tables runs one
    const size_t smem = Fp8Layout<G>::smem_bytes(a.batch, a.s_max);
    const size_t cta_smem = ((size_t)device_info().max_smem + 1024) / kCtasPerSm - 1024;
    const int ctas = smem <= cta_smem ? kCtasPerSm : 1;
    return launch_pdl(kern, dim3(grid * ctas), dim3(kThreads), smem, s, tm, tm_s, a);
}

template <int G>
cudaError_t launch_fp8_g(const DecodeArgs &a, int grid, cudaStream_t s) {
    return a.cache.dtype == 1 ? launch_fp8_t<G, true>(a, grid, s) : launch_fp8_t<G, false>(a, grid, s);
}

}  // namespace

cudaError_t launch_decode_fp8(const DecodeArgs &a, int grid, cudaStream_t s) {
    if (a.batch == 0) return cudaSuccess;
    if (a.cache.head_dim != kD || a.batch > kMaxBatch8) return cudaErrorInvalidValue;
    switch (a.num_q_heads / (a.cache.num_kv_heads * a.head_groups)) {  // query heads per unit
        case 1: return launch_fp8_g<1>(a, grid, s);
        case 2: return launch_fp8_g<2>(a, grid, s);
        case 4: return launch_fp8_g<4>(a, grid, s);
        case 8: return launch_fp8_g<8>(a, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv
