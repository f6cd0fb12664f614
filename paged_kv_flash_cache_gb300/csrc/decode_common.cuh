// decode_common.cuh -- pieces shared by the split-KV decode kernels: the work-unit numbering
// built in each CTA's prologue from the context lengths, and the cursor it gives for a unit.
//
// A unit is (sequence, KV head, split of `chunk` tokens). Units are numbered split-major: every
// unit of split 0, then of split 1, ...; inside a split by sequence (in order of decreasing split
// count, so split s is held by the first n_s sequences of that order, ties by index), then by KV
// head. Units are dealt round-robin, so the CTAs running at one time read the same token range
// of a few sequences, all KV heads of each: the heads of one page are one contiguous run of
// memory, and where block tables share pages (requests that open with the same cached prompt)
// the sequences read each shared page within a few microseconds of each other, the later reads
// from L2. Every CTA builds the same numbering: no step of it depends on thread timing.
#pragma once

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

struct UnitCursor {
    int b, kvh, split, t0, t1;
};

// Shared-memory tables of the numbering (all int):
//   lens  [batch]      context lengths clamped to the table's capacity
//   ord   [batch]      sequences by decreasing split count, ties by index
//   first [s_max + 1]  first[s] = sum over sequences of min(splits, s); split s's units start at
//                      first[s] * hkv and number n_s * hkv, n_s = first[s + 1] - first[s]
//   hist  [s_max + 1]  prologue scratch: sequences per split count, then a fill count
//   qrow  [batch]      the sequence's query / output row (b, or cu_q_lens[b] in a mixed batch)
//   misc  [kUnitMisc]  misc[0] the split size of the launch (see decode_scan_units); misc[1..]
//                      prologue scratch (unit counts of the candidate split sizes)
struct UnitTable {
    int *lens, *ord, *first, *hist, *qrow, *misc;
};

__host__ __device__ constexpr size_t unit_table_ints(int batch, int s_max) {
    return 3 * (size_t)batch + 2 * ((size_t)s_max + 1) + kUnitMisc;
}

__device__ __forceinline__ UnitTable unit_table(int *ints, int batch, int s_max) {
    UnitTable t;
    t.lens = ints;
    t.ord = ints + batch;
    t.first = ints + 2 * batch;
    t.hist = t.first + s_max + 1;
    t.qrow = t.hist + s_max + 1;
    t.misc = t.qrow + batch;
    return t;
}

__device__ __forceinline__ UnitCursor unit_of(int u, const UnitTable &t, int s_max, int hkv, int chunk) {
    int lo = 0, hi = s_max;  // the split: last s with first[s] * hkv <= u
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (t.first[mid] * hkv <= u) lo = mid; else hi = mid;
    }
    const int r = u - t.first[lo] * hkv;  // < n_lo * hkv
    const int rank = r / hkv;
    UnitCursor c;
    c.split = lo;
    c.kvh = r - rank * hkv;
    c.b = t.ord[rank];
    c.t0 = lo * chunk;
    const int end = c.t0 + chunk;
    const int len = t.lens[c.b];
    c.t1 = end < len ? end : len;
    return c;
}

// Page ids of up to 64 consecutive logical pages of one block-table row, two per lane of the
// producer warp (lane j holds pages first + j and first + 32 + j). The producer loads a unit's
// window one unit ahead, so the table read's latency is not on the path that issues the unit's
// copies; units of more than 64 pages load further windows as they go.
struct PageWindow {
    int first, count, p0, p1;
};

__device__ __forceinline__ PageWindow load_pages(const int *bt_row, int first, int count, int lane) {
    PageWindow w;
    w.first = first;
    w.count = count < 64 ? count : 64;
    w.p0 = lane < w.count ? __ldg(bt_row + first + lane) : 0;
    w.p1 = lane + 32 < w.count ? __ldg(bt_row + first + 32 + lane) : 0;
    return w;
}

// The first window of unit c (its pages from c.t0's page on).
__device__ __forceinline__ PageWindow unit_pages(const DecodeArgs &a, const UnitCursor &c, int lane) {
    const int *bt_row = a.block_tables + (size_t)c.b * a.max_blocks_per_seq;
    const int f = c.t0 >> a.cache.log2_block_size;
    const int l = (c.t1 - 1) >> a.cache.log2_block_size;
    return load_pages(bt_row, f, l - f + 1, lane);
}

// Page id of logical page `page` (inside the window) for the calling lane; all 32 lanes call,
// lanes whose page lies outside the window get an unspecified id they must not use.
__device__ __forceinline__ int window_page(const PageWindow &w, int page) {
    int rel = page - w.first;
    rel = rel < 0 ? 0 : (rel > 63 ? 63 : rel);
    const int lo = __shfl_sync(0xffffffffu, w.p0, rel & 31);
    const int hi = __shfl_sync(0xffffffffu, w.p1, rel & 31);
    return rel < 32 ? lo : hi;
}

// Merge rows: a consumer warp's D partial sums of one query head, then its m and l, padded to
// a multiple of four floats so that every row starts on a 16-byte boundary (vector reads below)
// and the rows of neighbouring heads start in different banks.
template <int D>
constexpr int kMergeRow = D + 4;

// Sum of x[0..N) in the order of a butterfly reduction over N lanes (pairs i, i + N/2 first), so
// that a lane-parallel sum and a per-lane sum round alike.
template <int N>
__device__ __forceinline__ float tree_sum(const float (&x)[N]) {
    if constexpr (N == 1) {
        return x[0];
    } else {
        float y[N / 2];
#pragma unroll
        for (int i = 0; i < N / 2; ++i) y[i] = x[i] + x[i + N / 2];
        return tree_sum<N / 2>(y);
    }
}

// The decode step's append, by the merge warp of each CTA before its first unit (a native cache):
// row r of the batch's 2 * batch * Hkv new rows -- sequence r / (2 Hkv), head (r / 2) % Hkv, K
// (even r) or V (odd r) -- goes to position context_lens[b] of its sequence, page
// block_table[b][pos / block_size], offset pos % block_size, as D / 8 16-byte vectors, one per
// lane. The attention of the same call reads positions below context_lens[b] only, so the two
// touch different rows (a page slice that a copy brings in whole holds the new row as one of the
// rows past the context end, which every kernel masks). A position outside the table or a page
// outside the pool is flagged (kErrDeviceRange) and skipped, as the append kernel does.
template <int D>
__device__ __forceinline__ void append_step_rows(const DecodeArgs &a, int lane) {
    constexpr int kVec = D / 8;            // 16-byte vectors a row
    constexpr int kRowsPerPass = 32 / kVec;
    const int hkv = a.cache.num_kv_heads, bs = a.cache.block_size;
    const int nrows = 2 * a.batch * hkv;
    const int sub = lane / kVec, e = lane % kVec;
    const long long cap = (long long)a.max_blocks_per_seq * bs;
    uint4 *cache = static_cast<uint4 *>(const_cast<void *>(a.cache.ptr));
    for (int r0 = blockIdx.x * kRowsPerPass; r0 < nrows; r0 += gridDim.x * kRowsPerPass) {
        const int r = r0 + sub;
        if (r >= nrows) continue;
        const int kv = r & 1, bh = r >> 1;
        const int b = bh / hkv, h = bh - b * hkv;
        const uint4 v = __ldg(static_cast<const uint4 *>(kv ? a.v_new : a.k_new) + (size_t)bh * kVec + e);
        const int pos = __ldg(a.context_lens + b);
        if (pos < 0 || pos >= cap) {
            if (e == 0) set_error(a.err, kErrDeviceRange);
            continue;
        }
        const int pb = __ldg(a.block_tables + (size_t)b * a.max_blocks_per_seq + (pos >> a.cache.log2_block_size));
        if (pb < 0 || pb >= a.cache.num_blocks) {
            if (e == 0) set_error(a.err, kErrDeviceRange);
            continue;
        }
        const size_t row = (((size_t)pb * 2 + kv) * hkv + h) * bs + (pos & (bs - 1));
        cache[row * kVec + e] = v;
    }
}

// The merge warp of a decode CTA. At the end of a unit each of the W token slices leaves its
// (acc[D], m, l) row per query head of the unit in merge buffer i ([W][G][kMergeRow<D>] floats; m
// in log2 units, acc and l relative to 2^m), the unit id is written (warp 0) and mfull[i] completes;
// this loop combines the rows -- M = max m, weights 2^(m_w - M), out = sum w acc / sum w l, lse =
// (M + log2 sum w l) ln 2 -- writes the final output of a single-split context or the split's
// partial, and frees the buffer on mempty[i]. NB buffers (1 or 2) take turns; unit id -1 ends the loop. Lane g
// finds the weights of head g (all heads at once); then each head's output is D / 32 consecutive
// dims per lane, read and written as vectors. Returns false if a wait gave up (the error word is
// set).
template <int D, int G, int W, int NB = 2>
__device__ __forceinline__ bool merge_warp_loop(const DecodeArgs &a, const UnitTable &ut, const float *merge,
                                                size_t buf_floats, uint64_t *mfull, uint64_t *mempty,
                                                const int *merge_unit, volatile int *abort_flag, int lane) {
    static_assert(G <= 32, "one lane per query head of a unit");
    static_assert(W == 1 || W == 2 || W == 4 || W == 8 || W == 16 || W == 32, "token slices: a power of two");
    constexpr int RS = kMergeRow<D>;
    constexpr int V = D / 32;  // consecutive dims per lane
    static_assert(V == 2 || V == 4, "head_dim 64 or 128");
    const int hkv = a.cache.num_kv_heads * a.head_groups, chunk = ut.misc[0];  // unit heads; split size
    if (a.k_new && !a.cache.fp8) append_step_rows<D>(a, lane);
    int mbuf = 0;
    uint32_t mphase = 0;
    for (;;) {
        if (!mbar_wait(&mfull[mbuf], mphase, abort_flag, a.err)) return false;
        const int u = merge_unit[mbuf];
        if (u < 0) return true;
        const UnitCursor c = unit_of(u, ut, a.s_max, hkv, chunk);
        const float *rows = merge + (size_t)mbuf * buf_floats;
        const int splits = (ut.lens[c.b] + chunk - 1) / chunk;
        const size_t prow0 = (size_t)c.b * a.num_q_heads + (size_t)c.kvh * G;          // partial rows
        const size_t orow0 = (size_t)ut.qrow[c.b] * a.num_q_heads + (size_t)c.kvh * G;  // output rows
        float wl[W];
        float inv_l = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) wl[w] = 0.f;
        if (lane < G) {
            float mw[W], lw[W];
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < W; ++w) {
                const float *r = rows + ((size_t)w * G + lane) * RS;
                mw[w] = r[D];
                lw[w] = r[D + 1];
                M = fmaxf(M, mw[w]);
            }
            float lt[W];
#pragma unroll
            for (int w = 0; w < W; ++w) {
                wl[w] = (mw[w] == -INFINITY) ? 0.f : exp2f(mw[w] - M);
                lt[w] = lw[w] * wl[w];
            }
            const float lsum = tree_sum<W>(lt);
            inv_l = lsum > 0.f ? 1.f / lsum : 0.f;
            const float lse_v = lsum > 0.f ? (M + log2f(lsum)) * kLn2 : -INFINITY;
            if (splits == 1) {
                if (a.lse) a.lse[orow0 + lane] = lse_v;
            } else {
                a.part_lse[(prow0 + lane) * a.s_max + c.split] = lse_v;
            }
        }
#pragma unroll(G < 4 ? G : 4)
        for (int g = 0; g < G; ++g) {
            float wv[W];
#pragma unroll
            for (int w = 0; w < W; ++w) wv[w] = __shfl_sync(0xffffffffu, wl[w], g);
            const float inv = __shfl_sync(0xffffffffu, inv_l, g);
            float acc[V];
#pragma unroll
            for (int v = 0; v < V; ++v) acc[v] = 0.f;
#pragma unroll
            for (int w = 0; w < W; ++w) {
                const float *r = rows + ((size_t)w * G + g) * RS + V * lane;
                if constexpr (V == 4) {
                    const float4 x = *reinterpret_cast<const float4 *>(r);
                    acc[0] += x.x * wv[w];
                    acc[1] += x.y * wv[w];
                    acc[2] += x.z * wv[w];
                    acc[3] += x.w * wv[w];
                } else {
                    const float2 x = *reinterpret_cast<const float2 *>(r);
                    acc[0] += x.x * wv[w];
                    acc[1] += x.y * wv[w];
                }
            }
#pragma unroll
            for (int v = 0; v < V; ++v) acc[v] *= inv;
            if (splits == 1) store_out_vec<V>(a.out, (orow0 + g) * D + V * lane, acc, a.out_dtype);
            else store_out_vec<V>(a.part_o, ((prow0 + g) * a.s_max + c.split) * D + V * lane, acc, 2);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&mempty[mbuf]);
        if (++mbuf == NB) {
            mbuf = 0;
            mphase ^= 1u;
        }
    }
}

// Split size of an automatic split (DecodeArgs::auto_chunk): the host's chunk c0 (which sizes the
// workspace: s_max splits of c0 at full capacity) or 1.5, 2, 3 or 4 times it, rounded up to the
// 128-token split alignment, whichever minimises the modelled time of the launch: units are dealt
// round-robin to the grid's CTAs, so a CTA runs about ceil(U / grid) units of up to c tokens, each
// costing its tokens plus a fixed kUnitCostTokens (the unit's set-up, pipeline refill and partial
// row). A larger split never needs more than s_max splits, so the workspace layout still holds.
// Every CTA computes the same choice from the same lengths.
constexpr int kSplitCandidates = 5;
constexpr int kUnitCostTokens = 150;

__device__ __forceinline__ int split_candidate(int c0, int k, int cap) {
    const int m = k == 0 ? 2 : k == 1 ? 3 : k == 2 ? 4 : k == 3 ? 6 : 8;  // halves of c0
    const long long c = ((long long)c0 * m / 2 + 127) / 128 * 128, top = ((long long)cap + 127) / 128 * 128;
    return (int)(c < top ? c : top);  // at most the capacity (one split a context), rounded
}

// Prologue run by all kThreads threads of a CTA: clamp the lengths (flagging out-of-range ones),
// choose the split size (automatic splits; misc[0], and *chunk_out from CTA 0 for the merge
// kernel) and build the tables above. Returns the number of units; ends with __syncthreads.
template <int kThreads>
__device__ __forceinline__ int decode_scan_units(const DecodeArgs &a, const UnitTable &t) {
    const int tid = threadIdx.x, lane = tid & 31;
    const int S = a.s_max;
    const int cap = a.max_blocks_per_seq * a.cache.block_size;
    // (the largest candidate, the capacity rounded up to 128, keeps len + chunk - 1 within int)
    const bool choose = a.auto_chunk && S > 1 && cap <= (1 << 30) - 128;
    for (int s = tid; s <= S; s += kThreads) t.hist[s] = 0;
    if (tid < kUnitMisc) t.misc[tid] = 0;
    __syncthreads();
    int cnt[kSplitCandidates];
#pragma unroll
    for (int k = 0; k < kSplitCandidates; ++k) cnt[k] = 0;
    for (int i = tid; i < a.batch; i += kThreads) {
        int len = __ldg(a.context_lens + i);
        if (len < 0 || len > cap) {
            set_error(a.err, kErrDeviceRange);
            len = len < 0 ? 0 : cap;
        }
        int qrow = i;
        if (a.cu_q_lens) {  // mixed batch: only single-row sequences are decoded here
            const int q0 = __ldg(a.cu_q_lens + i), q1 = __ldg(a.cu_q_lens + i + 1);
            qrow = q0;
            if (q1 - q0 != 1) len = 0;
        }
        t.lens[i] = len;
        t.qrow[i] = qrow;
        if (choose) {
#pragma unroll
            for (int k = 0; k < kSplitCandidates; ++k) {
                const int c = split_candidate(a.chunk, k, cap);
                cnt[k] += len > 0 ? (len - 1) / c + 1 : 0;
            }
        }
    }
    int chunk = a.chunk;
    if (choose) {
#pragma unroll
        for (int k = 0; k < kSplitCandidates; ++k) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) cnt[k] += __shfl_xor_sync(0xffffffffu, cnt[k], o);
            if (lane == 0 && cnt[k]) atomicAdd(&t.misc[1 + k], cnt[k]);
        }
        __syncthreads();
        if (tid < 32) {
            // lane k prices candidate k; the cheapest wins, the smaller split on a tie
            const long long hu = (long long)a.cache.num_kv_heads * a.head_groups, grid = gridDim.x;
            const int k = lane < kSplitCandidates ? lane : 0;
            const int c = split_candidate(a.chunk, k, cap);
            const long long units = (long long)t.misc[1 + k] * hu;
            long long key = ((units + grid - 1) / grid * (long long)(min(c, cap) + kUnitCostTokens)) * 8 + k;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) key = min(key, __shfl_xor_sync(0xffffffffu, key, o));
            if (lane == 0) {
                const int best = split_candidate(a.chunk, (int)(key & 7), cap);
                t.misc[0] = best;
                if (blockIdx.x == 0 && a.chunk_out) *a.chunk_out = best;
            }
        }
        __syncthreads();
        chunk = t.misc[0];
    } else if (tid == 0) {
        t.misc[0] = chunk;
        if (blockIdx.x == 0 && a.chunk_out) *a.chunk_out = chunk;
    }
    for (int i = tid; i < a.batch; i += kThreads)
        atomicAdd(&t.hist[(t.lens[i] + chunk - 1) / chunk], 1);  // split count <= S since len <= cap
    __syncthreads();
    if (tid < 32) {
        // n_s = batch - (sequences with at most s splits); first[s + 1] = first[s] + n_s
        int below = 0, run = 0;
        for (int s0 = 0; s0 < S; s0 += 32) {
            const int s = s0 + lane;
            int h = s < S ? t.hist[s] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, h, o);
                if (lane >= o) h += y;
            }
            int n = s < S ? a.batch - (below + h) : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, n, o);
                if (lane >= o) n += y;
            }
            if (s < S) t.first[s + 1] = run + n;
            below += __shfl_sync(0xffffffffu, h, 31);
            run += __shfl_sync(0xffffffffu, n, 31);
        }
        if (lane == 0) t.first[0] = 0;
        __syncwarp();
        // Stable placement, 32 sequences at a time in index order: a sequence with k splits goes
        // after the sequences with more than k splits and after those with k splits and a lower
        // index (hist[k] now counts those already placed).
        for (int s = lane; s <= S; s += 32) t.hist[s] = 0;
        __syncwarp();
        for (int i0 = 0; i0 < a.batch; i0 += 32) {
            const int i = i0 + lane;
            const int k = i < a.batch ? (t.lens[i] + chunk - 1) / chunk : -1;
            const unsigned same = __match_any_sync(0xffffffffu, k);
            const int rank = __popc(same & ((1u << lane) - 1u));
            if (i < a.batch) {
                const int above = k < S ? t.first[k + 1] - t.first[k] : 0;
                t.ord[above + t.hist[k] + rank] = i;
            }
            __syncwarp();
            if (i < a.batch && rank == __popc(same) - 1) t.hist[k] += __popc(same);
            __syncwarp();
        }
    }
    __syncthreads();
    return t.first[S] * a.cache.num_kv_heads * a.head_groups;
}

}  // namespace pkv
