// prefill_wide.cu -- paged_attn_prefill at head_dim 256 (16-bit cache) on the 5th-generation tensor
// cores.
//
// Same computation as prefill.cu: out = softmax(Q K^T * scale) V for every query row of the chunk
// and every query head ("为什么Attention是O(n²)", mathematics section; the prefill phase of its
// prefill / decode section), keys read through the block table ("企业官网建设流程全解析", section
// 2.1) from the cache [num_blocks, 2, Hkv, block_size, D] ("Flash Attention与Paged Attention如何共同
// 优化大模型推理？", section 3), running max / running sum of that page's section 2, causal (bottom-
// right aligned) or not. A row of 256 dims is twice prefill.cu's, so a CTA holds one 128-row query
// tile instead of two (TMEM: S_0, S_1 of 64 columns, O of 256) and key tiles of 64 tokens (a K or V
// tile is 32 KB, as a 128-token tile at head_dim 128):
//   warp 0     TMA producer: the Q tile once (3-D tensor map over [total_q, Hq, D], four 64-column
//              boxes), then for each key tile j its K item and its V item, alternately into a ring
//              of four 32 KB slots; each lane issues the boxes of one page of the tile;
//   warp 1     TMEM owner and MMA issuer (one thread), in the order QK(0), QK(1), PV(0), QK(2),
//              PV(1), ...: S_{j%2} = Q K_j^T, then O += P_j V_j once the softmax has written P_j
//              (the input type, 64 keys = 32 TMEM columns) over S_{j%2}, so the softmax of tile
//              j + 1 overlaps the P V of tile j;
//   warps 2-5  softmax of TMEM lanes 32 (w % 4) .. + 31 = query rows, one row per thread: scale,
//              causal / context masks, running max with the lazy rescale of prefill.cu (O rescaled
//              in TMEM only when the max grows by more than 2^8; exact at the final division),
//              exp2, row sum; epilogue O / l -> out, lse.
#include <cuda.h>
#include <cuda_runtime.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "prefill_common.cuh"
#include "tcgen05.cuh"
#include "warp_mma.cuh"

namespace pkv {
namespace {

constexpr int kD = 256;
constexpr int kBM = 128;                 // query rows per CTA
constexpr int kBN = 64;                  // keys per key tile
constexpr int kRing = 4;                 // ring slots (items alternate K, V)
constexpr int kHalves = kD / 64;         // 128-byte swizzle atoms along D
constexpr int kThreads = 6 * 32;
constexpr int kProducerWarp = 0, kMmaWarp = 1;  // warps 2-5: softmax
constexpr float kRescaleLog2 = 8.0f;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;            // S_0 [0, 64), S_1 [64, 128); P_j over S_{j%2}
constexpr uint32_t kColO = 256;          // O [256, 512)
constexpr uint32_t kQHalf = kBM * 128;   // a 64-column half of the Q tile: 128 rows x 128 bytes
constexpr uint32_t kQBytes = kHalves * kQHalf;
constexpr uint32_t kKVHalf = kBN * 128;  // a 64-column half of a K or V tile
constexpr uint32_t kKVBytes = kHalves * kKVHalf;
constexpr uint32_t kRingOff = kQBytes;
constexpr uint32_t kBarOff = kRingOff + kRing * kKVBytes;
constexpr uint32_t kSmemBytes = kBarOff + 256 + 1024;  // + 1024-byte alignment slack

struct WideParams {
    const int *cu_q_lens, *context_lens, *block_tables;
    int batch, mb, num_q_heads, num_kv_heads, group, bs, log2_bs, num_blocks;
    float scale_log2;
    int causal, skip_single;
    void *out;
    int out_dtype;
    float *lse;
    int *err;
};

__device__ __forceinline__ uint32_t pack_pair(float a, float b, bool bf16) {
    if (bf16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_wide_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                        WideParams p) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment: the 128-byte swizzle pattern is a function of address bits 4-9
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t *sQ = smem;
    uint8_t *sRing = smem + kRingOff;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kBarOff);
    uint64_t *kv_full = bars;            // [kRing] the item in the slot has landed
    uint64_t *kv_empty = bars + kRing;   // [kRing] its MMAs are done with it
    uint64_t *q_full = bars + 2 * kRing;
    uint64_t *s_full = q_full + 1;       // [2] S_i computed
    uint64_t *p_full = s_full + 2;       // [2] P written over S_i (and O rescaled)
    uint64_t *o_done = p_full + 2;       // [2] the P V of the last tile j with j % 2 == i is done
    uint64_t *drain = o_done + 2;        // every MMA issued has completed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // grid (heads, row blocks, sequences), row blocks last-first: CTAs start in linear order, so the
    // CTAs running together share one sequence's K/V (it stays in L2), and within it the blocks that
    // see the most keys (causal) start first
    // (a mixed batch: sequences by their rank among those with several query rows, so that no CTA
    // without work precedes one with work)
    const int mt = (int)gridDim.y - 1 - (int)blockIdx.y, h = blockIdx.x;
    pdl_wait();  // lengths, tables, q and the chunk's own K/V may come from the previous kernel
    const int b = p.skip_single ? nth_multi_row_sequence(p.cu_q_lens, p.batch, blockIdx.z) : (int)blockIdx.z;
    if (b < 0) return;  // uniform: past the mixed batch's last chunk
    const int q0 = __ldg(p.cu_q_lens + b);
    const int q_len = __ldg(p.cu_q_lens + b + 1) - q0;
    const int m_start = mt * kBM;
    if (m_start >= q_len || (p.skip_single && q_len == 1)) return;  // uniform: nothing allocated yet
    const int L = __ldg(p.context_lens + b);
    if (L > p.mb * p.bs || q_len > L || L < 0) {
        if (threadIdx.x == 0) set_error(p.err, kErrDeviceRange);
        return;
    }
    const int rows = min(kBM, q_len - m_start);
    const int qpos0 = L - q_len + m_start;           // absolute position of row 0
    const int kv_end = p.causal ? qpos0 + rows : L;  // keys [0, kv_end) are needed
    const int n_tiles = (kv_end + kBN - 1) / kBN;
    const int g = h / p.group;                       // the KV head

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRing; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        mbar_init(q_full, 1);
        for (int x = 0; x < 2; ++x) {
            mbar_init(&s_full[x], 1);
            mbar_init(&p_full[x], 4);
            mbar_init(&o_done[x], 1);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp) {
        // ===================================== TMA producer =====================================
        const int box_rows = p.bs < kBN ? p.bs : kBN;
        uint32_t issued = 0;  // ring items issued (for the abort drain)
        if (lane == 0) {
            tc::prefetch_tensormap(&tm_q);
            tc::prefetch_tensormap(&tm_kv);
            mbar_arrive_expect_tx(q_full, kQBytes);
#pragma unroll
            for (int hf = 0; hf < kHalves; ++hf)
                tc::tma_load_3d(sQ + hf * kQHalf, &tm_q, hf * 64, h, q0 + m_start, q_full);
        }
        const int *bt = p.block_tables + (size_t)b * p.mb;
        bool ok = true;
        for (int j = 0; j < n_tiles && ok; ++j) {
            const int kv_start = j * kBN;
            const int n_valid = min(kBN, L - kv_start);
            const int page0 = kv_start >> p.log2_bs;
            const int npages = p.bs < kBN ? (n_valid + p.bs - 1) / p.bs : 1;  // <= 8 (block size >= 8)
            const int off = p.bs < kBN ? 0 : (kv_start & (p.bs - 1));
            int pb = 0;
            if (lane < npages) {
                pb = __ldg(bt + page0 + lane);
                if (pb < 0 || pb >= p.num_blocks) {
                    set_error(p.err, kErrDeviceRange);
                    pb = 0;
                }
            }
            for (int kv = 0; kv < 2; ++kv) {
                const uint32_t u = 2u * j + kv, slot = u % kRing, ph = (u / kRing) & 1u;
                if (!mbar_wait(&kv_empty[slot], ph ^ 1u, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(&kv_full[slot], (uint32_t)npages * box_rows * 128u * kHalves);
                __syncwarp();
                if (lane < npages) {
                    const int row = ((pb * 2 + kv) * p.num_kv_heads + g) * p.bs + off;
                    uint8_t *dst = sRing + slot * kKVBytes + (uint32_t)lane * box_rows * 128u;
#pragma unroll
                    for (int hf = 0; hf < kHalves; ++hf)
                        tc::tma_load_2d(dst + hf * kKVHalf, &tm_kv, hf * 64, row, &kv_full[slot]);
                }
                ++issued;
            }
        }
        if (!ok) {
            // let the copies in flight land before the CTA exits (bounded)
            volatile int no_abort = 0;
            const uint32_t first = issued > (uint32_t)kRing ? issued - kRing : 0u;
            for (uint32_t u = first; u < issued; ++u) mbar_wait(&kv_full[u % kRing], (u / kRing) & 1u, &no_abort, nullptr);
            mbar_wait(q_full, 0, &no_abort, nullptr);
        }
    } else if (warp == kMmaWarp) {
        // ====================================== MMA issuer ======================================
        if (lane == 0) {
            const uint32_t id_qk = tc::idesc_f16(BF16, kBM, kBN, false);
            const uint32_t id_pv = tc::idesc_f16(BF16, kBM, kD, true);
            const uint32_t aQ = smem_addr(sQ), aRing = smem_addr(sRing);
            bool ok = mbar_wait(q_full, 0, abort_flag, p.err);
            tc::fence_after_sync();
            // O (+)= P_t V_t: P in the input type (kBN keys = kBN / 2 TMEM columns over S_{t%2}); V is
            // [tokens x D], D contiguous: MN-major B, 8-token groups 1024 B apart, 64-column halves
            // kKVHalf apart; 16 tokens = 8 TMEM columns of P
            auto pv = [&](int t) -> bool {
                const uint32_t uV = 2u * t + 1, vslot = uV % kRing;
                if (!mbar_wait(&p_full[t & 1], ((uint32_t)t >> 1) & 1u, abort_flag, p.err)) return false;
                if (!mbar_wait(&kv_full[vslot], (uV / kRing) & 1u, abort_flag, p.err)) return false;
                tc::fence_after_sync();
                const uint32_t tP = tmem + kColS + (uint32_t)kBN * (t & 1);
                const uint32_t aV = aRing + vslot * kKVBytes;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    tc::mma_f16_ts(tmem + kColO, tP + 8u * kk, tc::smem_desc(aV + (uint32_t)kk * 2048u, kKVHalf, 1024),
                                   id_pv, (t > 0 || kk > 0) ? 1u : 0u);
                tc::mma_commit(&o_done[t & 1]);
                tc::mma_commit(&kv_empty[vslot]);  // the V item is done
                return true;
            };
            for (int j = 0; ok && j < n_tiles; ++j) {
                // S_{j%2} = Q K_j^T
                const uint32_t uK = 2u * j, kslot = uK % kRing;
                if (!(ok = mbar_wait(&kv_full[kslot], (uK / kRing) & 1u, abort_flag, p.err))) break;
                tc::fence_after_sync();
                const uint32_t aK = aRing + kslot * kKVBytes;
                const uint32_t tS = tmem + kColS + (uint32_t)kBN * (j & 1);
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t oq = (uint32_t)(kk >> 2) * kQHalf + (uint32_t)(kk & 3) * 32u;
                    const uint32_t ok_ = (uint32_t)(kk >> 2) * kKVHalf + (uint32_t)(kk & 3) * 32u;
                    tc::mma_f16_ss(tS, tc::smem_desc(aQ + oq, 16, 1024), tc::smem_desc(aK + ok_, 16, 1024), id_qk,
                                   kk > 0 ? 1u : 0u);
                }
                tc::mma_commit(&s_full[j & 1]);
                tc::mma_commit(&kv_empty[kslot]);  // the K item is done once S_j is
                // the previous tile's P V (its softmax overlapped this QK)
                if (j > 0 && !(ok = pv(j - 1))) break;
            }
            if (ok) ok = pv(n_tiles - 1);
            tc::mma_commit(drain);
            volatile int no_abort = 0;
            mbar_wait(drain, 0, &no_abort, p.err);
        }
        __syncwarp();
    } else {
        // ================================= softmax + epilogue =================================
        const int quarter = warp & 3;                 // the warp's TMEM lane quarter
        const int r = quarter * 32 + lane;            // query row of the tile
        const bool row_ok = r < rows;
        const int qpos = qpos0 + r;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const uint32_t tO = tmem + kColO + lane_base;
        const float c = p.scale_log2;
        float m_use = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; ok && j < n_tiles; ++j) {
            const int kv_start = j * kBN;
            if (!(ok = mbar_wait(&s_full[j & 1], ((uint32_t)j >> 1) & 1u, abort_flag, p.err))) break;
            tc::fence_after_sync();
            const uint32_t tS = tmem + kColS + (uint32_t)kBN * (j & 1) + lane_base;
            float s[kBN];
#pragma unroll
            for (int cc = 0; cc < kBN / 32; ++cc)
                tc::tmem_ld32(tS + cc * 32, *reinterpret_cast<float(*)[32]>(&s[cc * 32]));
            tc::tmem_wait_ld();
            // last key index this row may see in this tile (-1: none, a padding row)
            int lim = L - 1 - kv_start;
            if (p.causal) lim = min(lim, qpos - kv_start);
            if (!row_ok) lim = -1;
            if (lim < kBN - 1) {
#pragma unroll
                for (int i = 0; i < kBN; ++i) s[i] = (i <= lim) ? s[i] : -INFINITY;
            }
            // row max as 8 independent chains
            float m8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) m8[k] = fmax3(s[k], s[k + 8], s[k + 16]);
#pragma unroll
            for (int i = 24; i < kBN; i += 16)
#pragma unroll
                for (int k = 0; k < 8; ++k) m8[k] = fmax3(m8[k], s[i + k], (i + 8 + k < kBN) ? s[i + 8 + k] : -INFINITY);
            const float mx = fmaxf(fmax3(m8[0], m8[1], m8[2]), fmax3(fmax3(m8[3], m8[4], m8[5]), m8[6], m8[7]));
            const float m_new = fmaxf(m_use, mx * c);
            const bool grow = m_new > m_use + kRescaleLog2;  // false when m_new = -inf
            const float alpha = grow ? ex2f(m_use - m_new) : 1.f;  // 0 when m_use = -inf
            if (grow) {
                m_use = m_new;
                l *= alpha;
            }
            // a row with a visible key has a finite max; a padding row uses 0, so ex2(-inf) = 0
            const float neg_m = (m_use == -INFINITY) ? 0.f : -m_use;
            const float2 c2 = make_float2(c, c), nm2 = make_float2(neg_m, neg_m);
            uint32_t pk[kBN / 2];
            float2 l4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
            for (int q = 0; q < kBN / 2; ++q) {
                const float2 xq = ffma2(make_float2(s[2 * q], s[2 * q + 1]), c2, nm2);
                const float2 e = make_float2(ex2f(xq.x), ex2f(xq.y));
                l4[q & 3] = fadd2(l4[q & 3], e);
                pk[q] = pack_pair(e.x, e.y, BF16);
            }
            const float2 l2 = fadd2(fadd2(l4[0], l4[1]), fadd2(l4[2], l4[3]));
            l += l2.x + l2.y;
            // O is touched only after P_{j-1} V_{j-1} is done
            if (j > 0) {
                if (!(ok = mbar_wait(&o_done[(j - 1) & 1], ((uint32_t)(j - 1) >> 1) & 1u, abort_flag, p.err))) break;
                tc::fence_after_sync();
                if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
                    for (int cc = 0; cc < kD / 32; ++cc) {
                        float o[32];
                        tc::tmem_ld32(tO + cc * 32, o);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= alpha;
                        tc::tmem_st32(tO + cc * 32, o);
                    }
                }
            }
#pragma unroll
            for (int cc = 0; cc < kBN / 32; ++cc)
                tc::tmem_st16(tS + cc * 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[cc * 16]));
            tc::tmem_wait_st();
            // keys at or beyond the context end may hold unwritten cache bytes: their V rows are
            // zeroed (thread r, row r) so that 0 * garbage cannot reach O
            const int n_valid = L - kv_start;
            if (n_valid < kBN) {
                const uint32_t uV = 2u * j + 1;
                if (!(ok = mbar_wait(&kv_full[uV % kRing], (uV / kRing) & 1u, abort_flag, p.err))) break;
                if (r >= n_valid && r < kBN) {
                    uint8_t *sV = sRing + (uV % kRing) * kKVBytes;
#pragma unroll
                    for (int hf = 0; hf < kHalves; ++hf)
#pragma unroll
                        for (int cc = 0; cc < 8; ++cc)
                            *reinterpret_cast<uint4 *>(sV + hf * kKVHalf + (uint32_t)r * 128u + cc * 16) = make_uint4(0, 0, 0, 0);
                }
                tc::fence_proxy_async_smem();
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[j & 1]);
        }
        // ---- epilogue: O / l ----
        const int jl = n_tiles - 1;
        if (ok && mbar_wait(&o_done[jl & 1], ((uint32_t)jl >> 1) & 1u, abort_flag, p.err)) {
            tc::fence_after_sync();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const size_t row_g = (size_t)(q0 + m_start + r);
            const size_t obase = (row_g * p.num_q_heads + h) * kD;
#pragma unroll
            for (int cc = 0; cc < kD / 32; ++cc) {
                float o[32];
                tc::tmem_ld32(tO + cc * 32, o);
                tc::tmem_wait_ld();
                if (row_ok) {
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        const float x[4] = {o[4 * v] * inv, o[4 * v + 1] * inv, o[4 * v + 2] * inv, o[4 * v + 3] * inv};
                        store_out_vec<4>(p.out, obase + cc * 32 + 4 * v, x, p.out_dtype);
                    }
                }
            }
            if (row_ok && p.lse) p.lse[row_g * p.num_q_heads + h] = l > 0.f ? (m_use + __log2f(l)) * kLn2 : -INFINITY;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    pdl_launch_dependents();
    if (warp == kMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

namespace {

template <bool BF16>
cudaError_t launch_wide_t(const PrefillArgs &a, cudaStream_t stream) {
    CUtensorMap tm_q, tm_kv;
    cudaError_t e = encode_q_heads_map(a.q, BF16 ? 1 : 0, a.total_q, a.num_q_heads, kD, kBM, &tm_q);
    if (e != cudaSuccess) return e;
    e = encode_cache_map(a.cache, a.cache.block_size < kBN ? a.cache.block_size : kBN, &tm_kv);
    if (e != cudaSuccess) return e;
    WideParams p;
    p.cu_q_lens = a.cu_q_lens;
    p.context_lens = a.context_lens;
    p.block_tables = a.block_tables;
    p.batch = a.batch;
    p.mb = a.max_blocks_per_seq;
    p.num_q_heads = a.num_q_heads;
    p.num_kv_heads = a.cache.num_kv_heads;
    p.group = a.num_q_heads / a.cache.num_kv_heads;
    p.bs = a.cache.block_size;
    p.log2_bs = a.cache.log2_block_size;
    p.num_blocks = a.cache.num_blocks;
    p.scale_log2 = a.scale * kLog2e;
    p.causal = a.causal;
    p.skip_single = a.skip_single;
    p.out = a.out;
    p.out_dtype = a.out_dtype;
    p.lse = a.lse;
    p.err = a.err;
    auto kern = prefill_wide_kernel<BF16>;
    static DeviceFlags configured;  // opt in to the kernel's shared memory once per device
    const int dev = device_info().device;
    if (dev >= 64 || !configured.test(dev)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev < 64) configured.set(dev);
    }
    const long long row_blocks = ((long long)a.max_q_len + kBM - 1) / kBM;
    if (row_blocks > 65535) return cudaErrorNotSupported;
    dim3 grid(a.num_q_heads, (unsigned)row_blocks, a.batch);
    return launch_pdl(kern, grid, dim3(kThreads), kSmemBytes, stream, tm_q, tm_kv, p);
}

}  // namespace

cudaError_t launch_prefill_wide(const PrefillArgs &a, cudaStream_t s) {
    if (a.max_q_len == 0) return cudaSuccess;
    if (a.cache.head_dim != kD || a.cache.fp8) return cudaErrorNotSupported;
    return a.cache.dtype == 1 ? launch_wide_t<true>(a, s) : launch_wide_t<false>(a, s);
}
}  // namespace pkv
