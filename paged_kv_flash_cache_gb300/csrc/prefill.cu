// prefill.cu -- paged_attn_prefill: a chunk of queries per sequence against its paged context,
// causal (bottom-right aligned) or not, on the 5th-generation tensor cores.
//
// What it computes: out = softmax(Q K^T * scale) V for every query row of the chunk and every
// query head ("为什么Attention是O(n²)", mathematics section), the keys read through the block table
// ("企业官网建设流程全解析", section 2.1) from the cache [num_blocks, 2, Hkv, block_size, D]
// ("Flash Attention与Paged Attention如何共同优化大模型推理？", section 3), with the running max /
// running sum of that page's section 2 so the score matrix never leaves the SM, and the causal
// flag of the library call quoted there.  Prefill is the matrix-matrix phase ("为什么Attention是
// O(n²)", prefill / decode section): Q K^T and P V are dense contractions and run as tcgen05.mma.
//
// CTA = one query head x 128 query rows of one sequence (192 threads):
//   warp 0     TMA producer: Q tile once (3-D tensor map over [total_q, Hq, D]); for each
//              128-key tile, the pages it covers are looked up in the block table by the
//              warp's lanes and each lane issues its page's K and V boxes (2-D tensor map over
//              the cache viewed as rows of D elements), 128-byte swizzle, into a 2-stage ring;
//   warp 1     TMEM owner and MMA issuer (one thread): S = Q K^T into TMEM columns [0, 128),
//              then O += P V into columns [128, 128 + D); S of tile j+1 is issued as soon as the
//              softmax has read S of tile j, so the tensor pipe works during the softmax;
//   warps 2-5  softmax / epilogue, one query row per thread (TMEM lane = row): scale, causal and
//              context masks, row max, exp2, row sum, P (input dtype) written to shared memory in
//              the swizzled K-major layout the MMA reads; O is rescaled in TMEM only when the
//              running max grows by more than 2^8 (the final O / l uses the same max, so the
//              result is exact); the epilogue reads O from TMEM, divides by l, writes out / lse.
// Every wait is bounded (a timeout sets the device error word and the CTA winds down).
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "tcgen05.cuh"

namespace pkv {
namespace {

constexpr int kBM = 128;       // query rows per CTA
constexpr int kBN = 128;       // keys per KV tile
constexpr int kStages = 2;     // KV ring depth
constexpr int kThreads = 192;  // 6 warps
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when the max grows by more than 2^8

template <int D>
struct PrefillLayout {
    static constexpr int kHalves = D / 64;                      // 128-byte swizzle atoms along D
    static constexpr uint32_t kTileHalf = 128 * 128;            // 128 rows x 128 bytes
    static constexpr uint32_t kQBytes = kHalves * kTileHalf;
    static constexpr uint32_t kKVBytes = kHalves * kTileHalf;   // one K (or V) tile
    static constexpr uint32_t kPBytes = 2 * kTileHalf;          // 128 rows x 128 keys
    static constexpr uint32_t kQOff = 0;
    static constexpr uint32_t kKVOff = kQOff + kQBytes;         // stage s: K at +2*s*kKVBytes, V after it
    static constexpr uint32_t kPOff = kKVOff + kStages * 2 * kKVBytes;
    static constexpr uint32_t kBarOff = kPOff + kPBytes;
    static constexpr uint32_t kSmemBytes = kBarOff + 128 + 1024;  // barriers + alignment slack
    static constexpr uint32_t kTmemCols = 256;                    // S: 128 columns, O: D columns
    static constexpr uint32_t kOCol = 128;
};

struct PrefillParams {
    const int *cu_q_lens, *context_lens, *block_tables;
    int batch, mb, num_q_heads, num_kv_heads, group, bs, log2_bs, num_blocks;
    float scale_log2;
    int causal;
    void *out;
    int out_dtype;
    float *lse;
    int *err;
};

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack2(float a, float b, bool bf16) {
    if (bf16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                   PrefillParams p) {
    using Lay = PrefillLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment: the 128-byte swizzle pattern is a function of address bits 4-9.
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t *sQ = smem + Lay::kQOff;
    uint8_t *sP = smem + Lay::kPOff;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::kBarOff);
    uint64_t *full = bars;        // [kStages] K/V tile landed
    uint64_t *empty = bars + 2;   // [kStages] K/V stage free again
    uint64_t *q_full = bars + 4;
    uint64_t *s_full = bars + 5;  // S_j in TMEM
    uint64_t *s_free = bars + 6;  // softmax has read S_j
    uint64_t *p_full = bars + 7;  // P_j in shared memory (and O rescaled)
    uint64_t *o_done = bars + 8;  // P_j V_j accumulated into O
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 9);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 10);
    uint64_t *drain = bars + 11;  // every MMA issued has completed (before TMEM is freed)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int q0 = __ldg(p.cu_q_lens + b);
    const int q_len = __ldg(p.cu_q_lens + b + 1) - q0;
    const int m_start = mt * kBM;
    if (m_start >= q_len) return;  // uniform: nothing allocated yet
    int L = __ldg(p.context_lens + b);
    const int cap = p.mb * p.bs;
    if (L > cap || q_len > L || L < 0) {
        if (threadIdx.x == 0) set_error(p.err, kErrDeviceRange);
        return;
    }
    const int rows = min(kBM, q_len - m_start);
    const int qpos0 = L - q_len + m_start;                // absolute position of row 0
    const int kv_end = p.causal ? qpos0 + rows : L;       // keys [0, kv_end) are needed
    const int n_tiles = (kv_end + kBN - 1) / kBN;
    const int g = h / p.group;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(q_full, 1);
        mbar_init(s_full, 1);
        mbar_init(s_free, 4);
        mbar_init(p_full, 4);
        mbar_init(o_done, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, Lay::kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ===================================== TMA producer =====================================
        const int box_rows = p.bs < kBN ? p.bs : kBN;
        uint32_t issued_mask = 0, issued_parity = 0;
        if (lane == 0) {
            tc::prefetch_tensormap(&tm_q);
            tc::prefetch_tensormap(&tm_kv);
            mbar_arrive_expect_tx(q_full, Lay::kQBytes);
#pragma unroll
            for (int hf = 0; hf < Lay::kHalves; ++hf)
                tc::tma_load_3d(sQ + hf * Lay::kTileHalf, &tm_q, hf * 64, h, q0 + m_start, q_full);
        }
        const int *bt = p.block_tables + (size_t)b * p.mb;
        for (int j = 0; j < n_tiles; ++j) {
            const int s = j % kStages;
            const uint32_t ph = (uint32_t)(j / kStages) & 1u;
            const int kv_start = j * kBN;
            const int n_valid = min(kBN, L - kv_start);
            const int page0 = kv_start >> p.log2_bs;
            const int npages = p.bs < kBN ? (n_valid + p.bs - 1) / p.bs : 1;
            const int off = p.bs < kBN ? 0 : (kv_start & (p.bs - 1));
            int pb = 0;
            if (lane < npages) {
                pb = __ldg(bt + page0 + lane);
                if (pb < 0 || pb >= p.num_blocks) {
                    set_error(p.err, kErrDeviceRange);
                    pb = 0;
                }
            }
            if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.err)) {
                for (int i = 0; i < kStages; ++i)
                    if (issued_mask & (1u << i)) {
                        volatile int no_abort = 0;
                        mbar_wait(&full[i], (issued_parity >> i) & 1u, &no_abort, nullptr);
                    }
                break;
            }
            uint8_t *sK = smem + Lay::kKVOff + (uint32_t)s * 2 * Lay::kKVBytes;
            uint8_t *sV = sK + Lay::kKVBytes;
            if (lane == 0)
                mbar_arrive_expect_tx(&full[s], (uint32_t)npages * box_rows * 128u * Lay::kHalves * 2u);
            __syncwarp();
            if (lane < npages) {
                const int rowK = ((pb * 2 + 0) * p.num_kv_heads + g) * p.bs + off;
                const int rowV = rowK + p.num_kv_heads * p.bs;
                const uint32_t dst = (uint32_t)lane * box_rows * 128u;
#pragma unroll
                for (int hf = 0; hf < Lay::kHalves; ++hf) {
                    tc::tma_load_2d(sK + hf * Lay::kTileHalf + dst, &tm_kv, hf * 64, rowK, &full[s]);
                    tc::tma_load_2d(sV + hf * Lay::kTileHalf + dst, &tm_kv, hf * 64, rowV, &full[s]);
                }
            }
            issued_mask |= 1u << s;
            issued_parity = (issued_parity & ~(1u << s)) | (ph << s);
        }
    } else if (warp == 1) {
        // ====================================== MMA issuer ======================================
        if (lane == 0) {
            const uint32_t id_qk = tc::idesc_f16(BF16, kBM, kBN, false);
            const uint32_t id_pv = tc::idesc_f16(BF16, kBM, D, true);
            const uint32_t tS = tmem, tO = tmem + Lay::kOCol;
            const uint32_t aQ = smem_addr(sQ), aP = smem_addr(sP);
            const uint32_t aKV = smem_addr(smem + Lay::kKVOff);
            bool ok = mbar_wait(q_full, 0, abort_flag, p.err);
            auto issue_qk = [&](int j) -> bool {
                const int s = j % kStages;
                if (!mbar_wait(&full[s], (uint32_t)(j / kStages) & 1u, abort_flag, p.err)) return false;
                tc::fence_after_sync();
                const uint32_t aK = aKV + (uint32_t)s * 2 * Lay::kKVBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t o = (uint32_t)(kk >> 2) * Lay::kTileHalf + (uint32_t)(kk & 3) * 32u;
                    tc::mma_f16_ss(tS, tc::smem_desc(aQ + o, 16, 1024), tc::smem_desc(aK + o, 16, 1024), id_qk,
                                   kk > 0 ? 1u : 0u);
                }
                tc::mma_commit(s_full);
                return true;
            };
            if (ok) ok = issue_qk(0);
            for (int j = 0; ok && j < n_tiles; ++j) {
                if (j + 1 < n_tiles) {
                    // S is single-buffered: wait until the softmax has read S_j
                    if (!mbar_wait(s_free, (uint32_t)j & 1u, abort_flag, p.err) || !issue_qk(j + 1)) break;
                }
                if (!mbar_wait(p_full, (uint32_t)j & 1u, abort_flag, p.err)) break;
                tc::fence_after_sync();
                const int s = j % kStages;
                const uint32_t aV = aKV + (uint32_t)s * 2 * Lay::kKVBytes + Lay::kKVBytes;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    const uint32_t oP = (uint32_t)(kk >> 2) * Lay::kTileHalf + (uint32_t)(kk & 3) * 32u;
                    // V is [keys x D] with D contiguous: MN-major B; 8-key groups 1024 B apart,
                    // 64-column halves kTileHalf apart
                    tc::mma_f16_ss(tO, tc::smem_desc(aP + oP, 16, 1024),
                                   tc::smem_desc(aV + (uint32_t)kk * 2048u, Lay::kTileHalf, 1024), id_pv,
                                   (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc::mma_commit(o_done);
                tc::mma_commit(&empty[s]);
            }
            tc::mma_commit(drain);
            volatile int no_abort = 0;
            mbar_wait(drain, 0, &no_abort, p.err);
        }
        __syncwarp();
    } else {
        // ================================ softmax + epilogue ================================
        const int quarter = warp & 3;                  // TMEM lanes 32*quarter .. +31
        const int r = quarter * 32 + lane;             // row within the tile
        const bool row_ok = r < rows;
        const int qpos = qpos0 + r;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_base, tO = tmem + Lay::kOCol + lane_base;
        float m_use = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_tiles && ok; ++j) {
            const int kv_start = j * kBN;
            if (!mbar_wait(s_full, (uint32_t)j & 1u, abort_flag, p.err)) { ok = false; break; }
            tc::fence_after_sync();
            float s[kBN];
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c) tc::tmem_ld32(tS + c * 32, *reinterpret_cast<float(*)[32]>(&s[c * 32]));
            tc::tmem_wait_ld();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free);
            // last key index this row may see in this tile (-1: none)
            int lim = L - 1 - kv_start;
            if (p.causal) lim = min(lim, qpos - kv_start);
            if (!row_ok) lim = -1;
            float mx = -INFINITY;
#pragma unroll
            for (int i = 0; i < kBN; ++i) {
                const float v = (i <= lim) ? s[i] * p.scale_log2 : -INFINITY;
                s[i] = v;
                mx = fmaxf(mx, v);
            }
            const float m_new = fmaxf(m_use, mx);
            const bool grow = m_new > m_use + kRescaleLog2;   // false when m_new = -inf
            const float alpha = grow ? fast_exp2(m_use - m_new) : 1.f;  // 0 when m_use = -inf
            if (grow) {
                m_use = m_new;
                l *= alpha;
            }
            // O and P are touched only after P_{j-1} V_{j-1} is done
            if (j > 0) {
                if (!mbar_wait(o_done, (uint32_t)(j - 1) & 1u, abort_flag, p.err)) { ok = false; break; }
                tc::fence_after_sync();
                if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        float o[32];
                        tc::tmem_ld32(tO + c * 32, o);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= alpha;
                        tc::tmem_st32(tO + c * 32, o);
                    }
                    tc::tmem_wait_st();
                }
            }
            float lsum = 0.f;
#pragma unroll
            for (int i = 0; i < kBN; ++i) {
                const float e = (s[i] == -INFINITY) ? 0.f : fast_exp2(s[i] - m_use);
                s[i] = e;
                lsum += e;
            }
            l += lsum;
            // P row -> shared memory, K-major, 128-byte swizzle (16-byte chunk c of row r at c ^ (r & 7))
#pragma unroll
            for (int c = 0; c < kBN / 8; ++c) {
                uint4 v;
                v.x = pack2(s[c * 8 + 0], s[c * 8 + 1], BF16);
                v.y = pack2(s[c * 8 + 2], s[c * 8 + 3], BF16);
                v.z = pack2(s[c * 8 + 4], s[c * 8 + 5], BF16);
                v.w = pack2(s[c * 8 + 6], s[c * 8 + 7], BF16);
                const uint32_t o = (uint32_t)(c >> 3) * Lay::kTileHalf + (uint32_t)r * 128u +
                                   ((uint32_t)((c & 7) ^ (r & 7)) << 4);
                *reinterpret_cast<uint4 *>(sP + o) = v;
            }
            // keys at or beyond the context end may hold unwritten cache bytes: zero those V rows
            const int n_valid = L - kv_start;
            if (n_valid < kBN && r >= n_valid) {
                uint8_t *sV = smem + Lay::kKVOff + (uint32_t)(j % kStages) * 2 * Lay::kKVBytes + Lay::kKVBytes;
#pragma unroll
                for (int hf = 0; hf < Lay::kHalves; ++hf)
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4 *>(sV + hf * Lay::kTileHalf + (uint32_t)r * 128u + c * 16) =
                            make_uint4(0, 0, 0, 0);
            }
            tc::fence_proxy_async_smem();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }
        // ---- epilogue: O / l ----
        if (ok && mbar_wait(o_done, (uint32_t)(n_tiles - 1) & 1u, abort_flag, p.err)) {
            tc::fence_after_sync();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const size_t row_g = (size_t)(q0 + m_start + r);
            const size_t obase = (row_g * p.num_q_heads + h) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float o[32];
                tc::tmem_ld32(tO + c * 32, o);
                tc::tmem_wait_ld();
                if (row_ok) {
                    if (p.out_dtype == 2) {
                        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + obase + c * 32);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv,
                                                 o[4 * i + 3] * inv);
                    } else {
                        const bool obf = p.out_dtype == 1;
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.out) + obase + c * 32);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            uint4 v;
                            v.x = pack2(o[8 * i + 0] * inv, o[8 * i + 1] * inv, obf);
                            v.y = pack2(o[8 * i + 2] * inv, o[8 * i + 3] * inv, obf);
                            v.z = pack2(o[8 * i + 4] * inv, o[8 * i + 5] * inv, obf);
                            v.w = pack2(o[8 * i + 6] * inv, o[8 * i + 7] * inv, obf);
                            dst[i] = v;
                        }
                    }
                }
            }
            if (row_ok && p.lse) p.lse[row_g * p.num_q_heads + h] = l > 0.f ? (m_use + __log2f(l)) * kLn2 : -INFINITY;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, Lay::kTmemCols);
    }
}

// ---- host side: tensor maps --------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

template <int D, bool BF16>
cudaError_t launch_t(const PrefillArgs &a, cudaStream_t stream) {
    using Lay = PrefillLayout<D>;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const CUtensorMapDataType dt = BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap tm_q, tm_kv;
    {
        // q [total_q, Hq, D]: x = d, y = head, z = token; box 64 x 1 x 128
        cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)a.num_q_heads, (cuuint64_t)a.total_q};
        cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.num_q_heads * D * 2};
        cuuint32_t box[3] = {64, 1, (cuuint32_t)kBM};
        cuuint32_t es[3] = {1, 1, 1};
        if (enc(&tm_q, dt, 3, const_cast<void *>(a.q), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        // cache viewed as rows of D elements: row ((pb*2 + kv)*Hkv + h)*bs + off
        const cuuint64_t nrows = (cuuint64_t)a.cache.num_blocks * 2 * a.cache.num_kv_heads * a.cache.block_size;
        if (nrows > 0x7fffffffull) return cudaErrorNotSupported;  // TMA row coordinates are int32
        cuuint64_t dims[2] = {(cuuint64_t)D, nrows};
        cuuint64_t strides[1] = {(cuuint64_t)D * 2};
        cuuint32_t box[2] = {64, (cuuint32_t)(a.cache.block_size < kBN ? a.cache.block_size : kBN)};
        cuuint32_t es[2] = {1, 1};
        if (enc(&tm_kv, dt, 2, const_cast<void *>(a.cache.ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    PrefillParams p;
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
    p.out = a.out;
    p.out_dtype = a.out_dtype;
    p.lse = a.lse;
    p.err = a.err;
    auto kern = prefill_kernel<D, BF16>;
    static bool configured[64] = {};
    const int dev = device_info().device;
    if (dev >= 64 || !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Lay::kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev < 64) configured[dev] = true;
    }
    dim3 grid((a.max_q_len + kBM - 1) / kBM, a.num_q_heads, a.batch);
    kern<<<grid, kThreads, Lay::kSmemBytes, stream>>>(tm_q, tm_kv, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t s) {
    if (a.max_q_len == 0) return cudaSuccess;
    const bool bf16 = a.cache.dtype == 1;
    if (a.cache.head_dim == 128) return bf16 ? launch_t<128, true>(a, s) : launch_t<128, false>(a, s);
    return bf16 ? launch_t<64, true>(a, s) : launch_t<64, false>(a, s);
}

}  // namespace pkv
