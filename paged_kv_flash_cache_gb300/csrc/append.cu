// append.cu -- kv_cache_append: scatter new tokens' K and V rows into their pages.
//
// A decode step appends the new token's K and V to the cache and prefill stores every
// prompt token's K and V ("为什么Attention是O(n²)", prefill / decode section); token i of a
// sequence lives in page block_table[i / block_size] at offset i % block_size
// ("企业官网建设流程全解析", section 2.1) of the cache [num_blocks, 2, num_heads, block_size,
// head_dim] ("Flash Attention与Paged Attention如何共同优化大模型推理？", section 3).
//
// One warp per (new token, group of 8 heads): the warp resolves (sequence, position, page), then
// moves those heads' K rows and V rows as 16-byte vectors. Reads of k_new / v_new are contiguous;
// each destination head row (D elements) is a contiguous 128 / 256-byte run. Small items keep
// every SM busy even when a call appends a few thousand tokens.
// Pure bandwidth: 2 reads + 2 writes of Hkv * D * 2 bytes per token (an FP8 cache: writes of
// Hkv * (D + 4) bytes for each of K and V).
#include <climits>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kAppendThreads = 256;

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

constexpr int kHeadsPerItem = 8;  // a work item is one token's K and V rows of up to 8 heads

// Page and in-page row of new token t (all lanes of the warp, same t). The sequence is the last b
// with cu_new_lens[b] <= t, i.e. the count of b in [1, batch) with cu_new_lens[b] <= t (lengths
// are non-negative): up to 32 sequences, one load per lane and a ballot, ctx_before read in the
// same round trip; more, a binary search; no cu_new_lens (a decode step), sequence t. Returns false (error word set) for a position outside
// the table or a page id outside the pool.
__device__ __forceinline__ bool token_slot(const AppendArgs &a, int t, int lane, int &pb, int &off) {
    int b;
    long long pos;
    if (!a.cu_new_lens) {  // one new token per sequence
        b = t;
        pos = __ldg(a.ctx_before + t);
    } else if (a.batch <= 32) {
        const int cu_j = (lane >= 1 && lane < a.batch) ? __ldg(a.cu_new_lens + lane) : INT_MAX;
        const int ctx_j = lane < a.batch ? __ldg(a.ctx_before + lane) : 0;
        const int cu_b_j = lane < a.batch ? __ldg(a.cu_new_lens + lane) : 0;
        b = __popc(__ballot_sync(0xffffffffu, cu_j <= t));
        pos = (long long)__shfl_sync(0xffffffffu, ctx_j, b) + (t - __shfl_sync(0xffffffffu, cu_b_j, b));
    } else {
        int lo = 0, hi = a.batch;  // answer in [lo, hi)
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(a.cu_new_lens + mid) <= t) lo = mid; else hi = mid;
        }
        b = lo;
        pos = (long long)__ldg(a.ctx_before + b) + (t - __ldg(a.cu_new_lens + b));
    }
    const long long logical = pos >> a.log2_block_size;
    if (pos < 0 || logical >= a.max_blocks_per_seq) {
        if (lane == 0) set_error(a.err, kErrDeviceRange);
        return false;
    }
    pb = __ldg(a.block_tables + (size_t)b * a.max_blocks_per_seq + logical);
    if (pb < 0 || pb >= a.num_blocks) {
        if (lane == 0) set_error(a.err, kErrDeviceRange);
        return false;
    }
    off = (int)(pos & (a.block_size - 1));
    return true;
}

template <int D>
__global__ void __launch_bounds__(kAppendThreads) append_kernel(AppendArgs a) {
    constexpr int kVecPerRow = D / 8;  // 16-byte vectors per head row
    constexpr int kUnroll = (kHeadsPerItem * kVecPerRow + 31) / 32;  // vectors per lane per item
    static_assert(kHeadsPerItem * kVecPerRow <= 32 * kUnroll, "one pass of the warp per item");
    const int lane = threadIdx.x & 31;
    const int warps_total = gridDim.x * (kAppendThreads / 32);
    const int hkv = a.num_kv_heads;
    const int chunks = (hkv + kHeadsPerItem - 1) / kHeadsPerItem;
    const long long items = (long long)a.num_new_tokens * chunks;
    const int vec_per_token = hkv * kVecPerRow;
    const uint4 *kn = static_cast<const uint4 *>(a.k_new);
    const uint4 *vn = static_cast<const uint4 *>(a.v_new);
    uint4 *cache = static_cast<uint4 *>(a.cache);
    // vectors between consecutive heads / between K and V of one page
    const size_t head_stride = (size_t)a.block_size * kVecPerRow;
    const size_t kv_stride = (size_t)hkv * head_stride;

    pdl_wait();  // the previous kernel may still read the pages this call writes
    for (long long it = (long long)blockIdx.x * (kAppendThreads / 32) + (threadIdx.x >> 5); it < items;
         it += warps_total) {
        const int t = (int)(it / chunks);
        const int h0 = (int)(it - (long long)t * chunks) * kHeadsPerItem;
        const int nvec = min(kHeadsPerItem, hkv - h0) * kVecPerRow;
        // the item's K and V vectors first: they depend only on the token, so their loads overlap
        // the lookup of its page
        const uint4 *ks = kn + (size_t)t * vec_per_token + (size_t)h0 * kVecPerRow;
        const uint4 *vs = vn + (size_t)t * vec_per_token + (size_t)h0 * kVecPerRow;
        uint4 kv[kUnroll], vv[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int c = lane + u * 32;
            if (c < nvec) {
                kv[u] = ld_stream(ks + c);
                vv[u] = ld_stream(vs + c);
            }
        }
        int pb, off;
        if (!token_slot(a, t, lane, pb, off)) continue;
        const size_t page_base = (size_t)pb * 2 * kv_stride + (size_t)off * kVecPerRow;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int c = lane + u * 32;
            if (c < nvec) {
                const int h = h0 + c / kVecPerRow;
                const int e = c % kVecPerRow;
                const size_t dst = page_base + (size_t)h * head_stride + e;
                cache[dst] = kv[u];
                cache[dst + kv_stride] = vv[u];
            }
        }
    }
    pdl_launch_dependents();
}

// FP8 cache: the warp's rows (up to 8 heads x K and V of one token) are quantised kRows at a
// time; D / 8 lanes hold one row (8 elements each), find its largest magnitude by shuffles and
// write 8 codes each, the row's first lane its scale. All arithmetic in FP32: scale = amax / 448,
// code = E4M3(x * (448 / amax)) rounded to nearest even and saturated.
template <int D, typename Tag>
__global__ void __launch_bounds__(kAppendThreads) append_fp8_kernel(AppendArgs a) {
    constexpr int kLanesPerRow = D / 8;
    constexpr int kRows = 32 / kLanesPerRow;  // rows quantised per pass of the warp
    const int lane = threadIdx.x & 31;
    const int sub = lane / kLanesPerRow, chk = lane % kLanesPerRow;
    const int warps_total = gridDim.x * (kAppendThreads / 32);
    const int hkv = a.num_kv_heads;
    const int chunks = (hkv + kHeadsPerItem - 1) / kHeadsPerItem;
    const long long items = (long long)a.num_new_tokens * chunks;
    const uint4 *kn = static_cast<const uint4 *>(a.k_new);
    const uint4 *vn = static_cast<const uint4 *>(a.v_new);
    uint8_t *codes = static_cast<uint8_t *>(a.cache);

    pdl_wait();  // the previous kernel may still read the pages this call writes
    for (long long it = (long long)blockIdx.x * (kAppendThreads / 32) + (threadIdx.x >> 5); it < items;
         it += warps_total) {
        const int t = (int)(it / chunks);
        const int h0 = (int)(it - (long long)t * chunks) * kHeadsPerItem;
        const int nh = min(kHeadsPerItem, hkv - h0);
        // all of this lane's loads first (one memory round trip per item, overlapping the lookup
        // of the token's page), then the rows
        constexpr int kPasses = 2 * kHeadsPerItem / kRows;
        uint4 raws[kPasses];
#pragma unroll
        for (int ps = 0; ps < kPasses; ++ps) {
            const int r = ps * kRows + sub;
            raws[ps] = make_uint4(0u, 0u, 0u, 0u);
            if (r < 2 * nh) {
                const int kv = r >= nh ? 1 : 0;
                const int h = h0 + r - kv * nh;
                raws[ps] = ld_stream((kv ? vn : kn) + ((size_t)t * hkv + h) * kLanesPerRow + chk);
            }
        }
        int pb, off;
        if (!token_slot(a, t, lane, pb, off)) continue;
#pragma unroll
        for (int ps = 0; ps < kPasses; ++ps) {
            const int r = ps * kRows + sub;  // row r: K (r < nh) or V of head h0 + r % nh
            const bool active = r < 2 * nh;
            const int kv = active && r >= nh ? 1 : 0;
            const int h = h0 + (active ? r - kv * nh : 0);
            float2 f[4];
            unpack8x2(raws[ps], f, Tag());
            float amax = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fmaxf(fabsf(f[j].x), fabsf(f[j].y)));
#pragma unroll
            for (int o = kLanesPerRow / 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            if (active) {
                const size_t row = (((size_t)pb * 2 + kv) * hkv + h) * a.block_size + off;
                uint2 c = make_uint2(0u, 0u);
                float scale = 0.f;
                if (amax > 0.f) {
                    scale = amax / 448.0f;
                    const float inv = 448.0f / amax;
                    c.x = pack_e4m3x2(f[0].x * inv, f[0].y * inv) | (pack_e4m3x2(f[1].x * inv, f[1].y * inv) << 16);
                    c.y = pack_e4m3x2(f[2].x * inv, f[2].y * inv) | (pack_e4m3x2(f[3].x * inv, f[3].y * inv) << 16);
                }
                *reinterpret_cast<uint2 *>(codes + row * D + chk * 8) = c;
                if (chk == 0) a.scales[row] = scale;
            }
        }
    }
    pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_append(const AppendArgs &a, cudaStream_t s) {
    if (a.num_new_tokens == 0 || a.batch == 0) return cudaSuccess;
    const int warps_per_cta = kAppendThreads / 32;
    const long long items = (long long)a.num_new_tokens * ((a.num_kv_heads + kHeadsPerItem - 1) / kHeadsPerItem);
    const long long want = (items + warps_per_cta - 1) / warps_per_cta;
    const int cap = device_info().num_sms * 8;
    const int grid = want < cap ? (int)want : cap;
    if (a.fp8) {
        if (a.dtype == 1) {
            if (a.head_dim == 128) return launch_pdl(append_fp8_kernel<128, BF16Tag>, dim3(grid), dim3(kAppendThreads), 0, s, a);
            return launch_pdl(append_fp8_kernel<64, BF16Tag>, dim3(grid), dim3(kAppendThreads), 0, s, a);
        }
        if (a.head_dim == 128) return launch_pdl(append_fp8_kernel<128, F16Tag>, dim3(grid), dim3(kAppendThreads), 0, s, a);
        return launch_pdl(append_fp8_kernel<64, F16Tag>, dim3(grid), dim3(kAppendThreads), 0, s, a);
    }
    if (a.head_dim == 256) return launch_pdl(append_kernel<256>, dim3(grid), dim3(kAppendThreads), 0, s, a);
    if (a.head_dim == 128) return launch_pdl(append_kernel<128>, dim3(grid), dim3(kAppendThreads), 0, s, a);
    return launch_pdl(append_kernel<64>, dim3(grid), dim3(kAppendThreads), 0, s, a);
}

}  // namespace pkv
