// pkv_internal.h -- host-side launcher interface between the C ABI (pkv_api.cu)
// and the kernel translation units.  Arguments arrive here already validated.
#pragma once

#include <atomic>
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/pkv.h"

namespace pkv {

struct CacheView {
    const void *ptr;
    int num_blocks, num_kv_heads, block_size, log2_block_size, head_dim;
    int dtype;  // 0 fp16, 1 bf16: q / k_new / v_new, and the elements of a native cache
    int fp8;    // 1: ptr holds E4M3 codes and `scales` one FP32 scale per row
    const float *scales;
};

struct AppendArgs {
    void *cache;
    int num_blocks, num_kv_heads, block_size, log2_block_size, head_dim;
    int dtype;      // type of k_new / v_new
    int fp8;        // 1: quantise into E4M3 codes + per-row scales
    float *scales;
    const void *k_new, *v_new;
    // cu_new_lens nullptr: one new token per sequence (a decode step), token t being sequence t's
    const int *cu_new_lens, *ctx_before, *block_tables;
    int batch, max_blocks_per_seq, num_new_tokens;
    int *err;
};

struct DecodeArgs {
    CacheView cache;
    const void *q;
    int num_q_heads;
    const int *block_tables, *context_lens;
    int batch, max_blocks_per_seq;
    float scale;
    int chunk;   // tokens per split (multiple of the decode tile); with auto_chunk the smallest
    int auto_chunk;  // 1: the kernel may take 1.5 - 4 times chunk (decode_scan_units), 0: chunk
    int *chunk_out;  // where CTA 0 stores the split size it took (for the merge kernel), or nullptr
    // Units per KV head when a KV head serves more query heads than one unit holds (the native
    // group kernel holds 32 (head_dim 128), 16 or 8, the largest that divides the group; the FP8
    // kernel 8; MQA, wide groups), else 1:
    // unit head v reads KV head v / head_groups and serves query heads n*v .. n*v + n-1.
    int head_groups;
    // Mixed batch (prefill chunks and decode rows in one call): cu_q_lens [batch + 1] of the call's
    // q / out rows; only sequences with exactly one query row are decoded here, their row being
    // cu_q_lens[b]. nullptr: every sequence has one query row, row b.
    const int *cu_q_lens;
    int q_rows;  // rows of q (and of out): batch, or the mixed call's total query rows
    int s_max;   // splits a full-capacity context uses: ceil(max_blocks_per_seq * block_size / chunk)
    int stages;  // pipeline stages of the group kernel (chosen at launch from the shared memory left)
    float *part_o;    // [batch, Hq, s_max, D]
    float *part_lse;  // [batch, Hq, s_max]
    void *out;
    int out_dtype;
    float *lse;
    int *err;
    // Decode step on the kernels with a merge warp (a native cache on the CUDA-core and mma.sync
    // paths): the new token's K and V rows [batch, Hkv, D], which the merge warps write at
    // position context_lens[b] of each sequence before their first unit. nullptr: no append.
    const void *k_new, *v_new;
};

struct CombineArgs {
    const float *part_o, *part_lse;
    int n_rows, num_splits, head_dim;
    // When context_lens is set, row r = b * rows_per_seq + h uses ceil(len_b / chunk)
    // splits; rows with exactly one split were finished by the decode kernel.
    const int *context_lens;
    int rows_per_seq, chunk;
    const int *chunk_dev;  // the split size the split kernel chose (read after it completes), or nullptr: chunk
    // mixed batch: row r = b * rows_per_seq + h goes to output row cu_q_lens[b] * rows_per_seq + h,
    // and only for sequences with exactly one query row (nullptr: output row r)
    const int *cu_q_lens;
    void *out;
    int out_dtype;
    float *lse;
};

struct PrefillArgs {
    CacheView cache;
    const void *q;
    int num_q_heads;
    const int *cu_q_lens, *context_lens, *block_tables;
    int batch, max_blocks_per_seq, total_q, max_q_len;
    float scale;
    int causal;
    int skip_single;  // mixed batch: sequences with one query row are the decode's
    void *out;
    int out_dtype;
    float *lse;
    int *err;
};

// Launch with programmatic stream serialization (the kernel calls pdl_wait() before touching
// memory the previous kernel may write).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// Opt a kernel in to `max_dynamic_smem` bytes of dynamic shared memory and to the largest shared
// memory carve-out of the L1 / shared array, so that as many of its CTAs as the shared memory allows
// are resident on an SM (the decode kernels that run two CTAs an SM rely on it).
template <typename K>
inline cudaError_t set_smem_attributes(K *kern, int max_dynamic_smem) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, max_dynamic_smem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
}

// Per-device facts cached on first use.
struct DeviceInfo {
    int device;
    int num_sms;
    int decode_ctas_per_sm;
    int max_smem;  // dynamic shared memory a CTA may opt in to (bytes)
};
const DeviceInfo &device_info();

// Once-per-device flags (devices 0..63) for a launcher's one-time cudaFuncSetAttribute opt-in.
// Setting the attribute twice is harmless, so threads that race on a first launch may both set
// it; the flags are atomic so that the race is not a data race.
struct DeviceFlags {
    std::atomic<unsigned long long> bits{0};
    bool test(int dev) const {
        return dev >= 0 && dev < 64 && ((bits.load(std::memory_order_acquire) >> dev) & 1ull) != 0;
    }
    void set(int dev) {
        if (dev >= 0 && dev < 64) bits.fetch_or(1ull << dev, std::memory_order_release);
    }
};
int *device_error_word();  // the current device's sticky error word (device address)

constexpr int kDecodeTile = 64;         // tokens per decode pipeline stage
constexpr int kSplitAlign = 128;        // decode splits start at multiples of this many tokens
constexpr int kDecodeMaxSplits = 2048;  // splits of one context (bounds the split size from below)
constexpr int kUnitMisc = 8;           // ints of a decode CTA's unit table beyond its per-sequence and per-split parts

cudaError_t launch_append(const AppendArgs &a, cudaStream_t s);
cudaError_t encode_cache_map(const CacheView &c, int box_rows, CUtensorMap *map);
// As encode_kv5_map with whole rows of D elements per box row and no swizzle (the CUDA-core
// decode reads plain rows).
cudaError_t encode_kv5_rows_map(const CacheView &c, int box_rows, CUtensorMap *map);
cudaError_t encode_kv5_map(const CacheView &c, int box_rows, CUtensorMap *map);
cudaError_t encode_fp8_maps(const CacheView &c, int box_rows, CUtensorMap *codes, CUtensorMap *scales);
// 2-D tensor map over `rows` rows of `cols` 16-bit elements (bf16 if bf16 != 0, else f16), rows
// contiguous; boxes of box_cols x box_rows, 128-byte swizzle (box_cols * 2 = 128).
cudaError_t encode_rows_map(const void *ptr, int bf16, long long rows, int cols, int box_cols, int box_rows,
                            CUtensorMap *map);
cudaError_t launch_decode_gqa(const DecodeArgs &a, int grid, cudaStream_t s);
// Tensor-core (tcgen05) decode for a unit of up to 128 query heads of one KV head.
cudaError_t launch_decode_tc(const DecodeArgs &a, int grid, cudaStream_t s);
cudaError_t launch_decode_fp8(const DecodeArgs &a, int grid, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs &a, int grid, cudaStream_t s);
cudaError_t launch_combine(const CombineArgs &a, cudaStream_t s);
cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t s);
// head_dim 256 (prefill_wide.cu): one 128-row query tile a CTA, 64-key tiles
cudaError_t launch_prefill_wide(const PrefillArgs &a, cudaStream_t s);
// q [total_q, Hq, D] as a 3-D tensor map (d, head, token), boxes of 64 columns x 1 head x box_rows
// tokens, 128-byte swizzle
cudaError_t encode_q_heads_map(const void *q, int bf16, int total_q, int num_q_heads, int head_dim, int box_rows,
                               CUtensorMap *map);
int decode_ctas_per_sm(int head_dim, int group, int dtype);
int decode_max_batch();

}  // namespace pkv
