// pkv_api.cu -- the C ABI of libpkv (declared in include/pkv.h): argument validation,
// launch configuration, workspace sizing, status codes and the device error word.
// No call here allocates device memory.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "pkv_internal.h"

namespace pkv {

// Sticky device error word (first range / timeout event wins); one per device context.
__device__ int g_device_error;

namespace {

// Per-device launch facts and the address of the device error word, filled once per device by
// the first call that finds the device usable. `ready` is stored with release order after the
// fields and loaded with acquire order, so a thread that sees it set also sees the fields.
struct DeviceSlot {
    std::atomic<bool> ready{false};
    DeviceInfo info{};
    int *err_ptr = nullptr;
};
constexpr int kMaxDevices = 64;
DeviceSlot g_slots[kMaxDevices];
std::mutex g_slot_lock;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }


int ilog2(int x) {
    int r = 0;
    while ((1 << r) < x) ++r;
    return r;
}

// The current device's slot, or nullptr when the device, its attributes or the address of its
// error word cannot be read. A failure is not cached: the next call tries again.
DeviceSlot *slot() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return nullptr;
    }
    DeviceSlot &s = g_slots[dev];
    if (s.ready.load(std::memory_order_acquire)) return &s;
    std::lock_guard<std::mutex> g(g_slot_lock);
    if (!s.ready.load(std::memory_order_relaxed)) {
        int sms = 0, smem = 0;
        void *p = nullptr;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess || p == nullptr || sms <= 0 || smem <= 0) {
            (void)cudaGetLastError();
            return nullptr;
        }
        s.info.device = dev;
        s.info.num_sms = sms;
        s.info.decode_ctas_per_sm = 1;
        s.info.max_smem = smem;
        s.err_ptr = static_cast<int *>(p);
        s.ready.store(true, std::memory_order_release);
    }
    return &s;
}

// Launch facts of a device that could not be queried: used only to size workspaces before any
// device is usable (the smallest split chunk, so the size is never too small).
const DeviceInfo kNoDevice = {-1, 1, 1, 48 * 1024};

pkv_status check_cache(const pkv_cache &c) {
    if (!c.ptr || !aligned16(c.ptr)) return PKV_ERR_INVALID_ARG;
    if (c.num_blocks < 0 || c.num_kv_heads <= 0 || c.block_size <= 0 || c.head_dim <= 0) return PKV_ERR_INVALID_ARG;
    if (c.format != PKV_KV_NATIVE && c.format != PKV_KV_FP8_E4M3) return PKV_ERR_UNSUPPORTED;
    if (c.format == PKV_KV_FP8_E4M3 && (!c.scales || !aligned16(c.scales))) return PKV_ERR_INVALID_ARG;
    if (c.dtype != PKV_F16 && c.dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (c.head_dim != 64 && c.head_dim != 128 && c.head_dim != 256) return PKV_ERR_UNSUPPORTED;
    if (c.format == PKV_KV_FP8_E4M3 && c.head_dim == 256) return PKV_ERR_UNSUPPORTED;
    if (!is_pow2(c.block_size) || c.block_size < 8 || c.block_size > 512) return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

pkv_status check_out_dtype(pkv_dtype out_dtype, pkv_dtype cache_dtype) {
    if (out_dtype != cache_dtype && out_dtype != PKV_F32) return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

CacheView view_of(const pkv_cache &c) {
    CacheView v;
    v.ptr = c.ptr;
    v.num_blocks = c.num_blocks;
    v.num_kv_heads = c.num_kv_heads;
    v.block_size = c.block_size;
    v.log2_block_size = ilog2(c.block_size);
    v.head_dim = c.head_dim;
    v.dtype = (int)c.dtype;
    v.fp8 = c.format == PKV_KV_FP8_E4M3 ? 1 : 0;
    v.scales = v.fp8 ? c.scales : nullptr;
    return v;
}

// Tokens per decode split.  Automatic: enough (sequence, KV head, split) units for about
// eight per CTA at full capacity, in [128, 512] tokens; explicit: capacity / num_splits
// rounded up to kSplitAlign (128, the tensor-core decode's key tile).  Either way at least
// capacity / kDecodeMaxSplits, rounded up, so that a full context has at most kDecodeMaxSplits
// splits.
int split_tokens(int batch, int num_kv_heads, int block_size, int max_blocks_per_seq, int num_splits) {
    const long long cap = (long long)max_blocks_per_seq * block_size;
    const long long tile = kSplitAlign;
    long long c;
    if (num_splits > 0) {
        c = (cap + num_splits - 1) / num_splits;
    } else {
        const DeviceSlot *s = slot();
        const DeviceInfo &d = s ? s->info : kNoDevice;
        const long long ctas = (long long)d.num_sms * d.decode_ctas_per_sm;
        const long long want = (long long)batch * num_kv_heads * cap / (ctas * 8 > 0 ? ctas * 8 : 1);
        // the largest of these at or below want (at least 128): 768-token splits measured best on
        // the streaming paths (7B-like, FP8 and mixed batches against 512, 640 and 1024)
        static const int kSizes[] = {768, 512, 384, 256, 128};
        int i = 0;
        while (kSizes[i] > 128 && kSizes[i] > want) ++i;
        c = kSizes[i];
    }
    const long long floor_c = (cap + kDecodeMaxSplits - 1) / kDecodeMaxSplits;
    if (c < floor_c) c = floor_c;
    c = (c + tile - 1) / tile * tile;
    return (int)(c < tile ? tile : c);
}

}  // namespace

const DeviceInfo &device_info() {
    const DeviceSlot *s = slot();
    return s ? s->info : kNoDevice;
}
int *device_error_word() {
    DeviceSlot *s = slot();
    return s ? s->err_ptr : nullptr;
}

}  // namespace pkv

using namespace pkv;

extern "C" {

int pkv_version(void) { return 101; }

const char *pkv_status_string(pkv_status s) {
    switch (s) {
        case PKV_OK: return "PKV_OK";
        case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
        case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
        case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE";
        case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
        case PKV_ERR_DEVICE_RANGE: return "PKV_ERR_DEVICE_RANGE";
        case PKV_ERR_TIMEOUT: return "PKV_ERR_TIMEOUT";
    }
    return "PKV_ERR_UNKNOWN";
}

pkv_status pkv_kv_cache_append(pkv_cache cache, const void *k_new, const void *v_new, const int *cu_new_lens,
                               const int *ctx_before, const int *block_tables, int batch, int max_blocks_per_seq,
                               int num_new_tokens, void *stream) {
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    if (batch < 0 || num_new_tokens < 0 || max_blocks_per_seq <= 0) return PKV_ERR_INVALID_ARG;
    if (batch == 0 || num_new_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !cu_new_lens || !ctx_before || !block_tables) return PKV_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new)) return PKV_ERR_INVALID_ARG;
    DeviceSlot *s = slot();
    if (!s) return PKV_ERR_CUDA;
    AppendArgs a;
    a.cache = cache.ptr;
    a.num_blocks = cache.num_blocks;
    a.num_kv_heads = cache.num_kv_heads;
    a.block_size = cache.block_size;
    a.log2_block_size = ilog2(cache.block_size);
    a.head_dim = cache.head_dim;
    a.dtype = (int)cache.dtype;
    a.fp8 = cache.format == PKV_KV_FP8_E4M3 ? 1 : 0;
    a.scales = a.fp8 ? cache.scales : nullptr;
    a.k_new = k_new;
    a.v_new = v_new;
    a.cu_new_lens = cu_new_lens;
    a.ctx_before = ctx_before;
    a.block_tables = block_tables;
    a.batch = batch;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_new_tokens = num_new_tokens;
    a.err = s->err_ptr;
    return launch_append(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int pkv_decode_split_tokens(int batch, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                            int max_blocks_per_seq, int num_splits) {
    (void)num_q_heads;
    (void)head_dim;
    if (batch <= 0 || num_kv_heads <= 0 || block_size <= 0 || max_blocks_per_seq <= 0) return kSplitAlign;
    return split_tokens(batch, num_kv_heads, block_size, max_blocks_per_seq, num_splits);
}

static size_t partial_bytes(int batch, int num_q_heads, long long s_max, int head_dim) {
    const size_t b = (size_t)batch * num_q_heads * s_max * (head_dim + 1) * sizeof(float);
    return (b + 15) & ~(size_t)15;
}

size_t pkv_decode_workspace_size(int batch, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                 int max_blocks_per_seq, int num_splits) {
    if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        max_blocks_per_seq <= 0)
        return 0;
    const long long cap = (long long)max_blocks_per_seq * block_size;
    const int chunk = split_tokens(batch, num_kv_heads, block_size, max_blocks_per_seq, num_splits);
    const long long s_max = (cap + chunk - 1) / chunk;
    if (s_max <= 1) return 0;
    // FP32 partials [batch, Hq, s_max, D] and their lse [batch, Hq, s_max], padded to 16 bytes, then
    // one 16-byte slot: the split size the split kernel took (read by the merge kernel)
    return partial_bytes(batch, num_q_heads, s_max, head_dim) + 16;
}

}  // extern "C"

namespace pkv {
namespace {

// The decode call; cu_q_lens != nullptr decodes only the single-row sequences of a mixed batch
// (their rows cu_q_lens[b]) and leaves the other rows untouched.
pkv_status decode_impl(const pkv_cache &cache, const void *q, int num_q_heads, const int *block_tables,
                       const int *context_lens, const int *cu_q_lens, int batch, int q_rows, int max_blocks_per_seq,
                       float scale, int num_splits, void *workspace, size_t workspace_bytes, void *out,
                       pkv_dtype out_dtype, float *lse, void *stream, const void *k_new = nullptr,
                       const void *v_new = nullptr) {
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    if ((st = check_out_dtype(out_dtype, cache.dtype)) != PKV_OK) return st;
    if (batch < 0 || max_blocks_per_seq <= 0 || num_q_heads <= 0 || num_splits < 0) return PKV_ERR_INVALID_ARG;
    if (num_q_heads % cache.num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    const int group = num_q_heads / cache.num_kv_heads;
    const bool fp8 = cache.format == PKV_KV_FP8_E4M3;
    // an FP8 cache: 1, 2, 4, or any multiple of 8 query heads per KV head (8 per unit; head_dim 64:
    // at most 8); a native cache: any group
    if (fp8 && group != 1 && group != 2 && group != 4 && group % 8 != 0) return PKV_ERR_UNSUPPORTED;
    if (fp8 && group > 8 && cache.head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (batch == 0) return PKV_OK;
    if (!q || !block_tables || !context_lens || !out) return PKV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || (lse && !aligned16(lse))) return PKV_ERR_INVALID_ARG;
    const long long cap = (long long)max_blocks_per_seq * cache.block_size;
    if (cap > (1ll << 30)) return PKV_ERR_UNSUPPORTED;
    DeviceSlot *s = slot();
    if (!s) return PKV_ERR_CUDA;
    const int chunk = split_tokens(batch, cache.num_kv_heads, cache.block_size, max_blocks_per_seq, num_splits);
    const int s_max = (int)((cap + chunk - 1) / chunk);
    const size_t need = pkv_decode_workspace_size(batch, num_q_heads, cache.num_kv_heads, cache.head_dim,
                                                  cache.block_size, max_blocks_per_seq, num_splits);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace))) return PKV_ERR_WORKSPACE;
    DecodeArgs a;
    a.cache = view_of(cache);
    a.q = q;
    a.num_q_heads = num_q_heads;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.batch = batch;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.scale = scale;
    a.chunk = chunk;
    a.chunk_out = need > 0 ? reinterpret_cast<int *>(static_cast<uint8_t *>(workspace) +
                                                     partial_bytes(batch, num_q_heads, s_max, cache.head_dim))
                           : nullptr;
    a.q_rows = q_rows;
    a.s_max = s_max;
    a.stages = 0;  // set by the group kernel's launcher
    // The kernel and the query heads of a unit (a KV head's group, or an equal share of it):
    //   FP8 cache: the FP8 kernels, at most 8 per unit;
    //   native cache, 1 or 2 heads per KV head: CUDA cores (decode.cu), the group as one unit;
    //   4 or 8: mma.sync units of the whole group (decode_gqa.cu);
    //   any other group: tcgen05 units (decode_tc.cu) of the group, or, above 128 heads, of its
    //   largest divisor up to 128.
    enum { kCudaCores, kMmaSync, kTcgen05, kFp8Tensor } path;
    int per_unit;
    if (fp8) {
        path = cache.head_dim == 128 ? kFp8Tensor : kCudaCores;
        per_unit = group < 8 ? group : 8;
    } else if (group <= 2 && cache.head_dim <= 128) {
        path = kCudaCores;
        per_unit = group;
    } else if ((group == 4 || group == 8) && cache.head_dim <= 128) {
        path = kMmaSync;
        per_unit = group;
    } else {
        path = kTcgen05;
        per_unit = group;
        for (int d = 128; per_unit > 128; --d)
            if (group % d == 0) per_unit = d;
    }
    a.head_groups = group / per_unit;
    // The tcgen05 units (many query heads each) run below the memory roofline, so how evenly the
    // units divide over the CTAs sets their time: with an automatic split the kernel picks the split
    // size from the lengths (decode_scan_units). The other paths stream at the copy rate, where the
    // host's split measured best; a requested split count is kept as given.
    a.auto_chunk = (num_splits == 0 && path == kTcgen05) ? 1 : 0;
    a.cu_q_lens = cu_q_lens;
    a.part_o = static_cast<float *>(workspace);
    a.part_lse = need > 0 ? a.part_o + (size_t)batch * num_q_heads * s_max * cache.head_dim : nullptr;
    a.out = out;
    a.out_dtype = (int)out_dtype;
    a.lse = lse;
    a.err = s->err_ptr;
    // a decode step's append goes with the kernels that have a merge warp (16-bit cache, CUDA-core
    // and mma.sync paths); the others get the append kernel after the decode
    const bool fused_append = k_new && !fp8 && path != kTcgen05;
    a.k_new = fused_append ? k_new : nullptr;
    a.v_new = fused_append ? v_new : nullptr;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const int grid = s->info.num_sms * s->info.decode_ctas_per_sm;
    // The kernels keep a launch's unit tables in shared memory, so a batch runs in slices of at
    // most decode_max_batch() sequences, each a decode of its own (the split size and the
    // workspace layout [batch, Hq, s_max, ...] are the whole batch's; a slice's partials start at
    // its first sequence's). A mixed batch's rows are absolute (cu_q_lens), so only cu_q_lens moves.
    const size_t qe = 2, oe = out_dtype == PKV_F32 ? 4 : 2;  // element sizes of q and out
    // sequences a launch: at most decode_max_batch(), and unit tables (3 ints a sequence, 2 a split, 8 more)
    // of at most 24 KB, which every decode kernel's shared-memory layout leaves room for
    int slice = (6144 - 2 * (s_max + 1) - kUnitMisc) / 3;
    slice = slice < 1 ? 1 : (slice > decode_max_batch() ? decode_max_batch() : slice);
    for (int b0 = 0; b0 < batch; b0 += slice) {
        const int nb = batch - b0 < slice ? batch - b0 : slice;
        DecodeArgs d = a;
        d.batch = nb;
        d.block_tables = block_tables + (size_t)b0 * max_blocks_per_seq;
        d.context_lens = context_lens + b0;
        if (cu_q_lens) {
            d.cu_q_lens = cu_q_lens + b0;
        } else {
            d.q = static_cast<const uint8_t *>(q) + (size_t)b0 * num_q_heads * cache.head_dim * qe;
            d.q_rows = nb;
            d.out = static_cast<uint8_t *>(out) + (size_t)b0 * num_q_heads * cache.head_dim * oe;
            d.lse = lse ? lse + (size_t)b0 * num_q_heads : nullptr;
        }
        if (need > 0) {
            d.part_o = a.part_o + (size_t)b0 * num_q_heads * s_max * cache.head_dim;
            d.part_lse = a.part_lse + (size_t)b0 * num_q_heads * s_max;
        }
        if (fused_append) {
            const size_t row_bytes = (size_t)cache.num_kv_heads * cache.head_dim * 2;
            d.k_new = static_cast<const uint8_t *>(k_new) + (size_t)b0 * row_bytes;
            d.v_new = static_cast<const uint8_t *>(v_new) + (size_t)b0 * row_bytes;
        }
        cudaError_t le;
        switch (path) {
            case kFp8Tensor: le = launch_decode_fp8(d, grid, cs); break;
            case kMmaSync: le = launch_decode_gqa(d, grid, cs); break;
            case kTcgen05: le = launch_decode_tc(d, grid, cs); break;
            default: le = launch_decode(d, grid, cs); break;
        }
        if (le != cudaSuccess) return PKV_ERR_CUDA;
        // Rows that span several splits (and empty rows) are finished by the merge.
        CombineArgs c;
        c.part_o = d.part_o;
        c.part_lse = d.part_lse;
        c.n_rows = nb * num_q_heads;
        c.num_splits = s_max;
        c.head_dim = cache.head_dim;
        c.context_lens = d.context_lens;
        c.rows_per_seq = num_q_heads;
        c.chunk = chunk;
        c.chunk_dev = a.auto_chunk ? a.chunk_out : nullptr;  // the kernel's own choice, else chunk
        c.cu_q_lens = d.cu_q_lens;
        c.out = d.out;
        c.out_dtype = (int)out_dtype;
        c.lse = d.lse;
        if (launch_combine(c, cs) != cudaSuccess) return PKV_ERR_CUDA;
    }
    if (k_new && !fused_append) {
        AppendArgs ap;
        ap.cache = const_cast<void *>(cache.ptr);
        ap.num_blocks = cache.num_blocks;
        ap.num_kv_heads = cache.num_kv_heads;
        ap.block_size = cache.block_size;
        ap.log2_block_size = ilog2(cache.block_size);
        ap.head_dim = cache.head_dim;
        ap.dtype = (int)cache.dtype;
        ap.fp8 = fp8 ? 1 : 0;
        ap.scales = fp8 ? cache.scales : nullptr;
        ap.k_new = k_new;
        ap.v_new = v_new;
        ap.cu_new_lens = nullptr;  // one token per sequence, at position context_lens[b]
        ap.ctx_before = context_lens;
        ap.block_tables = block_tables;
        ap.batch = batch;
        ap.max_blocks_per_seq = max_blocks_per_seq;
        ap.num_new_tokens = batch;
        ap.err = s->err_ptr;
        if (launch_append(ap, cs) != cudaSuccess) return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" {

pkv_status pkv_paged_attn_decode(pkv_cache cache, const void *q, int num_q_heads, const int *block_tables,
                                 const int *context_lens, int batch, int max_blocks_per_seq, float scale,
                                 int num_splits, void *workspace, size_t workspace_bytes, void *out,
                                 pkv_dtype out_dtype, float *lse, void *stream) {
    return decode_impl(cache, q, num_q_heads, block_tables, context_lens, nullptr, batch, batch, max_blocks_per_seq,
                       scale, num_splits, workspace, workspace_bytes, out, out_dtype, lse, stream);
}

pkv_status pkv_paged_attn_decode_step(pkv_cache cache, const void *q, int num_q_heads, const int *block_tables,
                                      const int *context_lens, int batch, int max_blocks_per_seq, float scale,
                                      int num_splits, void *workspace, size_t workspace_bytes, void *out,
                                      pkv_dtype out_dtype, float *lse, const void *k_new, const void *v_new,
                                      void *stream) {
    if (batch > 0 && (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))) return PKV_ERR_INVALID_ARG;
    return decode_impl(cache, q, num_q_heads, block_tables, context_lens, nullptr, batch, batch, max_blocks_per_seq,
                       scale, num_splits, workspace, workspace_bytes, out, out_dtype, lse, stream, k_new, v_new);
}

pkv_status pkv_attn_combine(const float *partial_o, const float *partial_lse, int n_rows, int num_splits,
                            int head_dim, void *out, pkv_dtype out_dtype, float *lse, void *stream) {
    if (n_rows < 0 || num_splits <= 0) return PKV_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return PKV_ERR_UNSUPPORTED;
    if (out_dtype != PKV_F16 && out_dtype != PKV_BF16 && out_dtype != PKV_F32) return PKV_ERR_UNSUPPORTED;
    if (n_rows == 0) return PKV_OK;
    if (!partial_o || !partial_lse || !out) return PKV_ERR_INVALID_ARG;
    if (!aligned16(partial_o) || !aligned16(out)) return PKV_ERR_INVALID_ARG;
    if (!slot()) return PKV_ERR_CUDA;
    CombineArgs c;
    c.part_o = partial_o;
    c.part_lse = partial_lse;
    c.n_rows = n_rows;
    c.num_splits = num_splits;
    c.head_dim = head_dim;
    c.context_lens = nullptr;
    c.cu_q_lens = nullptr;
    c.rows_per_seq = 1;
    c.chunk = 1;
    c.chunk_dev = nullptr;
    c.out = out;
    c.out_dtype = (int)out_dtype;
    c.lse = lse;
    return launch_combine(c, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // extern "C"

namespace pkv {
namespace {

// The prefill call; skip_single leaves the single-row sequences of a mixed batch to the decode.
pkv_status prefill_impl(const pkv_cache &cache, const void *q, int num_q_heads, const int *cu_q_lens,
                        const int *context_lens, const int *block_tables, int batch, int max_blocks_per_seq,
                        int total_q, int max_q_len, float scale, int causal, void *out, pkv_dtype out_dtype,
                        float *lse, void *stream, int skip_single) {
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    if ((st = check_out_dtype(out_dtype, cache.dtype)) != PKV_OK) return st;
    if (batch < 0 || max_blocks_per_seq <= 0 || num_q_heads <= 0 || total_q < 0 || max_q_len < 0)
        return PKV_ERR_INVALID_ARG;
    if (num_q_heads % cache.num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    if (batch == 0 || total_q == 0) return PKV_OK;
    if (!q || !cu_q_lens || !context_lens || !block_tables || !out) return PKV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || (lse && !aligned16(lse))) return PKV_ERR_INVALID_ARG;
    const long long cap = (long long)max_blocks_per_seq * cache.block_size;
    if (cap > (1ll << 30)) return PKV_ERR_UNSUPPORTED;
    // grid (heads, sequences, row blocks of 256 rows, 128 at head_dim 256): the last two dimensions
    // hold at most 65535
    const int block_rows = cache.head_dim == 256 ? 128 : 256;
    if (batch > 65535 || ((long long)max_q_len + block_rows - 1) / block_rows > 65535) return PKV_ERR_UNSUPPORTED;
    DeviceSlot *s = slot();
    if (!s) return PKV_ERR_CUDA;
    PrefillArgs a;
    a.cache = view_of(cache);
    a.q = q;
    a.num_q_heads = num_q_heads;
    a.cu_q_lens = cu_q_lens;
    a.context_lens = context_lens;
    a.block_tables = block_tables;
    a.batch = batch;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.total_q = total_q;
    a.max_q_len = max_q_len;
    a.scale = scale;
    a.causal = causal ? 1 : 0;
    a.skip_single = skip_single;
    a.out = out;
    a.out_dtype = (int)out_dtype;
    a.lse = lse;
    a.err = s->err_ptr;
    cudaError_t e = launch_prefill(a, static_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return PKV_ERR_UNSUPPORTED;
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace
}  // namespace pkv

extern "C" {

pkv_status pkv_paged_attn_prefill(pkv_cache cache, const void *q, int num_q_heads, const int *cu_q_lens,
                                  const int *context_lens, const int *block_tables, int batch,
                                  int max_blocks_per_seq, int total_q, int max_q_len, float scale, int causal,
                                  void *out, pkv_dtype out_dtype, float *lse, void *stream) {
    return prefill_impl(cache, q, num_q_heads, cu_q_lens, context_lens, block_tables, batch, max_blocks_per_seq,
                        total_q, max_q_len, scale, causal, out, out_dtype, lse, stream, 0);
}

pkv_status pkv_paged_attn_mixed(pkv_cache cache, const void *q, int num_q_heads, const int *cu_q_lens,
                                const int *context_lens, const int *block_tables, int batch, int max_blocks_per_seq,
                                int total_q, int max_q_len, float scale, int causal, int num_splits, void *workspace,
                                size_t workspace_bytes, void *out, pkv_dtype out_dtype, float *lse, void *stream) {
    if (!cu_q_lens && batch > 0) return PKV_ERR_INVALID_ARG;
    // decode rows first (split kernel + merge), then the prefill chunks; each kernel leaves the
    // other kind's rows alone
    if (total_q < 0) return PKV_ERR_INVALID_ARG;
    pkv_status st = decode_impl(cache, q, num_q_heads, block_tables, context_lens, cu_q_lens, batch, total_q,
                                max_blocks_per_seq, scale, num_splits, workspace, workspace_bytes, out, out_dtype,
                                lse, stream);
    if (st != PKV_OK) return st;
    return prefill_impl(cache, q, num_q_heads, cu_q_lens, context_lens, block_tables, batch, max_blocks_per_seq,
                        total_q, max_q_len, scale, causal, out, out_dtype, lse, stream, 1);
}

pkv_status pkv_get_device_error(void *stream, int *code) {
    if (!code) return PKV_ERR_INVALID_ARG;
    *code = PKV_OK;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return PKV_ERR_CUDA;
    DeviceSlot *s = slot();
    if (!s) return PKV_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, s->err_ptr, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return PKV_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpy(s->err_ptr, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return PKV_ERR_CUDA;
    }
    *code = v;
    return PKV_OK;
}

}  // extern "C"
