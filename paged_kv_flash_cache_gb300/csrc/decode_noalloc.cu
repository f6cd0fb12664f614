// decode_noalloc.cu -- pkv_paged_attn_decode_noalloc: paged decode attention that needs no
// caller-provided workspace and allocates nothing.
//
// Who needs it: some callers cannot call cudaMalloc. A plugin invoked through a host
// framework's interface may be handed only its input and output buffers, with no workspace
// argument and no allocator to ask; a serving runtime may reserve all device memory up front in
// its own pool, so an extra cudaMalloc would fail or fragment what it planned. For them this
// entry point keeps the split-KV partial results in a fixed-size array that the library itself
// holds in device memory.
//
// How: the array below is a file-scope __device__ variable, so every GPU that loads this
// library reserves it (once its module is loaded) until the process exits. Host code cannot
// use the array's name as a device address -- on the host that name is only a stand-in -- so on
// the first call on each device (with that device current) cudaGetSymbolAddress fetches the
// real address, which is kept per device once the lookup succeeds and passed to the kernels.
// The rest is the regular decode path (pkv_paged_attn_decode) unchanged, with this array as its
// workspace.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "pkv_internal.h"

namespace pkv {
namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[PKV_DECODE_NOALLOC_SCRATCH_BYTES];

// The array's device address on each device, once looked up (nullptr: not yet). Only a
// successful lookup is kept; a failed one (made during a stream capture, say) is retried by the
// next call.
constexpr int kMaxDevices = 64;
std::atomic<void *> g_scratch[kMaxDevices];
std::mutex g_scratch_lock;

// Device address of g_decode_scratch on the current device.
cudaError_t scratch_address(void **out) {
    *out = nullptr;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void *p = g_scratch[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        std::lock_guard<std::mutex> g(g_scratch_lock);
        p = g_scratch[dev].load(std::memory_order_relaxed);
        if (p == nullptr) {
            e = cudaGetSymbolAddress(&p, g_decode_scratch);
            if (e != cudaSuccess || p == nullptr) {
                (void)cudaGetLastError();  // leave no error behind for the caller's next check
                return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
            }
            g_scratch[dev].store(p, std::memory_order_release);
        }
    }
    *out = p;
    return cudaSuccess;
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_paged_attn_decode_noalloc(pkv_cache cache, const void *q, int num_q_heads,
                                                    const int *block_tables, const int *context_lens, int batch,
                                                    int max_blocks_per_seq, float scale, int num_splits, void *out,
                                                    pkv_dtype out_dtype, float *lse, void *stream) {
    const size_t need = pkv_decode_workspace_size(batch, num_q_heads, cache.num_kv_heads, cache.head_dim,
                                                  cache.block_size, max_blocks_per_seq, num_splits);
    if (need > (size_t)PKV_DECODE_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (pkv::scratch_address(&scratch) != cudaSuccess || scratch == nullptr) return PKV_ERR_CUDA;
    return pkv_paged_attn_decode(cache, q, num_q_heads, block_tables, context_lens, batch, max_blocks_per_seq, scale,
                                 num_splits, scratch, (size_t)PKV_DECODE_NOALLOC_SCRATCH_BYTES, out, out_dtype, lse,
                                 stream);
}
