// decode_common.cuh -- pieces shared by the split-KV decode kernels: the work-unit cursor and
// the prologue that numbers the units from the context lengths.
#pragma once

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

struct UnitCursor {
    int b, kvh, split, t0, t1;
};

// Unit u -> (b, kv head, split); prefix[b] = units of sequences < b, units ordered with the KV
// head fastest so consecutive CTAs share block-table rows.
__device__ __forceinline__ UnitCursor unit_of(int u, const int *prefix, const int *lens, int batch, int hkv,
                                              int chunk) {
    int lo = 0, hi = batch;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= u) lo = mid; else hi = mid;
    }
    UnitCursor c;
    c.b = lo;
    const int r = u - prefix[lo];
    c.kvh = r % hkv;
    c.split = r / hkv;
    c.t0 = c.split * chunk;
    const int end = c.t0 + chunk;
    c.t1 = end < lens[lo] ? end : lens[lo];
    return c;
}

// Clamp the context lengths into shared memory (flagging out-of-range ones), and write the
// exclusive prefix of units per sequence (ceil(len / chunk) splits x KV heads) to prefix[0..batch];
// prefix[batch] is the total. All kThreads threads of the CTA take part; ends with __syncthreads.
template <int kThreads>
__device__ __forceinline__ void decode_scan_units(const DecodeArgs &a, int *lens, int *prefix, int *scan_tmp) {
    constexpr int kDecodeThreads = kThreads;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hkv = a.cache.num_kv_heads, chunk = a.chunk;
    const int cap = a.max_blocks_per_seq * a.cache.block_size;
    const int per = (a.batch + kDecodeThreads - 1) / kDecodeThreads;
    const int i0 = tid * per;
    int local = 0;
    for (int i = i0; i < i0 + per && i < a.batch; ++i) {
        int len = __ldg(a.context_lens + i);
        if (len < 0 || len > cap) {
            set_error(a.err, kErrDeviceRange);
            len = len < 0 ? 0 : cap;
        }
        lens[i] = len;
        local += ((len + chunk - 1) / chunk) * hkv;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) scan_tmp[warp] = incl;
    __syncthreads();
    int warp_base = 0;
    for (int w = 0; w < warp; ++w) warp_base += scan_tmp[w];
    int run = warp_base + incl - local;
    for (int i = i0; i < i0 + per && i < a.batch; ++i) {
        prefix[i] = run;
        run += ((lens[i] + chunk - 1) / chunk) * hkv;
    }
    if (tid == kDecodeThreads - 1) prefix[a.batch] = warp_base + incl;
    __syncthreads();
}

}  // namespace pkv
