// pkv_device.cuh -- device helpers shared by the libpkv kernels (sm_103a):
// mbarrier and bulk-copy (TMA engine) wrappers in inline PTX, bounded waits
// that report a timeout instead of hanging, the sticky device error word, and
// fp16 / bf16 <-> fp32 conversions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <string.h>

namespace pkv {

// Codes written into the device error word (same values as pkv_status).
constexpr int kErrDeviceRange = 5;
constexpr int kErrTimeout = 6;

// A bounded wait gives up after this many nanoseconds of %globaltimer.
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;

__device__ __forceinline__ void set_error(int *err, int code) {
    if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- mbarrier -----------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for phase `parity` of `bar` to complete.  Gives up (returns false) when
// *abort becomes non-zero or after timeout_ns (default kWaitTimeoutNs), in which case it
// records kErrTimeout and raises *abort so the CTA's other roles stop too.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort, int *err,
                                          unsigned long long timeout_ns = kWaitTimeoutNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 63u) == 0) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > timeout_ns) {
                set_error(err, kErrTimeout);
                *abort = 1;
                return false;
            }
        }
    }
}

// ---- bulk copies (non-tensor TMA): global -> shared, completion on an mbarrier -------------
// Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_addr(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Programmatic dependent launch. A kernel launched with programmatic stream serialization may
// start while the previous kernel on its stream drains: before pdl_wait() it touches only its
// kernel parameters and its own shared memory (any global input may have been written by the
// previous kernel, the caller's included); pdl_wait() returns once the previous kernel has
// completed and its writes are visible. pdl_launch_dependents() lets the next such kernel start
// launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Named barrier among `nthreads` threads (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_barrier(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---- element types --------------------------------------------------------------------------
struct F16Tag {
    using T = __half;
};
struct BF16Tag {
    using T = __nv_bfloat16;
};

// Eight packed 16-bit values (one 16-byte vector) to fp32.
__device__ __forceinline__ void unpack8(const uint4 &raw, float (&f)[8], F16Tag) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h;
        memcpy(&h, &w[i], 4);
        const float2 x = __half22float2(h);
        f[2 * i] = x.x;
        f[2 * i + 1] = x.y;
    }
}

__device__ __forceinline__ void unpack8(const uint4 &raw, float (&f)[8], BF16Tag) {
    // bf16 is the upper half of an fp32: the conversion is a shift / mask.
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Eight packed 16-bit values to four fp32 pairs (element 2i in .x, 2i+1 in .y).
__device__ __forceinline__ void unpack8x2(const uint4 &raw, float2 (&f)[4], F16Tag) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h;
        memcpy(&h, &w[i], 4);
        f[i] = __half22float2(h);
    }
}

__device__ __forceinline__ void unpack8x2(const uint4 &raw, float2 (&f)[4], BF16Tag) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
}

// OCP FP8 E4M3 codes, one byte per element, in increasing element order. Eight codes (one
// 8-byte load) to four fp32 pairs: every E4M3 value is exact in fp16, and fp16 in fp32.
__device__ __forceinline__ void unpack_e4m3x8(const uint2 &raw, float2 (&f)[4]) {
    const uint32_t w[2] = {raw.x, raw.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        uint32_t lo, hi;
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"((unsigned short)(w[i] & 0xffffu)));
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"((unsigned short)(w[i] >> 16)));
        __half2 h0, h1;
        memcpy(&h0, &lo, 4);
        memcpy(&h1, &hi, 4);
        f[2 * i] = __half22float2(h0);
        f[2 * i + 1] = __half22float2(h1);
    }
}

// Two fp32 values to two E4M3 codes (round to nearest even, magnitudes beyond 448 saturated);
// x0 goes to the low byte.
__device__ __forceinline__ uint32_t pack_e4m3x2(float x0, float x1) {
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(x1), "f"(x0));
    return r;
}

// Paired FP32 arithmetic of sm_100-class GPUs (one instruction for two lanes of a float2).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rc, ra, rb, rc;\n\tmov.b64 {%0, %1}, rc;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 ra, ra, rb;\n\tmov.b64 {%0, %1}, ra;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 ra, ra, rb;\n\tmov.b64 {%0, %1}, ra;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 fsub2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 ra, ra, rb;\n\tmov.b64 {%0, %1}, ra;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Output element store with a single round-to-nearest-even conversion.
// out_dtype: 0 = fp16, 1 = bf16, 2 = fp32.
__device__ __forceinline__ void store_out(void *out, size_t idx, float v, int out_dtype) {
    if (out_dtype == 2) {
        static_cast<float *>(out)[idx] = v;
    } else if (out_dtype == 1) {
        static_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(v);
    } else {
        static_cast<__half *>(out)[idx] = __float2half_rn(v);
    }
}

// V (2, 4 or 8) consecutive outputs from element idx on (idx a multiple of V, the base 16-byte
// aligned): vector stores (one; two for 8 FP32 values), rounded as store_out rounds each value.
template <int V>
__device__ __forceinline__ void store_out_vec(void *out, size_t idx, const float (&v)[V], int out_dtype) {
    static_assert(V == 2 || V == 4 || V == 8, "vectors of 2, 4 or 8");
    if constexpr (V == 8) {
        if (out_dtype == 2) {
            float *o = static_cast<float *>(out) + idx;
            *reinterpret_cast<float4 *>(o) = make_float4(v[0], v[1], v[2], v[3]);
            *reinterpret_cast<float4 *>(o + 4) = make_float4(v[4], v[5], v[6], v[7]);
            return;
        }
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (out_dtype == 1) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
                memcpy(&w[i], &h, 4);
            } else {
                const __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
                memcpy(&w[i], &h, 4);
            }
        }
        *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + idx) = make_uint4(w[0], w[1], w[2], w[3]);
        return;
    } else {
    if (out_dtype == 2) {
        float *o = static_cast<float *>(out) + idx;
        if constexpr (V == 4) *reinterpret_cast<float4 *>(o) = make_float4(v[0], v[1], v[2], v[3]);
        else *reinterpret_cast<float2 *>(o) = make_float2(v[0], v[1]);
        return;
    }
    uint32_t w[V / 2];
#pragma unroll
    for (int i = 0; i < V / 2; ++i) {
        if (out_dtype == 1) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            memcpy(&w[i], &h, 4);
        } else {
            const __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
            memcpy(&w[i], &h, 4);
        }
    }
    uint16_t *o = static_cast<uint16_t *>(out) + idx;
    if constexpr (V == 4) *reinterpret_cast<uint2 *>(o) = make_uint2(w[0], w[1]);
    else *reinterpret_cast<uint32_t *>(o) = w[0];
    }
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

}  // namespace pkv
