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
// CTA = one query head x 256 query rows of one sequence, as two 128-row tiles A and B that share
// every K/V tile (384 threads, three warpgroups). Over an FP8 cache (head_dim 128) the E4M3 codes
// are converted in place to f16 (exactly, as code * 2^-8, on the integer pipe): K tiles by warps
// 2-3, V tiles by the softmax warps between key tiles; the products run in f16; the
// softmax multiplies each score column by its K row scale and each P column by its V row scale
// over W (a power of two warp 2 keeps at or above every V scale so far; O carries the factor W);
// otherwise as below:
//   warp 0     TMA producer: both Q tiles once (3-D tensor map over [total_q, Hq, D]); then for
//              each 128-key tile j the K tile and the V tile, each into one slot of a 4-slot ring:
//              the pages a tile covers are looked up in the block table by the warp's lanes and each
//              lane issues its page's boxes (2-D tensor map over the cache viewed as rows of D
//              elements, 128-byte swizzle);
//   warp 1     TMEM owner and MMA issuer (one thread). TMEM columns: S_A [0,128), S_B [128,256),
//              O_A [256,256+D), O_B [384,384+D); P_x is written over the first 64 columns of S_x.
//              Ping-pong issue order per key tile j: O_A += P_A V_j, S_A = Q_A K_{j+1}^T,
//              O_B += P_B V_j, S_B = Q_B K_{j+1}^T, so one tile's softmax overlaps the other tile's
//              MMAs; P is the A operand straight from TMEM, so only K and V come from shared memory;
//   WG 1, 2    softmax of tile A / tile B, one query row per thread (TMEM lane = row): scale,
//              causal / context masks, running max (O rescaled in TMEM only when the max grows by
//              more than 2^8; the final O / l uses the same max, so the result is exact), exp2, row
//              sum, P in the input dtype written to TMEM; epilogue O / l -> out, lse.
// Warpgroup 0 gives registers to the two softmax warpgroups (setmaxnreg).
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "prefill_common.cuh"
#include "tcgen05.cuh"

namespace pkv {
namespace {

constexpr int kBM = 128;       // query rows per tile
constexpr int kRows = 256;     // query rows per CTA (tiles A and B)
constexpr int kBN = 128;       // keys per KV tile
constexpr int kRing = 4;       // K/V ring slots
constexpr int kThreads = 384;  // 3 warpgroups
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when the max grows by more than 2^8
// TMEM columns: S_A (and P_A over its first 64 columns) [0,128), S_B / P_B [128,256),
// O_A [256,384), O_B [384,512).
constexpr uint32_t kColS = 0, kColO = 256;

template <int D, bool FP8 = false>
struct PrefillLayout {
    static constexpr int kHalves = D / 64;                      // 128-byte swizzle atoms along D
    static constexpr uint32_t kTileHalf = 128 * 128;            // 128 rows x 128 bytes
    static constexpr uint32_t kQBytes = kHalves * kTileHalf;    // one 128-row Q tile
    static constexpr uint32_t kKVBytes = kHalves * kTileHalf;   // one K or V tile
    static constexpr uint32_t kQOff = 0;
    static constexpr uint32_t kRingOff = 2 * kQBytes;
    static constexpr uint32_t kBarOff = kRingOff + kRing * kKVBytes;
    // FP8 cache: the codes of a ring item (128 rows of D bytes) land, for D = 128, in its slot's
    // upper half (where the f16 tile's second 64-column half goes; converted in place), for D = 64
    // in a code buffer of their own (64-byte rows, unswizzled); its row scales in a scale slot
    static constexpr bool kCodesApart = FP8 && D == 64;
    static constexpr uint32_t kCodeOff = kTileHalf;             // within a ring slot (D = 128)
    static constexpr uint32_t kScaleOff = kBarOff + 256;        // [kRing][128] FP32
    // the K row scales of key tile j times the softmax's log2 scale, at [j % 4][128] FP32
    static constexpr uint32_t kKScaleOff = kScaleOff + kRing * 128 * 4;
    static constexpr uint32_t kCodeBufOff = kKScaleOff + kRing * 128 * 4;  // [kRing][128 x 64 B] (D = 64)
    static constexpr uint32_t kSmemBytes = kBarOff + 256 + (FP8 ? 2 * kRing * 128 * 4 : 0) +
                                           (kCodesApart ? kRing * 128 * 64 : 0) + 1024;  // + alignment slack
    // the codes of ring slot `slot`
    __device__ static uint8_t *codes(uint8_t *smem, uint8_t *ring, int slot) {
        return kCodesApart ? smem + kCodeBufOff + slot * (128 * 64) : ring + slot * kKVBytes + kCodeOff;
    }
    static constexpr uint32_t kTmemCols = 512;
};

struct PrefillParams {
    const int *cu_q_lens, *context_lens, *block_tables;
    int batch, mb, num_q_heads, num_kv_heads, group, bs, log2_bs, num_blocks;
    float scale_log2;
    int causal;
    int skip_single;      // mixed batch: leave sequences with one query row to the decode kernels
    const float *scales;  // FP8 cache: FP32 row scales [NB, 2, Hkv, bs]
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

// exp2 on the FMA pipe for two values at once (the MUFU exp2 rate of an SM equals its bf16 tensor
// rate per score element at head_dim 128, so a share of the exponentials is evaluated here).
// Cody-Waite range reduction 2^x = 2^j 2^f, j = round(x) by the 1.5*2^23 magic-number addition,
// f in [-1/2, 1/2]; 2^f by a minimax polynomial (relative error, Remez exchange, constant term
// pinned to 1 so exp2(0) = 1 exactly; coefficients from csrc/exp2_poly.py): degree 3 (max
// relative error 4.3e-4) when P is rounded to bf16, degree 4 (3.6e-6) when P is fp16; 2^j is
// added to the exponent field. Inputs are clamped to >= -125 (2^-125 ~ 0 against the row sum).
template <bool BF16>
__device__ __forceinline__ float2 exp2_fma2(float2 x) {
    constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
    x.x = fmaxf(x.x, -125.f);
    x.y = fmaxf(x.y, -125.f);
    const float2 t = fadd2(x, make_float2(kMagic, kMagic));
    const float2 f = fsub2(x, fsub2(t, make_float2(kMagic, kMagic)));
    float2 p;
    if (BF16) {
        p = ffma2(make_float2(4.169875011e-02f, 4.169875011e-02f), f, make_float2(2.420305163e-01f, 2.420305163e-01f));
        p = ffma2(p, f, make_float2(6.957668066e-01f, 6.957668066e-01f));
    } else {
        p = ffma2(make_float2(9.782912210e-03f, 9.782912210e-03f), f, make_float2(5.597688258e-02f, 5.597688258e-02f));
        p = ffma2(p, f, make_float2(2.402071059e-01f, 2.402071059e-01f));
        p = ffma2(p, f, make_float2(6.931136250e-01f, 6.931136250e-01f));
    }
    p = ffma2(p, f, make_float2(1.f, 1.f));
    // t's low mantissa bits hold j (offset by the magic number, whose bits shift out)
    return make_float2(__uint_as_float(__float_as_uint(p.x) + (__float_as_uint(t.x) << 23)),
                       __uint_as_float(__float_as_uint(p.y) + (__float_as_uint(t.y) << 23)));
}

// Pairs q of a 128-key row with (q % 8) < kEmuPerEight take exp2_fma2, the others MUFU ex2.
// 0: every exponential on MUFU. Moving a quarter of them to the FMA pipe timed slower on this
// kernel, whose bound is the hand-off between the MMA thread and the softmax warps, not ex2.
constexpr int kEmuPerEight = 0;

__device__ __forceinline__ uint32_t pack2(float a, float b, bool bf16) {
    if (bf16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Four E4M3 codes (one 32-bit word, lowest byte first) to two f16x2 words holding the codes'
// values times 2^-8, exactly, on the integer pipe. An E4M3 code s.eeee.mmm (bias 7) placed as the
// f16 bits s.0eeee.mmm0000000 (bias 15) is its value times 2^(7 - 15) = 2^-8: normal codes map to
// normal f16 values and subnormal codes (eeee = 0, value m * 2^-9) to f16 subnormals m * 2^-17,
// both exact. Per pair of codes: a byte permute, then (t + (t & sign bits)) << 7, where the
// addition moves each sign bit from bit 7 to bit 8 of its 16-bit half. (The f16 conversion
// instruction would do the same work on the pipe that also packs P, which the softmax keeps busy:
// measured, the whole pass then took 3.38 ms against 3.18 ms.)
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t tl = __byte_perm(w, 0u, 0x4140), th = __byte_perm(w, 0u, 0x4342);
    lo = (tl + (tl & 0x00800080u)) << 7;
    hi = (th + (th & 0x00800080u)) << 7;
}
// The factor the converted codes carry (2^-8), undone in FP32 by the K scales and the epilogue.
constexpr float kCodeFactorInv = 256.f;

// Smallest power of two >= x, for finite x >= 0 (0 for 0; 2^-126 for subnormal x).
__device__ __forceinline__ float pow2_ceil(float x) {
    uint32_t b = __float_as_uint(x);
    if (b == 0u) return 0.f;
    if (b & 0x7fffffu) b = (b & 0x7f800000u) + 0x800000u;
    return __uint_as_float(b);
}

// Over an FP8 cache: the E4M3 codes of row r of a ring item become the f16 row r (values times
// 2^-8, see e4m3x4_to_f16) of the layout TMA writes for a 16-bit cache (64-column halves of
// 128-byte rows, 128-byte swizzle); rows at or beyond zero_from become zero. A pass takes 8 rows
// g .. g + 7 (g a multiple of 8), and every swizzled address is a lane constant plus 1 KB a pass.
//   D = 128: the codes (128 bytes a row, swizzled like an f16 half by TMA) sit where the row's
//   second f16 half goes, so the pass converts in place: lane -> rows rr and rr + 4 (rr = lane /
//   8), 16-code chunk c = lane % 8; a row is read entirely before any of it is written. The lanes
//   of the two halves store opposite chunks first: the 8 stores of a row in one instruction then
//   fill all 32 banks once.
//   D = 64: the codes come from a buffer of their own (64 bytes a row, unswizzled): lane -> row
//   rr = lane / 4, 16-code chunk c = lane % 4, written as f16 chunks 2c and 2c + 1.
template <int D, uint32_t kTileHalf>
struct RowConverter;

template <uint32_t kTileHalf>
struct RowConverter<128, kTileHalf> {
    uint32_t ld[2], sta[2], stb[2];
    int rr, hf;
    __device__ __forceinline__ explicit RowConverter(int lane) {
        const int c = lane & 7;
        rr = lane >> 3;
        hf = c >> 2;
        const int k0 = 2 * (c & 3);
        const int ka = hf ? k0 + 1 : k0, kb = hf ? k0 : k0 + 1;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int rw = rr + 4 * i;  // == row & 7
            ld[i] = rw * 128u + ((c ^ rw) << 4);
            sta[i] = hf * kTileHalf + rw * 128u + ((ka ^ rw) << 4);
            stb[i] = hf * kTileHalf + rw * 128u + ((kb ^ rw) << 4);
        }
    }
    __device__ __forceinline__ void pass(const uint8_t *codes, uint8_t *f16, int g, int zero_from) const {
        const uint32_t grp = (uint32_t)g * 128u;
        uint4 raw[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) raw[i] = *reinterpret_cast<const uint4 *>(codes + grp + ld[i]);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            uint32_t h16[8];  // f16 pairs of dims 16c .. 16c+15
            e4m3x4_to_f16(raw[i].x, h16[0], h16[1]);
            e4m3x4_to_f16(raw[i].y, h16[2], h16[3]);
            e4m3x4_to_f16(raw[i].z, h16[4], h16[5]);
            e4m3x4_to_f16(raw[i].w, h16[6], h16[7]);
            if (g + rr + 4 * i >= zero_from) {
#pragma unroll
                for (int k = 0; k < 8; ++k) h16[k] = 0u;
            }
            const uint4 v0 = make_uint4(h16[0], h16[1], h16[2], h16[3]);
            const uint4 v1 = make_uint4(h16[4], h16[5], h16[6], h16[7]);
            *reinterpret_cast<uint4 *>(f16 + grp + sta[i]) = hf ? v1 : v0;
            *reinterpret_cast<uint4 *>(f16 + grp + stb[i]) = hf ? v0 : v1;
        }
    }
};

template <uint32_t kTileHalf>
struct RowConverter<64, kTileHalf> {
    uint32_t ld, sta, stb;
    int rr;
    __device__ __forceinline__ explicit RowConverter(int lane) {
        const int c = lane & 3;
        rr = lane >> 2;  // == row & 7
        ld = rr * 64u + c * 16u;
        sta = rr * 128u + (((2 * c) ^ rr) << 4);
        stb = rr * 128u + (((2 * c + 1) ^ rr) << 4);
    }
    __device__ __forceinline__ void pass(const uint8_t *codes, uint8_t *f16, int g, int zero_from) const {
        const uint4 raw = *reinterpret_cast<const uint4 *>(codes + (uint32_t)g * 64u + ld);
        uint32_t h16[8];
        e4m3x4_to_f16(raw.x, h16[0], h16[1]);
        e4m3x4_to_f16(raw.y, h16[2], h16[3]);
        e4m3x4_to_f16(raw.z, h16[4], h16[5]);
        e4m3x4_to_f16(raw.w, h16[6], h16[7]);
        if (g + rr >= zero_from) {
#pragma unroll
            for (int k = 0; k < 8; ++k) h16[k] = 0u;
        }
        const uint32_t grp = (uint32_t)g * 128u;
        *reinterpret_cast<uint4 *>(f16 + grp + sta) = make_uint4(h16[0], h16[1], h16[2], h16[3]);
        *reinterpret_cast<uint4 *>(f16 + grp + stb) = make_uint4(h16[4], h16[5], h16[6], h16[7]);
    }
};

// BF16: type of q and the default output. FP8: the cache holds E4M3 codes with one FP32 scale per
// row; the tensor-core products then run in f16 (MMA below), which holds every code exactly.
template <int D, bool BF16, bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                   PrefillParams p) {
    using Lay = PrefillLayout<D, FP8>;
    constexpr bool MMA_BF16 = BF16 && !FP8;  // operand type of the tcgen05 products and of P
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment: the 128-byte swizzle pattern is a function of address bits 4-9.
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t *sQ = smem + Lay::kQOff;
    uint8_t *sRing = smem + Lay::kRingOff;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::kBarOff);
    uint64_t *kv_full = bars;            // [kRing]
    uint64_t *kv_empty = bars + 4;       // [kRing]
    uint64_t *q_full = bars + 8;
    uint64_t *s_full = bars + 9;         // [2] S_A / S_B computed
    uint64_t *p_full = bars + 13;        // [2] P_A / P_B in TMEM (and O rescaled)
    uint64_t *o_done = bars + 15;        // [2] P V accumulated into O_A / O_B
    uint64_t *drain = bars + 17;         // every MMA issued has completed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 18);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 19);
    uint64_t *kv_code = bars + 20;       // [kRing] FP8: codes and scales of a ring item have landed
    uint64_t *q_ready = bars + 24;       // FP8: Q converted to f16 (or left as it is for f16 q)
    const float *sScale = reinterpret_cast<const float *>(smem + Lay::kScaleOff);  // FP8: [kRing][128]
    float *sW = reinterpret_cast<float *>(bars + 25);  // FP8: [kRing] W of each V item (see the converter)
    uint64_t *ks_ready = bars + 27;      // [4] FP8: K scales of key tile j in sKS[j % 4]
    uint64_t *r_ready = bars + 11;       // [2] FP8: r and W of the V item in ring slot 2i + 1
    float *sKS = reinterpret_cast<float *>(smem + Lay::kKScaleOff);  // FP8: [4][128]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // grid (heads, batch, row blocks) with the row blocks last-first: CTAs start in linear order, so
    // the row blocks that see the most keys (causal) start in the first wave and the short ones
    // fill in behind them. A mixed batch: (heads, row blocks last-first, sequences by their rank
    // among those with several query rows), so that no CTA without work precedes one with work.
    const int h = blockIdx.x;
    const int mt = p.skip_single ? (int)gridDim.y - 1 - (int)blockIdx.y : (int)gridDim.z - 1 - (int)blockIdx.z;
    pdl_wait();  // lengths, tables, q and the chunk's own K/V may come from the previous kernel
    const int b = p.skip_single ? nth_multi_row_sequence(p.cu_q_lens, p.batch, blockIdx.z) : (int)blockIdx.y;
    if (b < 0) return;  // uniform: past the mixed batch's last chunk
    const int q0 = __ldg(p.cu_q_lens + b);
    const int q_len = __ldg(p.cu_q_lens + b + 1) - q0;
    const int m_start = mt * kRows;
    if (m_start >= q_len || (p.skip_single && q_len == 1)) return;  // uniform: nothing allocated yet
    const int L = __ldg(p.context_lens + b);
    if (L > p.mb * p.bs || q_len > L || L < 0) {
        if (threadIdx.x == 0) set_error(p.err, kErrDeviceRange);
        return;
    }
    const int rows = min(kRows, q_len - m_start);
    const int qpos0 = L - q_len + m_start;                // absolute position of row 0
    const int kv_end = p.causal ? qpos0 + rows : L;       // keys [0, kv_end) are needed
    const int n_tiles = (kv_end + kBN - 1) / kBN;
    const int g = h / p.group;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRing; ++s) {
            // FP8: a K slot (even: items alternate K, V) is full once both converter warps have
            // converted it, a V slot once the 8 softmax warps have; the K row scales leave the
            // ring slot for sKS, so every slot is free once its MMAs are done
            mbar_init(&kv_full[s], FP8 ? ((s & 1) ? 8 : 2) : 1);
            mbar_init(&kv_empty[s], 1);
            if (FP8) {
                mbar_init(&kv_code[s], 1);
                mbar_init(&ks_ready[s], 1);
                if (s < 2) mbar_init(&r_ready[s], 1);
            }
        }
        mbar_init(q_full, 1);
        if (FP8) mbar_init(q_ready, 2);
        for (int x = 0; x < 2; ++x) {
            mbar_init(&s_full[x], 1);
            mbar_init(&p_full[x], 4);
            mbar_init(&o_done[x], 1);
        }
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

    if (warp < 4) {
        tc::regs_dec<72>();
        if (warp == 0) {
            // ==================================== TMA producer ====================================
            const int box_rows = p.bs < kBN ? p.bs : kBN;
            uint32_t issued = 0;  // ring items issued (for the abort drain)
            if (lane == 0) {
                tc::prefetch_tensormap(&tm_q);
                tc::prefetch_tensormap(&tm_kv);
                mbar_arrive_expect_tx(q_full, 2 * Lay::kQBytes);
#pragma unroll
                for (int x = 0; x < 2; ++x)
#pragma unroll
                    for (int hf = 0; hf < Lay::kHalves; ++hf)
                        tc::tma_load_3d(sQ + x * Lay::kQBytes + hf * Lay::kTileHalf, &tm_q, hf * 64, h,
                                        q0 + m_start + x * kBM, q_full);
            }
            const int *bt = p.block_tables + (size_t)b * p.mb;
            bool ok = true;
            for (int j = 0; j < n_tiles && ok; ++j) {
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
                for (int kv = 0; kv < 2; ++kv) {
                    const uint32_t u = 2u * j + kv, slot = u % kRing, ph = (u / kRing) & 1u;
                    if (!mbar_wait(&kv_empty[slot], ph ^ 1u, abort_flag, p.err)) { ok = false; break; }
                    uint8_t *dst0 = sRing + slot * Lay::kKVBytes;
                    if constexpr (FP8) {
                        // codes (one 128-byte box row per token) and row scales of each page slice
                        if (lane == 0) mbar_arrive_expect_tx(&kv_code[slot], (uint32_t)npages * box_rows * (D + 4u));
                        __syncwarp();
                        if (lane < npages) {
                            const int row = ((pb * 2 + kv) * p.num_kv_heads + g) * p.bs + off;
                            const uint32_t dst = (uint32_t)lane * box_rows;
                            tc::tma_load_2d(Lay::codes(smem, sRing, slot) + dst * D, &tm_kv, 0, row, &kv_code[slot]);
                            bulk_g2s(smem + Lay::kScaleOff + (slot * 128u + dst) * 4u, p.scales + row,
                                     (uint32_t)box_rows * 4u, &kv_code[slot], l2_policy_evict_first());
                        }
                    } else {
                        if (lane == 0)
                            mbar_arrive_expect_tx(&kv_full[slot], (uint32_t)npages * box_rows * 128u * Lay::kHalves);
                        __syncwarp();
                        if (lane < npages) {
                            const int row = ((pb * 2 + kv) * p.num_kv_heads + g) * p.bs + off;
                            const uint32_t dst = (uint32_t)lane * box_rows * 128u;
#pragma unroll
                            for (int hf = 0; hf < Lay::kHalves; ++hf)
                                tc::tma_load_2d(dst0 + hf * Lay::kTileHalf + dst, &tm_kv, hf * 64, row, &kv_full[slot]);
                        }
                    }
                    ++issued;
                }
            }
            if (!ok) {
                // let copies in flight land before the CTA exits (bounded)
                const uint32_t first = issued > (uint32_t)kRing ? issued - kRing : 0u;
                for (uint32_t u = first; u < issued; ++u) {
                    volatile int no_abort = 0;
                    mbar_wait(FP8 ? &kv_code[u % kRing] : &kv_full[u % kRing], (u / kRing) & 1u, &no_abort, nullptr);
                }
            }
        } else if (FP8 && warp >= 2) {
            // ================================ FP8 converter warps ================================
            // Per K item: the codes become f16 in place (RowConverter), warp 2 rows 0-63 and warp 3
            // rows 64-127; warp 3 also copies the K row scales, times the log2 scale and 2^8 (the
            // converted codes' factor), to sKS. The V items' codes are converted by the 8 softmax
            // warps, each after its previous key tile (V_j is needed only after the softmax of
            // tile j); here warp 2 turns each V item's row scales w into r = w / W in place, W a
            // power of two at or above every V scale seen so far in this CTA (kept in sW[slot]):
            // the softmax folds r into P, and O carries the factor W (rescaled exactly when W
            // grows).
            const int cw = warp - 2;
            const RowConverter<D, Lay::kTileHalf> conv(lane);
            bool cok = mbar_wait(q_full, 0, abort_flag, p.err);
            if (BF16 && cok) {
                // q to f16 in place (exact for |q| within f16's range)
                uint4 *q4 = reinterpret_cast<uint4 *>(sQ);
                for (int i = cw * 32 + lane; i < 2 * (int)Lay::kQBytes / 16; i += 64) {
                    const uint4 v = q4[i];
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                    uint32_t o[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) o[k] = pack2(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xffff0000u), false);
                    q4[i] = make_uint4(o[0], o[1], o[2], o[3]);
                }
                tc::fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0 && cok) mbar_arrive(q_ready);
            float w_run = 0.f;  // warp 2: W so far
            for (int u = 0; cok && u < 2 * n_tiles; ++u) {
                const int slot = u % kRing, kv = u & 1;
                if (kv == 1 && cw == 1) continue;  // V codes: converted by the softmax warps
                if (!(cok = mbar_wait(&kv_code[slot], (uint32_t)(u / kRing) & 1u, abort_flag, p.err))) break;
                const int n_valid = L - (u >> 1) * kBN;
                if (kv == 0) {
                    if (cw == 1) {
                        // the K row scales of this key tile, times the softmax's log2 scale, to
                        // sKS[tile % 4] (read there by the softmax warps, so that the ring slot is
                        // free as soon as its QK MMAs are done)
                        const float4 k4 = reinterpret_cast<const float4 *>(sScale + slot * 128)[lane];
                        const float sl2 = p.scale_log2 * kCodeFactorInv;
                        reinterpret_cast<float4 *>(sKS + ((u >> 1) & 3) * 128)[lane] =
                            make_float4(k4.x * sl2, k4.y * sl2, k4.z * sl2, k4.w * sl2);
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&ks_ready[(u >> 1) & 3]);
                    }
                    for (int g = cw * 64; g < cw * 64 + 64; g += 8)
                        conv.pass(Lay::codes(smem, sRing, slot), sRing + slot * Lay::kKVBytes, g, kBN);
                    tc::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&kv_full[slot]);
                } else {
                    // warp 2: r = w / W for this V item's rows (0 beyond the context), W = max(W so
                    // far, 2^ceil(log2 max w)); each lane rewrites the 4 scales it read
                    float *sc = const_cast<float *>(sScale) + slot * 128;
                    float4 w4 = reinterpret_cast<const float4 *>(sc)[lane];
                    const int r0 = 4 * lane;
                    w4.x = r0 < n_valid ? w4.x : 0.f;
                    w4.y = r0 + 1 < n_valid ? w4.y : 0.f;
                    w4.z = r0 + 2 < n_valid ? w4.z : 0.f;
                    w4.w = r0 + 3 < n_valid ? w4.w : 0.f;
                    float vmax = fmaxf(fmaxf(w4.x, w4.y), fmaxf(w4.z, w4.w));
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
                    w_run = fmaxf(w_run, pow2_ceil(vmax));
                    const float inv_w = w_run > 0.f ? __frcp_rn(w_run) : 0.f;  // exact: W is a power of two
                    reinterpret_cast<float4 *>(sc)[lane] = make_float4(w4.x * inv_w, w4.y * inv_w, w4.z * inv_w, w4.w * inv_w);
                    if (lane == 0) sW[slot] = w_run;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&r_ready[slot >> 1]);
                }
            }
        } else if (warp == 1) {
            // ===================================== MMA issuer =====================================
            if (lane == 0) {
                const uint32_t id_qk = tc::idesc_f16(MMA_BF16, kBM, kBN, false);
                const uint32_t id_pv = tc::idesc_f16(MMA_BF16, kBM, D, true);
                const uint32_t aQ = smem_addr(sQ), aRing = smem_addr(sRing);
                auto ring_wait = [&](uint32_t u) {
                    return mbar_wait(&kv_full[u % kRing], (u / kRing) & 1u, abort_flag, p.err);
                };
                auto qk = [&](int x, uint32_t aK) {
                    const uint32_t aQx = aQ + (uint32_t)x * Lay::kQBytes;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t o = (uint32_t)(kk >> 2) * Lay::kTileHalf + (uint32_t)(kk & 3) * 32u;
                        tc::mma_f16_ss(tmem + kColS + 128u * x, tc::smem_desc(aQx + o, 16, 1024), tc::smem_desc(aK + o, 16, 1024),
                                       id_qk, kk > 0 ? 1u : 0u);
                    }
                    tc::mma_commit(&s_full[x]);
                };
                auto pv = [&](int x, uint32_t aV, int j) {
                    const uint32_t tP = tmem + kColS + 128u * x, tO = tmem + kColO + 128u * x;
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk) {
                        // V is [keys x D], D contiguous: MN-major B; 8-key groups 1024 B apart,
                        // 64-column halves kTileHalf apart. P: 16 keys = 8 TMEM columns.
                        tc::mma_f16_ts(tO, tP + 8u * kk, tc::smem_desc(aV + (uint32_t)kk * 2048u, Lay::kTileHalf, 1024),
                                       id_pv, (j > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc::mma_commit(&o_done[x]);
                };
                bool ok = mbar_wait(FP8 ? q_ready : q_full, 0, abort_flag, p.err) && ring_wait(0);
                if (ok) {
                    tc::fence_after_sync();
                    qk(0, aRing);  // S_A = Q_A K_0^T
                    qk(1, aRing);  // S_B = Q_B K_0^T
                    tc::mma_commit(&kv_empty[0]);
                }
                // Ping-pong: tile A's P V_j then its next S, then tile B's. P_x sits in S_x's columns;
                // the tensor pipe runs the MMAs of this thread in issue order, so S_x(j+1) is
                // written only after P_x(j) V_j has read P_x(j).
                for (int j = 0; ok && j < n_tiles; ++j) {
                    const uint32_t uK = 2u * j, uV = uK + 1, uKn = uK + 2;
                    const uint32_t aV = aRing + (uV % kRing) * Lay::kKVBytes;
                    const uint32_t aKn = aRing + (uKn % kRing) * Lay::kKVBytes;
                    const uint32_t ph = (uint32_t)j & 1u;
                    const bool more = j + 1 < n_tiles;
                    if (!(ok = ring_wait(uV) && mbar_wait(&p_full[0], ph, abort_flag, p.err))) break;
                    tc::fence_after_sync();
                    pv(0, aV, j);
                    if (more) {
                        if (!(ok = ring_wait(uKn))) break;
                        qk(0, aKn);
                    }
                    if (!(ok = mbar_wait(&p_full[1], ph, abort_flag, p.err))) break;
                    tc::fence_after_sync();
                    pv(1, aV, j);
                    tc::mma_commit(&kv_empty[uV % kRing]);
                    if (more) {
                        qk(1, aKn);
                        tc::mma_commit(&kv_empty[uKn % kRing]);
                    }
                }
                tc::mma_commit(drain);
                volatile int no_abort = 0;
                mbar_wait(drain, 0, &no_abort, p.err);
            }
            __syncwarp();
        }
    } else {
        tc::regs_inc<208>();
        // ================================= softmax + epilogue =================================
        const int x = (warp >> 2) - 1;                 // 0: tile A, 1: tile B
        const int quarter = warp & 3;                  // TMEM lanes 32*quarter .. +31
        const int r = quarter * 32 + lane;             // row within the tile
        const int row = x * kBM + r;                   // row within the CTA block
        const bool row_ok = row < rows;
        const int qpos = qpos0 + row;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + kColS + 128u * x + lane_base;   // S_x, and P_x over its first 64 columns
        const uint32_t tO = tmem + kColO + 128u * x + lane_base;
        // over an FP8 cache the log2 scale is folded into the K row scales (sKS)
        const float c = FP8 ? 1.f : p.scale_log2;
        float m_use = -INFINITY, l = 0.f;
        float w_cur = 0.f;  // FP8: the factor W that O carries (the converter's, as of the last V item)
        bool ok = true;
        // FP8: the 8 softmax warps convert the codes of V item jv in place, 16 rows each (2 passes
        // of 8 rows; rows beyond the context zeroed), V_0 before the first key tile and V_{j+1}
        // right after tile j: V_{j+1}'s codes land while the softmax works on tile j, and the P
        // V_{j+1} MMAs need it only after the softmax of tile j + 1
        const RowConverter<D, Lay::kTileHalf> vconv(lane);
        auto convert_v = [&](int jv) -> bool {
            const uint32_t uV = 2u * jv + 1, vslot = uV % kRing;
            if (!mbar_wait(&kv_code[vslot], (uV / kRing) & 1u, abort_flag, p.err)) return false;
            const int g = (x * 4 + quarter) * 16;
            uint8_t *vb = sRing + vslot * Lay::kKVBytes;
            const uint8_t *vc = Lay::codes(smem, sRing, vslot);
            vconv.pass(vc, vb, g, L - jv * kBN);
            vconv.pass(vc, vb, g + 8, L - jv * kBN);
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&kv_full[vslot]);
            return true;
        };
        if constexpr (FP8) ok = convert_v(0);
        for (int j = 0; ok && j < n_tiles; ++j) {
            const int kv_start = j * kBN;
            const uint32_t ph = (uint32_t)j & 1u;
            if (!(ok = mbar_wait(&s_full[x], ph, abort_flag, p.err))) break;
            tc::fence_after_sync();
            float s[kBN];
#pragma unroll
            for (int cc = 0; cc < kBN / 32; ++cc)
                tc::tmem_ld32(tS + cc * 32, *reinterpret_cast<float(*)[32]>(&s[cc * 32]));
            tc::tmem_wait_ld();
            if constexpr (FP8) {
                // K row scales (times the log2 scale) multiply the score columns, in FP32. sKS[j % 4]
                // is next written for tile j + 4, whose K item cannot arrive before both softmax
                // warpgroups are done with tile j + 1
                if (!(ok = mbar_wait(&ks_ready[j & 3], (uint32_t)(j >> 2) & 1u, abort_flag, p.err))) break;
                const float4 *ks4 = reinterpret_cast<const float4 *>(sKS + (j & 3) * 128);
#pragma unroll
                for (int i = 0; i < kBN / 4; ++i) {
                    const float4 k4 = ks4[i];
                    const float2 a = fmul2(make_float2(s[4 * i], s[4 * i + 1]), make_float2(k4.x, k4.y));
                    const float2 b = fmul2(make_float2(s[4 * i + 2], s[4 * i + 3]), make_float2(k4.z, k4.w));
                    s[4 * i] = a.x;
                    s[4 * i + 1] = a.y;
                    s[4 * i + 2] = b.x;
                    s[4 * i + 3] = b.y;
                }
            }
            // last key index this row may see in this tile (-1: none)
            int lim = L - 1 - kv_start;
            if (p.causal) lim = min(lim, qpos - kv_start);
            if (!row_ok) lim = -1;
            const bool masked = lim < kBN - 1;
            if (masked) {
#pragma unroll
                for (int i = 0; i < kBN; ++i) s[i] = (i <= lim) ? s[i] : -INFINITY;
            }
            // row max as 8 independent chains (two warps per scheduler cannot hide a 64-deep chain)
            float m8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) m8[k] = fmax3(s[k], s[k + 8], s[k + 16]);
#pragma unroll
            for (int i = 24; i < kBN; i += 16)
#pragma unroll
                for (int k = 0; k < 8; ++k) m8[k] = fmax3(m8[k], s[i + k], (i + 8 + k < kBN) ? s[i + 8 + k] : -INFINITY);
            const float mx = fmaxf(fmax3(m8[0], m8[1], m8[2]), fmax3(fmax3(m8[3], m8[4], m8[5]), m8[6], m8[7]));
            const float m_new = fmaxf(m_use, mx * c);
            const bool grow = m_new > m_use + kRescaleLog2;   // false when m_new = -inf
            const float alpha = grow ? fast_exp2(m_use - m_new) : 1.f;  // 0 when m_use = -inf
            if (grow) {
                m_use = m_new;
                l *= alpha;
            }
            // masked entries are -inf; m_use is finite for a row with a visible key, and a row
            // without one (padding row) uses 0 so that exp2(-inf) = 0 instead of a NaN
            const float neg_m = (m_use == -INFINITY) ? 0.f : -m_use;
            uint32_t pk[kBN / 2];
            float2 l4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
            const float2 c2 = make_float2(c, c), nm2 = make_float2(neg_m, neg_m);
            // FP8: P' = p * r (r = V row scale / W, FP32) enters the P.V product, so the V tile
            // holds the exact codes; l sums p. W is the converter's for this V item.
            bool w_grow = false;
            float w_ratio = 1.f;
            const float4 *r4 = nullptr;
            if constexpr (FP8) {
                const uint32_t uV = 2u * j + 1, vslot = uV % kRing;
                if (!(ok = mbar_wait(&r_ready[vslot >> 1], (uV / kRing) & 1u, abort_flag, p.err))) break;
                const float w_j = sW[vslot];
                w_grow = w_j > w_cur;  // the same for every thread of the CTA
                if (w_grow) {
                    w_ratio = w_cur / w_j;  // exact: powers of two (0 while O is still 0)
                    w_cur = w_j;
                }
                r4 = reinterpret_cast<const float4 *>(sScale + vslot * 128);
            }
            if (masked) {
                // boundary tiles: -inf entries, MUFU only (ex2(-inf) = 0)
#pragma unroll
                for (int q = 0; q < kBN / 2; ++q) {
                    const float2 xq = ffma2(make_float2(s[2 * q], s[2 * q + 1]), c2, nm2);
                    const float2 e = make_float2(fast_exp2(xq.x), fast_exp2(xq.y));
                    l4[q & 3] = fadd2(l4[q & 3], e);
                    if constexpr (FP8) {
                        const float4 rv = r4[q >> 1];
                        const float2 er = fmul2(e, (q & 1) ? make_float2(rv.z, rv.w) : make_float2(rv.x, rv.y));
                        pk[q] = pack2(er.x, er.y, false);
                    } else {
                        pk[q] = pack2(e.x, e.y, MMA_BF16);
                    }
                }
            } else {
#pragma unroll
                for (int q = 0; q < kBN / 2; ++q) {
                    const float2 xq = ffma2(make_float2(s[2 * q], s[2 * q + 1]), c2, nm2);
                    const float2 e = ((q & 7) < kEmuPerEight) ? exp2_fma2<MMA_BF16>(xq)
                                                              : make_float2(fast_exp2(xq.x), fast_exp2(xq.y));
                    l4[q & 3] = fadd2(l4[q & 3], e);
                    if constexpr (FP8) {
                        const float4 rv = r4[q >> 1];
                        const float2 er = fmul2(e, (q & 1) ? make_float2(rv.z, rv.w) : make_float2(rv.x, rv.y));
                        pk[q] = pack2(er.x, er.y, false);
                    } else {
                        pk[q] = pack2(e.x, e.y, MMA_BF16);
                    }
                }
            }
            const float2 l2 = fadd2(fadd2(l4[0], l4[1]), fadd2(l4[2], l4[3]));
            const float lsum = l2.x + l2.y;
            l += lsum;
            // P_x and O_x are touched only after P_x V_{j-1} is done
            if (j > 0) {
                if (!(ok = mbar_wait(&o_done[x], (uint32_t)(j - 1) & 1u, abort_flag, p.err))) break;
                tc::fence_after_sync();
                if (__any_sync(0xffffffffu, grow) || w_grow) {
                    const float o_scale = alpha * w_ratio;
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) {
                        float o[32];
                        tc::tmem_ld32(tO + cc * 32, o);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= o_scale;
                        tc::tmem_st32(tO + cc * 32, o);
                    }
                }
            }
#pragma unroll
            for (int cc = 0; cc < kBN / 32; ++cc)
                tc::tmem_st16(tS + cc * 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[cc * 16]));
            tc::tmem_wait_st();
            // keys at or beyond the context end may hold unwritten cache bytes: tile A zeroes those V rows
            const int n_valid = L - kv_start;
            if (!FP8 && x == 0 && n_valid < kBN) {  // (an FP8 cache's converter writes zeros there)
                const uint32_t uV = 2u * j + 1;
                if (!(ok = mbar_wait(&kv_full[uV % kRing], (uV / kRing) & 1u, abort_flag, p.err))) break;
                if (r >= n_valid) {
                    uint8_t *sV = sRing + (uV % kRing) * Lay::kKVBytes;
#pragma unroll
                    for (int hf = 0; hf < Lay::kHalves; ++hf)
#pragma unroll
                        for (int cc = 0; cc < 8; ++cc)
                            *reinterpret_cast<uint4 *>(sV + hf * Lay::kTileHalf + (uint32_t)r * 128u + cc * 16) =
                                make_uint4(0, 0, 0, 0);
                }
                tc::fence_proxy_async_smem();
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[x]);
            if constexpr (FP8) {
                if (j + 1 < n_tiles && !(ok = convert_v(j + 1))) break;
            }
        }
        // ---- epilogue: O / l ----
        if (ok && mbar_wait(&o_done[x], (uint32_t)(n_tiles - 1) & 1u, abort_flag, p.err)) {
            tc::fence_after_sync();
            // O / l; over an FP8 cache O carries the factor W (0 only when every V scale is 0) and
            // the converted codes' 2^-8
            const float inv = l > 0.f ? (FP8 ? w_cur * kCodeFactorInv : 1.f) / l : 0.f;
            const size_t row_g = (size_t)(q0 + m_start + row);
            const size_t obase = (row_g * p.num_q_heads + h) * D;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                float o[32];
                tc::tmem_ld32(tO + cc * 32, o);
                tc::tmem_wait_ld();
                if (row_ok) {
                    if (p.out_dtype == 2) {
                        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + obase + cc * 32);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv,
                                                 o[4 * i + 3] * inv);
                    } else {
                        const bool obf = p.out_dtype == 1;
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.out) + obase + cc * 32);
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
    pdl_launch_dependents();
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

}  // namespace

// 2-D tensor map over the cache viewed as rows of D elements (row ((pb*2 + kv)*Hkv + h)*bs + off),
// boxes of 64 columns x box_rows rows, 128-byte swizzle.
cudaError_t encode_cache_map(const CacheView &c, int box_rows, CUtensorMap *map) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    // 16-bit elements: boxes of 64 columns (128 bytes); FP8 codes, head_dim 128: boxes of 128
    // one-byte columns, so every box row is one 128-byte swizzle atom either way; FP8 codes,
    // head_dim 64: boxes of 64-byte rows, unswizzled
    const bool codes64 = c.fp8 && c.head_dim == 64;
    if (c.fp8 && c.head_dim != 128 && !codes64) return cudaErrorNotSupported;
    const CUtensorMapDataType dt = c.fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : c.dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const cuuint64_t nrows = (cuuint64_t)c.num_blocks * 2 * c.num_kv_heads * c.block_size;
    if (nrows > 0x7fffffffull || nrows == 0) return cudaErrorNotSupported;  // TMA row coordinates are int32
    cuuint64_t dims[2] = {(cuuint64_t)c.head_dim, nrows};
    cuuint64_t strides[1] = {(cuuint64_t)c.head_dim * (c.fp8 ? 1 : 2)};
    cuuint32_t box[2] = {c.fp8 ? (cuuint32_t)c.head_dim : 64u, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    if (enc(map, dt, 2, const_cast<void *>(c.ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            codes64 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    return cudaSuccess;
}

cudaError_t encode_q_heads_map(const void *q, int bf16, int total_q, int num_q_heads, int head_dim, int box_rows,
                               CUtensorMap *map) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    if (total_q <= 0 || box_rows <= 0 || box_rows > 256) return cudaErrorNotSupported;
    // q [total_q, Hq, D]: x = d, y = head, z = token; box 64 x 1 x box_rows
    cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_q_heads, (cuuint64_t)total_q};
    cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)num_q_heads * head_dim * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(q),
            dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    return cudaSuccess;
}

cudaError_t encode_rows_map(const void *ptr, int bf16, long long rows, int cols, int box_cols, int box_rows,
                            CUtensorMap *map) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    if (rows <= 0 || rows > 0x7fffffffll || box_rows <= 0 || box_rows > 256 || box_cols * 2 != 128)
        return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    if (enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(ptr),
            dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    return cudaSuccess;
}

// The cache viewed as the 5-D tensor [NB][2][Hkv][bs][D] so that one box holds a page slice of K
// and of V: box = 128 bytes of columns (64 16-bit elements, or 128 FP8 codes) x box_rows x 1 head
// x 2 (K, V) x 1 page, 128-byte swizzle; shared memory receives the K rows, then the V rows.
cudaError_t encode_kv5_map(const CacheView &c, int box_rows, CUtensorMap *map) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t D = (cuuint64_t)c.head_dim, bs = (cuuint64_t)c.block_size, h = (cuuint64_t)c.num_kv_heads;
    const cuuint64_t nb = (cuuint64_t)c.num_blocks, es_bytes = c.fp8 ? 1 : 2;
    if (nb == 0 || nb > 0x7fffffffull) return cudaErrorNotSupported;
    if (c.fp8 && D != 128) return cudaErrorNotSupported;
    const CUtensorMapDataType dt = c.fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : c.dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    cuuint64_t dims[5] = {D, bs, h, 2, nb};
    cuuint64_t strides[4] = {D * es_bytes, D * bs * es_bytes, D * bs * h * es_bytes, D * bs * h * 2 * es_bytes};
    cuuint32_t box[5] = {(cuuint32_t)(128 / es_bytes), (cuuint32_t)box_rows, 1, 2, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    if (enc(map, dt, 5, const_cast<void *>(c.ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    return cudaSuccess;
}

cudaError_t encode_kv5_rows_map(const CacheView &c, int box_rows, CUtensorMap *map) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    if (c.fp8) return cudaErrorNotSupported;
    const cuuint64_t D = (cuuint64_t)c.head_dim, bs = (cuuint64_t)c.block_size, h = (cuuint64_t)c.num_kv_heads;
    const cuuint64_t nb = (cuuint64_t)c.num_blocks;
    if (nb == 0 || nb > 0x7fffffffull || D > 256) return cudaErrorNotSupported;
    const CUtensorMapDataType dt = c.dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    cuuint64_t dims[5] = {D, bs, h, 2, nb};
    cuuint64_t strides[4] = {D * 2, D * bs * 2, D * bs * h * 2, D * bs * h * 2 * 2};
    cuuint32_t box[5] = {(cuuint32_t)D, (cuuint32_t)box_rows, 1, 2, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    if (enc(map, dt, 5, const_cast<void *>(c.ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    return cudaSuccess;
}

// An FP8 cache: the codes as encode_kv5_map, the scales as the 4-D tensor [NB][2][Hkv][bs]
// (box box_rows x 1 x 2 x 1: K scales, then V scales).
cudaError_t encode_fp8_maps(const CacheView &c, int box_rows, CUtensorMap *codes, CUtensorMap *scales) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    if (!c.fp8 || c.head_dim != 128) return cudaErrorNotSupported;
    const cuuint64_t bs = (cuuint64_t)c.block_size, h = (cuuint64_t)c.num_kv_heads;
    const cuuint64_t nb = (cuuint64_t)c.num_blocks;
    {
        const cudaError_t e = encode_kv5_map(c, box_rows, codes);
        if (e != cudaSuccess) return e;
    }
    {
        cuuint64_t dims[4] = {bs, h, 2, nb};
        cuuint64_t strides[3] = {bs * 4, bs * h * 4, bs * h * 2 * 4};
        cuuint32_t box[4] = {(cuuint32_t)box_rows, 1, 2, 1};
        cuuint32_t es[4] = {1, 1, 1, 1};
        if (enc(scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(c.scales), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

namespace {

template <int D, bool BF16, bool FP8>
cudaError_t launch_t(const PrefillArgs &a, cudaStream_t stream) {
    using Lay = PrefillLayout<D, FP8>;
    CUtensorMap tm_q, tm_kv;
    {
        const cudaError_t e = encode_q_heads_map(a.q, BF16 ? 1 : 0, a.total_q, a.num_q_heads, D, kBM, &tm_q);
        if (e != cudaSuccess) return e;
    }
    {
        const cudaError_t e = encode_cache_map(a.cache, a.cache.block_size < kBN ? a.cache.block_size : kBN, &tm_kv);
        if (e != cudaSuccess) return e;
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
    p.skip_single = a.skip_single;
    p.scales = a.cache.scales;
    p.out = a.out;
    p.out_dtype = a.out_dtype;
    p.lse = a.lse;
    p.err = a.err;
    auto kern = prefill_kernel<D, BF16, FP8>;
    static DeviceFlags configured;
    const int dev = device_info().device;
    if (!configured.test(dev)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Lay::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured.set(dev);
    }
    const unsigned row_blocks = (unsigned)((a.max_q_len + kRows - 1) / kRows);
    const dim3 grid = a.skip_single ? dim3(a.num_q_heads, row_blocks, a.batch) : dim3(a.num_q_heads, a.batch, row_blocks);
    return launch_pdl(kern, grid, dim3(kThreads), Lay::kSmemBytes, stream, tm_q, tm_kv, p);
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t s) {
    if (a.max_q_len == 0) return cudaSuccess;
    if (a.cache.head_dim == 256) return a.cache.fp8 ? cudaErrorNotSupported : launch_prefill_wide(a, s);
    if (a.cache.head_dim != 64 && a.cache.head_dim != 128) return cudaErrorNotSupported;
    const bool bf16 = a.cache.dtype == 1;
    if (a.cache.fp8) {
        if (a.cache.head_dim == 128) return bf16 ? launch_t<128, true, true>(a, s) : launch_t<128, false, true>(a, s);
        return bf16 ? launch_t<64, true, true>(a, s) : launch_t<64, false, true>(a, s);
    }
    if (a.cache.head_dim == 128) return bf16 ? launch_t<128, true, false>(a, s) : launch_t<128, false, false>(a, s);
    return bf16 ? launch_t<64, true, false>(a, s) : launch_t<64, false, false>(a, s);
}

}  // namespace pkv
