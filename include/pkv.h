/*
 * pkv.h -- C ABI of libpkv: attention over a paged KV cache on NVIDIA GB300 (sm_103a).
 *
 * The operations follow the subject's web pages (cited by page title and section):
 *  [FAPA] "Flash Attention与Paged Attention如何共同优化大模型推理？" (ipipp.com)
 *         s2: tiled attention with a running max m and running sum l, old output
 *             rescaled by exp(m_old - m_new), final division by l; the library
 *             call's causal flag.  s3: pages of block_size tokens, cache shape
 *             [num_blocks, 2, num_heads, block_size, head_dim], per-sequence page
 *             table, each page's valid-token count.
 *  [CHUNK] "企业官网建设流程全解析" (cf-1.com) s2.1: logical block = i / block_size,
 *             physical block = block_table[logical], offset = i % block_size;
 *             s2.3: one launch for the whole batch instead of one per request.
 *  [ON2]  "为什么Attention是O(n²)" (answer.freetools.me): softmax(QK^T/sqrt(d_k))V
 *             (mathematics section); prefill writes every prompt token's K/V into
 *             the cache, a decode step attends one query to all cached K/V and
 *             appends the new token's K/V (prefill / decode section); grouped-query
 *             attention, several query heads sharing one KV head (GQA section).
 *  [BLK]  "从一次压测翻车说起：分块 attention ..." (pwwt.cn) s3.3, s5.3: parallelise
 *             over batch x head and over key/value blocks (here: split-KV with a
 *             log-sum-exp merge instead of atomics); s3.4, s5.4: FP32 accumulation.
 *
 * Conventions shared by every call
 *  - All data pointers are DEVICE pointers owned by the caller; the library never
 *    allocates, frees or keeps them.  Every pointer must be 16-byte aligned.
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL is
 *    the legacy default stream).  A returned PKV_OK means the launch was queued.
 *  - Arguments are validated on the host before anything is launched; an invalid
 *    call returns an error and launches nothing.
 *  - Values that live on the device (page ids, lengths) are range-checked by the
 *    kernels: a bad one never faults, the affected token or tile is skipped or
 *    read from page 0, and a sticky device error word records the first such
 *    event (read it with pkv_get_device_error).
 *  - Cache layout (row-major): cache[pb][kv][h][off][d] over
 *    [num_blocks, 2, num_kv_heads, block_size, head_dim]; kv = 0 is K, 1 is V;
 *    element offset ((((pb*2 + kv)*Hkv + h)*bs + off)*D + d).
 *  - Query head h reads KV head h / (Hq / Hkv).
 *  - Block tables are int32 [batch, max_blocks_per_seq]; entry [b][i / bs] holds
 *    the page of token i of sequence b.  Unused entries are never read.
 *  - Arithmetic: fp16 / bf16 inputs, FP32 products, sums and softmax; the output is
 *    rounded once (round-to-nearest-even) to out_dtype.
 *  - lse outputs are natural-log log-sum-exp of the scaled scores, FP32
 *    (-inf for an empty context).
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>

/* Exported symbols (the library is built with hidden visibility by default). */
#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,   /* null / misaligned pointer, negative size, inconsistent shapes */
    PKV_ERR_UNSUPPORTED = 2,   /* head_dim, block_size, dtype or head grouping outside the supported set */
    PKV_ERR_WORKSPACE = 3,     /* workspace missing or smaller than pkv_decode_workspace_size() */
    PKV_ERR_CUDA = 4,          /* a CUDA runtime call failed (launch, attribute, sync) */
    PKV_ERR_DEVICE_RANGE = 5,  /* device error word: a page id, table slot or length was out of range */
    PKV_ERR_TIMEOUT = 6        /* device error word: a bounded wait inside a kernel expired */
} pkv_status;

typedef enum { PKV_F16 = 0, PKV_BF16 = 1, PKV_F32 = 2 } pkv_dtype;

/* How the cache stores K and V.
 *  PKV_KV_NATIVE    ptr holds dtype elements (2 bytes each).
 *  PKV_KV_FP8_E4M3  ptr holds one-byte OCP FP8 E4M3 codes (1 sign, 4 exponent bits
 *                   with bias 7, 3 fraction bits; no infinities; largest finite
 *                   448) and `scales` one FP32 scale per cached row, i.e. per
 *                   (page, K/V, KV head, token): element = decode(code) * scale.
 *                   A row is written by pkv_kv_cache_append as scale = amax / 448,
 *                   code = round-to-nearest-even, saturating, of x * (448 / amax),
 *                   in FP32 (amax = largest |x| of the row; an all-zero row stores
 *                   scale 0 and zero codes).  The pages name KV-cache compression
 *                   ([ON2]) without a scheme; this per-row scaling is the library's
 *                   reading of it. */
typedef enum { PKV_KV_NATIVE = 0, PKV_KV_FP8_E4M3 = 1 } pkv_kv_format;

/* The paged KV cache [num_blocks, 2, num_kv_heads, block_size, head_dim] ([FAPA] s3).
 * dtype (PKV_F16 or PKV_BF16) is the type of q, k_new and v_new, of the default
 * output, and of the elements of a native cache.  Supported: head_dim 64, 128 or
 * 256 (256: a native cache only; an FP8 cache with head_dim 256 returns
 * PKV_ERR_UNSUPPORTED); block_size a power of two in [8, 512].  format and scales
 * are as above (scales [num_blocks, 2, num_kv_heads, block_size], 16-byte aligned;
 * NULL for a native cache).  Every call accepts an FP8 cache.  Over an FP8 cache
 * the tensor-core products run in f16 on the exact codes (the row scales are
 * applied in FP32): q must lie within f16's range (|q| < 65504; magnitudes below
 * 2^-24 count as 0). */
typedef struct {
    void *ptr;
    int num_blocks;
    int num_kv_heads;
    int block_size;
    int head_dim;
    pkv_dtype dtype;
    pkv_kv_format format;
    float *scales;
} pkv_cache;

/* kv_cache_append -- write new tokens' K and V into their pages ([ON2] prefill /
 * decode; [CHUNK] s2.1 addressing); an FP8 cache receives each row's codes and
 * scale, computed as described at pkv_kv_format.
 *   k_new, v_new      [num_new_tokens, Hkv, D] in the cache dtype, packed by
 *                     sequence: sequence b owns rows cu_new_lens[b] .. cu_new_lens[b+1]-1.
 *   cu_new_lens       int32 [batch+1], cu_new_lens[0] = 0, non-decreasing,
 *                     cu_new_lens[batch] = num_new_tokens.
 *   ctx_before        int32 [batch]: tokens already cached; the j-th new token of
 *                     sequence b goes to position ctx_before[b] + j.
 *   block_tables      int32 [batch, max_blocks_per_seq]; pages for every written
 *                     position must already be assigned.
 * A native cache receives a bit-exact copy.  Positions whose table slot is beyond max_blocks_per_seq,
 * or whose page id is outside [0, num_blocks), are skipped and flag
 * PKV_ERR_DEVICE_RANGE.  Nothing else in the cache is modified. */
PKV_API pkv_status pkv_kv_cache_append(pkv_cache cache, const void *k_new, const void *v_new,
                               const int *cu_new_lens, const int *ctx_before,
                               const int *block_tables, int batch, int max_blocks_per_seq,
                               int num_new_tokens, void *stream);

/* Bytes of workspace pkv_paged_attn_decode needs for these sizes: the FP32 split
 * partials (padded to 16 bytes) and a 16-byte slot, or 0 when no context can span several
 * splits.  num_splits as passed to pkv_paged_attn_decode (0 = automatic). */
PKV_API size_t pkv_decode_workspace_size(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                 int block_size, int max_blocks_per_seq, int num_splits);

/* Tokens per split that pkv_paged_attn_decode uses for these sizes (a multiple of
 * 128, and at least capacity / 2048 so that a context has at most 2048 splits); a
 * context of L tokens is cut into ceil(L / chunk) splits.  With num_splits = 0 this is the
 * smallest split: the split kernel, which sees the context lengths, may take 1.5, 2, 3 or
 * 4 times it (rounded up to a multiple of 128) where its model of the launch's time says
 * the work divides better over its CTAs; the workspace size holds for every choice. */
PKV_API int pkv_decode_split_tokens(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                            int block_size, int max_blocks_per_seq, int num_splits);

/* paged_attn_decode -- one query per sequence against its whole paged context
 * ([ON2] decode; [FAPA] s2 online softmax, s3 paging; [BLK] s5.3 split over
 * key/value blocks).
 *   q             [batch, Hq, D] in the cache dtype.
 *   context_lens  int32 [batch]: cached tokens of each sequence (0 allowed: the
 *                 output is 0 and lse is -inf); must not exceed
 *                 max_blocks_per_seq * block_size (else flagged and clamped).
 *   scale         multiplies q.k (1/sqrt(D) for the textbook definition).
 *   num_splits    0 = automatic; else the context capacity
 *                 max_blocks_per_seq * block_size is cut into this many splits.
 *   workspace     device scratch of at least pkv_decode_workspace_size() bytes
 *                 (FP32 partial outputs and their lse); contents need no init.
 *   out           [batch, Hq, D] in out_dtype (the cache dtype or PKV_F32).
 *   lse           FP32 [batch, Hq] or NULL.
 *   num_q_heads   any multiple of the cache's num_kv_heads (any group size); over an
 *                 FP8 cache the group must be 1, 2, 4 or a multiple of 8 (head_dim 64:
 *                 at most 8), else PKV_ERR_UNSUPPORTED.
 *   batch         any size: batches run in slices of up to 2048 sequences.
 * Launches the split kernel and, when some context spans several splits, the
 * merge of pkv_attn_combine on the same stream (once per slice). */
PKV_API pkv_status pkv_paged_attn_decode(pkv_cache cache, const void *q, int num_q_heads,
                                 const int *block_tables, const int *context_lens, int batch,
                                 int max_blocks_per_seq, float scale, int num_splits,
                                 void *workspace, size_t workspace_bytes,
                                 void *out, pkv_dtype out_dtype, float *lse, void *stream);

/* paged_attn_decode_step -- one decode step in one call: the attention of
 * pkv_paged_attn_decode over each sequence's context_lens[b] cached tokens, and the
 * append of the step's new token, whose K and V go to position context_lens[b] (attend,
 * then append: [ON2] decode; position -> page and offset as pkv_kv_cache_append).
 * Arguments as pkv_paged_attn_decode, plus
 *   k_new, v_new  [batch, Hkv, D] in the cache's 16-bit type (over an FP8 cache: quantised
 *                 to E4M3 codes + row scales as pkv_kv_cache_append does); device, 16-byte
 *                 aligned, required when batch > 0 (else PKV_ERR_INVALID_ARG).
 * The attention reads positions below context_lens[b] only, so the result is that of
 * pkv_paged_attn_decode followed by pkv_kv_cache_append of one token per sequence, bit for
 * bit (outputs, lse and every cache element). The caller advances context_lens by one for
 * the next step. A position context_lens[b] outside the table (the table full) or a page id
 * outside the pool is skipped and flags PKV_ERR_DEVICE_RANGE; the attention still runs.
 * Launches: on a 16-bit cache with 1, 2, 4 or 8 query heads per KV head (head_dim 64 or
 * 128) the split kernel writes the new rows itself (its merge warps, before their first
 * unit), so the call is the split kernel and its merge; otherwise the append kernel
 * follows the decode on the same stream. */
PKV_API pkv_status pkv_paged_attn_decode_step(pkv_cache cache, const void *q, int num_q_heads,
                                      const int *block_tables, const int *context_lens, int batch,
                                      int max_blocks_per_seq, float scale, int num_splits,
                                      void *workspace, size_t workspace_bytes,
                                      void *out, pkv_dtype out_dtype, float *lse,
                                      const void *k_new, const void *v_new, void *stream);

/* paged_attn_prefill -- a chunk of queries per sequence against its paged context,
 * causal or not ([ON2] prefill; [FAPA] s2 causal flag; [BLK] s2.2 chunked queries).
 * "Append first, then attend": the chunk's own K/V must already be in the cache.
 *   q             [total_q, Hq, D] in the cache dtype, packed by sequence:
 *                 sequence b owns rows cu_q_lens[b] .. cu_q_lens[b+1]-1.
 *   cu_q_lens     int32 [batch+1] (q_len_b = cu_q_lens[b+1] - cu_q_lens[b]).
 *   context_lens  int32 [batch]: tokens in the cache INCLUDING the chunk, with
 *                 q_len_b <= context_lens[b].
 *   causal        non-zero: query r of sequence b sits at absolute position
 *                 context_lens[b] - q_len_b + r and sees keys 0 .. that position
 *                 (bottom-right alignment); zero: every query sees the whole context.
 *   max_q_len     an upper bound of q_len_b over the batch (sizes the grid; batch and
 *                 ceil(max_q_len / 256), or ceil(max_q_len / 128) at head_dim 256, at most
 *                 65535 each, else PKV_ERR_UNSUPPORTED).
 *   out           [total_q, Hq, D] in out_dtype; lse FP32 [total_q, Hq] or NULL. */
PKV_API pkv_status pkv_paged_attn_prefill(pkv_cache cache, const void *q, int num_q_heads,
                                  const int *cu_q_lens, const int *context_lens,
                                  const int *block_tables, int batch, int max_blocks_per_seq,
                                  int total_q, int max_q_len, float scale, int causal,
                                  void *out, pkv_dtype out_dtype, float *lse, void *stream);

/* paged_attn_mixed -- one call over a batch that mixes decode sequences (exactly one query
 * row) and prefill chunks (several query rows, their K/V already appended): prefill and
 * decode in one step, as a continuously batched serving loop issues them ([ON2] continuous
 * batching; "Prefill/Decode mixed execution"). Arguments as pkv_paged_attn_prefill (q, out,
 * lse indexed by the rows of cu_q_lens; causal applies to the chunks, a single row sees its
 * whole context either way) plus num_splits / workspace as pkv_paged_attn_decode, sized by
 * pkv_decode_workspace_size(batch, ...). The single-row sequences run on the decode kernels
 * (split-KV, one unit per KV head's query group), the others on the prefill kernel; each
 * kernel leaves the other kind's rows untouched. The decode constraint on head grouping (an
 * FP8 cache) applies to the whole call. */
PKV_API pkv_status pkv_paged_attn_mixed(pkv_cache cache, const void *q, int num_q_heads,
                                const int *cu_q_lens, const int *context_lens,
                                const int *block_tables, int batch, int max_blocks_per_seq,
                                int total_q, int max_q_len, float scale, int causal,
                                int num_splits, void *workspace, size_t workspace_bytes,
                                void *out, pkv_dtype out_dtype, float *lse, void *stream);

/* attn_combine -- log-sum-exp merge of split-KV partial results ([FAPA] s2: the
 * same rescale-by-exp(m_old - m_new) identity applied to whole splits).
 *   partial_o     FP32 [n_rows, num_splits, head_dim]: each split's output,
 *                 already divided by that split's own softmax sum.
 *   partial_lse   FP32 [n_rows, num_splits]: natural-log lse of each split's
 *                 scaled scores; -inf marks an empty split (weight 0).
 *   out           [n_rows, head_dim] in out_dtype; lse FP32 [n_rows] or NULL.
 * A row whose splits are all empty gets output 0 and lse -inf. */
PKV_API pkv_status pkv_attn_combine(const float *partial_o, const float *partial_lse, int n_rows,
                            int num_splits, int head_dim, void *out, pkv_dtype out_dtype,
                            float *lse, void *stream);

/* paged_attn_decode_noalloc -- the same computation and arguments as
 * pkv_paged_attn_decode, for callers that cannot allocate device memory: a plugin
 * that its host framework hands only input and output buffers (no workspace, no
 * allocator), or a runtime that reserves all device memory in its own pool up front.
 * The paper has no counterpart: this is a deployment convenience, not part of the
 * method.
 *   - Allocates nothing (no cudaMalloc, cudaFree or allocating library call).  The
 *     split partials live in a fixed array of PKV_DECODE_NOALLOC_SCRATCH_BYTES that
 *     the library keeps in device memory; every GPU that loads the library holds it
 *     until the process exits.
 *   - Sizes whose workspace (pkv_decode_workspace_size) exceeds that array are
 *     rejected with PKV_ERR_WORKSPACE before anything is launched.
 *   - The first call on each device (that device current) looks up the array's device
 *     address with cudaGetSymbolAddress; make that first call before any stream
 *     capture.  A lookup that fails returns PKV_ERR_CUDA and is not remembered: the
 *     next call looks again.
 *   - All calls share the one array, which keeps the last call's contents.  Nothing
 *     in it has to start at zero: each call writes every partial it later reads.
 *     Calls that overlap on the GPU (concurrent streams, or several host threads)
 *     race on the array: serialise them. */
#define PKV_DECODE_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
PKV_API pkv_status pkv_paged_attn_decode_noalloc(pkv_cache cache, const void *q, int num_q_heads,
                                         const int *block_tables, const int *context_lens, int batch,
                                         int max_blocks_per_seq, float scale, int num_splits,
                                         void *out, pkv_dtype out_dtype, float *lse, void *stream);

/* selftest_wait_timeout -- failure-detection check. Every wait inside the kernels is bounded:
 * after its limit it records PKV_ERR_TIMEOUT in the device error word and the kernel winds
 * down instead of hanging. This launches one warp that waits, the same way, on an mbarrier
 * nothing will complete, with a limit of timeout_us microseconds (1..1000000); read the
 * result with pkv_get_device_error (PKV_ERR_TIMEOUT expected). The pages have no
 * counterpart; it exists to test the failure path without faulting the GPU. */
PKV_API pkv_status pkv_selftest_wait_timeout(unsigned int timeout_us, void *stream);

/* Synchronise `stream`, then read and clear the sticky device error word of the
 * current device.  *code receives PKV_OK, PKV_ERR_DEVICE_RANGE or PKV_ERR_TIMEOUT.
 * Returns PKV_ERR_CUDA if the synchronisation or the read fails. */
PKV_API pkv_status pkv_get_device_error(void *stream, int *code);

/* Human-readable name of a status code (static storage). */
PKV_API const char *pkv_status_string(pkv_status status);

/* Library ABI version (major * 100 + minor). */
PKV_API int pkv_version(void);  /* 101: pkv_cache carries format and scales */

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
