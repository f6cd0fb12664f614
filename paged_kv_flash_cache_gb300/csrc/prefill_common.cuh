// prefill_common.cuh -- pieces shared by the two prefill kernels (prefill.cu, prefill_wide.cu).
#pragma once

#include <stdint.h>

namespace pkv {

// Mixed batch (prefill chunks and decode rows in one call, the decode rows being the decode
// kernels'): the n-th sequence (from 0) with more than one query row, or -1 when there are at
// most n of them. The prefill grid numbers its CTAs by this rank, so the CTAs with work come
// first in launch order and the ones past the last chunk, which return at once, last. Called by
// every thread of the CTA with the same n (four 32-sequence ballots a round, their loads in
// flight together).
__device__ __forceinline__ int nth_multi_row_sequence(const int *cu_q_lens, int batch, int n) {
    const int lane = threadIdx.x & 31;
    int before = 0;
    for (int g0 = 0; g0 < batch; g0 += 128) {
        unsigned m[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int i = g0 + k * 32 + lane;
            const bool multi = i < batch && __ldg(cu_q_lens + i + 1) - __ldg(cu_q_lens + i) > 1;
            m[k] = __ballot_sync(0xffffffffu, multi);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int c = __popc(m[k]);
            if (n < before + c) {
                const int r = n - before;  // the r-th set bit of m[k]
                const bool mine = ((m[k] >> lane) & 1u) && __popc(m[k] & ((1u << lane) - 1u)) == r;
                return g0 + k * 32 + __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
            }
            before += c;
        }
    }
    return -1;
}

}  // namespace pkv
