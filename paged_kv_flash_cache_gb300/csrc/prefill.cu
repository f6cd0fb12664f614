// prefill.cu -- paged_attn_prefill (placeholder until the tcgen05 kernel lands).
#include "pkv_internal.h"

namespace pkv {

cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t s) {
    (void)a;
    (void)s;
    return cudaErrorNotSupported;
}

}  // namespace pkv
