// selftest.cu -- failure-detection check of the bounded waits every kernel here relies on.
//
// Kernels never spin without a limit: each mbarrier wait gives up after a time limit, records
// PKV_ERR_TIMEOUT in the device error word and winds its CTA down, so a lost arrival (a copy that
// never lands, a role that stopped early) surfaces as a status instead of a hung GPU. This entry
// point exercises that path on purpose and safely: one warp waits on an mbarrier that nothing
// will ever complete, with a short limit, and returns.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

__global__ void __launch_bounds__(32, 1) wait_timeout_kernel(unsigned long long timeout_ns, int *err) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // one arrival expected; none will come
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncwarp();
    mbar_wait(&bar, 0, &abort_flag, err, timeout_ns);
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_selftest_wait_timeout(unsigned int timeout_us, void *stream) {
    if (timeout_us == 0 || timeout_us > 1000000u) return PKV_ERR_INVALID_ARG;
    int *err = device_error_word();
    if (!err) return PKV_ERR_CUDA;
    wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(1000ull * timeout_us, err);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
