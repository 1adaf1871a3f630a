// la_selftest_wait_timeout (contract in include/linattn.h): exercises the bounded-wait
// path every kernel of the library relies on, without any fault. One block waits on an
// mbarrier that nothing ever arrives on; the wait gives up after the given number of
// clock cycles, records a timeout in the device status word and the kernel returns.
#include "la_internal.h"

namespace la {

__global__ void selftest_wait_kernel(unsigned long long limit, int* status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // expects one arrival that never comes
        fence_mbar_init();
    }
    __syncthreads();
    bool done = false;
    const unsigned long long t0 = clock64();
    while (!(done = mbar_try_wait(&bar, 0))) {
        if (clock64() - t0 > limit) break;
    }
    if (!done && threadIdx.x == 0) atomicOr(status, STATUS_TIMEOUT);
}

}  // namespace la

extern "C" int la_selftest_wait_timeout(unsigned long long limit_cycles, la_stream_t stream) {
    if (limit_cycles == 0 || limit_cycles > (1ull << 32)) return LA_ERR_INVALID_ARG;
    int* status = nullptr;
    const int rc = la::device_status_word(&status);
    if (rc != LA_OK) return rc;
    la::selftest_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(limit_cycles, status);
    return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}
