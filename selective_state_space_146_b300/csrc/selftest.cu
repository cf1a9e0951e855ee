// selftest.cu -- exercises the library's failure path on the device without
// faulting it: a kernel waits, with a caller-given time limit, on an mbarrier
// that nothing arrives on, records the same error bit the scan kernels record
// when a bounded wait gives up, and returns.  ss_get_device_error then reports
// SS_ERR_TIMEOUT and clears the word, and the context stays usable.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"
#include "ssscan.h"

namespace ss {

__global__ void __launch_bounds__(32) selftest_wait(unsigned long long limit_ns, unsigned* err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // one arrival expected; none will come
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x != 0) return;
    const unsigned long long start = globaltimer();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(&bar, 0)) return;  // never: nothing arrives
        if ((it & 63u) == 0 && globaltimer() - start > limit_ns) {
            atomicOr(err, ERR_WAIT_TIMEOUT);
            return;
        }
    }
}

int launch_selftest_wait(unsigned limit_us, unsigned* err, cudaStream_t st) {
    selftest_wait<<<1, 32, 0, st>>>((unsigned long long)limit_us * 1000ull, err);
    count_launch(1);
    return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_LAUNCH;
}

}  // namespace ss
