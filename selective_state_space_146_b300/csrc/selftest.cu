// selftest.cu -- two diagnostics.
//
// selftest_wait exercises the library's failure path on the device without
// faulting it: a kernel waits, with a caller-given time limit, on an mbarrier
// that nothing arrives on, records the same error bit the scan kernels record
// when a bounded wait gives up, and returns.  ss_get_device_error then reports
// SS_ERR_TIMEOUT and clears the word, and the context stays usable.
//
// probe_ex2 measures the MUFU pipe's ex2.approx.f32 throughput, the pipe that
// bounds the selective scan's exponentials: one 1024-thread CTA per SM, each
// thread running eight independent chains x <- 2^(x * c), timed with clock64
// on each SM.
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

// Eight independent chains per thread keep enough ex2 in flight to fill the
// pipe; the multiply that feeds each ex2 runs on the FMA pipe, which has four
// times the lanes.  Each CTA writes its cycle count and a checksum that keeps
// the chains alive.
constexpr int kProbeChains = 8;
__device__ unsigned long long g_probe_cycles[1024];
__device__ float g_probe_sink[1024];

__global__ void __launch_bounds__(1024, 1) probe_ex2(int iters) {
    float v[kProbeChains];
#pragma unroll
    for (int k = 0; k < kProbeChains; ++k) v[k] = -0.25f * (k + 1) - 1e-3f * (threadIdx.x & 31);
    __syncthreads();
    const unsigned long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int k = 0; k < kProbeChains; ++k) v[k] = ex2_approx(v[k] * -0.75f) - 1.0f;
    }
    __syncthreads();
    const unsigned long long t1 = clock64();
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < kProbeChains; ++k) s += v[k];
    if (threadIdx.x == 0 && blockIdx.x < 1024) {
        g_probe_cycles[blockIdx.x] = t1 - t0;
        g_probe_sink[blockIdx.x] = s;
    }
}

int probe_ex2_rate(double* per_sm_clk, cudaStream_t st) {
    const int sms = sm_count_current();
    const int ctas = sms < 1024 ? sms : 1024;
    const int iters = 4096;
    probe_ex2<<<ctas, 1024, 0, st>>>(iters);
    count_launch(1);
    if (cudaGetLastError() != cudaSuccess) return SS_ERR_LAUNCH;
    unsigned long long cyc[1024];
    if (cudaMemcpyFromSymbolAsync(cyc, g_probe_cycles, sizeof(unsigned long long) * ctas, 0,
                                  cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return SS_ERR_CUDA;
    unsigned long long worst = 1;
    for (int i = 0; i < ctas; ++i) worst = cyc[i] > worst ? cyc[i] : worst;
    *per_sm_clk = 1024.0 * iters * kProbeChains / (double)worst;
    return SS_OK;
}

}  // namespace ss
