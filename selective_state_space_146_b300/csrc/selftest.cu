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
//
// probe_scan_forms measures the two ways of running the recurrence over a
// 32-step tile of one channel with 16 states (page "Mamba模型笔记" §4.5, the
// parallel scan over (A_bar, B_bar u) pairs with (a1, b1) o (a2, b2) =
// (a1 a2, a2 b1 + b2)): `seq`, one lane per channel stepping through t with
// the states in registers (the form the scan kernels use), and `shfl`, one
// lane per step, the 32 steps composed by a five-level warp-shuffle
// (Kogge-Stone) scan per state, then the carry from the previous tile applied
// and the readout taken.  Both read the same B | C table from shared memory
// and produce the same y; the probe reports channel-steps per second of each.
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

__device__ float g_probe_scan_sink[4096];

template <bool SHFL>
__global__ void __launch_bounds__(256) probe_scan(int tiles) {
    // B | C table of one 32-step tile, as the scan kernels keep it:
    // row t = (B0 B1 C0 C1 | B2 B3 C2 C3 | ...), 128 bytes
    __shared__ float4 tab[32][8];
    for (int i = threadIdx.x; i < 256; i += blockDim.x) {
        const float v = 0.1f * (float)((i * 37) % 19) - 0.9f;
        tab[i / 8][i % 8] = make_float4(v, 0.5f * v, 0.25f - v, v * v);
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    float A2[16];
#pragma unroll
    for (int n = 0; n < 16; ++n) A2[n] = -(float)(n + 1) * kLog2e;
    float sink = 0.f;
    if constexpr (!SHFL) {
        // one lane = one channel, 32 steps in sequence
        float h[16] = {};
        for (int k = 0; k < tiles; ++k) {
#pragma unroll 4
            for (int t = 0; t < 32; ++t) {
                const float dl = 0.01f + 1e-4f * (float)((lane + t + k) & 15);
                const float du = dl * (0.5f - 0.03f * (float)((lane * 3 + t) & 31));
                float y = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 bc = tab[t][j];
                    h[2 * j] = fmaf(ex2_approx(dl * A2[2 * j]), h[2 * j], du * bc.x);
                    h[2 * j + 1] = fmaf(ex2_approx(dl * A2[2 * j + 1]), h[2 * j + 1], du * bc.y);
                    y = fmaf(bc.z, h[2 * j], fmaf(bc.w, h[2 * j + 1], y));
                }
                sink += y;
            }
        }
    } else {
        // one lane = one step of the tile; the warp scans one channel's
        // sequence tile after tile, carrying the state across tiles (the same
        // channel-steps as above)
        const float4* row = tab[lane];
        float hin[16] = {};  // the state entering the tile: the previous tile's last
        for (int k = 0; k < tiles; ++k) {
            for (int c = 0; c < 32; ++c) {
                const float dl = 0.01f + 1e-4f * (float)((c + lane + k) & 15);
                const float du = dl * (0.5f - 0.03f * (float)((c * 3 + lane) & 31));
                float a[16], b[16];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 bc = row[j];
                    a[2 * j] = ex2_approx(dl * A2[2 * j]);
                    a[2 * j + 1] = ex2_approx(dl * A2[2 * j + 1]);
                    b[2 * j] = du * bc.x;
                    b[2 * j + 1] = du * bc.y;
                }
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
                    for (int n = 0; n < 16; ++n) {
                        const float ap = __shfl_up_sync(0xffffffffu, a[n], o);
                        const float bp = __shfl_up_sync(0xffffffffu, b[n], o);
                        if (lane >= o) {
                            b[n] = fmaf(a[n], bp, b[n]);
                            a[n] *= ap;
                        }
                    }
                }
                float y = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 bc = row[j];
                    const float h0v = fmaf(a[2 * j], hin[2 * j], b[2 * j]);
                    const float h1v = fmaf(a[2 * j + 1], hin[2 * j + 1], b[2 * j + 1]);
                    y = fmaf(bc.z, h0v, fmaf(bc.w, h1v, y));
                    hin[2 * j] = __shfl_sync(0xffffffffu, h0v, 31);
                    hin[2 * j + 1] = __shfl_sync(0xffffffffu, h1v, 31);
                }
                sink += y + hin[0];
            }
        }
    }
    g_probe_scan_sink[(blockIdx.x * blockDim.x + threadIdx.x) & 4095] = sink;
}

int probe_scan_forms(double* seq_steps_per_s, double* shfl_steps_per_s, cudaStream_t st) {
    const int sms = sm_count_current();
    const int ctas = sms * 4, threads = 256, tiles = 64;
    // channel-steps of one launch: every lane owns (seq) or walks (shfl) 32
    // channels' tiles of 32 steps, `tiles` times
    const double steps = (double)ctas * threads * 32.0 * tiles;
    cudaEvent_t e0, e1;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) return SS_ERR_CUDA;
    double out[2] = {0.0, 0.0};
    for (int form = 0; form < 2; ++form) {
        for (int rep = 0; rep < 2; ++rep) {  // the first launch warms up
            cudaEventRecord(e0, st);
            if (form == 0) probe_scan<false><<<ctas, threads, 0, st>>>(tiles);
            else probe_scan<true><<<ctas, threads, 0, st>>>(tiles);
            cudaEventRecord(e1, st);
            count_launch(1);
        }
        float ms = 0.f;
        if (cudaGetLastError() != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
            cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess) {
            cudaEventDestroy(e0);
            cudaEventDestroy(e1);
            return SS_ERR_CUDA;
        }
        out[form] = steps / (ms * 1e-3);
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    *seq_steps_per_s = out[0];
    *shfl_steps_per_s = out[1];
    return SS_OK;
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
