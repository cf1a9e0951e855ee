// ssd.cu -- the Mamba-2 SSD scan on sm_103a.
//
// What is computed (page "Mamba模型笔记" §5; state-spaces/mamba README §4.3):
// per batch row b and head h (group g = h / (H/G)), with a = exp(dt A_h),
//   S[p][n] <- a S[p][n] + dt x[p] B[g][n],   y[p] = sum_n C[g][n] S[p][n] + D_h x[p].
//
// This file holds the general CUDA-core kernel (one thread per (b, h, p),
// state row in registers, sequential over t): any strides, dtypes, P and
// N <= 256.  The chunked tensor-core kernel lives in ssd_tc.cu.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>

#include "internal.h"
#include "ptx.cuh"
#include "ssscan.h"

namespace ss {

template <typename T, int NMAX>
__global__ void __launch_bounds__(128) ssd_general(SSDArgs a) {
    const int64_t unit = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t units = (int64_t)a.Bsz * a.H * a.P;
    if (unit >= units) return;
    const int p = (int)(unit % a.P);
    const int h = (int)((unit / a.P) % a.H);
    const int b = (int)(unit / ((int64_t)a.P * a.H));
    const int g = h / (a.H / a.G);
    const int N = a.N;
    float S[NMAX];
#pragma unroll
    for (int n = 0; n < NMAX; ++n)
        S[n] = (a.h0 && n < N) ? a.h0[b * a.sh_b + h * a.sh_h + p * a.sh_p + n * a.sh_n] : 0.f;
    const float A2 = a.A[h * a.sA] * kLog2e;
    const float Dh = a.Dv ? a.Dv[h * a.sD] : 0.f;
    const T* x = static_cast<const T*>(a.x) + b * a.sx_b + h * a.sx_h + p * a.sx_p;
    const T* dt = static_cast<const T*>(a.dt) + b * a.sdt_b + h * a.sdt_h;
    const T* Bp = static_cast<const T*>(a.Bm) + b * a.sB_b + g * a.sB_g;
    const T* Cp = static_cast<const T*>(a.Cm) + b * a.sC_b + g * a.sC_g;
    T* y = static_cast<T*>(a.y) + b * a.sy_b + h * a.sy_h + p * a.sy_p;
    for (int t = 0; t < a.L; ++t) {
        const float dtv = Elem<T>::to_f(dt[t * a.sdt_l]);
        const float xv = Elem<T>::to_f(x[t * a.sx_l]);
        const float decay = ex2_approx(dtv * A2);
        const float dx = dtv * xv;
        const T* br = Bp + t * a.sB_l;
        const T* cr = Cp + t * a.sC_l;
        float acc = 0.f;
#pragma unroll
        for (int n = 0; n < NMAX; ++n) {
            if (n < N) {
                S[n] = fmaf(decay, S[n], dx * Elem<T>::to_f(br[n * a.sB_n]));
                acc = fmaf(Elem<T>::to_f(cr[n * a.sC_n]), S[n], acc);
            }
        }
        y[t * a.sy_l] = Elem<T>::from_f(fmaf(Dh, xv, acc));
    }
    if (a.last) {
        float* ls = a.last + b * a.sl_b + h * a.sl_h + p * a.sl_p;
        for (int n = 0; n < N; ++n) ls[n * a.sl_n] = S[n];
    }
}

template <typename T>
static int run_ssd_general(const SSDArgs& a, cudaStream_t st) {
    const int64_t units = (int64_t)a.Bsz * a.H * a.P;
    const int threads = 128;
    const unsigned blocks = (unsigned)((units + threads - 1) / threads);
    if (a.N <= 16) ssd_general<T, 16><<<blocks, threads, 0, st>>>(a);
    else if (a.N <= 64) ssd_general<T, 64><<<blocks, threads, 0, st>>>(a);
    else if (a.N <= 128) ssd_general<T, 128><<<blocks, threads, 0, st>>>(a);
    else ssd_general<T, 256><<<blocks, threads, 0, st>>>(a);
    count_launch(1);
    return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_LAUNCH;
}

int launch_ssd_tc(const SSDArgs& a, cudaStream_t st, const Scratch& scratch, bool* taken);

int launch_ssd(const SSDArgs& a, cudaStream_t st, const Scratch& scratch) {
    const char* force = getenv("SS_SSD_PATH");
    const bool general_only = force && !strcmp(force, "general");
    if (!general_only) {
        bool taken = false;
        int rc = launch_ssd_tc(a, st, scratch, &taken);
        if (taken) return rc;
    }
    return a.dtype == SS_BF16 ? run_ssd_general<__nv_bfloat16>(a, st) : run_ssd_general<float>(a, st);
}

// One recurrent step (decode): one warp per (b, h, p) state row; lanes split
// the N states and the readout is a warp sum.
template <typename T>
__global__ void __launch_bounds__(128) ssd_step(SSDStepArgs a) {
    const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= (int64_t)a.Bsz * a.H * a.P) return;
    const int p = (int)(row % a.P);
    const int h = (int)((row / a.P) % a.H);
    const int b = (int)(row / ((int64_t)a.P * a.H));
    const int g = h / (a.H / a.G);
    const float dtv = Elem<T>::to_f(static_cast<const T*>(a.dt)[b * a.sdt_b + h * a.sdt_h]);
    const float xv = Elem<T>::to_f(static_cast<const T*>(a.x)[b * a.sx_b + h * a.sx_h + p * a.sx_p]);
    const float decay = ex2_approx(dtv * a.A[h * a.sA] * kLog2e);
    const float dx = dtv * xv;
    const T* Bp = static_cast<const T*>(a.Bm) + b * a.sB_b + g * a.sB_g;
    const T* Cp = static_cast<const T*>(a.Cm) + b * a.sC_b + g * a.sC_g;
    float* st = a.state + b * a.ss_b + h * a.ss_h + p * a.ss_p;
    float acc = 0.f;
    for (int n = lane; n < a.N; n += 32) {
        const float sn = fmaf(decay, st[n * a.ss_n], dx * Elem<T>::to_f(Bp[n * a.sB_n]));
        st[n * a.ss_n] = sn;
        acc = fmaf(Elem<T>::to_f(Cp[n * a.sC_n]), sn, acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0)
        static_cast<T*>(a.y)[b * a.sy_b + h * a.sy_h + p * a.sy_p] =
            Elem<T>::from_f(fmaf(a.Dv ? a.Dv[h * a.sD] : 0.f, xv, acc));
}

// N = 128 with contiguous, 16-byte aligned state rows: lane l keeps states
// 4l .. 4l+3, so each warp moves its 512-byte row with one vector load and
// one vector store.
template <typename T>
__global__ void __launch_bounds__(128) ssd_step128(SSDStepArgs a) {
    const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= (int64_t)a.Bsz * a.H * a.P) return;
    const int p = (int)(row % a.P);
    const int h = (int)((row / a.P) % a.H);
    const int b = (int)(row / ((int64_t)a.P * a.H));
    const int g = h / (a.H / a.G);
    float4* st = reinterpret_cast<float4*>(a.state + b * a.ss_b + h * a.ss_h + p * a.ss_p) + lane;
    const float4 s4 = *st;
    const float dtv = Elem<T>::to_f(static_cast<const T*>(a.dt)[b * a.sdt_b + h * a.sdt_h]);
    const float xv = Elem<T>::to_f(static_cast<const T*>(a.x)[b * a.sx_b + h * a.sx_h + p * a.sx_p]);
    const float decay = ex2_approx(dtv * a.A[h * a.sA] * kLog2e);
    const float dx = dtv * xv;
    const T* Bp = static_cast<const T*>(a.Bm) + b * a.sB_b + g * a.sB_g + 4 * lane * a.sB_n;
    const T* Cp = static_cast<const T*>(a.Cm) + b * a.sC_b + g * a.sC_g + 4 * lane * a.sC_n;
    float bv[4], cv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        bv[i] = Elem<T>::to_f(Bp[i * a.sB_n]);
        cv[i] = Elem<T>::to_f(Cp[i * a.sC_n]);
    }
    float4 n4;
    n4.x = fmaf(decay, s4.x, dx * bv[0]);
    n4.y = fmaf(decay, s4.y, dx * bv[1]);
    n4.z = fmaf(decay, s4.z, dx * bv[2]);
    n4.w = fmaf(decay, s4.w, dx * bv[3]);
    *st = n4;
    float acc = fmaf(cv[0], n4.x, fmaf(cv[1], n4.y, fmaf(cv[2], n4.z, cv[3] * n4.w)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0)
        static_cast<T*>(a.y)[b * a.sy_b + h * a.sy_h + p * a.sy_p] =
            Elem<T>::from_f(fmaf(a.Dv ? a.Dv[h * a.sD] : 0.f, xv, acc));
}

int launch_ssd_step(const SSDStepArgs& a, cudaStream_t st) {
    const int64_t threads = (int64_t)a.Bsz * a.H * a.P * 32;
    const unsigned blocks = (unsigned)((threads + 127) / 128);
    const bool vec = a.N == 128 && a.ss_n == 1 && reinterpret_cast<uintptr_t>(a.state) % 16 == 0 &&
                     a.ss_p % 4 == 0 && a.ss_h % 4 == 0 && a.ss_b % 4 == 0;
    if (vec) {
        if (a.dtype == SS_BF16) ssd_step128<__nv_bfloat16><<<blocks, 128, 0, st>>>(a);
        else ssd_step128<float><<<blocks, 128, 0, st>>>(a);
    } else {
        if (a.dtype == SS_BF16) ssd_step<__nv_bfloat16><<<blocks, 128, 0, st>>>(a);
        else ssd_step<float><<<blocks, 128, 0, st>>>(a);
    }
    count_launch(1);
    return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_LAUNCH;
}

}  // namespace ss
