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
    // SS_DEBUG_SSD_PATH: 0 the CUDA-core kernel only; 1 / 2 the tensor-core
    // kernels only (no fallback: SS_ERR_UNSUPPORTED where they do not apply)
    const int path = debug_path(SS_DEBUG_SSD_PATH);
    if (path != 0) {
        bool taken = false;
        int rc = launch_ssd_tc(a, st, scratch, &taken);
        if (taken) return rc;
        if (path == 1 || path == 2) return SS_ERR_UNSUPPORTED;
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

// Four consecutive elements of B or C (lane l takes n = 4l .. 4l+3): one
// 8- or 16-byte load when the rows are unit-stride and aligned, else four
// strided loads.
template <typename T, bool VEC>
__device__ __forceinline__ void load4(const T* p, int64_t s, float (&v)[4]) {
    if constexpr (VEC && sizeof(T) == 4) {
        const float4 q = *reinterpret_cast<const float4*>(p);
        v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    } else if constexpr (VEC) {
        const uint2 q = *reinterpret_cast<const uint2*>(p);
        const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.x));
        const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.y));
        v[0] = lo.x; v[1] = lo.y; v[2] = hi.x; v[3] = hi.y;
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = Elem<T>::to_f(p[i * s]);
    }
}

// N = 128 with contiguous, 16-byte aligned state rows: lane l keeps states
// 4l .. 4l+3 of a row, so a warp moves a 512-byte state row with one vector
// load and one vector store.  A warp takes ROWS consecutive (b, h, p) rows:
// their state loads go out before any arithmetic, the walk over (b, h, p)
// divides only once, and the head's step, decay, D and B, C are fetched
// again only when the walk enters another head (or group).
template <typename T, int ROWS, bool VBC>
__global__ void __launch_bounds__(128) ssd_step128(SSDStepArgs a) {
    const int lane = threadIdx.x & 31;
    const int rows = a.Bsz * a.H * a.P;  // below 2^31, checked by the launcher
    const int row0 = (int)(((unsigned)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * ROWS;
    if (row0 >= rows) return;
    const int hpg = a.H / a.G;
    int p = row0 % a.P, h = (row0 / a.P) % a.H, b = row0 / (a.P * a.H);
    float4 s4[ROWS];
    {
        int pp = p, hh = h, bb = b;
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            if (row0 + r < rows)
                s4[r] = reinterpret_cast<const float4*>(a.state + bb * a.ss_b + hh * a.ss_h +
                                                        pp * a.ss_p)[lane];
            if (++pp == a.P) { pp = 0; if (++hh == a.H) { hh = 0; ++bb; } }
        }
    }
    int hc = -1, gc = -1, bc = -1;
    float dtv = 0.f, decay = 0.f, Dh = 0.f, bv[4] = {}, cv[4] = {};
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        if (row0 + r >= rows) break;  // warp-uniform
        if (h != hc || b != bc) {
            const int g = h / hpg;
            dtv = Elem<T>::to_f(static_cast<const T*>(a.dt)[b * a.sdt_b + h * a.sdt_h]);
            decay = ex2_approx(dtv * a.A[h * a.sA] * kLog2e);
            Dh = a.Dv ? a.Dv[h * a.sD] : 0.f;
            if (g != gc || b != bc) {
                load4<T, VBC>(static_cast<const T*>(a.Bm) + b * a.sB_b + g * a.sB_g +
                              4 * lane * a.sB_n, a.sB_n, bv);
                load4<T, VBC>(static_cast<const T*>(a.Cm) + b * a.sC_b + g * a.sC_g +
                              4 * lane * a.sC_n, a.sC_n, cv);
                gc = g;
            }
            hc = h; bc = b;
        }
        const float xv = Elem<T>::to_f(static_cast<const T*>(a.x)[b * a.sx_b + h * a.sx_h +
                                                                  p * a.sx_p]);
        const float dx = dtv * xv;
        float4 n4;
        n4.x = fmaf(decay, s4[r].x, dx * bv[0]);
        n4.y = fmaf(decay, s4[r].y, dx * bv[1]);
        n4.z = fmaf(decay, s4[r].z, dx * bv[2]);
        n4.w = fmaf(decay, s4[r].w, dx * bv[3]);
        reinterpret_cast<float4*>(a.state + b * a.ss_b + h * a.ss_h + p * a.ss_p)[lane] = n4;
        float acc = fmaf(cv[0], n4.x, fmaf(cv[1], n4.y, fmaf(cv[2], n4.z, cv[3] * n4.w)));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0)
            static_cast<T*>(a.y)[b * a.sy_b + h * a.sy_h + p * a.sy_p] =
                Elem<T>::from_f(fmaf(Dh, xv, acc));
        if (++p == a.P) { p = 0; if (++h == a.H) { h = 0; ++b; } }
    }
}

template <typename T, int ROWS>
static void launch_step128(const SSDStepArgs& a, bool vbc, cudaStream_t st) {
    const int64_t warps = ((int64_t)a.Bsz * a.H * a.P + ROWS - 1) / ROWS;
    const unsigned blocks = (unsigned)((warps * 32 + 127) / 128);
    if (vbc) ssd_step128<T, ROWS, true><<<blocks, 128, 0, st>>>(a);
    else ssd_step128<T, ROWS, false><<<blocks, 128, 0, st>>>(a);
}

int launch_ssd_step(const SSDStepArgs& a, cudaStream_t st) {
    const int64_t rows = (int64_t)a.Bsz * a.H * a.P;
    const bool vec = a.N == 128 && a.ss_n == 1 && reinterpret_cast<uintptr_t>(a.state) % 16 == 0 &&
                     a.ss_p % 4 == 0 && a.ss_h % 4 == 0 && a.ss_b % 4 == 0 &&
                     rows * 32 < ((int64_t)1 << 31);
    if (vec) {
        const size_t esz = a.dtype == SS_BF16 ? 2 : 4;
        auto aligned4 = [&](const void* ptr, int64_t sb, int64_t sg, int64_t sn) {
            return sn == 1 && reinterpret_cast<uintptr_t>(ptr) % (4 * esz) == 0 && sb % 4 == 0 &&
                   sg % 4 == 0;
        };
        const bool vbc = aligned4(a.Bm, a.sB_b, a.sB_g, a.sB_n) &&
                         aligned4(a.Cm, a.sC_b, a.sC_g, a.sC_n);
        // four rows per warp: 1.5x faster than one at 4 x 64 heads x 64
        if (a.dtype == SS_BF16) launch_step128<__nv_bfloat16, 4>(a, vbc, st);
        else launch_step128<float, 4>(a, vbc, st);
    } else {
        const unsigned blocks = (unsigned)((rows * 32 + 127) / 128);
        if (a.dtype == SS_BF16) ssd_step<__nv_bfloat16><<<blocks, 128, 0, st>>>(a);
        else ssd_step<float><<<blocks, 128, 0, st>>>(a);
    }
    count_launch(1);
    return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_LAUNCH;
}

}  // namespace ss
