// selective_scan_bwd.cu -- backward pass of the selective scan (training).
//
// Reverse-mode derivative of the forward scan (page "Mamba模型笔记" §2.2
// recurrence, §4.3 gate; 0539edu paper talk §2.3 discretisation; §5.4:
// intermediate states are recomputed instead of stored).  Given the gradient
// dout of the scan's output, with pre_t = sum_n C h_t + D u_t:
//
//   dpre_t = dout_t silu(z_t);  dz_t = dout_t pre_t silu'(z_t)
//   g_t    = C_t dpre_t + abar_{t+1} g_{t+1}                 (adjoint state)
//   dC_t  += dpre_t h_t;  dB_t += g_t dl_t u_t;  dD += dpre_t u_t
//   du_t   = D dpre_t + sum_n g_t dl_t B_t
//   dA    += g_t h_{t-1} abar_t dl_t
//   ddl_t  = sum_n g_t (h_{t-1} abar_t A + B_t u_t);  ddelta_t = ddl_t softplus'(.)
//
// One CTA = 16 channels of one batch row x 16 lanes (one state each, N <= 16).
// Sweep 1 runs the recurrence forward and stores the state every K = 32 steps
// (stream-ordered scratch).  Sweep 2 walks the chunks backwards: it recomputes
// the chunk's states into registers from the stored one, then steps t down
// with the adjoint.  Sums over n are 16-lane shuffles; dB and dC are reduced
// over the CTA's channels in shared memory and added to global memory
// atomically, dA, dD and ddelta_bias are added atomically over batch rows.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"
#include "ssscan.h"

namespace ss {

namespace bwd {

constexpr int NL = 16;      // lanes (states) per channel
constexpr int CH = 16;      // channels per CTA
constexpr int K = 32;       // steps per recompute chunk
constexpr int NTHREADS = NL * CH;

__device__ __forceinline__ float sum16(float v) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <typename T>
__global__ void __launch_bounds__(NTHREADS) scan_bwd(BwdArgs a) {
    // per warp (two channels, summed by one shuffle) and step of the chunk
    __shared__ float sdB[CH / 2][NL][K];
    __shared__ float sdC[CH / 2][NL][K];

    const int tid = threadIdx.x, n = tid % NL, ch = tid / NL;
    const int dgroups = (a.D + CH - 1) / CH;
    const int b = blockIdx.x / dgroups;
    const int d = (blockIdx.x % dgroups) * CH + ch;
    const bool valid = d < a.D;
    const bool live = valid && n < a.N;
    const int L = a.L;
    const int nchunk = (L + K - 1) / K;

    const float An = live ? a.A[d * a.sA_d + n * a.sA_n] : 0.f;
    const float A2 = An * kLog2e;
    const float Dd = (valid && a.Dv) ? a.Dv[d * a.sD] : 0.f;
    const float bd = (valid && a.bias) ? a.bias[d * a.sbias] : 0.f;
    const int dsafe = valid ? d : 0;
    const T* u = static_cast<const T*>(a.u) + b * a.su_b + dsafe * a.su_d;
    const T* dl = static_cast<const T*>(a.dl) + b * a.sdl_b + dsafe * a.sdl_d;
    const T* z = a.z ? static_cast<const T*>(a.z) + b * a.sz_b + dsafe * a.sz_d : nullptr;
    const T* go = static_cast<const T*>(a.dout) + b * a.sg_b + dsafe * a.sg_d;
    const T* Bp = static_cast<const T*>(a.Bm) + b * a.sB_b + (live ? n : 0) * a.sB_n;
    const T* Cp = static_cast<const T*>(a.Cm) + b * a.sC_b + (live ? n : 0) * a.sC_n;
    // checkpoints: state before chunk c at ck[c * NL]
    float* ck = a.ckpt + (((int64_t)b * a.D + dsafe) * (nchunk + 1)) * NL + n;

    auto delta_at = [&](int t) {
        float x = Elem<T>::to_f(dl[t * a.sdl_t]) + bd;
        return a.softplus ? softplus_f(x) : x;
    };

    // ---- sweep 1: forward, storing the state at every chunk start
    {
        float h = 0.f;
        if (valid) ck[0] = 0.f;
        for (int c = 0; c < nchunk; ++c) {
            const int t0 = c * K, tn = min(K, L - t0);
#pragma unroll 4
            for (int j = 0; j < tn; ++j) {
                const int t = t0 + j;
                const float dd = delta_at(t);
                const float bn = live ? Elem<T>::to_f(Bp[t * a.sB_t]) : 0.f;
                h = fmaf(ex2_approx(dd * A2), h, dd * bn * Elem<T>::to_f(u[t * a.su_t]));
            }
            if (valid) ck[(c + 1) * NL] = h;
        }
    }

    // ---- sweep 2: backward
    float g = 0.f, dAacc = 0.f, dDacc = 0.f, dbacc = 0.f;
    for (int c = nchunk - 1; c >= 0; --c) {
        const int t0 = c * K, tn = min(K, L - t0);
        const float hprev = valid ? ck[c * NL] : 0.f;
        float hs[K], ds[K];
        {
            float h = hprev;
#pragma unroll
            for (int j = 0; j < K; ++j) {
                if (j < tn) {
                    const int t = t0 + j;
                    const float dd = delta_at(t);
                    const float bn = live ? Elem<T>::to_f(Bp[t * a.sB_t]) : 0.f;
                    h = fmaf(ex2_approx(dd * A2), h, dd * bn * Elem<T>::to_f(u[t * a.su_t]));
                    ds[j] = dd;
                } else {
                    ds[j] = 0.f;
                }
                hs[j] = h;
            }
        }
#pragma unroll
        for (int j = K - 1; j >= 0; --j) {
            if (j < tn) {
                const int t = t0 + j;
                const float dd = ds[j];
                const float ht = hs[j];
                const float hm = j > 0 ? hs[j - 1] : hprev;
                const float abar = ex2_approx(dd * A2);
                const float uu = Elem<T>::to_f(u[t * a.su_t]);
                const float bn = live ? Elem<T>::to_f(Bp[t * a.sB_t]) : 0.f;
                const float cn = live ? Elem<T>::to_f(Cp[t * a.sC_t]) : 0.f;
                const float gout = Elem<T>::to_f(go[t * a.sg_t]);
                const float pre = sum16(cn * ht) + Dd * uu;
                float dpre = gout, dzv = 0.f;
                if (z) {
                    const float zz = Elem<T>::to_f(z[t * a.sz_t]);
                    const float sg = sigmoid_accurate(zz);
                    dpre = gout * zz * sg;
                    dzv = gout * pre * (sg + zz * sg * (1.f - sg));
                }
                g = fmaf(cn, dpre, g);
                float vc = dpre * ht, vb = g * dd * uu;
                vc += __shfl_xor_sync(0xffffffffu, vc, 16);
                vb += __shfl_xor_sync(0xffffffffu, vb, 16);
                if (ch % 2 == 0) {
                    sdC[ch / 2][n][j] = vc;
                    sdB[ch / 2][n][j] = vb;
                }
                const float dut = sum16(g * dd * bn) + Dd * dpre;
                const float ddl = sum16(g * fmaf(hm * abar, An, bn * uu));
                dAacc = fmaf(g * hm * abar, dd, dAacc);
                float ddx = ddl;
                if (a.softplus) {
                    const float x = Elem<T>::to_f(dl[t * a.sdl_t]) + bd;
                    ddx = ddl * sigmoid_accurate(x);
                }
                if (n == 0 && valid) {
                    dDacc = fmaf(dpre, uu, dDacc);
                    dbacc += ddx;
                    static_cast<T*>(a.du)[b * a.sdu_b + d * a.sdu_d + t * a.sdu_t] = Elem<T>::from_f(dut);
                    static_cast<T*>(a.ddl)[b * a.sddl_b + d * a.sddl_d + t * a.sddl_t] =
                        Elem<T>::from_f(ddx);
                    if (z)
                        static_cast<T*>(a.dz)[b * a.sdz_b + d * a.sdz_d + t * a.sdz_t] =
                            Elem<T>::from_f(dzv);
                }
                g *= abar;
            }
        }
        __syncthreads();
        // dB, dC of this chunk: sum over the CTA's channels, then one atomic add
        for (int idx = tid; idx < NL * K; idx += NTHREADS) {
            const int nn = idx / K, j = idx % K;
            if (nn < a.N && j < tn) {
                float sb = 0.f, sc = 0.f;
#pragma unroll
                for (int q = 0; q < CH / 2; ++q) {
                    sb += sdB[q][nn][j];
                    sc += sdC[q][nn][j];
                }
                atomicAdd(a.dB + ((int64_t)b * a.N + nn) * L + t0 + j, sb);
                atomicAdd(a.dC + ((int64_t)b * a.N + nn) * L + t0 + j, sc);
            }
        }
        __syncthreads();
    }
    if (live) atomicAdd(a.dA + d * a.N + n, dAacc);
    if (valid && n == 0) {
        if (a.dD) atomicAdd(a.dD + d, dDacc);
        if (a.dbias) atomicAdd(a.dbias + d, dbacc);
    }
}

}  // namespace bwd

int launch_selective_bwd(const BwdArgs& args, cudaStream_t st, const Scratch& scratch) {
    BwdArgs a = args;
    // the fp32 sums start from zero (and stay zero when there is nothing to scan)
    const size_t nA = (size_t)a.D * a.N, nBC = (size_t)a.Bsz * a.N * a.L;
    if ((nA && cudaMemsetAsync(a.dA, 0, sizeof(float) * nA, st) != cudaSuccess) ||
        (nBC && cudaMemsetAsync(a.dB, 0, sizeof(float) * nBC, st) != cudaSuccess) ||
        (nBC && cudaMemsetAsync(a.dC, 0, sizeof(float) * nBC, st) != cudaSuccess) ||
        (a.dD && a.D && cudaMemsetAsync(a.dD, 0, sizeof(float) * a.D, st) != cudaSuccess) ||
        (a.dbias && a.D && cudaMemsetAsync(a.dbias, 0, sizeof(float) * a.D, st) != cudaSuccess))
        return SS_ERR_CUDA;
    if (a.L == 0 || a.Bsz == 0 || a.D == 0) return SS_OK;
    const int nchunk = (a.L + bwd::K - 1) / bwd::K;
    const size_t bytes = (size_t)a.Bsz * a.D * (nchunk + 1) * bwd::NL * sizeof(float);
    void* ck = scratch.alloc(bytes, st, scratch.ctx);
    if (!ck) return SS_ERR_ALLOC;
    a.ckpt = static_cast<float*>(ck);
    const int dgroups = (a.D + bwd::CH - 1) / bwd::CH;
    const unsigned grid = (unsigned)((int64_t)a.Bsz * dgroups);
    if (a.dtype == SS_BF16) bwd::scan_bwd<__nv_bfloat16><<<grid, bwd::NTHREADS, 0, st>>>(a);
    else bwd::scan_bwd<float><<<grid, bwd::NTHREADS, 0, st>>>(a);
    count_launch(1);
    const cudaError_t e = cudaGetLastError();
    scratch.release(ck, st, scratch.ctx);
    return e == cudaSuccess ? SS_OK : SS_ERR_LAUNCH;
}

}  // namespace ss
