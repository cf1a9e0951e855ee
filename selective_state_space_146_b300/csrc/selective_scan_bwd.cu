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
// Two kernels:
//  * scan_bwd_fast (N = 16, unit t-stride, 16-byte aligned rows): one CTA per
//    32 channels of a batch row, four lanes per channel, each lane keeping four
//    states.  Activations arrive as 128-byte-swizzled TMA tiles (64 bf16 or 32
//    fp32 steps), double buffered.  Pass 1 runs the recurrence forward over the
//    tiles and stores the state every 8 steps (stream-ordered scratch); given
//    those states from the forward (ss_selective_scan_bwd_ckpt) it skips this
//    pass.  Pass 2 walks the tiles backwards; for each 8-step sub-chunk it
//    recomputes the states into registers from the stored one (loaded two
//    sub-chunks ahead), then steps t down with the adjoint.  Sums over the
//    four lanes of a channel are two xor-shuffles; dB
//    and dC are reduce-scattered over the eight channels of a warp, summed over
//    the CTA's warps in shared memory and written as per-CTA partial sums;
//    du / ddelta / dz leave through TMA stores.  scan_bwd_finish then adds the
//    partials of dB, dC (over channel blocks) and of dA, dD, ddelta_bias (over
//    batch rows) in a fixed order, so the result does not depend on timing.
//  * scan_bwd (any strides, N <= 16): one lane per state, 16 channels per CTA,
//    dB / dC reduced in shared memory and added with atomics.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>

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


// ---------------------------------------------------------------------------
// scan_bwd_fast

namespace bwdf {

template <typename T>
struct Cfg {
    static constexpr int ES = (int)sizeof(T);
    static constexpr int N = 16;
    static constexpr int TT = 128 / ES;        // steps per tile: one swizzle row
    static constexpr int KS = 8;               // steps per recompute sub-chunk
    static constexpr int NSUB = TT / KS;
    static constexpr int CH = 32;              // channels per CTA
    static constexpr int NTHREADS = CH * 4;    // four lanes per channel
    static constexpr int NWARPS = NTHREADS / 32;
    static constexpr int ACT = CH * 128;       // one activation tile
    static constexpr int RAWBC = N * 128;      // one raw B or C tile ([n][t])
    static constexpr int OFF_U = 0, OFF_DL = ACT, OFF_Z = 2 * ACT, OFF_G = 3 * ACT;
    static constexpr int OFF_B = 4 * ACT, OFF_C = 4 * ACT + RAWBC;
    static constexpr int STAGE = 4 * ACT + 2 * RAWBC;
    static constexpr int OFF_TAB = 2 * STAGE;               // fp32 [t][B 0..15 | C 0..15]
    static constexpr int OFF_OUT = OFF_TAB + TT * 128;      // du, ddelta, dz tiles
    static constexpr int RED = NWARPS * KS * 32 * 4;        // [warp][KS][32] fp32
    static constexpr int OFF_RED = OFF_OUT + 3 * ACT;       // two of them, alternating
    static constexpr int OFF_BAR = OFF_RED + 2 * RED;
    static constexpr int SMEM = OFF_BAR + 64 + 1024;
    static constexpr int NV = 2 * N;                        // dB and dC values per step
    static_assert(STAGE % 1024 == 0 && OFF_OUT % 1024 == 0, "swizzled tiles 1024-aligned");
    static_assert(3 * SMEM <= 228 * 1024, "three CTAs per SM");
};

struct Params {
    int Bsz, D, L, ntiles, dgroups, softplus;
    const float* A; int64_t sA_d, sA_n;
    const float* Dv; int64_t sD;
    const float* bias; int64_t sbias;
    float* ckpt;      // [b][d][L/8 rounded up][16]: the state before each sub-chunk
    int ck_given;     // ckpt holds the forward's states: no forward pass here
    float* part;      // [dgroup][b][t][32]: dB (n) then dC (n), summed over a CTA
    float* partA;     // [b][d][16]
    float* partD;     // [b][d]
    float* partbias;  // [b][d]
    unsigned* err;
};

// Raw B (and C) of one tile, [n][t] in T, into the fp32 table [t][32]
// (B[0..15] then C[0..15]).  Warp w converts rows n = (lane + it) & 15 for
// it = w, w + NWARPS, ...: a lane reads one 32-bit word of a raw row (distinct
// banks across the warp) and writes its one or two steps.
template <typename T, int NWARPS>
__device__ __forceinline__ void convert_table(uint32_t rawB, uint32_t rawC, uint32_t tab,
                                              bool with_c, int warp, int lane) {
    for (int it = warp; it < (with_c ? 32 : 16); it += NWARPS) {
        const int n = (lane + it) & 15;
        const uint32_t src = (it < 16 ? rawB : rawC) + n * 128 + lane * 4;
        const uint32_t col = ((it < 16 ? 0 : 16) + n) * 4;
        const uint32_t w = lds32(src);
        if constexpr (sizeof(T) == 2) {
            asm volatile("st.shared.b32 [%0], %1;" ::"r"(tab + (2 * lane) * 128 + col),
                         "r"(w << 16) : "memory");
            asm volatile("st.shared.b32 [%0], %1;" ::"r"(tab + (2 * lane + 1) * 128 + col),
                         "r"(w & 0xffff0000u) : "memory");
        } else {
            asm volatile("st.shared.b32 [%0], %1;" ::"r"(tab + lane * 128 + col), "r"(w)
                         : "memory");
        }
    }
}

// One round of a reduce-scatter across lanes lane and lane ^ m: keep one half
// of v (the upper one if `upper`), add the partner's copy of that half.
template <int LEN>
__device__ __forceinline__ void rs_half(const float* v, float* out, bool upper, int m) {
#pragma unroll
    for (int e = 0; e < LEN / 2; ++e) {
        const float lo = v[e], hi = v[LEN / 2 + e];
        out[e] = (upper ? hi : lo) + __shfl_xor_sync(0xffffffffu, upper ? lo : hi, m);
    }
}

template <typename T, bool HAS_Z>
__global__ void __launch_bounds__(Cfg<T>::NTHREADS, 3)
scan_bwd_fast(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_dl,
              const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_g,
              const __grid_constant__ CUtensorMap tm_B, const __grid_constant__ CUtensorMap tm_C,
              const __grid_constant__ CUtensorMap tm_du, const __grid_constant__ CUtensorMap tm_ddl,
              const __grid_constant__ CUtensorMap tm_dz, const Params p) {
    using C = Cfg<T>;
    constexpr int ES = C::ES, TT = C::TT, KS = C::KS, NSUB = C::NSUB, NT = C::NTHREADS;
    static_assert(NT == 128, "four warps of eight channels");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t s0 = smem_u32(smem);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int sub = lane & 3;                 // states 4 sub .. 4 sub + 3
    const int ci = warp * 8 + (lane >> 2);    // channel row within the tile
    const int b = blockIdx.x / p.dgroups, dg = blockIdx.x % p.dgroups;
    const int d0 = dg * C::CH, d = d0 + ci;
    const bool valid = d < p.D;
    const int L = p.L, ntiles = p.ntiles, nkc = (L + KS - 1) / KS;

    float A2[4], An[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        An[s] = valid ? p.A[d * p.sA_d + (4 * sub + s) * p.sA_n] : 0.f;
        A2[s] = An[s] * kLog2e;
    }
    const float Dd = (valid && p.Dv) ? p.Dv[d * p.sD] : 0.f;
    const float biasd = (valid && p.bias) ? p.bias[d * p.sbias] : 0.f;
    const bool sp = p.softplus != 0;
    float* ck = p.ckpt + ((int64_t)b * p.D + (valid ? d : 0)) * nkc * 16 + 4 * sub;

    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        fence_mbar_init();
    }
    __syncthreads();

    // load q of 2 ntiles: pass 1 tile q, then pass 2 tile 2 ntiles - 1 - q.
    // With the forward's states given, pass 1 is skipped and the loads start
    // at q0 = ntiles; stages and barrier phases count from q0.
    const int q0 = p.ck_given ? ntiles : 0;
    auto issue = [&](int q) {
        if (q >= 2 * ntiles) return;
        const uint32_t st = C::STAGE * ((q - q0) & 1);
        uint64_t* bar = &full[(q - q0) & 1];
        uint8_t* base = smem + st;
        if (q < ntiles) {
            const int t0 = q * TT;
            mbar_arrive_expect_tx(bar, 2 * C::ACT + C::RAWBC);
            tma_load_3d(base + C::OFF_U, &tm_u, bar, t0, d0, b);
            tma_load_3d(base + C::OFF_DL, &tm_dl, bar, t0, d0, b);
            tma_load_3d(base + C::OFF_B, &tm_B, bar, t0, 0, b);
        } else {
            const int t0 = (2 * ntiles - 1 - q) * TT;
            mbar_arrive_expect_tx(bar, (HAS_Z ? 4 : 3) * C::ACT + 2 * C::RAWBC);
            tma_load_3d(base + C::OFF_U, &tm_u, bar, t0, d0, b);
            tma_load_3d(base + C::OFF_DL, &tm_dl, bar, t0, d0, b);
            if (HAS_Z) tma_load_3d(base + C::OFF_Z, &tm_z, bar, t0, d0, b);
            tma_load_3d(base + C::OFF_G, &tm_g, bar, t0, d0, b);
            tma_load_3d(base + C::OFF_B, &tm_B, bar, t0, 0, b);
            tma_load_3d(base + C::OFF_C, &tm_C, bar, t0, 0, b);
        }
    };
    if (tid == 0) {
        tma_prefetch_desc(&tm_u);
        tma_prefetch_desc(&tm_dl);
        tma_prefetch_desc(&tm_g);
        tma_prefetch_desc(&tm_B);
        tma_prefetch_desc(&tm_C);
        if (HAS_Z) tma_prefetch_desc(&tm_z);
        issue(q0);
        issue(q0 + 1);
    }

    const uint32_t tab = s0 + C::OFF_TAB;
    const uint32_t red = s0 + C::OFF_RED;
    int nred = 0;  // sub-chunks flushed so far (selects the reduction buffer)
    const uint32_t out = s0 + C::OFF_OUT;
    float dDacc = 0.f, dbacc = 0.f;
    // value this lane holds after the reduce-scatter over the warp's channels:
    // kind (lane bit 4: 0 = dB, 1 = dC) of state 4 sub + (lane bits 3..2)
    const int vidx = ((lane >> 4) & 1) * 16 + 4 * sub + ((lane >> 2) & 3);

    int consumed = q0;  // loads waited for
    // start of load q: wait for it (and, in pass 2, for the previous tile's
    // output stores to have left the out tiles), then build the B|C table
    auto begin = [&](int q) -> bool {
        bool ok = true;
        if (tid == 0) {
            ok = mbar_wait(&full[(q - q0) & 1], ((q - q0) >> 1) & 1, p.err);
            if (q >= ntiles + 1) bulk_wait_read<0>();
        }
        if (!__syncthreads_and(ok)) return false;
        consumed = q + 1;
        const uint32_t st = s0 + C::STAGE * ((q - q0) & 1);
        convert_table<T, C::NWARPS>(st + C::OFF_B, st + C::OFF_C, tab, q >= ntiles, warp, lane);
        __syncthreads();
        return true;
    };
    auto finish = [&](int q) {
        __syncthreads();  // the stage and the table are free
        if (tid == 0) issue(q + 2);
    };

    // Per 8-step sub-chunk kc of a tile, lane `sub` computes delta (and the
    // softplus slope) of steps 2 sub, 2 sub + 1 and the four lanes of the
    // channel exchange them.  Steps past the end get delta = 0 (no update) and
    // slope 0 (no gradient).
    auto deltas = [&](uint32_t st, int kc, int tn, float* dd, float* sg) {
        float x[2];
        if constexpr (ES == 2) {
            const uint32_t w = lds32(st + C::OFF_DL + (ci << 7) + ((kc ^ (ci & 7)) << 4) + sub * 4);
            x[0] = __uint_as_float(w << 16);
            x[1] = __uint_as_float(w & 0xffff0000u);
        } else {
            const uint2 w = lds64(st + C::OFF_DL + (ci << 7) + (((2 * kc + (sub >> 1)) ^ (ci & 7)) << 4) +
                                  (sub & 1) * 8);
            x[0] = __uint_as_float(w.x);
            x[1] = __uint_as_float(w.y);
        }
        float own_d[2], own_s[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const float xb = x[e] + biasd;
            const bool live = kc * KS + 2 * sub + e < tn;
            const float v = sp ? softplus_f(xb) : xb;
            own_d[e] = live ? v : 0.f;
            // softplus'(x) = sigmoid(x) = 1 - exp(-softplus(x))
            own_s[e] = live ? (sp ? 1.f - ex2_approx(-v * kLog2e) : 1.f) : 0.f;
        }
        const int gbase = lane & ~3;
#pragma unroll
        for (int j = 0; j < KS; ++j) {
            dd[j] = __shfl_sync(0xffffffffu, own_d[j & 1], gbase + (j >> 1));
            if (sg) sg[j] = __shfl_sync(0xffffffffu, own_s[j & 1], gbase + (j >> 1));
        }
    };
    // the KS elements of an activation tile row for sub-chunk kc, widened
    auto load8 = [&](uint32_t tile, int kc, float* v) {
        if constexpr (ES == 2) {
            const uint4 w = lds128(tile + (ci << 7) + ((kc ^ (ci & 7)) << 4));
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[2 * i] = __uint_as_float(ww[i] << 16);
                v[2 * i + 1] = __uint_as_float(ww[i] & 0xffff0000u);
            }
        } else {
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const float4 w = lds128f(tile + (ci << 7) + (((2 * kc + h2) ^ (ci & 7)) << 4));
                v[4 * h2] = w.x; v[4 * h2 + 1] = w.y; v[4 * h2 + 2] = w.z; v[4 * h2 + 3] = w.w;
            }
        }
    };
    const float2 A2p[2] = {make_float2(A2[0], A2[1]), make_float2(A2[2], A2[3])};
    const float2 Anp[2] = {make_float2(An[0], An[1]), make_float2(An[2], An[3])};

    bool ok = true;
    {
        // ---- pass 1: forward, store the state before every sub-chunk
        float2 h2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        for (int q = 0; q < ntiles && ok && !p.ck_given; ++q) {
            if (!(ok = begin(q))) break;
            const uint32_t st = s0 + C::STAGE * (q & 1);
            const int t0 = q * TT, tn = min(TT, L - t0);
#pragma unroll 1
            for (int kc = 0; kc < NSUB; ++kc) {
                if (t0 + kc * KS >= L) break;
                if (valid)
                    *reinterpret_cast<float4*>(ck + (int64_t)(t0 / KS + kc) * 16) =
                        make_float4(h2[0].x, h2[0].y, h2[1].x, h2[1].y);
                float dd[KS], uf[KS];
                deltas(st, kc, tn, dd, nullptr);
                load8(st + C::OFF_U, kc, uf);
#pragma unroll
                for (int jj = 0; jj < KS; ++jj) {
                    const int j = kc * KS + jj;
                    const float4 Bv = lds128f(tab + j * 128 + sub * 16);
                    const float du = dd[jj] * uf[jj];
                    const float2 d2 = make_float2(dd[jj], dd[jj]), du2 = make_float2(du, du);
                    const float2 bv2[2] = {make_float2(Bv.x, Bv.y), make_float2(Bv.z, Bv.w)};
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const float2 ar = __fmul2_rn(d2, A2p[k]);
                        const float2 ab = make_float2(ex2_approx(ar.x), ex2_approx(ar.y));
                        h2[k] = __ffma2_rn(ab, h2[k], __fmul2_rn(du2, bv2[k]));
                    }
                }
            }
            finish(q);
        }
    }
    float2 g2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    float2 dA2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    // the stored states of the next two sub-chunks to process (sub-chunks go
    // from the last to the first), loaded two sub-chunks ahead: one ahead
    // left the load's latency exposed (0.93 -> 0.86 ms at the layer shape)
    auto load_ck = [&](int kcg) {
        return (valid && kcg >= 0) ? *reinterpret_cast<const float4*>(ck + (int64_t)kcg * 16)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    float4 ck_next = load_ck(nkc - 1), ck_next2 = load_ck(nkc - 2);
    for (int q = ntiles; q < 2 * ntiles && ok; ++q) {
        if (!(ok = begin(q))) break;
        const uint32_t st = s0 + C::STAGE * ((q - q0) & 1);
        const int tile = 2 * ntiles - 1 - q;
        const int t0 = tile * TT, tn = min(TT, L - t0);
        // ---- pass 2: backward over the tile's sub-chunks, last first
#pragma unroll 1
        for (int kc = NSUB - 1; kc >= 0; --kc) {
            const int tb = kc * KS;
            if (t0 + tb >= L) continue;
            const uint32_t redb = red + (nred & 1) * C::RED;
            const float2 hc2[2] = {make_float2(ck_next.x, ck_next.y),
                                   make_float2(ck_next.z, ck_next.w)};
            ck_next = ck_next2;
            ck_next2 = load_ck(t0 / KS + kc - 2);
            float ds[KS], sg[KS], uf[KS], gf[KS], zf[KS];
            deltas(st, kc, tn, ds, sg);
            load8(st + C::OFF_U, kc, uf);
            load8(st + C::OFF_G, kc, gf);
            if (HAS_Z) load8(st + C::OFF_Z, kc, zf);
            // recompute the sub-chunk's states
            float2 hs2[2][KS];
            {
                float2 hr[2] = {hc2[0], hc2[1]};
#pragma unroll
                for (int jj = 0; jj < KS; ++jj) {
                    const float4 Bv = lds128f(tab + (tb + jj) * 128 + sub * 16);
                    const float du = ds[jj] * uf[jj];
                    const float2 d2 = make_float2(ds[jj], ds[jj]), du2 = make_float2(du, du);
                    const float2 bv2[2] = {make_float2(Bv.x, Bv.y), make_float2(Bv.z, Bv.w)};
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const float2 ar = __fmul2_rn(d2, A2p[k]);
                        const float2 ab = make_float2(ex2_approx(ar.x), ex2_approx(ar.y));
                        hr[k] = __ffma2_rn(ab, hr[k], __fmul2_rn(du2, bv2[k]));
                        hs2[k][jj] = hr[k];
                    }
                }
            }
            // adjoint sweep, t descending; lane `sub` keeps output `sub` of each
            // step (du, ddelta, dz)
            float outv[KS];
#pragma unroll
            for (int jj = KS - 1; jj >= 0; --jj) {
                const int j = tb + jj;
                const float dd = ds[jj], uu = uf[jj], go = gf[jj];
                const float4 Bv = lds128f(tab + j * 128 + sub * 16);
                const float4 Cv = lds128f(tab + j * 128 + 64 + sub * 16);
                const float2 bv2[2] = {make_float2(Bv.x, Bv.y), make_float2(Bv.z, Bv.w)};
                const float2 cv2[2] = {make_float2(Cv.x, Cv.y), make_float2(Cv.z, Cv.w)};
                float dpre = go, zz = 0.f, sz = 0.f;
                if (HAS_Z) {
                    zz = zf[jj];
                    sz = sigmoid_accurate(zz);
                    dpre = go * zz * sz;
                }
                const float ddu = dd * uu;
                const float2 d2 = make_float2(dd, dd), dpre2 = make_float2(dpre, dpre);
                const float2 ddu2 = make_float2(ddu, ddu);
                float2 pre2 = make_float2(0.f, 0.f), gb2 = pre2, ga2 = pre2;
                float v[8];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const float2 ht = hs2[k][jj];
                    const float2 hm = jj > 0 ? hs2[k][jj > 0 ? jj - 1 : 0] : hc2[k];
                    const float2 ar = __fmul2_rn(d2, A2p[k]);
                    const float2 ab = make_float2(ex2_approx(ar.x), ex2_approx(ar.y));
                    pre2 = __ffma2_rn(cv2[k], ht, pre2);
                    g2[k] = __ffma2_rn(cv2[k], dpre2, g2[k]);
                    const float2 qv = __fmul2_rn(g2[k], __fmul2_rn(hm, ab));  // g h_{t-1} abar
                    dA2[k] = __ffma2_rn(qv, d2, dA2[k]);
                    ga2 = __ffma2_rn(qv, Anp[k], ga2);
                    gb2 = __ffma2_rn(g2[k], bv2[k], gb2);
                    const float2 vb = __fmul2_rn(g2[k], ddu2);   // dB
                    const float2 vc = __fmul2_rn(dpre2, ht);      // dC
                    v[2 * k] = vb.x; v[2 * k + 1] = vb.y;
                    v[4 + 2 * k] = vc.x; v[4 + 2 * k + 1] = vc.y;
                    g2[k] = __fmul2_rn(g2[k], ab);
                }
                float pre_p = pre2.x + pre2.y, gb = gb2.x + gb2.y, ga = ga2.x + ga2.y;
#pragma unroll
                for (int m = 1; m <= 2; m <<= 1) {
                    pre_p += __shfl_xor_sync(0xffffffffu, pre_p, m);
                    gb += __shfl_xor_sync(0xffffffffu, gb, m);
                    ga += __shfl_xor_sync(0xffffffffu, ga, m);
                }
                const float dut = fmaf(dd, gb, Dd * dpre);
                const float ddx = fmaf(uu, gb, ga) * sg[jj];
                dDacc = fmaf(dpre, uu, dDacc);
                dbacc += ddx;
                float dzv = 0.f;
                if (HAS_Z) dzv = go * fmaf(Dd, uu, pre_p) * (sz + zz * sz * (1.f - sz));
                outv[jj] = sub == 0 ? dut : (sub == 1 ? ddx : dzv);
                float v4[4], vv2[2], v1[1];
                rs_half<8>(v, v4, lane & 16, 16);
                rs_half<4>(v4, vv2, lane & 8, 8);
                rs_half<2>(vv2, v1, lane & 4, 4);
                asm volatile("st.shared.b32 [%0], %1;"
                             ::"r"(redb + ((warp * KS + jj) * 32 + vidx) * 4),
                             "r"(__float_as_uint(v1[0])) : "memory");
            }
            if (sub < (HAS_Z ? 3 : 2)) {
                const uint32_t row = out + sub * C::ACT + (ci << 7);
                if constexpr (ES == 2) {
                    uint32_t w[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        __nv_bfloat162 h = __floats2bfloat162_rn(outv[2 * i], outv[2 * i + 1]);
                        w[i] = *reinterpret_cast<uint32_t*>(&h);
                    }
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                                 ::"r"(row + ((kc ^ (ci & 7)) << 4)), "r"(w[0]), "r"(w[1]),
                                 "r"(w[2]), "r"(w[3]) : "memory");
                } else {
                    sts128f(row + (((2 * kc) ^ (ci & 7)) << 4),
                            make_float4(outv[0], outv[1], outv[2], outv[3]));
                    sts128f(row + (((2 * kc + 1) ^ (ci & 7)) << 4),
                            make_float4(outv[4], outv[5], outv[6], outv[7]));
                }
            }
            __syncthreads();
            // this sub-chunk's dB / dC, summed over the CTA's warps
            for (int e = tid; e < KS * 32; e += NT) {
                const int jj = e >> 5, vv = e & 31;
                const int t = t0 + tb + jj;
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < C::NWARPS; ++w)
                    sum += __uint_as_float(lds32(redb + ((w * KS + jj) * 32 + vv) * 4));
                if (t < L) p.part[(((int64_t)dg * p.Bsz + b) * L + t) * 32 + vv] = sum;
            }
            // no barrier here: the next sub-chunk writes the other buffer, and
            // the barrier after it orders this flush before the one after that
            ++nred;
        }
        // du / ddelta / dz of the tile leave through TMA stores (clipped at
        // the tensor's edges)
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            tma_store_3d(&tm_du, smem + C::OFF_OUT, t0, d0, b);
            tma_store_3d(&tm_ddl, smem + C::OFF_OUT + C::ACT, t0, d0, b);
            if (HAS_Z) tma_store_3d(&tm_dz, smem + C::OFF_OUT + 2 * C::ACT, t0, d0, b);
            bulk_commit();
        }
        finish(q);
    }
    const float dA[4] = {dA2[0].x, dA2[0].y, dA2[1].x, dA2[1].y};
    if (tid == 0) bulk_wait<0>();
    if (!ok) {
        // a load never arrived: wait (bounded) for the ones still in flight
        if (tid == 0)
            for (int k = consumed; k < min(consumed + 2, 2 * ntiles); ++k)
                mbar_wait(&full[(k - q0) & 1], ((k - q0) >> 1) & 1, p.err);
        return;
    }
    if (!valid) return;
    const int64_t bd = (int64_t)b * p.D + d;
    *reinterpret_cast<float4*>(p.partA + bd * 16 + 4 * sub) = make_float4(dA[0], dA[1], dA[2], dA[3]);
    if (sub == 0) {
        p.partD[bd] = dDacc;
        p.partbias[bd] = dbacc;
    }
}

// dB, dC summed over channel blocks; dA, dD, ddelta_bias over batch rows.
__global__ void __launch_bounds__(256) scan_bwd_finish(Params p, int dgroups, float* dB, float* dC,
                                                      float* dAo, float* dDo, float* dbo) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nbc = (int64_t)p.Bsz * p.L * 32;
    const int64_t L = p.L;
    if (i < nbc) {
        const int v = (int)(i & 31);
        const int64_t bt = i >> 5;  // b * L + t
        float sum = 0.f;
        for (int k = 0; k < dgroups; ++k) sum += p.part[((int64_t)k * p.Bsz * L) * 32 + i];
        const int64_t b = bt / L, t = bt % L;
        float* dst = v < 16 ? dB : dC;
        dst[(b * 16 + (v & 15)) * L + t] = sum;
        return;
    }
    int64_t r = i - nbc;
    if (r < (int64_t)p.D * 16) {
        float sum = 0.f;
        for (int bb = 0; bb < p.Bsz; ++bb) sum += p.partA[(int64_t)bb * p.D * 16 + r];
        dAo[r] = sum;
        return;
    }
    r -= (int64_t)p.D * 16;
    if (r < p.D) {
        float sd = 0.f, sb = 0.f;
        for (int bb = 0; bb < p.Bsz; ++bb) {
            sd += p.partD[(int64_t)bb * p.D + r];
            sb += p.partbias[(int64_t)bb * p.D + r];
        }
        if (dDo) dDo[r] = sd;
        if (dbo) dbo[r] = sb;
    }
}

}  // namespace bwdf

static bool bwd_fast_ok(const BwdArgs& a) {
    if (a.N != 16 || a.L >= (1 << 30)) return false;
    const int es = a.dtype == SS_BF16 ? 2 : 4;
    auto row_ok = [&](const void* ptr, int64_t sb, int64_t sr, int64_t st) {
        if (!ptr) return true;
        if (st != 1 && a.L > 1) return false;
        if (reinterpret_cast<uintptr_t>(ptr) % 16) return false;
        if ((sr * es) % 16 || (sb * es) % 16) return false;
        return sr * es < (int64_t(1) << 40) && sb * es < (int64_t(1) << 40);
    };
    return row_ok(a.u, a.su_b, a.su_d, a.su_t) && row_ok(a.dl, a.sdl_b, a.sdl_d, a.sdl_t) &&
           row_ok(a.z, a.sz_b, a.sz_d, a.sz_t) && row_ok(a.dout, a.sg_b, a.sg_d, a.sg_t) &&
           row_ok(a.Bm, a.sB_b, a.sB_n, a.sB_t) && row_ok(a.Cm, a.sC_b, a.sC_n, a.sC_t) &&
           row_ok(a.du, a.sdu_b, a.sdu_d, a.sdu_t) && row_ok(a.ddl, a.sddl_b, a.sddl_d, a.sddl_t) &&
           row_ok(a.dz, a.sdz_b, a.sdz_d, a.sdz_t);
}

template <typename T>
static int run_bwd_fast(const BwdArgs& a, cudaStream_t st, const Scratch& scratch) {
    using C = bwdf::Cfg<T>;
    const int TT = C::TT;
    CUtensorMap m[9];
    const bool has_z = a.z != nullptr;
    if (!make_map_3d(&m[0], a.u, a.dtype, a.L, a.D, a.Bsz, a.su_d, a.su_b, TT, C::CH) ||
        !make_map_3d(&m[1], a.dl, a.dtype, a.L, a.D, a.Bsz, a.sdl_d, a.sdl_b, TT, C::CH) ||
        !make_map_3d(&m[3], a.dout, a.dtype, a.L, a.D, a.Bsz, a.sg_d, a.sg_b, TT, C::CH) ||
        !make_map_3d(&m[4], a.Bm, a.dtype, a.L, 16, a.Bsz, a.sB_n, a.sB_b, TT, 16, false) ||
        !make_map_3d(&m[5], a.Cm, a.dtype, a.L, 16, a.Bsz, a.sC_n, a.sC_b, TT, 16, false) ||
        !make_map_3d(&m[6], a.du, a.dtype, a.L, a.D, a.Bsz, a.sdu_d, a.sdu_b, TT, C::CH) ||
        !make_map_3d(&m[7], a.ddl, a.dtype, a.L, a.D, a.Bsz, a.sddl_d, a.sddl_b, TT, C::CH))
        return -1;
    if (has_z) {
        if (!make_map_3d(&m[2], a.z, a.dtype, a.L, a.D, a.Bsz, a.sz_d, a.sz_b, TT, C::CH) ||
            !make_map_3d(&m[8], a.dz, a.dtype, a.L, a.D, a.Bsz, a.sdz_d, a.sdz_b, TT, C::CH))
            return -1;
    } else {
        m[2] = m[0];
        m[8] = m[6];  // never used without z
    }
    const int dgroups = (a.D + C::CH - 1) / C::CH;
    const int nkc = (a.L + C::KS - 1) / C::KS;
    const size_t n_ck = a.ckpt_in ? 0 : (size_t)a.Bsz * a.D * nkc * 16;
    const size_t n_part = (size_t)dgroups * a.Bsz * a.L * 32;
    const size_t n_pa = (size_t)a.Bsz * a.D * 16, n_pd = (size_t)a.Bsz * a.D;
    const size_t bytes = sizeof(float) * (n_ck + n_part + n_pa + 2 * n_pd);
    float* base = static_cast<float*>(scratch.alloc(bytes, st, scratch.ctx));
    if (!base) return SS_ERR_ALLOC;
    bwdf::Params p{};
    p.Bsz = a.Bsz; p.D = a.D; p.L = a.L; p.ntiles = (a.L + TT - 1) / TT; p.dgroups = dgroups;
    p.softplus = a.softplus;
    p.A = a.A; p.sA_d = a.sA_d; p.sA_n = a.sA_n;
    p.Dv = a.Dv; p.sD = a.sD;
    p.bias = a.bias; p.sbias = a.sbias;
    p.ckpt = a.ckpt_in ? const_cast<float*>(a.ckpt_in) : base;  // given: only read
    p.ck_given = a.ckpt_in ? 1 : 0;
    p.part = base + n_ck;
    p.partA = p.part + n_part;
    p.partD = p.partA + n_pa;
    p.partbias = p.partD + n_pd;
    p.err = a.err;
    auto kern = has_z ? bwdf::scan_bwd_fast<T, true> : bwdf::scan_bwd_fast<T, false>;
    static bool attr_set[2][64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    const int zi = has_z ? 1 : 0;
    if (dev < 0 || dev >= 64 || !attr_set[zi][dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
                cudaSuccess ||
            cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) !=
                cudaSuccess) {
            scratch.release(base, st, scratch.ctx);
            return SS_ERR_LAUNCH;
        }
        if (dev >= 0 && dev < 64) attr_set[zi][dev] = true;
    }
    kern<<<(unsigned)((int64_t)a.Bsz * dgroups), C::NTHREADS, C::SMEM, st>>>(
        m[0], m[1], m[2], m[3], m[4], m[5], m[6], m[7], m[8], p);
    const int64_t total = (int64_t)a.Bsz * a.L * 32 + (int64_t)a.D * 16 + a.D;
    bwdf::scan_bwd_finish<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(p, dgroups, a.dB, a.dC,
                                                                          a.dA, a.dD, a.dbias);
    count_launch(2);
    const cudaError_t e = cudaGetLastError();
    scratch.release(base, st, scratch.ctx);
    return e == cudaSuccess ? SS_OK : SS_ERR_LAUNCH;
}

// A call with unit t-strides whose rows are not 16-byte aligned (an odd L in
// bf16, for one) runs scan_bwd_fast on padded copies: u, delta, z, dout, B
// and C go into stream-ordered scratch with the row pitch rounded up to 16
// bytes, du, ddelta and dz come back from padded rows into the caller's (dA,
// dB, dC, dD and ddelta_bias are written in place: their layout does not
// depend on the row pitch).  The forward's checkpoints keep their layout.
// *taken stays false when the rows need no padding, when a stride or the
// scratch does not allow it, or when no tensor map fits the padded layout.
template <typename T>
static int run_bwd_repacked(const BwdArgs& a, cudaStream_t st, const Scratch& scratch, bool* taken) {
    *taken = false;
    if (a.N != 16 || a.L < (a.ckpt_in ? 1 : 2) || a.L >= (1 << 30) || scratch.limit != ~size_t(0))
        return SS_OK;
    const int64_t es = sizeof(T), L = a.L, Lp = padded_len(L, (int)es);
    auto unit_t = [](const void* p, int64_t stt) { return !p || stt == 1; };
    if (!unit_t(a.u, a.su_t) || !unit_t(a.dl, a.sdl_t) || !unit_t(a.z, a.sz_t) ||
        !unit_t(a.dout, a.sg_t) || !unit_t(a.Bm, a.sB_t) || !unit_t(a.Cm, a.sC_t) ||
        !unit_t(a.du, a.sdu_t) || !unit_t(a.ddl, a.sddl_t) || !unit_t(a.dz, a.sdz_t))
        return SS_OK;
    if (bwd_fast_ok(a)) return SS_OK;  // already the fast kernel's layout
    // every row must be a full row of L elements (no overlap)
    auto rows_ok = [&](const void* p, int64_t sr) { return !p || a.D < 2 || sr >= L; };
    if (!rows_ok(a.u, a.su_d) || !rows_ok(a.dl, a.sdl_d) || !rows_ok(a.z, a.sz_d) ||
        !rows_ok(a.dout, a.sg_d) || !rows_ok(a.du, a.sdu_d) || !rows_ok(a.ddl, a.sddl_d) ||
        !rows_ok(a.dz, a.sdz_d) || a.sB_n < L || a.sC_n < L)
        return SS_OK;
    const size_t act = (size_t)a.Bsz * a.D * Lp * es, bc = (size_t)a.Bsz * 16 * Lp * es;
    auto r256 = [](size_t n) { return (n + 255) & ~size_t(255); };
    const int nact = a.z ? 7 : 5;  // u, delta, dout, du, ddelta (+ z, dz)
    uint8_t* base = static_cast<uint8_t*>(scratch.alloc(r256(act) * nact + 2 * r256(bc), st,
                                                        scratch.ctx));
    if (!base) return SS_OK;  // no room: the general kernel
    uint8_t* pu = base;
    uint8_t* pdl = pu + r256(act);
    uint8_t* pg = pdl + r256(act);
    uint8_t* pdu = pg + r256(act);
    uint8_t* pddl = pdu + r256(act);
    uint8_t* pz = a.z ? pddl + r256(act) : nullptr;
    uint8_t* pdz = a.z ? pz + r256(act) : nullptr;
    uint8_t* pB = pddl + r256(act) * (a.z ? 3 : 1);
    uint8_t* pC = pB + r256(bc);
    BwdArgs c = a;
    const int64_t sb = (int64_t)a.D * Lp;
    c.u = pu;     c.su_b = sb;   c.su_d = Lp;
    c.dl = pdl;   c.sdl_b = sb;  c.sdl_d = Lp;
    c.dout = pg;  c.sg_b = sb;   c.sg_d = Lp;
    c.du = pdu;   c.sdu_b = sb;  c.sdu_d = Lp;
    c.ddl = pddl; c.sddl_b = sb; c.sddl_d = Lp;
    if (a.z) {
        c.z = pz;   c.sz_b = sb;  c.sz_d = Lp;
        c.dz = pdz; c.sdz_b = sb; c.sdz_d = Lp;
    }
    c.Bm = pB; c.sB_b = 16 * Lp; c.sB_n = Lp;
    c.Cm = pC; c.sC_b = 16 * Lp; c.sC_n = Lp;
    if (!bwd_fast_ok(c)) {
        scratch.release(base, st, scratch.ctx);
        return SS_OK;
    }
    RowPacker pk(a.dtype, L, Lp, st);
    pk.add(pu, a.u, a.Bsz, a.su_b, a.D, a.su_d, true);
    pk.add(pdl, a.dl, a.Bsz, a.sdl_b, a.D, a.sdl_d, true);
    pk.add(pg, a.dout, a.Bsz, a.sg_b, a.D, a.sg_d, true);
    if (a.z) pk.add(pz, a.z, a.Bsz, a.sz_b, a.D, a.sz_d, true);
    pk.add(pB, a.Bm, a.Bsz, a.sB_b, 16, a.sB_n, true);
    pk.add(pC, a.Cm, a.Bsz, a.sC_b, 16, a.sC_n, true);
    int rc = pk.flush();
    if (rc == SS_OK) {
        rc = run_bwd_fast<T>(c, st, scratch);
        if (rc == -1) {  // no tensor map for the padded layout: nothing was launched on it
            scratch.release(base, st, scratch.ctx);
            return SS_OK;
        }
    }
    *taken = true;
    if (rc == SS_OK) {
        pk.add(pdu, a.du, a.Bsz, a.sdu_b, a.D, a.sdu_d, false);
        pk.add(pddl, a.ddl, a.Bsz, a.sddl_b, a.D, a.sddl_d, false);
        if (a.z) pk.add(pdz, a.dz, a.Bsz, a.sdz_b, a.D, a.sdz_d, false);
        rc = pk.flush();
    }
    scratch.release(base, st, scratch.ctx);
    return rc;
}

int launch_selective_bwd(const BwdArgs& args, cudaStream_t st, const Scratch& scratch) {
    BwdArgs a = args;
    const bool empty = a.L == 0 || a.Bsz == 0 || a.D == 0;
    const bool force_general = debug_path(SS_DEBUG_BWD_PATH) == 0;
    auto repacked = [&](bool* taken) {
        return a.dtype == SS_BF16 ? run_bwd_repacked<__nv_bfloat16>(a, st, scratch, taken)
                                  : run_bwd_repacked<float>(a, st, scratch, taken);
    };
    if (a.ckpt_in && !empty) {
        // the forward's states come in the fast kernel's layout only
        if (a.N != 16) return SS_ERR_UNSUPPORTED;
        if (!bwd_fast_ok(a)) {
            bool taken = false;
            const int rc = repacked(&taken);
            return taken ? rc : SS_ERR_UNSUPPORTED;
        }
        const int rc = a.dtype == SS_BF16 ? run_bwd_fast<__nv_bfloat16>(a, st, scratch)
                                          : run_bwd_fast<float>(a, st, scratch);
        return rc == -1 ? SS_ERR_UNSUPPORTED : rc;
    }
    if (!empty && !force_general && bwd_fast_ok(a)) {
        const int rc = a.dtype == SS_BF16 ? run_bwd_fast<__nv_bfloat16>(a, st, scratch)
                                          : run_bwd_fast<float>(a, st, scratch);
        if (rc != -1) return rc;  // -1: no tensor map for this layout, take the general kernel
    }
    if (!empty && !force_general) {
        bool taken = false;
        const int rc = repacked(&taken);
        if (taken) return rc;
    }
    // the general kernel adds into the fp32 sums; with nothing to scan they stay zero
    const size_t nA = (size_t)a.D * a.N, nBC = (size_t)a.Bsz * a.N * a.L;
    if ((nA && cudaMemsetAsync(a.dA, 0, sizeof(float) * nA, st) != cudaSuccess) ||
        (nBC && cudaMemsetAsync(a.dB, 0, sizeof(float) * nBC, st) != cudaSuccess) ||
        (nBC && cudaMemsetAsync(a.dC, 0, sizeof(float) * nBC, st) != cudaSuccess) ||
        (a.dD && a.D && cudaMemsetAsync(a.dD, 0, sizeof(float) * a.D, st) != cudaSuccess) ||
        (a.dbias && a.D && cudaMemsetAsync(a.dbias, 0, sizeof(float) * a.D, st) != cudaSuccess))
        return SS_ERR_CUDA;
    if (empty) return SS_OK;
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
