// selective_scan.cu -- the Mamba selective scan on sm_103a.
//
// What is computed (page "Mamba模型笔记" §2.2 and §4.1-§4.4; 0539edu paper
// talk §2.3): per batch row b and channel d, with dl = softplus(delta + bias),
//   h[n] <- exp(dl * A[d,n]) * h[n] + dl * B[b,n,t] * u,
//   y     = (sum_n C[b,n,t] h[n] + D[d] u) * z * sigmoid(z).
//
// Kernels here (the grouped-B/C kernels live in selective_scan_grouped.cu,
// the N = 32 / 64 / 128 kernel in selective_scan_wide.cu):
//
//  * scan_general: one thread per (b, d), any strides, any N <= 256.  Used for
//    what the faster kernels do not take (odd lengths, non-unit t strides,
//    other N).
//
//  * scan_fast: N = 16, unit t stride, 16-byte aligned rows.  One CTA owns a
//    tile of channels of one batch row over one time segment:
//      warp 0      lane 0 issues the TMA (cp.async.bulk.tensor) loads of the
//                  u / delta / z tiles (128 bytes of t per channel row,
//                  128-byte swizzle) and of the raw B / C tiles into a ring of
//                  stages; all lanes convert B and C of each landed tile to an
//                  fp32 table shared by all channels of the CTA;
//      warps 1..   consumers: NSPLIT lanes per channel, each keeping N/NSPLIT
//                  states in registers and stepping through t sequentially
//                  with packed f32x2 arithmetic.  delta (softplus) is computed
//                  once per channel and step and all-gathered in the lane
//                  group; the partial readouts are reduce-scattered so each
//                  lane finishes (skip, gate) and stores its own steps of y.
//                  With the conv in front the tile holds x and the lanes
//                  compute u = silu(conv(x)) in fp32 the same way as delta.
//    All hand-offs are mbarriers; every wait is bounded (ERR_WAIT_TIMEOUT).
//    When the channels alone cannot fill the GPU the sequence is split into
//    segments: a summary pass records, per segment, prod_t exp(dl A) =
//    exp(A sum_t dl) and the end state from zero; the main pass seeds each
//    segment with the fold of its predecessors' summaries.  For a training
//    step (CKPT) each lane also stores its four states at every 8-step
//    sub-chunk start, in the backward kernel's layout.
//
//  * scan_step: one recurrent step (decode), four lanes per (b, d).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <initializer_list>
#include <type_traits>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "internal.h"
#include "ptx.cuh"
#include "scan_common.cuh"
#include "ssscan.h"

namespace ss {

// ---------------------------------------------------------------------------
// General kernel.

template <typename T, int NMAX>
__global__ void __launch_bounds__(128) scan_general(ScanArgs a) {
    int64_t unit = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (unit >= (int64_t)a.Bsz * a.D) return;
    const int b = (int)(unit / a.D), d = (int)(unit % a.D);
    const int N = a.N;
    float h[NMAX], A2[NMAX];
#pragma unroll
    for (int n = 0; n < NMAX; ++n) {
        h[n] = (a.h0 && n < N) ? a.h0[b * a.sh_b + d * a.sh_d + n * a.sh_n] : 0.f;
        A2[n] = n < N ? a.A[d * a.sA_d + n * a.sA_n] * kLog2e : 0.f;
    }
    const float Dd = a.Dv ? a.Dv[d * a.sD] : 0.f;
    const float bd = a.bias ? a.bias[d * a.sbias] : 0.f;
    const T* u = static_cast<const T*>(a.u) + b * a.su_b + d * a.su_d;
    const T* dl = static_cast<const T*>(a.dl) + b * a.sdl_b + d * a.sdl_d;
    const T* z = a.z ? static_cast<const T*>(a.z) + b * a.sz_b + d * a.sz_d : nullptr;
    T* y = static_cast<T*>(a.y) + b * a.sy_b + d * a.sy_d;
    const int g = a.G > 1 ? d / (a.D / a.G) : 0;  // this channel's B, C group
    const T* Bp = static_cast<const T*>(a.Bm) + b * a.sB_b + g * a.sB_g;
    const T* Cp = static_cast<const T*>(a.Cm) + b * a.sC_b + g * a.sC_g;
    // conv in front (optional): u = silu(bias + sum_k w[k] x[t - W + 1 + k])
    float wk[4] = {0.f, 0.f, 0.f, 0.f}, xh[3] = {0.f, 0.f, 0.f}, cbias = 0.f;
    if (a.cw) {
        for (int k = 0; k < a.cwidth; ++k) wk[4 - a.cwidth + k] = a.cw[d * a.scw_d + k * a.scw_k];
        cbias = a.cb ? a.cb[d * a.scb] : 0.f;
    }
    for (int t = 0; t < a.L; ++t) {
        float uu = Elem<T>::to_f(u[t * a.su_t]);
        if (a.cw) {
            const float pre = fmaf(wk[0], xh[0], fmaf(wk[1], xh[1], fmaf(wk[2], xh[2],
                                   fmaf(wk[3], uu, cbias))));
            xh[0] = xh[1]; xh[1] = xh[2]; xh[2] = uu;
            uu = pre * sigmoid_accurate(pre);
        }
        float dd = Elem<T>::to_f(dl[t * a.sdl_t]) + bd;
        if (a.softplus) dd = softplus_f(dd);
        const float du = dd * uu;
        float acc = 0.f;
#pragma unroll
        for (int n = 0; n < NMAX; ++n) {
            if (n < N) {
                const float bn = Elem<T>::to_f(Bp[n * a.sB_n + t * a.sB_t]);
                const float cn = Elem<T>::to_f(Cp[n * a.sC_n + t * a.sC_t]);
                h[n] = fmaf(ex2_approx(dd * A2[n]), h[n], du * bn);
                acc = fmaf(cn, h[n], acc);
            }
        }
        acc = fmaf(Dd, uu, acc);
        if (z) {
            const float zz = Elem<T>::to_f(z[t * a.sz_t]);
            acc *= zz * sigmoid_accurate(zz);
        }
        y[t * a.sy_t] = Elem<T>::from_f(acc);
    }
    if (a.last) {
        float* ls = a.last + b * a.sl_b + d * a.sl_d;
        for (int n = 0; n < N; ++n) ls[n * a.sl_n] = h[n];
    }
}

// ---------------------------------------------------------------------------
// Fast kernel.

struct FastParams {
    int Bsz, D, L;
    int dtiles;     // channel tiles per batch row
    int seg_len;    // multiple of the t tile
    int nseg;
    const float* A; int64_t sA_d, sA_n;
    const float* Dv; int64_t sD;
    const float* bias; int64_t sbias;
    float* last; int64_t sl_b, sl_d, sl_n;
    const float* h0; int64_t sh_b, sh_d, sh_n;  // initial state, may be null
    void* y; int64_t sy_b, sy_d;  // y rows are contiguous in t
    // causal conv1d + SiLU in front of the scan (CONV kernels): u = silu(conv(x))
    const void* x; int64_t sx_b, sx_d;  // x rows contiguous in t (the "u" tensor map)
    const float* cw; int64_t scw_d, scw_k;  // taps (D, W), W <= 4
    const float* cb; int64_t scb;           // bias (D), may be null
    int cwidth;
    float* summ;    // [nseg-1][Bsz*D][2][N]: prod of decays, end state from zero
    int bc_groups;  // B, C groups per batch row (1: shared)
    int bc_dpg;     // channels per group, a multiple of the channel tile
    int softplus;
    unsigned* err;
    float* ckpt;    // CKPT kernels: [Bsz*D][nkc][16] states at every 8-step sub-chunk start
    int nkc;
};

template <typename T, int NSPLIT, int CWARPS, int STAGES, bool HAS_Z, bool SUMMARY>
struct FastCfg {
    static constexpr int N = 16;
    static constexpr int ES = sizeof(T);
    static constexpr int VEC = 16 / ES;          // elements per 16-byte chunk
    static constexpr int TT = 128 / ES;          // t per tile (one 128-byte row)
    static constexpr int CHUNKS = TT / VEC;      // = 8
    static constexpr int CPW = 32 / NSPLIT;      // channels per consumer warp
    static constexpr int DT = CWARPS * CPW;      // channels per CTA
    static constexpr int NS = N / NSPLIT;        // states per thread
    static constexpr int NCONS = CWARPS * 32;
    static constexpr int NTHREADS = NCONS + 32;  // + one warp: TMA issue and B|C conversion
    static constexpr bool LOAD_Z = HAS_Z && !SUMMARY;
    static constexpr bool LOAD_C = !SUMMARY;
    static constexpr int TILE_BYTES = DT * 128;  // one [DT][TT] tile of u, delta, z or y
    static constexpr int RAW_BYTES = N * 128;    // one [N][TT] tile of B or C as loaded
    static constexpr int BC_BYTES = TT * 2 * N * 4;
    // stage: u, delta, [z], raw B, [raw C], fp32 B|C table
    static constexpr int OFF_DL = TILE_BYTES;
    static constexpr int OFF_Z = 2 * TILE_BYTES;
    static constexpr int OFF_RAWB = (LOAD_Z ? 3 : 2) * TILE_BYTES;
    static constexpr int OFF_RAWC = OFF_RAWB + RAW_BYTES;
    static constexpr int OFF_BC = OFF_RAWC + (LOAD_C ? RAW_BYTES : 0);
    static constexpr int STAGE_BYTES = OFF_BC + BC_BYTES;
    static constexpr int TILE_TX = TILE_BYTES * (LOAD_Z ? 3 : 2);
    static constexpr int RAW_TX = RAW_BYTES * (LOAD_C ? 2 : 1);
    static constexpr int SMEM_BYTES = STAGE_BYTES * STAGES + 256 /*barriers*/ + 1024 /*align*/;
    static_assert(TILE_BYTES % 1024 == 0, "tile must keep 1024-byte swizzle alignment");
    static_assert(STAGE_BYTES % 1024 == 0, "stage must keep 1024-byte alignment");
    static_assert(NS % 2 == 0, "states per lane come in pairs");
    static_assert(VEC % NSPLIT == 0, "each lane owns whole steps of a chunk");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

// Store K floats as T (K * sizeof(T) in {4, 8, 16} bytes) to shared memory.
template <typename T, int K>
__device__ __forceinline__ void sts_elems(uint32_t a, const float* v) {
    constexpr int BYTES = K * (int)sizeof(T);
    uint32_t w[4];
    if constexpr (sizeof(T) == 2) {
#pragma unroll
        for (int i = 0; i < K / 2; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t*>(&h);
        }
    } else {
#pragma unroll
        for (int i = 0; i < K; ++i) w[i] = __float_as_uint(v[i]);
    }
    if constexpr (BYTES == 16)
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(w[0]), "r"(w[1]),
                     "r"(w[2]), "r"(w[3]) : "memory");
    else if constexpr (BYTES == 8)
        asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(a), "r"(w[0]), "r"(w[1]) : "memory");
    else
        asm volatile("st.shared.b32 [%0], %1;" ::"r"(a), "r"(w[0]) : "memory");
}

template <typename T, int NSPLIT, int CWARPS, int STAGES, bool HAS_Z, bool SUMMARY, bool CONV,
          bool CKPT = false>
__global__ void __launch_bounds__(FastCfg<T, NSPLIT, CWARPS, STAGES, HAS_Z, SUMMARY>::NTHREADS, 3)
scan_fast(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_dl,
          const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_B,
          const __grid_constant__ CUtensorMap tm_C, const FastParams p) {
    using Cfg = FastCfg<T, NSPLIT, CWARPS, STAGES, HAS_Z, SUMMARY>;
    constexpr int N = Cfg::N, TT = Cfg::TT, VEC = Cfg::VEC, NS = Cfg::NS, DT = Cfg::DT;
    constexpr int ES = Cfg::ES;
    constexpr int K = VEC / NSPLIT;  // t per chunk whose delta and y this lane owns

    // Align to 1024 bytes (128-byte swizzle atoms) by pointer arithmetic on the
    // shared array itself, so every access below stays a shared-memory access.
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::STAGE_BYTES * STAGES);
    uint64_t* full = bars;             // u / delta / z landed (TMA bytes)
    uint64_t* raw = bars + STAGES;     // raw B / C landed (TMA bytes)
    uint64_t* table = bars + 2 * STAGES;  // fp32 B|C table written
    uint64_t* empty = bars + 3 * STAGES;  // consumers done; the stage may be refilled

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x / p.dtiles;
    const int d0 = (blockIdx.x % p.dtiles) * DT;
    const int seg = blockIdx.y;
    const int tbeg = seg * p.seg_len;
    const int tend = min(p.L, tbeg + p.seg_len);
    const int ntiles = (tend - tbeg + TT - 1) / TT;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&raw[s], 1);
            mbar_init(&table[s], 32);
            mbar_init(&empty[s], Cfg::NCONS);
        }
        fence_mbar_init();
    }
    __syncthreads();

    auto stage = [&](int s) { return smem + s * Cfg::STAGE_BYTES; };

    if (warp == 0) {
        // ---------------- TMA loads (lane 0) and the B|C table (all lanes) ----------------
        // One warp does both so a CTA has one helper warp: with three CTAs per
        // SM that keeps four warps per SM sub-partition (the register cap).
        // Tile k + STAGES - 1 is issued into the stage of tile k - 1 right after
        // tile k's table is written, once the consumers have released it.
        const int bc_row = b * p.bc_groups + d0 / p.bc_dpg;  // B / C rows of the tile
        auto issue = [&](int k) {
            const int s = k % STAGES;
            const int t0 = tbeg + k * TT;
            uint8_t* st = stage(s);
            mbar_arrive_expect_tx(&raw[s], Cfg::RAW_TX);
            tma_load_3d(st + Cfg::OFF_RAWB, &tm_B, &raw[s], t0, 0, bc_row);
            if (Cfg::LOAD_C) tma_load_3d(st + Cfg::OFF_RAWC, &tm_C, &raw[s], t0, 0, bc_row);
            mbar_arrive_expect_tx(&full[s], Cfg::TILE_TX);
            tma_load_3d(st, &tm_u, &full[s], t0, d0, b);
            tma_load_3d(st + Cfg::OFF_DL, &tm_dl, &full[s], t0, d0, b);
            if (Cfg::LOAD_Z) tma_load_3d(st + Cfg::OFF_Z, &tm_z, &full[s], t0, d0, b);
        };
        if (lane == 0) {
            tma_prefetch_desc(&tm_u);
            tma_prefetch_desc(&tm_dl);
            tma_prefetch_desc(&tm_B);
            if (Cfg::LOAD_Z) tma_prefetch_desc(&tm_z);
            if (Cfg::LOAD_C) tma_prefetch_desc(&tm_C);
            for (int k = 0; k < STAGES && k < ntiles; ++k) issue(k);
        }
        for (int k = 0; k < ntiles; ++k) {
            const int s = k % STAGES;
            if (!__all_sync(0xffffffffu, mbar_wait(&raw[s], (k / STAGES) & 1, p.err))) break;
            const uint32_t st = smem_u32(stage(s));
            convert_bc<T, Cfg::LOAD_C>(st + Cfg::OFF_RAWB, st + Cfg::OFF_RAWC, st + Cfg::OFF_BC,
                                       lane);
            mbar_arrive(&table[s]);
            const int kn = k - 1 + STAGES;
            bool ok = true;
            if (lane == 0 && k >= 1 && kn < ntiles) {
                ok = mbar_wait(&empty[kn % STAGES], ((kn / STAGES) - 1) & 1, p.err);
                if (ok) issue(kn);
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        }
        return;
    }

    // ---------------- consumers ----------------
    // NSPLIT consecutive lanes share one channel; lane `part` of the group keeps
    // states [part*NS, part*NS + NS), computes delta for t in its K-slot of
    // every chunk, and owns the outputs of that slot.
    const int cw = warp - 1;
    const int ci = cw * Cfg::CPW + lane / NSPLIT;  // channel row within the tile
    const int part = lane % NSPLIT;
    const int gbase = lane - part;
    const int d = d0 + ci;
    const bool valid = d < p.D;
    const int64_t bd = (int64_t)b * p.D + d;

    float2 A2[NS / 2], h2[NS / 2];
    // the summary pass always starts from zero; the main pass from the
    // caller's initial state (if any)
    const bool from_h0 = !SUMMARY && valid && p.h0;
#pragma unroll
    for (int j = 0; j < NS / 2; ++j) {
        const int n = part * NS + 2 * j;
        A2[j] = valid ? make_float2(p.A[d * p.sA_d + n * p.sA_n] * kLog2e,
                                    p.A[d * p.sA_d + (n + 1) * p.sA_n] * kLog2e)
                      : make_float2(0.f, 0.f);
        h2[j] = from_h0 ? make_float2(p.h0[b * p.sh_b + d * p.sh_d + n * p.sh_n],
                                      p.h0[b * p.sh_b + d * p.sh_d + (n + 1) * p.sh_n])
                        : make_float2(0.f, 0.f);
    }
    const float Dd = (valid && p.Dv) ? p.Dv[d * p.sD] : 0.f;
    const float biasd = (valid && p.bias) ? p.bias[d * p.sbias] : 0.f;
    const bool sp = p.softplus != 0;

    if (!SUMMARY && seg > 0 && valid) {
        // state entering this segment: fold the summaries of segments 0..seg-1
        const int64_t per = (int64_t)p.Bsz * p.D * 2 * N;
        for (int j = 0; j < seg; ++j) {
            const float* sm = p.summ + j * per + bd * 2 * N;
#pragma unroll
            for (int q = 0; q < NS / 2; ++q) {
                const int n = part * NS + 2 * q;
                h2[q] = __ffma2_rn(make_float2(sm[n], sm[n + 1]), h2[q],
                                   make_float2(sm[N + n], sm[N + n + 1]));
            }
        }
    }

    // conv in front (CONV): taps right-aligned, wk[3] multiplies x[t] and
    // wk[4-W] x[t-W+1]; xc holds x at the three steps before the current tile
    [[maybe_unused]] float wk[4] = {0.f, 0.f, 0.f, 0.f}, xc[3] = {0.f, 0.f, 0.f};
    [[maybe_unused]] float cbias = 0.f;
    if constexpr (CONV) {
        if (valid) {
            for (int k = 0; k < p.cwidth; ++k)
                wk[4 - p.cwidth + k] = p.cw[(int64_t)d * p.scw_d + k * p.scw_k];
            cbias = p.cb ? p.cb[(int64_t)d * p.scb] : 0.f;
            const T* xr = static_cast<const T*>(p.x) + (int64_t)b * p.sx_b + (int64_t)d * p.sx_d;
            for (int j = 0; j < 3; ++j) {
                const int t = tbeg - 3 + j;
                xc[j] = t >= 0 ? Elem<T>::to_f(xr[t]) : 0.f;
            }
        }
    }
    // x at tile-local step j of this lane's row (j >= -3; the carry before 0)
    [[maybe_unused]] auto x_at = [&](uint32_t su, int j) -> float {
        if (j < 0) return j == -3 ? xc[0] : (j == -2 ? xc[1] : xc[2]);
        const uint32_t a = su + swz(ci, j / VEC) + (j % VEC) * ES;
        return ES == 2 ? __uint_as_float(lds16(a) << 16) : __uint_as_float(lds32(a));
    };

    float dsum = 0.f;  // sum of delta over the segment (summary pass)
    T* yrow = static_cast<T*>(p.y) + (int64_t)b * p.sy_b + (int64_t)(valid ? d : 0) * p.sy_d;

    // The three parts of one 16-byte chunk (VEC steps) of this lane's channel:
    //   prep:   delta of the own K-slot (softplus), all-gathered in the group,
    //           and u of the whole chunk;
    //   core:   the recurrence over the chunk's steps (partial readouts);
    //   finish: reduce-scatter of the readouts, skip and gate, store of y.
    // Tiles are processed as prep(c+1) | core(c) | finish(c-1) so the three
    // independent streams interleave.
    auto prep = [&](uint32_t su, int c, int tcount, float* dd, float* uf, float* uo, auto tail) {
        constexpr bool TAIL = decltype(tail)::value;
        const int off = swz(ci, c);
        if constexpr (CONV) {
            // u = silu(conv(x)) in fp32 for the own K-slot, all-gathered like delta
            const int j0 = c * VEC + part * K;
            float xw[K + 3];
#pragma unroll
            for (int m = 0; m < K + 3; ++m) xw[m] = x_at(su, j0 - 3 + m);
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const float pre = fmaf(wk[0], xw[k], fmaf(wk[1], xw[k + 1],
                                       fmaf(wk[2], xw[k + 2], fmaf(wk[3], xw[k + 3], cbias))));
                uo[k] = pre * sigmoid_accurate(pre);
            }
#pragma unroll
            for (int j = 0; j < VEC; ++j)
                uf[j] = NSPLIT == 1 ? uo[j % K] : __shfl_sync(0xffffffffu, uo[j % K], gbase + j / K);
        } else {
            lds_elems<T, VEC>(su + off, uf);
        }
        float dv[K];
        lds_elems<T, K>(su + Cfg::OFF_DL + off + part * K * ES, dv);
#pragma unroll
        for (int k = 0; k < K; ++k) {
            float x = dv[k] + biasd;
            x = softplus_if(x, sp);
            if (TAIL && c * VEC + part * K + k >= tcount) x = 0.f;  // past the end: no update
            dv[k] = x;
        }
#pragma unroll
        for (int j = 0; j < VEC; ++j)
            dd[j] = NSPLIT == 1 ? dv[j % K] : __shfl_sync(0xffffffffu, dv[j % K], gbase + j / K);
    };
    // CKPT: the state at the start of every 8-step sub-chunk goes to p.ckpt
    // (lane `part` holds states 4 part .. 4 part + 3), for the backward
    static_assert(!CKPT || (NSPLIT == 4 && !SUMMARY && !CONV), "checkpoints: 4 lanes per channel");
    int ck_t0 = 0;  // first step of the tile being scanned
    auto core = [&](uint32_t bcp, int c, const float* dd, const float* uf, float* yv) {
        if constexpr (CKPT) {
            const int tg = ck_t0 + c * VEC;
            if (valid && tg % 8 == 0)
                *reinterpret_cast<float4*>(p.ckpt + ((int64_t)bd * p.nkc + tg / 8) * 16 + part * NS) =
                    make_float4(h2[0].x, h2[0].y, h2[1].x, h2[1].y);
        }
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            if (SUMMARY) dsum += dd[i];
            const float2 d2 = make_float2(dd[i], dd[i]);
            const float du = dd[i] * uf[i];
            const float2 du2 = make_float2(du, du);
            const uint32_t row = bcp + (c * VEC + i) * 128;
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < NS / 2; ++j) {
                const float4 bc = lds128f(row + j * 16);  // B pair, C pair
                const float2 ar = __fmul2_rn(d2, A2[j]);
                const float2 a = make_float2(ex2_approx(ar.x), ex2_approx(ar.y));
                h2[j] = __ffma2_rn(a, h2[j], __fmul2_rn(du2, make_float2(bc.x, bc.y)));
                if constexpr (!SUMMARY) acc = __ffma2_rn(make_float2(bc.z, bc.w), h2[j], acc);
            }
            yv[i] = acc.x + acc.y;
        }
    };
    auto finish = [&](uint32_t su, int tile_t0, int c, const float* yv, const float* uo,
                      auto tail) {
        [[maybe_unused]] constexpr bool TAIL = decltype(tail)::value;
        if constexpr (!SUMMARY) {
            // reduce-scatter: lane `part` ends with the full sums of its K steps
            float yo[K];
            if constexpr (NSPLIT == 1) {
#pragma unroll
                for (int k = 0; k < K; ++k) yo[k] = yv[k];
            } else if constexpr (NSPLIT == 2) {
                reduce_half<VEC>(yv, yo, part & 1, 1);
            } else if constexpr (NSPLIT == 4) {
                float w[VEC / 2];
                reduce_half<VEC>(yv, w, (part >> 1) & 1, 2);
                reduce_half<VEC / 2>(w, yo, part & 1, 1);
            } else {
                float w[VEC / 2], x[VEC / 4];
                reduce_half<VEC>(yv, w, (part >> 2) & 1, 4);
                reduce_half<VEC / 2>(w, x, (part >> 1) & 1, 2);
                reduce_half<VEC / 4>(x, yo, part & 1, 1);
            }
            const int own = swz(ci, c) + part * K * ES;
            // u of the own K-slot for the skip: still in the tile, or (CONV,
            // where the tile holds x) computed by prep
            float us[K];
            if constexpr (CONV) {
#pragma unroll
                for (int k = 0; k < K; ++k) us[k] = uo[k];
            } else {
                lds_elems<T, K>(su + own, us);
            }
            [[maybe_unused]] float zo[K];
            if constexpr (HAS_Z) lds_elems<T, K>(su + Cfg::OFF_Z + own, zo);
#pragma unroll
            for (int k = 0; k < K; ++k) {
                float o = fmaf(Dd, us[k], yo[k]);
                if constexpr (HAS_Z) o *= zo[k] * sigmoid_accurate(zo[k]);
                yo[k] = o;
            }
            if (valid) {
                const int tg = tile_t0 + c * VEC + part * K;
                stg_elems<T, K>(yrow + tg, yo, TAIL ? tend - tg : K);
            }
        }
    };
    // A full tile: 8 chunks, software-pipelined so that every trip holds
    // core(c) | prep(c+1) | finish(c-1) in one branch-free block.
    auto full_tile = [&](uint32_t su, int tile_t0) {
        static_assert(Cfg::CHUNKS == 8, "pipeline below assumes 8 chunks per tile");
        const uint32_t bcp = su + Cfg::OFF_BC + part * (NS / 2) * 16;
        float ddA[VEC], ufA[VEC], ddB[VEC], ufB[VEC], yA[VEC], yB[VEC], uoA[K], uoB[K];
        prep(su, 0, TT, ddA, ufA, uoA, std::false_type{});
        core(bcp, 0, ddA, ufA, yA);
        prep(su, 1, TT, ddB, ufB, uoB, std::false_type{});
#pragma unroll 1
        for (int c = 1; c < 7; c += 2) {
            core(bcp, c, ddB, ufB, yB);
            if constexpr (CONV) {
                finish(su, tile_t0, c - 1, yA, uoA, std::false_type{});  // before uoA is refilled
                prep(su, c + 1, TT, ddA, ufA, uoA, std::false_type{});
            } else {
                prep(su, c + 1, TT, ddA, ufA, uoA, std::false_type{});
                finish(su, tile_t0, c - 1, yA, uoA, std::false_type{});
            }
            core(bcp, c + 1, ddA, ufA, yA);
            if constexpr (CONV) {
                finish(su, tile_t0, c, yB, uoB, std::false_type{});
                prep(su, c + 2, TT, ddB, ufB, uoB, std::false_type{});
            } else {
                prep(su, c + 2, TT, ddB, ufB, uoB, std::false_type{});
                finish(su, tile_t0, c, yB, uoB, std::false_type{});
            }
        }
        core(bcp, 7, ddB, ufB, yB);
        finish(su, tile_t0, 6, yA, uoA, std::false_type{});
        finish(su, tile_t0, 7, yB, uoB, std::false_type{});
    };
    // The last, partial tile of a sequence: one chunk at a time, with checks.
    auto tail_tile = [&](uint32_t su, int tile_t0, int tcount) {
        const uint32_t bcp = su + Cfg::OFF_BC + part * (NS / 2) * 16;
        const int nch = (tcount + VEC - 1) / VEC;
        float dd[VEC], uf[VEC], yv[VEC], uo[K];
#pragma unroll 1
        for (int c = 0; c < nch; ++c) {
            prep(su, c, tcount, dd, uf, uo, std::true_type{});
            core(bcp, c, dd, uf, yv);
            finish(su, tile_t0, c, yv, uo, std::true_type{});
        }
    };

    bool ok = true;
    for (int k = 0; k < ntiles; ++k) {
        const int s = k % STAGES;
        if (!mbar_wait(&full[s], (k / STAGES) & 1, p.err) ||
            !mbar_wait(&table[s], (k / STAGES) & 1, p.err)) {
            ok = false;
            break;
        }
        const int tile_t0 = tbeg + k * TT;
        const int tcount = min(TT, tend - tile_t0);
        const uint32_t su = smem_u32(stage(s));
        ck_t0 = tile_t0;
        if (tcount == TT) full_tile(su, tile_t0);
        else tail_tile(su, tile_t0, tcount);
        if constexpr (CONV) {
            // the next tile's first steps look back at the last three of this one
            const float x0 = x_at(su, TT - 3), x1 = x_at(su, TT - 2), x2 = x_at(su, TT - 1);
            xc[0] = x0; xc[1] = x1; xc[2] = x2;
        }
        mbar_arrive(&empty[s]);
    }
    if (!ok || !valid) return;

    if constexpr (SUMMARY) {
        const int64_t per = (int64_t)p.Bsz * p.D * 2 * N;
        float* sm = p.summ + seg * per + bd * 2 * N;
#pragma unroll
        for (int q = 0; q < NS / 2; ++q) {
            const int n = part * NS + 2 * q;
            sm[n] = ex2_approx(A2[q].x * dsum);
            sm[n + 1] = ex2_approx(A2[q].y * dsum);
            sm[N + n] = h2[q].x;
            sm[N + n + 1] = h2[q].y;
        }
    } else {
        if (p.last && seg == p.nseg - 1) {
            float* ls = p.last + (int64_t)b * p.sl_b + (int64_t)d * p.sl_d;
#pragma unroll
            for (int q = 0; q < NS / 2; ++q) {
                const int n = part * NS + 2 * q;
                ls[n * p.sl_n] = h2[q].x;
                ls[(n + 1) * p.sl_n] = h2[q].y;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Host side.

bool make_map_3d(CUtensorMap* m, const void* base, int dtype, int64_t L, int64_t D, int64_t Bsz,
                 int64_t sd, int64_t sb, int box_t, int box_d, bool swizzle) {
    return make_map_3d_sw(m, base, dtype, L, D, Bsz, sd, sb, box_t, box_d, swizzle ? 128 : 0);
}

bool make_map_3d_sw(CUtensorMap* m, const void* base, int dtype, int64_t L, int64_t D, int64_t Bsz,
                    int64_t sd, int64_t sb, int box_t, int box_d, int swizzle_bytes) {
    auto enc = reinterpret_cast<EncodeFn>(tensor_map_encoder());
    if (!enc) return false;
    const int es = dtype == SS_BF16 ? 2 : 4;
    cuuint64_t dims[3] = {(cuuint64_t)L, (cuuint64_t)D, (cuuint64_t)Bsz};
    cuuint64_t strides[2] = {(cuuint64_t)(sd * es), (cuuint64_t)(sb * es)};
    cuuint32_t box[3] = {(cuuint32_t)box_t, (cuuint32_t)box_d, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, dtype == SS_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                     3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                     : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                           : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool fast_layout_ok(const ScanArgs& a) {
    if (a.N != 16) return false;
    const int es = a.dtype == SS_BF16 ? 2 : 4;
    auto row_ok = [&](const void* ptr, int64_t sb, int64_t sd, int64_t st) {
        if (!ptr) return true;
        if (st != 1 && a.L > 1) return false;
        if (reinterpret_cast<uintptr_t>(ptr) % 16) return false;
        if ((sd * es) % 16 || (sb * es) % 16) return false;
        if (sd * es >= (int64_t(1) << 40) || sb * es >= (int64_t(1) << 40)) return false;
        return true;
    };
    if (a.D > 1 && a.su_d == 0) return false;
    if (a.G > 1) {
        // every channel tile (32 channels; 64 with one lane per channel, which
        // is then not used) inside one group, and the (batch, group) rows of
        // B / C evenly spaced so one tensor map covers them
        if ((a.D / a.G) % 32 != 0) return false;
        if (a.sB_b != a.G * a.sB_g || a.sC_b != a.G * a.sC_g) return false;
        if ((a.sB_g * es) % 16 || (a.sC_g * es) % 16) return false;
    }
    return row_ok(a.u, a.su_b, a.su_d, a.su_t) && row_ok(a.dl, a.sdl_b, a.sdl_d, a.sdl_t) &&
           row_ok(a.z, a.sz_b, a.sz_d, a.sz_t) && row_ok(a.y, a.sy_b, a.sy_d, a.sy_t) &&
           row_ok(a.Bm, a.sB_b, a.sB_n, a.sB_t) && row_ok(a.Cm, a.sC_b, a.sC_n, a.sC_t) &&
           a.L < (1 << 30);
}

template <typename T, int NSPLIT, int CWARPS, int STAGES, bool HAS_Z, bool SUMMARY, bool CONV,
          bool CKPT = false>
static cudaError_t launch_fast_kernel(const CUtensorMap* maps, const FastParams& fp, dim3 grid,
                                      cudaStream_t st) {
    using Cfg = FastCfg<T, NSPLIT, CWARPS, STAGES, HAS_Z, SUMMARY>;
    auto kern = scan_fast<T, NSPLIT, CWARPS, STAGES, HAS_Z, SUMMARY, CONV, CKPT>;
    static bool attr_set[64] = {};  // the attribute is set once per device
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Cfg::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        // all of the unified L1 / shared storage as shared memory: 3 CTAs per SM
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    kern<<<grid, Cfg::NTHREADS, Cfg::SMEM_BYTES, st>>>(maps[0], maps[1], maps[2], maps[3], maps[4],
                                                       fp);
    count_launch(1);
    return cudaGetLastError();
}

// Tuning of the fast path: lanes per channel (NSPLIT) and consumer warps per
// CTA are paired so a CTA always holds 32 (NSPLIT = 2, 4) or 64 (NSPLIT = 1)
// channels; three stages fit three CTAs in one SM's shared memory.
constexpr int kStages = 3;

template <typename T, int NSPLIT, int kCWarps, bool CONV, bool CKPT = false>
static int run_fast(const ScanArgs& a, cudaStream_t st, const Scratch& scratch) {
    using CfgM = FastCfg<T, NSPLIT, kCWarps, kStages, true, false>;
    constexpr int TT = CfgM::TT, DT = CfgM::DT;
    FastParams fp{};
    fp.Bsz = a.Bsz; fp.D = a.D; fp.L = a.L;
    fp.dtiles = (a.D + DT - 1) / DT;
    fp.A = a.A; fp.sA_d = a.sA_d; fp.sA_n = a.sA_n;
    fp.Dv = a.Dv; fp.sD = a.sD; fp.bias = a.bias; fp.sbias = a.sbias;
    fp.last = a.last; fp.sl_b = a.sl_b; fp.sl_d = a.sl_d; fp.sl_n = a.sl_n;
    fp.y = a.y; fp.sy_b = a.sy_b; fp.sy_d = a.sy_d;
    fp.h0 = a.h0; fp.sh_b = a.sh_b; fp.sh_d = a.sh_d; fp.sh_n = a.sh_n;
    fp.x = a.u; fp.sx_b = a.su_b; fp.sx_d = a.su_d;
    fp.cw = a.cw; fp.scw_d = a.scw_d; fp.scw_k = a.scw_k; fp.cb = a.cb; fp.scb = a.scb;
    fp.cwidth = a.cwidth;
    fp.softplus = a.softplus; fp.err = a.err;
    fp.ckpt = a.ckpt; fp.nkc = (a.L + 7) / 8;
    const bool grouped = a.G > 1;
    fp.bc_groups = grouped ? a.G : 1;
    fp.bc_dpg = grouped ? a.D / a.G : a.D;

    // Segments along t when the channels alone leave the GPU short of CTAs.
    // Each extra segment adds a summary pass over its predecessors' steps
    // (about 0.65 of a main step), so the split pays only where the sequence
    // is long enough; the thresholds below were measured on the B300 over
    // 48..640 channel tiles and 16..4096 tiles of t (3 CTAs per SM resident):
    //   >= 2 CTAs per SM already                  -> no split;
    //   >= 128 tiles of t                         -> about 4 waves of CTAs,
    //                                                segments >= 8 tiles;
    //   >= 1 CTA per SM and a shorter sequence    -> no split;
    //   64..127 tiles                             -> about 2 waves, >= 4 tiles;
    //   fewer                                     -> about 2 CTAs per SM, >= 4 tiles
    //                                                (shorter where that leaves SMs idle).
    const int64_t sms = sm_count_current();
    const int64_t slots = sms * 3;
    const int64_t ctas = (int64_t)a.Bsz * fp.dtiles;
    const int64_t tiles = (a.L + TT - 1) / TT;
    auto cdiv = [](int64_t x, int64_t y) { return (x + y - 1) / y; };
    int64_t nseg64 = 1;
    if (ctas >= 2 * sms) nseg64 = 1;
    else if (tiles >= 128) nseg64 = std::min(cdiv(4 * slots, ctas), tiles / 8);
    else if (ctas >= sms) nseg64 = 1;
    else if (tiles >= 64) nseg64 = std::min(cdiv(2 * slots, ctas), tiles / 4);
    else nseg64 = std::min(cdiv(2 * sms, ctas), std::max(tiles / 4, cdiv(sms, ctas)));
    // the summaries ((nseg - 1) x channels x 2N floats) must fit the scratch
    const size_t per_seg = (size_t)a.Bsz * a.D * 2 * 16 * sizeof(float);
    nseg64 = std::min<int64_t>(nseg64, 1 + (int64_t)(scratch.limit / per_seg));
    int nseg = (int)std::max<int64_t>(1, std::min<int64_t>(64, nseg64));
    int64_t seg_tiles = (tiles + nseg - 1) / nseg;
    nseg = (int)((tiles + seg_tiles - 1) / seg_tiles);
    fp.seg_len = (int)(seg_tiles * TT);
    fp.nseg = nseg;

    // maps: 0 u, 1 delta, 2 z, 3 B, 4 C
    CUtensorMap maps[5];
    if (!make_map_3d(&maps[0], a.u, a.dtype, a.L, a.D, a.Bsz, a.su_d, a.su_b, TT, DT) ||
        !make_map_3d(&maps[1], a.dl, a.dtype, a.L, a.D, a.Bsz, a.sdl_d, a.sdl_b, TT, DT) ||
        // grouped B / C: (batch, group) rows merged, row stride = group stride
        !make_map_3d(&maps[3], a.Bm, a.dtype, a.L, a.N, (int64_t)a.Bsz * fp.bc_groups, a.sB_n,
                     grouped ? a.sB_g : a.sB_b, TT, 16, false) ||
        !make_map_3d(&maps[4], a.Cm, a.dtype, a.L, a.N, (int64_t)a.Bsz * fp.bc_groups, a.sC_n,
                     grouped ? a.sC_g : a.sC_b, TT, 16, false))
        return SS_ERR_CUDA;
    if (a.z) {
        if (!make_map_3d(&maps[2], a.z, a.dtype, a.L, a.D, a.Bsz, a.sz_d, a.sz_b, TT, DT))
            return SS_ERR_CUDA;
    } else {
        maps[2] = maps[0];
    }

    void* summ = nullptr;
    if (nseg > 1) {
        size_t bytes = (size_t)(nseg - 1) * a.Bsz * a.D * 2 * 16 * sizeof(float);
        summ = scratch.alloc(bytes, st, scratch.ctx);
        if (!summ) return SS_ERR_ALLOC;
        fp.summ = static_cast<float*>(summ);
        cudaError_t e = launch_fast_kernel<T, NSPLIT, kCWarps, kStages, false, true, CONV>(
            maps, fp, dim3((unsigned)ctas, nseg - 1), st);
        if (e != cudaSuccess) {
            scratch.release(summ, st, scratch.ctx);
            return SS_ERR_LAUNCH;
        }
    }
    cudaError_t e = a.z ? launch_fast_kernel<T, NSPLIT, kCWarps, kStages, true, false, CONV, CKPT>(
                              maps, fp, dim3((unsigned)ctas, nseg), st)
                        : launch_fast_kernel<T, NSPLIT, kCWarps, kStages, false, false, CONV, CKPT>(
                              maps, fp, dim3((unsigned)ctas, nseg), st);
    if (summ) scratch.release(summ, st, scratch.ctx);
    return e == cudaSuccess ? SS_OK : SS_ERR_LAUNCH;
}

template <typename T>
static int run_general(const ScanArgs& a, cudaStream_t st) {
    const int64_t units = (int64_t)a.Bsz * a.D;
    const int threads = 128;
    const unsigned blocks = (unsigned)((units + threads - 1) / threads);
    if (a.N <= 16) scan_general<T, 16><<<blocks, threads, 0, st>>>(a);
    else if (a.N <= 64) scan_general<T, 64><<<blocks, threads, 0, st>>>(a);
    else scan_general<T, 256><<<blocks, threads, 0, st>>>(a);
    count_launch(1);
    return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_LAUNCH;
}

// Up to kMaxRowCopies row copies in one launch (blockIdx.y picks the copy):
// copy q moves rows[q] rows of L elements, row r = i * n1[q] + j at
// i * s0 + j * s1 on either side.  Rows of kShortRow elements or more: a block
// copies two rows at a time, sixteen loads in flight per thread before the
// stores (enough bytes in flight per SM to cover the DRAM latency with 2-byte
// accesses), every warp access contiguous whatever the alignment of the rows.
// Shorter rows: consecutive threads take consecutive elements of the rows
// laid end to end.
constexpr int kShortRow = 256;
template <typename T>
__global__ void __launch_bounds__(256) copy_rows(const __grid_constant__ RowCopyList p) {
    const int q = blockIdx.y;
    const T* __restrict__ src = static_cast<const T*>(p.src[q]);
    T* __restrict__ dst = static_cast<T*>(p.dst[q]);
    const int n1 = p.n1[q], L = p.L;
    const int64_t rows = p.rows[q];
    if (L < kShortRow) {
        const int64_t total = rows * L;
        for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
             e += (int64_t)gridDim.x * blockDim.x) {
            const int64_t r = e / L, i = r / n1, j = r % n1;
            const int t = (int)(e - r * L);
            dst[i * p.ds0[q] + j * p.ds1[q] + t] = src[i * p.ss0[q] + j * p.ss1[q] + t];
        }
        return;
    }
    for (int64_t r = blockIdx.x; r < rows; r += 2 * (int64_t)gridDim.x) {
        // rows r and r + gridDim.x (when there is one)
        const int64_t r2 = r + gridDim.x;
        const bool two = r2 < rows;
        const int64_t i = r / n1, j = r % n1, i2 = two ? r2 / n1 : i, j2 = two ? r2 % n1 : j;
        const T* sp = src + i * p.ss0[q] + j * p.ss1[q];
        const T* sp2 = src + i2 * p.ss0[q] + j2 * p.ss1[q];
        T* dp = dst + i * p.ds0[q] + j * p.ds1[q];
        T* dp2 = dst + i2 * p.ds0[q] + j2 * p.ds1[q];
        for (int t0 = 0; t0 < L; t0 += 8 * 256) {
            T v[8], w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int t = t0 + e * 256 + (int)threadIdx.x;
                if (t < L) {
                    v[e] = sp[t];
                    if (two) w[e] = sp2[t];
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int t = t0 + e * 256 + (int)threadIdx.x;
                if (t < L) {
                    dp[t] = v[e];
                    if (two) dp2[t] = w[e];
                }
            }
        }
    }
}

RowPacker::RowPacker(int dtype, int64_t L, int64_t Lp, cudaStream_t st)
    : dtype_(dtype), Lp_(Lp), st_(st) {
    list_.L = (int)L;
}

void RowPacker::add(void* padded, const void* other, int64_t n0, int64_t s0, int64_t n1,
                    int64_t s1, bool in) {
    if (!other || rc_ != SS_OK) return;
    if (list_.count == kMaxRowCopies) flush();
    const int q = list_.count++;
    list_.src[q] = in ? other : padded;
    list_.dst[q] = in ? padded : const_cast<void*>(other);
    list_.ss0[q] = in ? s0 : n1 * Lp_;
    list_.ss1[q] = in ? s1 : Lp_;
    list_.ds0[q] = in ? n1 * Lp_ : s0;
    list_.ds1[q] = in ? Lp_ : s1;
    list_.rows[q] = n0 * n1;
    list_.n1[q] = (int)n1;
    max_rows_ = std::max(max_rows_, n0 * n1);
}

int RowPacker::flush() {
    if (rc_ == SS_OK && list_.count > 0 && max_rows_ > 0) {
        const int64_t sms = sm_count_current();
        const int64_t blocks = list_.L < kShortRow
                                   ? std::min<int64_t>((max_rows_ * list_.L + 255) / 256, sms * 8)
                                   : std::min<int64_t>((max_rows_ + 1) / 2, sms * 8);
        const dim3 grid((unsigned)blocks, (unsigned)list_.count);
        if (dtype_ == SS_BF16) copy_rows<__nv_bfloat16><<<grid, 256, 0, st_>>>(list_);
        else copy_rows<float><<<grid, 256, 0, st_>>>(list_);
        count_launch(1);
        if (cudaGetLastError() != cudaSuccess) rc_ = SS_ERR_LAUNCH;
    }
    list_.count = 0;
    max_rows_ = 0;
    return rc_;
}

// A call whose rows the fast kernels cannot map although every t-stride is 1
// (a row pitch or base that is not a multiple of 16 bytes: odd sequence
// lengths in bf16, for one) runs them on padded copies: u, delta, z and B, C
// go into stream-ordered scratch with rows padded to 16 bytes (row copies on
// the stream), the scan writes a padded y, which is copied back into the
// caller's y.  That moves about twice the bytes of the scan itself, against
// the general kernel's 19x (8 x 1536 x 2047) to 80x (1 x 2048 x 16383) of its
// time.  *taken stays false when the call needs no repacking, when a stride
// does not allow it, or with a fixed (size-limited) scratch.
static int run_repacked(const ScanArgs& a, cudaStream_t st, const Scratch& scratch, bool* taken) {
    *taken = false;
    // (one step: the general kernel is as fast, except for the checkpointing
    // forward, which has no general kernel)
    if (a.L < (a.ckpt ? 1 : 2) || scratch.limit != ~size_t(0)) return SS_OK;
    if (a.N != 16 && a.N != 32 && a.N != 64 && a.N != 128) return SS_OK;
    const int64_t es = a.dtype == SS_BF16 ? 2 : 4;
    const int64_t G = a.G > 1 ? a.G : 1;
    auto unit_t = [](const void* p, int64_t stt) { return !p || stt == 1; };
    if (!unit_t(a.u, a.su_t) || !unit_t(a.dl, a.sdl_t) || !unit_t(a.z, a.sz_t) ||
        !unit_t(a.y, a.sy_t) || !unit_t(a.Bm, a.sB_t) || !unit_t(a.Cm, a.sC_t))
        return SS_OK;
    auto aligned = [&](const void* p, int64_t s0, int64_t s1) {
        return !p || (reinterpret_cast<uintptr_t>(p) % 16 == 0 && (s0 * es) % 16 == 0 &&
                      (s1 * es) % 16 == 0);
    };
    const bool bc_ok = aligned(a.Bm, a.sB_b, a.sB_n) && aligned(a.Cm, a.sC_b, a.sC_n) &&
                       (G == 1 || ((a.sB_g * es) % 16 == 0 && (a.sC_g * es) % 16 == 0));
    if (aligned(a.u, a.su_b, a.su_d) && aligned(a.dl, a.sdl_b, a.sdl_d) &&
        aligned(a.z, a.sz_b, a.sz_d) && aligned(a.y, a.sy_b, a.sy_d) && bc_ok)
        return SS_OK;  // already the fast kernels' layout: nothing to gain
    // every source row must be a full row of L elements (no overlap)
    const int64_t L = a.L, Lp = padded_len(L, (int)es);
    if ((a.D > 1 && (a.su_d < L || a.sdl_d < L || (a.z && a.sz_d < L) || a.sy_d < L)) ||
        (a.N > 1 && (a.sB_n < L || a.sC_n < L)))
        return SS_OK;

    // the padded call's layout (pointers stand in until the scratch exists):
    // repack only when a fast kernel takes it
    ScanArgs c = a;
    void* const fake = reinterpret_cast<void*>(uintptr_t(256));
    c.u = fake; c.su_b = (int64_t)a.D * Lp; c.su_d = Lp;
    c.dl = fake; c.sdl_b = (int64_t)a.D * Lp; c.sdl_d = Lp;
    if (a.z) { c.z = fake; c.sz_b = (int64_t)a.D * Lp; c.sz_d = Lp; }
    c.y = fake; c.sy_b = (int64_t)a.D * Lp; c.sy_d = Lp;
    c.Bm = fake; c.sB_b = G * a.N * Lp; c.sB_n = Lp; c.sB_g = a.N * Lp;
    c.Cm = fake; c.sC_b = G * a.N * Lp; c.sC_n = Lp; c.sC_g = a.N * Lp;
    // (the checkpointing forward runs scan_fast only: N = 16, B, C per row)
    const bool fast = a.ckpt ? (a.N == 16 && G == 1 && !a.cw && fast_layout_ok(c))
                             : a.N == 16 ? fast_layout_ok(c)
                                         : (G == 1 && !a.cw && !(a.N == 32 && a.dtype != SS_BF16));
    if (!fast) return SS_OK;

    const size_t act = (size_t)a.Bsz * a.D * Lp * es, bc = (size_t)a.Bsz * G * a.N * Lp * es;
    auto r256 = [](size_t n) { return (n + 255) & ~size_t(255); };
    const size_t bytes = r256(act) * (a.z ? 4 : 3) + 2 * r256(bc);
    uint8_t* base = static_cast<uint8_t*>(scratch.alloc(bytes, st, scratch.ctx));
    if (!base) return SS_OK;  // no room: the general kernel, as before
    *taken = true;
    uint8_t* pu = base;
    uint8_t* pdl = pu + r256(act);
    uint8_t* py = pdl + r256(act);
    uint8_t* pz = a.z ? py + r256(act) : nullptr;
    uint8_t* pB = py + r256(act) * (a.z ? 2 : 1);
    uint8_t* pC = pB + r256(bc);
    const size_t dp = (size_t)Lp * es;
    RowPacker pk(a.dtype, L, Lp, st);
    auto pack = [&](uint8_t* dst, const void* src, int64_t sb, int64_t sd, bool in) {
        pk.add(dst, src, a.Bsz, sb, a.D, sd, in);
    };
    // (b, g, n) rows of B or C: one copy when the (b, g) rows are evenly
    // spaced, else one per batch row
    auto pack_bc = [&](uint8_t* dst, const void* src, int64_t sb, int64_t sg, int64_t sn) {
        if (G == 1 || sb == G * sg) {
            pk.add(dst, src, a.Bsz * G, G == 1 ? sb : sg, a.N, sn, true);
        } else {
            for (int64_t b = 0; b < a.Bsz; ++b)
                pk.add(dst + (size_t)b * G * a.N * dp,
                       static_cast<const uint8_t*>(src) + (size_t)(b * sb * es), G, sg, a.N, sn, true);
        }
    };
    pack(pu, a.u, a.su_b, a.su_d, true);
    pack(pdl, a.dl, a.sdl_b, a.sdl_d, true);
    if (a.z) pack(pz, a.z, a.sz_b, a.sz_d, true);
    pack_bc(pB, a.Bm, a.sB_b, G > 1 ? a.sB_g : 0, a.sB_n);
    pack_bc(pC, a.Cm, a.sC_b, G > 1 ? a.sC_g : 0, a.sC_n);
    int rc = pk.flush();
    if (rc == SS_OK) {
        c.u = pu; c.dl = pdl; c.z = pz; c.y = py; c.Bm = pB; c.Cm = pC;
        rc = launch_selective(c, st, scratch);
        if (rc == SS_OK) {  // y back to the caller's rows
            pack(py, a.y, a.sy_b, a.sy_d, false);
            rc = pk.flush();
        }
    }
    scratch.release(base, st, scratch.ctx);
    return rc;
}

// Path selection (ss_debug_set_path): SS_DEBUG_SCAN_PATH 0 forces the general
// kernel, 1 the fast kernel with SS_DEBUG_SCAN_SPLIT lanes per channel (1, 2,
// 4 or 8; 8 only for bf16, fp32 chunks hold 4 steps), 2 scan_seq.
int launch_selective(const ScanArgs& a, cudaStream_t st, const Scratch& scratch) {
    const int path = debug_path(SS_DEBUG_SCAN_PATH);
    const int split_req = debug_path(SS_DEBUG_SCAN_SPLIT);
    const int force = path == 0 ? 0 : (path == 1 ? split_req : -1);
    const bool bf = a.dtype == SS_BF16;
    // scan_seq takes every d_state-16 call in the TMA layout except small
    // calls that need time segments (scan_fast's two launches are faster
    // there) and the checkpointing forward (scan_fast keeps it: its states
    // are the backward's own, bit for bit)
    if ((path == 2 || path < 0) && !a.ckpt && a.L > 0) {
        bool taken = false;
        const int rc = launch_selective_seq(a, st, scratch, &taken);
        if (taken) return rc;
    }
    if (a.ckpt && a.L > 0) {  // (with L = 0 there are no checkpoints to write)
        // checkpoints for the backward come from the fast kernel with four
        // lanes per channel (the backward's layout of states across lanes)
        if (a.cw || a.G > 1) return SS_ERR_UNSUPPORTED;
        if (!fast_layout_ok(a)) {
            bool taken = false;
            const int rc = run_repacked(a, st, scratch, &taken);
            return taken ? rc : SS_ERR_UNSUPPORTED;
        }
        return bf ? run_fast<__nv_bfloat16, 4, 4, false, true>(a, st, scratch)
                  : run_fast<float, 4, 4, false, true>(a, st, scratch);
    }
    if (force != 0 && a.L > 0 && fast_layout_ok(a)) {
        // The fewest lanes per channel (at most 4) that give every SM 16
        // consumer warps.  Eight lanes per channel gives more warps but costs
        // more instructions per step than it recovers in latency (measured on
        // the Mamba-130M and -2.8B layer shapes); it stays available for tests.
        const int sms = sm_count_current();
        const int64_t ch = (int64_t)a.Bsz * a.D, want = (int64_t)sms * 512;
        int split = 1;
        while (split < 4 && ch * split < want) split *= 2;
        if (force == 1 || force == 2 || force == 4 || (force == 8 && bf)) split = force;
        // one lane per channel makes 64-channel tiles: groups of 32 need two lanes
        if (a.G > 1 && (a.D / a.G) % 64 != 0 && split == 1) split = 2;
        if (a.cw) {
            // conv in front: the conversion warp owns one channel row per lane
            if (split == 8) split = 4;
            if (bf) {
                if (split == 1) return run_fast<__nv_bfloat16, 1, 1, true>(a, st, scratch);
                if (split == 2) return run_fast<__nv_bfloat16, 2, 2, true>(a, st, scratch);
                return run_fast<__nv_bfloat16, 4, 4, true>(a, st, scratch);
            }
            if (split == 1) return run_fast<float, 1, 1, true>(a, st, scratch);
            if (split == 2) return run_fast<float, 2, 2, true>(a, st, scratch);
            return run_fast<float, 4, 4, true>(a, st, scratch);
        }
        if (bf) {
            if (split == 1) return run_fast<__nv_bfloat16, 1, 2, false>(a, st, scratch);
            if (split == 2) return run_fast<__nv_bfloat16, 2, 2, false>(a, st, scratch);
            if (split == 4) return run_fast<__nv_bfloat16, 4, 4, false>(a, st, scratch);
            return run_fast<__nv_bfloat16, 8, 8, false>(a, st, scratch);
        }
        if (split == 1) return run_fast<float, 1, 2, false>(a, st, scratch);
        if (split == 2) return run_fast<float, 2, 2, false>(a, st, scratch);
        return run_fast<float, 4, 4, false>(a, st, scratch);
    }
    if (force != 0 && a.L > 0 && a.G > 1) {
        bool taken = false;
        const int rc = launch_selective_grouped(a, st, &taken);
        if (taken) return rc;
    }
    if (force != 0 && a.L > 0) {
        bool taken = false;
        const int rc = launch_selective_wide(a, st, &taken);
        if (taken) return rc;
    }
    if (force != 0) {
        bool taken = false;
        const int rc = run_repacked(a, st, scratch, &taken);
        if (taken) return rc;
    }
    return bf ? run_general<__nv_bfloat16>(a, st) : run_general<float>(a, st);
}

// ---------------------------------------------------------------------------
// One recurrent step (decode): four threads per (b, d), the channel's state
// row read and written once.

template <typename T>
__global__ void __launch_bounds__(128) scan_step(StepArgs a) {
    // four lanes per (b, d): lane `sub` updates states sub, sub + 4, ...; the
    // readout is summed over the four lanes (they sit in one warp)
    const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t units = (int64_t)a.Bsz * a.D;
    const int64_t unit_raw = gt >> 2;
    const int sub = (int)(gt & 3);
    const bool valid = unit_raw < units;
    const int64_t unit = valid ? unit_raw : 0;
    const int b = (int)(unit / a.D), d = (int)(unit % a.D);
    const float uu = Elem<T>::to_f(static_cast<const T*>(a.u)[b * a.su_b + d * a.su_d]);
    float dd = Elem<T>::to_f(static_cast<const T*>(a.dl)[b * a.sdl_b + d * a.sdl_d]) +
               (a.bias ? a.bias[d * a.sbias] : 0.f);
    if (a.softplus) dd = softplus_f(dd);
    const float du = dd * uu;
    const T* Bp = static_cast<const T*>(a.Bm) + b * a.sB_b;
    const T* Cp = static_cast<const T*>(a.Cm) + b * a.sC_b;
    float* st = a.state + b * a.ss_b + d * a.ss_d;
    float acc = 0.f;
    if (valid) {
#pragma unroll 4
        for (int n = sub; n < a.N; n += 4) {
            const float hn = fmaf(ex2_approx(dd * a.A[d * a.sA_d + n * a.sA_n] * kLog2e),
                                  st[n * a.ss_n], du * Elem<T>::to_f(Bp[n * a.sB_n]));
            st[n * a.ss_n] = hn;
            acc = fmaf(Elem<T>::to_f(Cp[n * a.sC_n]), hn, acc);
        }
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    if (!valid || sub != 0) return;
    acc = fmaf(a.Dv ? a.Dv[d * a.sD] : 0.f, uu, acc);
    if (a.z) {
        const float zz = Elem<T>::to_f(static_cast<const T*>(a.z)[b * a.sz_b + d * a.sz_d]);
        acc *= zz * sigmoid_accurate(zz);
    }
    static_cast<T*>(a.y)[b * a.sy_b + d * a.sy_d] = Elem<T>::from_f(acc);
}

int launch_selective_step(const StepArgs& a, cudaStream_t st) {
    const int64_t threads = (int64_t)a.Bsz * a.D * 4;
    const unsigned blocks = (unsigned)((threads + 127) / 128);
    if (a.dtype == SS_BF16) scan_step<__nv_bfloat16><<<blocks, 128, 0, st>>>(a);
    else scan_step<float><<<blocks, 128, 0, st>>>(a);
    count_launch(1);
    return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_LAUNCH;
}

}  // namespace ss
