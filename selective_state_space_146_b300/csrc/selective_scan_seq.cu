// selective_scan_seq.cu -- the selective scan (d_state 16) on sm_103a with
// lean per-step arithmetic, for sequences of any length.
//
// What is computed (page "Mamba模型笔记" §2.2 and §4.1-§4.4; 0539edu paper
// talk §2.3): per batch row b and channel d, with dl = softplus(delta + bias),
//   h[n] <- exp(dl * A[d,n]) * h[n] + dl * B[b,n,t] * u,
//   y     = (sum_n C[b,n,t] h[n] + D[d] u) * z * sigmoid(z).
//
// scan_seq: one CTA = one work item over a tile of DT channels of one batch
// row and one time segment.
//   loads      one thread issues the TMA loads of the u / delta / z tiles (ROWB =
//              64 or 128 bytes of t per channel row, swizzled over ROWB) and of
//              the raw B, C tiles into a ring of stages; B and C of each landed
//              tile are converted into an fp32 table shared by all channels of
//              the CTA.  With HELPER, warp 0 does both and the consumers follow
//              it through mbarriers; without it the consumer warps share the
//              conversion of each tile between two block barriers and thread
//              0 refills the stage they have all left (a smaller CTA, one
//              more per SM);
//   consumers  NSPLIT lanes per channel (1, 2 or 4), each keeping
//              16 / NSPLIT states in registers and stepping through t with
//              packed f32x2 arithmetic; exp on the MUFU pipe, softplus with one
//              MUFU exponential and a polynomial for log1p on the FMA pipe.
//
// Time segments (page 0539edu paper talk §5.3-§5.4: a long sequence is cut
// into chunks and the state is passed on).  When the channels alone cannot
// fill the GPU the sequence is cut into nseg segments.  The launch then holds
// two kinds of items, numbered in this order (tile by tile):
//   summaries  (tile, segment s < nseg - 1): over the segment's steps, the end
//              state E from a zero state and P = prod_t exp(dl A) = exp(A sum dl).
//              The last summary of a tile to finish (a per-tile arrival
//              counter) folds the tile's summaries in segment order,
//              h_{s+1} = P_s h_s + E_s from the caller's initial state h_0, stores
//              every h_{s+1} and raises the tile's ready flag;
//   mains      (tile, segment s): the scan proper, from h_s (after the ready
//              flag for s > 0).
// The fold runs in one fixed order, so results do not depend on timing.  Each
// CTA takes its item number from a counter in global memory: a main only
// waits on summaries, which have smaller numbers, were taken by CTAs that are
// already running and never wait themselves, so every wait ends.  Waits are
// bounded all the same (ERR_WAIT_TIMEOUT after 2 s).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "scan_common.cuh"
#include "ssscan.h"

namespace ss {

struct SeqParams {
    int Bsz, D, L;
    int dtiles;   // channel tiles per batch row
    int ntile;    // Bsz * dtiles
    int seg_len;  // steps per segment, a multiple of the t tile
    int nseg;
    const float* A; int64_t sA_d, sA_n;
    const float* Dv; int64_t sD;
    const float* bias; int64_t sbias;
    float* last; int64_t sl_b, sl_d, sl_n;
    const float* h0; int64_t sh_b, sh_d, sh_n;  // initial state, may be null
    void* y; int64_t sy_b, sy_d;                // y rows are contiguous in t
    float* summ;        // [nseg-1][Bsz*D][2][16]: prod of decays, end state from zero
                        // (the end state is overwritten by h_{s+1} once the tile is folded)
    unsigned* ready;    // [ntile]: the tile's states h_1 .. h_{nseg-1} are stored
    unsigned* done;     // [ntile]: summaries of the tile finished so far
    unsigned* counter;  // next item number
    // causal conv1d + SiLU in front of the scan (CONV kernels): the u tiles
    // hold x and u = silu(bias + sum_k w[k] x[t - W + 1 + k]) is computed in fp32
    const void* x; int64_t sx_b, sx_d;       // x rows contiguous in t
    const float* cw; int64_t scw_d, scw_k;   // taps (D, W), W <= 4
    const float* cb; int64_t scb;            // bias (D), may be null
    int cwidth;
    int bc_groups;      // B, C groups per batch row (1: shared)
    int bc_dpg;         // channels per group, a multiple of the channel tile
    int softplus;
    unsigned* err;
};

template <typename T, int NSPLIT, int CWARPS, int STAGES, bool HAS_Z, int ROWB, bool HELPER>
struct SeqCfg {
    static constexpr int N = 16;
    static constexpr int ES = sizeof(T);
    static constexpr int VEC = 16 / ES;          // steps per 16-byte chunk
    static constexpr int TT = ROWB / ES;         // steps per tile (one ROWB-byte row)
    static constexpr int CHUNKS = TT / VEC;      // 4 or 8
    static constexpr int CPW = 32 / NSPLIT;      // channels per consumer warp
    static constexpr int DT = CWARPS * CPW;      // channels per CTA
    static constexpr int NS = N / NSPLIT;        // states per lane
    static constexpr int K = VEC / NSPLIT;       // steps of a chunk whose y a lane owns
    static constexpr int NCONS = CWARPS * 32;
    // + the TMA / table warp (HELPER), else the consumers take its work in turn
    static constexpr int NTHREADS = NCONS + (HELPER ? 32 : 0);
    static constexpr int WARP0 = HELPER ? 1 : 0;    // first consumer warp
    static constexpr int LEAD = WARP0 * 32;         // the consumer thread that waits and signals
    static constexpr int TILE_BYTES = DT * ROWB;  // one [DT][TT] tile of u, delta, z
    static constexpr int RAW_BYTES = N * ROWB;    // one [N][TT] tile of B or C as loaded
    static constexpr int BC_BYTES = TT * 2 * N * 4;
    // stage: u, delta, [z], raw B, raw C, fp32 B|C table
    static constexpr int OFF_DL = TILE_BYTES;
    static constexpr int OFF_Z = 2 * TILE_BYTES;
    static constexpr int OFF_RAWB = (HAS_Z ? 3 : 2) * TILE_BYTES;
    static constexpr int OFF_RAWC = OFF_RAWB + RAW_BYTES;
    static constexpr int OFF_BC = OFF_RAWC + RAW_BYTES;
    static constexpr int STAGE_BYTES = OFF_BC + BC_BYTES;
    static constexpr int SMEM_BYTES = STAGE_BYTES * STAGES + 128 /*barriers, item*/ + 1024 /*align*/;
    static_assert(TILE_BYTES % 1024 == 0, "tile must keep 1024-byte swizzle alignment");
    static_assert(STAGE_BYTES % 1024 == 0, "stage must keep 1024-byte alignment");
    static_assert(NS % 2 == 0 && K >= 1, "states per lane come in pairs; each lane owns steps");
    static_assert(DT <= 256, "TMA box rows");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

// log1p(e) / e on [0, 1] by a degree-7 polynomial: a near-minimax fit of the
// relative error (weighted least squares, refined until the error levels),
// max relative error of e * P(e) 3.5e-7 in fp32 Horner evaluation.
__device__ __forceinline__ float2 log1p_poly2(float2 e) {
    float2 p = make_float2(-0.008558019064366817f, -0.008558019064366817f);
    p = __ffma2_rn(p, e, make_float2(0.04416628181934357f, 0.04416628181934357f));
    p = __ffma2_rn(p, e, make_float2(-0.10780498385429382f, -0.10780498385429382f));
    p = __ffma2_rn(p, e, make_float2(0.177551731467247f, 0.177551731467247f));
    p = __ffma2_rn(p, e, make_float2(-0.24499653279781342f, -0.24499653279781342f));
    p = __ffma2_rn(p, e, make_float2(0.33276355266571045f, 0.33276355266571045f));
    p = __ffma2_rn(p, e, make_float2(-0.49997478723526f, -0.49997478723526f));
    p = __ffma2_rn(p, e, make_float2(0.9999998211860657f, 0.9999998211860657f));
    return __fmul2_rn(p, e);
}

// softplus(x) = max(x, 0) + log1p(e^-|x|) for K values at once (pairs packed):
// one MUFU exponential per value, the logarithm on the FMA pipe.  With `on`
// false the values are only shifted by the bias.
template <int K>
__device__ __forceinline__ void softplus_vals(float* v, float bias, bool on) {
#pragma unroll
    for (int k = 0; k + 1 < K; k += 2) {
        const float2 x = __fadd2_rn(make_float2(v[k], v[k + 1]), make_float2(bias, bias));
        const float2 e = make_float2(ex2_approx(-fabsf(x.x) * kLog2e), ex2_approx(-fabsf(x.y) * kLog2e));
        const float2 s = __fadd2_rn(make_float2(fmaxf(x.x, 0.f), fmaxf(x.y, 0.f)), log1p_poly2(e));
        v[k] = sel_f(on, s.x, x.x);
        v[k + 1] = sel_f(on, s.y, x.y);
    }
    if constexpr (K % 2 == 1) {
        const float x = v[K - 1] + bias;
        const float e = ex2_approx(-fabsf(x) * kLog2e);
        const float s = fmaxf(x, 0.f) + log1p_poly2(make_float2(e, e)).x;
        v[K - 1] = sel_f(on, s, x);
    }
}

// Bounded wait for a flag raised by another CTA (acquire at GPU scope).
__device__ __forceinline__ bool wait_flag(const unsigned* f, unsigned* err) {
    auto ld = [&]() {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
        return v;
    };
    if (ld()) return true;
    const unsigned long long start = globaltimer();
    unsigned sleep_ns = 64;
    for (uint32_t it = 1;; ++it) {
        __nanosleep(sleep_ns);  // back off: the flag's L2 line is shared by many waiters
        sleep_ns = sleep_ns < 1024 ? 2 * sleep_ns : sleep_ns;
        if (ld()) return true;
        if ((it & 15u) == 0 && globaltimer() - start > kWaitLimitNs) {
            atomicOr(err, ERR_WAIT_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ float2 lds64f(uint32_t a) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
    return v;
}

// One work item: SUMM is a segment summary, otherwise the scan proper.
template <typename T, int NSPLIT, int CWARPS, int STAGES, bool HAS_Z, int ROWB, bool HELPER, bool CONV, bool SUMM>
__device__ __forceinline__ void seq_item(const CUtensorMap* tm_u, const CUtensorMap* tm_dl,
                                         const CUtensorMap* tm_z, const CUtensorMap* tm_B,
                                         const CUtensorMap* tm_C, const SeqParams& p,
                                         uint8_t* smem, uint64_t* bars, int seg, int tile) {
    using Cfg = SeqCfg<T, NSPLIT, CWARPS, STAGES, HAS_Z, ROWB, HELPER>;
    constexpr int N = Cfg::N, TT = Cfg::TT, VEC = Cfg::VEC, NS = Cfg::NS, DT = Cfg::DT;
    constexpr int ES = Cfg::ES, K = Cfg::K;
    constexpr bool LOAD_Z = HAS_Z && !SUMM;
    uint64_t* full = bars;                // u / delta / z landed
    uint64_t* raw = bars + STAGES;        // raw B / C landed
    uint64_t* table = bars + 2 * STAGES;  // fp32 B|C table written (HELPER)
    uint64_t* empty = bars + 3 * STAGES;  // consumers done with the stage (HELPER)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = tile / p.dtiles;
    const int d0 = (tile % p.dtiles) * DT;
    const int tbeg = seg * p.seg_len;
    const int tend = min(p.L, tbeg + p.seg_len);
    const int ntiles = (tend - tbeg + TT - 1) / TT;
    auto stage = [&](int s) { return smem + s * Cfg::STAGE_BYTES; };

    // TMA loads of tile k of the segment into stage k % STAGES (one thread)
    const int bc_row = b * p.bc_groups + d0 / p.bc_dpg;
    auto issue = [&](int k) {
        const int s = k % STAGES;
        const int t0 = tbeg + k * TT;
        uint8_t* st = stage(s);
        mbar_arrive_expect_tx(&raw[s], Cfg::RAW_BYTES * (SUMM ? 1 : 2));
        tma_load_3d(st + Cfg::OFF_RAWB, tm_B, &raw[s], t0, 0, bc_row);
        if (!SUMM) tma_load_3d(st + Cfg::OFF_RAWC, tm_C, &raw[s], t0, 0, bc_row);
        mbar_arrive_expect_tx(&full[s], Cfg::TILE_BYTES * (LOAD_Z ? 3 : 2));
        tma_load_3d(st, tm_u, &full[s], t0, d0, b);
        tma_load_3d(st + Cfg::OFF_DL, tm_dl, &full[s], t0, d0, b);
        if (LOAD_Z) tma_load_3d(st + Cfg::OFF_Z, tm_z, &full[s], t0, d0, b);
    };
    if (threadIdx.x == 0)
        for (int k = 0; k < STAGES && k < ntiles; ++k) issue(k);

    if (HELPER && warp == 0) {
        // ---------------- the B|C table (all lanes) and the later loads (lane 0) ----------------
        for (int k = 0; k < ntiles; ++k) {
            const int s = k % STAGES;
            if (!__all_sync(0xffffffffu, mbar_wait(&raw[s], (k / STAGES) & 1, p.err))) break;
            const uint32_t st = smem_u32(stage(s));
            if constexpr (ROWB == 128)
                convert_bc<T, !SUMM>(st + Cfg::OFF_RAWB, st + Cfg::OFF_RAWC, st + Cfg::OFF_BC, lane);
            else
                convert_bc64<T, !SUMM>(st + Cfg::OFF_RAWB, st + Cfg::OFF_RAWC, st + Cfg::OFF_BC, lane);
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
    // NSPLIT consecutive lanes share one channel; lane `part` keeps states
    // [part*NS, part*NS + NS), computes delta for its K-slot of every chunk and
    // owns the outputs of that slot.
    const int ci = (warp - Cfg::WARP0) * Cfg::CPW + lane / NSPLIT;
    const int part = lane % NSPLIT;
    const int gbase = lane - part;
    const int d = d0 + ci;
    const bool valid = d < p.D;
    const int64_t bd = (int64_t)b * p.D + d;

    float2 A2[NS / 2], h2[NS / 2];
#pragma unroll
    for (int j = 0; j < NS / 2; ++j) {
        const int n = part * NS + 2 * j;
        A2[j] = valid ? make_float2(p.A[d * p.sA_d + n * p.sA_n] * kLog2e,
                                    p.A[d * p.sA_d + (n + 1) * p.sA_n] * kLog2e)
                      : make_float2(0.f, 0.f);
        h2[j] = (!SUMM && valid && p.h0)
                    ? make_float2(p.h0[b * p.sh_b + d * p.sh_d + n * p.sh_n],
                                  p.h0[b * p.sh_b + d * p.sh_d + (n + 1) * p.sh_n])
                    : make_float2(0.f, 0.f);
    }
    const float Dd = (valid && p.Dv) ? p.Dv[d * p.sD] : 0.f;
    const float biasd = (valid && p.bias) ? p.bias[d * p.sbias] : 0.f;
    const bool sp = p.softplus != 0;

    const int64_t per = (int64_t)p.Bsz * p.D * 2 * N;  // floats per segment of summaries
    if (!SUMM && seg > 0) {
        // the state entering this segment, stored by the tile's fold: one
        // thread waits for the flag (acquire), the consumers meet at a named
        // barrier, and every lane reads its state from L2, not this SM's L1
        if (threadIdx.x == Cfg::LEAD) wait_flag(p.ready + tile, p.err);
        named_sync(1, Cfg::NCONS);
        __threadfence();
        if (valid) {
            const float* sm = p.summ + (seg - 1) * per + bd * 2 * N + N;
#pragma unroll
            for (int q = 0; q < NS / 2; ++q)
                h2[q] = __ldcg(reinterpret_cast<const float2*>(sm + part * NS + 2 * q));
        }
    }

    float dsum = 0.f;  // sum of delta over the segment (summary)
    T* yrow = static_cast<T*>(p.y) + (int64_t)b * p.sy_b + (int64_t)(valid ? d : 0) * p.sy_d;

    // conv in front (CONV): taps right-aligned, wk[3] multiplies x[t] and
    // wk[4-W] x[t-W+1]; xc holds x at the three steps before the current tile
    // (read from global memory at the start of a segment)
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
        const uint32_t a = su + swz_rows<ROWB>(ci, j / VEC) + (j % VEC) * ES;
        return ES == 2 ? __uint_as_float(lds16(a) << 16) : __uint_as_float(lds32(a));
    };

    // The three parts of one 16-byte chunk (VEC steps) of this lane's channel:
    //   prep:   delta of the own K-slot (softplus), all-gathered in the lane
    //           group; u of the chunk (with the conv in front: u of the own
    //           K-slot computed from x, all-gathered like delta); du = delta * u;
    //   core:   the recurrence over the chunk's steps (partial readouts);
    //   finish: reduce-scatter of the readouts, skip and gate, store of y.
    // A full tile runs the chunks in a short loop (unrolled by two with
    // several lanes per channel): the loop body stays in the instruction
    // cache, and with 16 states per lane a chunk alone has ample independent
    // work.  With the conv in front, prep is a long chain (x loads, the taps,
    // SiLU, the all-gather), so the chunks run prep(c+1) | core(c) |
    // finish(c-1) instead.
    auto prep = [&](uint32_t su, int c, int tcount, float* dd, float* du, float* uf, float* uo,
                    auto tail) {
        constexpr bool TAIL = decltype(tail)::value;
        const int off = swz_rows<ROWB>(ci, c);
        if constexpr (CONV) {
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
        softplus_vals<K>(dv, biasd, sp);
        if constexpr (TAIL) {
#pragma unroll
            for (int k = 0; k < K; ++k)
                if (c * VEC + part * K + k >= tcount) dv[k] = 0.f;  // past the end: no update
        }
#pragma unroll
        for (int j = 0; j < VEC; ++j)
            dd[j] = NSPLIT == 1 ? dv[j] : __shfl_sync(0xffffffffu, dv[j % K], gbase + j / K);
#pragma unroll
        for (int j = 0; j < VEC; j += 2) {
            const float2 m = __fmul2_rn(make_float2(dd[j], dd[j + 1]), make_float2(uf[j], uf[j + 1]));
            du[j] = m.x;
            du[j + 1] = m.y;
        }
    };
    auto core = [&](uint32_t bcp, int c, const float* dd, const float* du, float* yv) {
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            if constexpr (SUMM) dsum += dd[i];
            const float2 d2 = make_float2(dd[i], dd[i]);
            const float2 du2 = make_float2(du[i], du[i]);
            const uint32_t row = bcp + (c * VEC + i) * 128;
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < NS / 2; ++j) {
                const float2 ar = __fmul2_rn(d2, A2[j]);
                const float2 a = make_float2(ex2_approx(ar.x), ex2_approx(ar.y));
                if constexpr (SUMM) {
                    const float2 bb = lds64f(row + j * 16);
                    h2[j] = __ffma2_rn(a, h2[j], __fmul2_rn(du2, bb));
                } else {
                    const float4 bc = lds128f(row + j * 16);  // B pair, C pair
                    h2[j] = __ffma2_rn(a, h2[j], __fmul2_rn(du2, make_float2(bc.x, bc.y)));
                    acc = __ffma2_rn(make_float2(bc.z, bc.w), h2[j], acc);
                }
            }
            if constexpr (!SUMM) yv[i] = acc.x + acc.y;
        }
    };
    auto finish = [&](uint32_t su, int tile_t0, int c, const float* yv, const float* uf,
                      const float* uo, auto tail) {
        [[maybe_unused]] constexpr bool TAIL = decltype(tail)::value;
        if constexpr (!SUMM) {
            float yo[K];
            if constexpr (NSPLIT == 1) {
#pragma unroll
                for (int k = 0; k < K; ++k) yo[k] = yv[k];
            } else if constexpr (NSPLIT == 2) {
                reduce_half<VEC>(yv, yo, part & 1, 1);
            } else {
                float w[VEC / 2];
                reduce_half<VEC>(yv, w, (part >> 1) & 1, 2);
                reduce_half<VEC / 2>(w, yo, part & 1, 1);
            }
            const int own = swz_rows<ROWB>(ci, c) + part * K * ES;
            float us[K];
            if constexpr (NSPLIT == 1 || CONV) {
#pragma unroll
                for (int k = 0; k < K; ++k) us[k] = NSPLIT == 1 ? uf[k] : uo[k];
            } else {
                lds_elems<T, K>(su + own, us);
            }
            [[maybe_unused]] float zo[K];
            if constexpr (LOAD_Z) lds_elems<T, K>(su + Cfg::OFF_Z + own, zo);
#pragma unroll
            for (int k = 0; k + 1 < K; k += 2) {
                float2 o = __ffma2_rn(make_float2(Dd, Dd), make_float2(us[k], us[k + 1]),
                                      make_float2(yo[k], yo[k + 1]));
                if constexpr (LOAD_Z) {
                    const float2 zz = make_float2(zo[k], zo[k + 1]);
                    const float2 ez = __fmul2_rn(zz, make_float2(-kLog2e, -kLog2e));
                    const float2 den = __fadd2_rn(make_float2(ex2_approx(ez.x), ex2_approx(ez.y)),
                                                  make_float2(1.f, 1.f));
                    const float2 g = __fmul2_rn(zz, make_float2(rcp_approx(den.x), rcp_approx(den.y)));
                    o = __fmul2_rn(o, g);
                }
                yo[k] = o.x;
                yo[k + 1] = o.y;
            }
            if constexpr (K % 2 == 1) {
                float o = fmaf(Dd, us[K - 1], yo[K - 1]);
                if constexpr (LOAD_Z) o *= zo[K - 1] * rcp_approx(1.f + ex2_approx(-zo[K - 1] * kLog2e));
                yo[K - 1] = o;
            }
            if (valid) {
                const int tg = tile_t0 + c * VEC + part * K;
                stg_elems<T, K>(yrow + tg, yo, TAIL ? tend - tg : K);
            }
        }
    };
    auto full_tile = [&](uint32_t su, int tile_t0) {
        const uint32_t bcp = su + Cfg::OFF_BC + part * (NS / 2) * 16;
        if constexpr (CONV) {
            // prep(c+1) | core(c) | finish(c-1): the conv's chain of loads,
            // FMAs and SiLU hides behind the recurrence of the chunk before
            float ddA[VEC], duA[VEC], ufA[VEC], yA[VEC], uoA[K];
            float ddB[VEC], duB[VEC], ufB[VEC], yB[VEC], uoB[K];
            prep(su, 0, TT, ddA, duA, ufA, uoA, std::false_type{});
            core(bcp, 0, ddA, duA, yA);
            prep(su, 1, TT, ddB, duB, ufB, uoB, std::false_type{});
#pragma unroll 1
            for (int c = 1; c < Cfg::CHUNKS - 1; c += 2) {
                core(bcp, c, ddB, duB, yB);
                finish(su, tile_t0, c - 1, yA, ufA, uoA, std::false_type{});
                prep(su, c + 1, TT, ddA, duA, ufA, uoA, std::false_type{});
                core(bcp, c + 1, ddA, duA, yA);
                finish(su, tile_t0, c, yB, ufB, uoB, std::false_type{});
                prep(su, c + 2, TT, ddB, duB, ufB, uoB, std::false_type{});
            }
            core(bcp, Cfg::CHUNKS - 1, ddB, duB, yB);
            finish(su, tile_t0, Cfg::CHUNKS - 2, yA, ufA, uoA, std::false_type{});
            finish(su, tile_t0, Cfg::CHUNKS - 1, yB, ufB, uoB, std::false_type{});
            return;
        }
        float dd[VEC], du[VEC], uf[VEC], yv[VEC], uo[K];
        if constexpr (NSPLIT == 1) {
#pragma unroll 1
            for (int c = 0; c < Cfg::CHUNKS; ++c) {
                prep(su, c, TT, dd, du, uf, uo, std::false_type{});
                core(bcp, c, dd, du, yv);
                finish(su, tile_t0, c, yv, uf, uo, std::false_type{});
            }
        } else {
#pragma unroll 2
            for (int c = 0; c < Cfg::CHUNKS; ++c) {
                prep(su, c, TT, dd, du, uf, uo, std::false_type{});
                core(bcp, c, dd, du, yv);
                finish(su, tile_t0, c, yv, uf, uo, std::false_type{});
            }
        }
    };
    auto tail_tile = [&](uint32_t su, int tile_t0, int tcount) {
        const uint32_t bcp = su + Cfg::OFF_BC + part * (NS / 2) * 16;
        const int nch = (tcount + VEC - 1) / VEC;
        float dd[VEC], du[VEC], uf[VEC], yv[VEC], uo[K];
#pragma unroll 1
        for (int c = 0; c < nch; ++c) {
            prep(su, c, tcount, dd, du, uf, uo, std::true_type{});
            core(bcp, c, dd, du, yv);
            finish(su, tile_t0, c, yv, uf, uo, std::true_type{});
        }
    };

    bool ok = true;
    for (int k = 0; k < ntiles; ++k) {
        const int s = k % STAGES;
        if constexpr (HELPER) {
            if (!mbar_wait(&full[s], (k / STAGES) & 1, p.err) ||
                !mbar_wait(&table[s], (k / STAGES) & 1, p.err)) {
                ok = false;
                break;
            }
        } else {
            // no helper warp: the consumers build the B|C table, a share of
            // the passes per warp, and meet; past that barrier every thread
            // is done with tile k - 1, whose stage then takes tile k - 1 + STAGES
            const bool got = mbar_wait(&full[s], (k / STAGES) & 1, p.err) &&
                             mbar_wait(&raw[s], (k / STAGES) & 1, p.err);
            if (!__syncthreads_and(got)) {
                ok = false;
                break;
            }
            const uint32_t st = smem_u32(stage(s));
            constexpr int PASSES = ROWB == 128 ? 8 : 4;
#pragma unroll
            for (int it = warp; it < PASSES; it += CWARPS) {
                if constexpr (ROWB == 128)
                    convert_bc_part<T, !SUMM>(st + Cfg::OFF_RAWB, st + Cfg::OFF_RAWC, st + Cfg::OFF_BC, lane, it);
                else
                    convert_bc64_part<T, !SUMM>(st + Cfg::OFF_RAWB, st + Cfg::OFF_RAWC, st + Cfg::OFF_BC, lane, it);
            }
            __syncthreads();
            if (threadIdx.x == 0 && k >= 1 && k - 1 + STAGES < ntiles) issue(k - 1 + STAGES);
        }
        const int tile_t0 = tbeg + k * TT;
        const int tcount = min(TT, tend - tile_t0);
        const uint32_t su = smem_u32(stage(s));
        if (tcount == TT) full_tile(su, tile_t0);
        else tail_tile(su, tile_t0, tcount);
        if constexpr (CONV) {
            // the next tile's first steps look back at the last three of this one
            const float x0 = x_at(su, TT - 3), x1 = x_at(su, TT - 2), x2 = x_at(su, TT - 1);
            xc[0] = x0; xc[1] = x1; xc[2] = x2;
        }
        if constexpr (HELPER) mbar_arrive(&empty[s]);
    }

    if constexpr (SUMM) {
        if (valid) {
            float* sm = p.summ + seg * per + bd * 2 * N;
#pragma unroll
            for (int q = 0; q < NS / 2; ++q) {
                const int n = part * NS + 2 * q;
                __stcg(reinterpret_cast<float2*>(sm + n),
                       make_float2(ex2_approx(A2[q].x * dsum), ex2_approx(A2[q].y * dsum)));
                __stcg(reinterpret_cast<float2*>(sm + N + n), h2[q]);
            }
        }
        // every consumer's summary is written (also after a failed wait, so
        // that the mains report the error instead of waiting): count this
        // summary in; the tile's last one folds them all
        int* s_last = reinterpret_cast<int*>(bars + 4 * STAGES) + 1;
        named_sync(1, Cfg::NCONS);
        if (threadIdx.x == Cfg::LEAD) {
            __threadfence();
            *s_last = atomicAdd(p.done + tile, 1u) == (unsigned)(p.nseg - 2);
        }
        named_sync(1, Cfg::NCONS);
        if (*s_last) {
            __threadfence();
            // h_{s+1} = P_s h_s + E_s from h_0, h_{s+1} replacing E_s.  Spread over
            // the consumer threads by (channel, state) so each warp access is two
            // contiguous 64-byte runs: thread c of the consumers folds state
            // c % 16 of channels c / 16 + i * CPP; the loads of BATCH segments
            // are issued before their fold so that their L2 latencies overlap.
            constexpr int CPP = Cfg::NCONS / 16;  // channels per pass
            constexpr int PASSES = DT / CPP;      // (channel, state) pairs per thread
            constexpr int BATCH = PASSES >= 16 ? 1 : 16 / PASSES;
            const int tc = threadIdx.x - Cfg::LEAD, n = tc & 15;
            const int64_t bd0 = (int64_t)b * p.D + d0;
            float hp[PASSES];
#pragma unroll
            for (int k = 0; k < PASSES; ++k) {
                const int dk = d0 + tc / 16 + k * CPP;
                hp[k] = (p.h0 && dk < p.D) ? p.h0[b * p.sh_b + dk * p.sh_d + n * p.sh_n] : 0.f;
            }
            const int nsum = p.nseg - 1;
            for (int j0 = 0; j0 < nsum; j0 += BATCH) {
                float P[BATCH][PASSES], E[BATCH][PASSES];
#pragma unroll
                for (int jb = 0; jb < BATCH; ++jb) {
#pragma unroll
                    for (int k = 0; k < PASSES; ++k) {
                        const int ck = tc / 16 + k * CPP;
                        if (j0 + jb < nsum && d0 + ck < p.D) {
                            const float* sm = p.summ + (j0 + jb) * per + (bd0 + ck) * 2 * N + n;
                            P[jb][k] = __ldcg(sm);
                            E[jb][k] = __ldcg(sm + N);
                        }
                    }
                }
#pragma unroll
                for (int jb = 0; jb < BATCH; ++jb) {
#pragma unroll
                    for (int k = 0; k < PASSES; ++k) {
                        const int ck = tc / 16 + k * CPP;
                        if (j0 + jb < nsum && d0 + ck < p.D) {
                            hp[k] = fmaf(P[jb][k], hp[k], E[jb][k]);
                            __stcg(p.summ + (j0 + jb) * per + (bd0 + ck) * 2 * N + N + n, hp[k]);
                        }
                    }
                }
            }
            named_sync(1, Cfg::NCONS);
            if (threadIdx.x == Cfg::LEAD) {
                __threadfence();
                asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p.ready + tile), "r"(1u)
                             : "memory");
            }
        }
    } else {
        if (ok && valid && p.last && seg == p.nseg - 1) {
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

template <typename T, int NSPLIT, int CWARPS, int STAGES, bool HAS_Z, int ROWB, bool HELPER, bool CONV, int MINB>
__global__ void __launch_bounds__(SeqCfg<T, NSPLIT, CWARPS, STAGES, HAS_Z, ROWB, HELPER>::NTHREADS, MINB)
scan_seq(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_dl,
         const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_B,
         const __grid_constant__ CUtensorMap tm_C, const SeqParams p) {
    using Cfg = SeqCfg<T, NSPLIT, CWARPS, STAGES, HAS_Z, ROWB, HELPER>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::STAGE_BYTES * STAGES);
    int* s_item = reinterpret_cast<int*>(bars + 4 * STAGES);  // [0] item, [1] last-summary flag

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&bars[s], 1);                       // full
            mbar_init(&bars[STAGES + s], 1);              // raw
            mbar_init(&bars[2 * STAGES + s], 32);         // table
            mbar_init(&bars[3 * STAGES + s], Cfg::NCONS); // empty
        }
        fence_mbar_init();
        *s_item = p.nseg == 1 ? (int)blockIdx.x : (int)atomicAdd(p.counter, 1u);
        if (p.nseg > 1 || blockIdx.x == 0) {
            tma_prefetch_desc(&tm_u);
            tma_prefetch_desc(&tm_dl);
            tma_prefetch_desc(&tm_B);
        }
    }
    __syncthreads();
    const int item = *s_item;
    const int S = p.nseg;
    if (S > 1 && item < p.ntile * (S - 1)) {  // summaries, tile by tile
        seq_item<T, NSPLIT, CWARPS, STAGES, HAS_Z, ROWB, HELPER, CONV, true>(&tm_u, &tm_dl, &tm_z, &tm_B, &tm_C, p, smem,
                                                         bars, item % (S - 1), item / (S - 1));
    } else {                                  // mains, tile by tile
        const int m = S > 1 ? item - p.ntile * (S - 1) : item;
        seq_item<T, NSPLIT, CWARPS, STAGES, HAS_Z, ROWB, HELPER, CONV, false>(&tm_u, &tm_dl, &tm_z, &tm_B, &tm_C, p, smem,
                                                          bars, m % S, m / S);
    }
}

// ---------------------------------------------------------------------------
// Host side.

namespace {

template <typename T, int NSPLIT, int CWARPS, int STAGES, bool HAS_Z, int ROWB, bool HELPER, bool CONV, int MINB>
struct SeqKernel {
    using Cfg = SeqCfg<T, NSPLIT, CWARPS, STAGES, HAS_Z, ROWB, HELPER>;
    static constexpr auto fn = scan_seq<T, NSPLIT, CWARPS, STAGES, HAS_Z, ROWB, HELPER, CONV, MINB>;
    // set the shared-memory attributes once per device; returns the resident
    // CTAs per SM (0 on failure)
    static int prepare() {
        static int occ[64] = {};
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
        if (!occ[dev]) {
            if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     Cfg::SMEM_BYTES) != cudaSuccess ||
                cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100) !=
                    cudaSuccess)
                return 0;
            int v = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, fn, Cfg::NTHREADS,
                                                              Cfg::SMEM_BYTES) != cudaSuccess ||
                v < 1)
                return 0;
            occ[dev] = v;
        }
        return occ[dev];
    }
    static cudaError_t launch(const CUtensorMap* maps, const SeqParams& sp, unsigned grid,
                              cudaStream_t st) {
        fn<<<grid, Cfg::NTHREADS, Cfg::SMEM_BYTES, st>>>(maps[0], maps[1], maps[2], maps[3], maps[4],
                                                          sp);
        count_launch(1);
        return cudaGetLastError();
    }
};

template <typename T, int NSPLIT, int CWARPS, int STAGES, int ROWB, int MINB, bool HELPER, bool CONV = false>
static int run_seq(const ScanArgs& a, cudaStream_t st, const Scratch& scratch,
                   int min_tiles_per_seg) {
    using KZ = SeqKernel<T, NSPLIT, CWARPS, STAGES, true, ROWB, HELPER, CONV, MINB>;
    using KN = SeqKernel<T, NSPLIT, CWARPS, STAGES, false, ROWB, HELPER, CONV, MINB>;
    using Cfg = typename KZ::Cfg;
    constexpr int TT = Cfg::TT, DT = Cfg::DT;
    const int occ = a.z ? KZ::prepare() : KN::prepare();
    if (!occ) return SS_ERR_CUDA;

    SeqParams sp{};
    sp.Bsz = a.Bsz; sp.D = a.D; sp.L = a.L;
    sp.dtiles = (a.D + DT - 1) / DT;
    sp.ntile = a.Bsz * sp.dtiles;
    sp.A = a.A; sp.sA_d = a.sA_d; sp.sA_n = a.sA_n;
    sp.Dv = a.Dv; sp.sD = a.sD; sp.bias = a.bias; sp.sbias = a.sbias;
    sp.last = a.last; sp.sl_b = a.sl_b; sp.sl_d = a.sl_d; sp.sl_n = a.sl_n;
    sp.h0 = a.h0; sp.sh_b = a.sh_b; sp.sh_d = a.sh_d; sp.sh_n = a.sh_n;
    sp.y = a.y; sp.sy_b = a.sy_b; sp.sy_d = a.sy_d;
    sp.softplus = a.softplus; sp.err = a.err;
    sp.x = a.u; sp.sx_b = a.su_b; sp.sx_d = a.su_d;
    sp.cw = a.cw; sp.scw_d = a.scw_d; sp.scw_k = a.scw_k; sp.cb = a.cb; sp.scb = a.scb;
    sp.cwidth = a.cwidth;
    const bool grouped = a.G > 1;
    sp.bc_groups = grouped ? a.G : 1;
    sp.bc_dpg = grouped ? a.D / a.G : a.D;

    // Segments (measured on the B300 over 2048..20480 channels and 1024..262144
    // steps): none while the channel tiles fill at least 60% of the resident
    // CTA slots; otherwise about three main items per slot (the dynamic order
    // evens out the end of the launch), segments of at least
    // `min_tiles_per_seg` tiles of t, at most 128 segments, and no more than
    // the scratch can hold.
    const int64_t slots = (int64_t)sm_count_current() * occ;
    const int64_t tiles = (a.L + TT - 1) / TT;
    int64_t nseg = 1;
    if (sp.ntile * 10 < slots * 6) {
        nseg = (3 * slots + sp.ntile - 1) / sp.ntile;
        nseg = std::min<int64_t>(nseg, std::max<int64_t>(1, tiles / min_tiles_per_seg));
    }
    const int forced = debug_path(SS_DEBUG_SCAN_SEGMENTS);
    if (forced > 0) nseg = forced;
    nseg = std::max<int64_t>(1, std::min<int64_t>(nseg, 128));
    auto scratch_bytes = [&](int64_t ns) {
        const size_t summ = (size_t)(ns - 1) * a.Bsz * a.D * 2 * 16 * sizeof(float);
        const size_t flags = ((size_t)2 * sp.ntile + 1) * sizeof(unsigned);
        return ((summ + 255) & ~size_t(255)) + ((flags + 255) & ~size_t(255));
    };
    while (nseg > 1 && scratch_bytes(nseg) > scratch.limit) --nseg;
    int64_t seg_tiles = (tiles + nseg - 1) / nseg;
    nseg = (tiles + seg_tiles - 1) / seg_tiles;
    sp.seg_len = (int)(seg_tiles * TT);
    sp.nseg = (int)nseg;

    // maps: 0 u, 1 delta, 2 z, 3 B, 4 C
    CUtensorMap maps[5];
    if (!make_map_3d_sw(&maps[0], a.u, a.dtype, a.L, a.D, a.Bsz, a.su_d, a.su_b, TT, DT, ROWB) ||
        !make_map_3d_sw(&maps[1], a.dl, a.dtype, a.L, a.D, a.Bsz, a.sdl_d, a.sdl_b, TT, DT, ROWB) ||
        !make_map_3d(&maps[3], a.Bm, a.dtype, a.L, a.N, (int64_t)a.Bsz * sp.bc_groups, a.sB_n,
                     grouped ? a.sB_g : a.sB_b, TT, 16, false) ||
        !make_map_3d(&maps[4], a.Cm, a.dtype, a.L, a.N, (int64_t)a.Bsz * sp.bc_groups, a.sC_n,
                     grouped ? a.sC_g : a.sC_b, TT, 16, false))
        return SS_ERR_CUDA;
    if (a.z) {
        if (!make_map_3d_sw(&maps[2], a.z, a.dtype, a.L, a.D, a.Bsz, a.sz_d, a.sz_b, TT, DT, ROWB))
            return SS_ERR_CUDA;
    } else {
        maps[2] = maps[0];
    }

    void* scr = nullptr;
    unsigned grid = (unsigned)sp.ntile;
    if (nseg > 1) {
        const size_t bytes = scratch_bytes(nseg);
        scr = scratch.alloc(bytes, st, scratch.ctx);
        if (!scr) return SS_ERR_ALLOC;
        const size_t summ_bytes =
            ((size_t)(nseg - 1) * a.Bsz * a.D * 2 * 16 * sizeof(float) + 255) & ~size_t(255);
        sp.summ = static_cast<float*>(scr);
        sp.ready = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(scr) + summ_bytes);
        sp.done = sp.ready + sp.ntile;
        sp.counter = sp.done + sp.ntile;
        // flags, arrival counts and the item counter start at zero (summaries
        // are written before they are read)
        if (cudaMemsetAsync(sp.ready, 0, bytes - summ_bytes, st) != cudaSuccess) {
            scratch.release(scr, st, scratch.ctx);
            return SS_ERR_CUDA;
        }
        grid = (unsigned)(sp.ntile * (2 * nseg - 1));
    }
    const cudaError_t e = a.z ? KZ::launch(maps, sp, grid, st) : KN::launch(maps, sp, grid, st);
    if (scr) scratch.release(scr, st, scratch.ctx);
    return e == cudaSuccess ? SS_OK : SS_ERR_LAUNCH;
}

}  // namespace

// Launch shapes by code (SS_DEBUG_SCAN_SHAPE): lanes per channel, consumer
// warps (channels per CTA), stages, row bytes of t per tile, CTAs per SM the
// launch bounds aim at, and whether a helper warp builds the B|C table and
// issues the loads (else the consumers do, in step with each other).
struct SeqShape {
    int nsplit, dt;
};
static constexpr SeqShape kShapes[] = {
    {0, 0},
    {1, 128},  // 1: one lane, 4 warps (128 channels), 2 stages, 64-byte rows, 4 per SM, no helper
    {1, 128},  // 2: one lane, 4 warps, 2 stages, 128-byte rows, 2 per SM, helper
    {2, 64},   // 3: two lanes, 4 warps (64 channels), 2 stages, 128-byte rows, 3 per SM, no helper
    {4, 32},   // 4: four lanes, 4 warps (32 channels), 3 stages, 128-byte rows, 3 per SM, helper
    {2, 64},   // 5: two lanes, 4 warps, 2 stages, 64-byte rows, 4 per SM, helper
    {1, 128},  // 6: one lane, 4 warps, 3 stages, 64-byte rows, 3 per SM, helper
    {2, 64},   // 7: shape 3 with the helper warp
};
constexpr int kNumShapes = 7;

//
// The library's choice (measured on the B300, d_state 16):
//   - enough channels for the 64-channel tiles of two lanes per channel
//     (shape 3) to fill 60% of the 3 x SM CTA slots: shape 3, no segments
//     (the Mamba-2.8B layer, 4 x 5120 channels; without the helper warp
//     0.920 ms, with it 0.949 ms);
//   - enough for the 32-channel tiles of four lanes (shape 4): shape 4, no
//     segments (the Mamba-130M layer, 8 x 1536 channels; here the helper
//     warp's overlap of the table build with the scan wins by 1%);
//   - fewer channels, so the sequence is cut into segments: one lane per
//     channel over 128 channels (shape 1, 4 CTAs/SM without the helper warp:
//     3.05 against 3.24 ms with it) from 512 tiles of 64 steps (the
//     long-context workload), two lanes from 32 tiles (shape 7: the helper
//     warp, whose overlap counts in items of a few tiles; without it
//     1 x 2048 x 4096 took 0.099 against 0.078 ms), four lanes below; no tile
//     much wider than the channels (64 or fewer channels: two lanes, 32 or
//     fewer: four); segments of at least two tiles.
int launch_selective_seq(const ScanArgs& a, cudaStream_t st, const Scratch& scratch, bool* taken) {
    *taken = false;
    if (a.N != 16 || a.ckpt || a.L <= 0 || !fast_layout_ok(a)) return SS_OK;
    const bool bf = a.dtype == SS_BF16;
    int shape = debug_path(SS_DEBUG_SCAN_SHAPE);
    if (shape < 1 || shape > kNumShapes) {
        const int64_t ch = (int64_t)a.Bsz * a.D, slots = (int64_t)sm_count_current() * 3;
        const int64_t tiles64 = ((int64_t)a.L + 63) / 64;
        const bool segmented = (ch / 32) * 10 < slots * 6;
        // a segmented call of under 2^22 channel-steps has items of a few
        // thousand channel-steps, whose fixed costs (the flag clear, the
        // per-tile fold on the critical path) outweigh the one launch: the
        // two-launch scan_fast is faster there (measured 0.038 against 0.052
        // ms at 1 x 512 x 4096); the caller takes it when *taken stays false
        if (segmented && ch * a.L < (int64_t(1) << 22) && debug_path(SS_DEBUG_SCAN_PATH) != 2)
            return SS_OK;
        if ((ch / 64) * 10 >= slots * 6) shape = 3;
        else if ((ch / 32) * 10 >= slots * 6) shape = 4;
        else if (tiles64 >= 512 && ch > 64) shape = 1;  // no tile wider than the channels
        else shape = tiles64 >= 32 && ch > 32 ? 7 : 4;
        // B, C per channel group: the tile must lie within one group
        while (a.G > 1 && (a.D / a.G) % kShapes[shape].dt != 0 && shape != 4)
            shape = shape == 1 ? 7 : 4;
    }
    const int dt = kShapes[shape].dt;
    if (a.G > 1 && (a.D / a.G) % dt != 0) return SS_OK;
    const int mtps = debug_path(SS_DEBUG_SCAN_SEG_TILES) > 0 ? debug_path(SS_DEBUG_SCAN_SEG_TILES) : 2;
    if (a.cw) {
        // the fused conv: the library's shapes, all with the helper warp
        // (others go to scan_fast)
        if (shape == 7) shape = 3;
        if (shape != 1 && shape != 3 && shape != 4) return SS_OK;
        *taken = true;
        if (shape == 1)
            return bf ? run_seq<__nv_bfloat16, 1, 4, 2, 64, 3, true, true>(a, st, scratch, mtps)
                      : run_seq<float, 1, 4, 2, 64, 3, true, true>(a, st, scratch, mtps);
        if (shape == 3)
            return bf ? run_seq<__nv_bfloat16, 2, 4, 2, 128, 3, true, true>(a, st, scratch, mtps)
                      : run_seq<float, 2, 4, 2, 128, 3, true, true>(a, st, scratch, mtps);
        return bf ? run_seq<__nv_bfloat16, 4, 4, 3, 128, 3, true, true>(a, st, scratch, mtps)
                  : run_seq<float, 4, 4, 3, 128, 3, true, true>(a, st, scratch, mtps);
    }
    *taken = true;
    switch (shape) {
        case 1: return bf ? run_seq<__nv_bfloat16, 1, 4, 2, 64, 4, false>(a, st, scratch, mtps)
                          : run_seq<float, 1, 4, 2, 64, 4, false>(a, st, scratch, mtps);
        case 2: return bf ? run_seq<__nv_bfloat16, 1, 4, 2, 128, 2, true>(a, st, scratch, mtps)
                          : run_seq<float, 1, 4, 2, 128, 2, true>(a, st, scratch, mtps);
        case 3: return bf ? run_seq<__nv_bfloat16, 2, 4, 2, 128, 3, false>(a, st, scratch, mtps)
                          : run_seq<float, 2, 4, 2, 128, 3, false>(a, st, scratch, mtps);
        case 4: return bf ? run_seq<__nv_bfloat16, 4, 4, 3, 128, 3, true>(a, st, scratch, mtps)
                          : run_seq<float, 4, 4, 3, 128, 3, true>(a, st, scratch, mtps);
        case 5: return bf ? run_seq<__nv_bfloat16, 2, 4, 2, 64, 4, true>(a, st, scratch, mtps)
                          : run_seq<float, 2, 4, 2, 64, 4, true>(a, st, scratch, mtps);
        case 7: return bf ? run_seq<__nv_bfloat16, 2, 4, 2, 128, 3, true>(a, st, scratch, mtps)
                          : run_seq<float, 2, 4, 2, 128, 3, true>(a, st, scratch, mtps);
        default: return bf ? run_seq<__nv_bfloat16, 1, 4, 3, 64, 3, true>(a, st, scratch, mtps)
                           : run_seq<float, 1, 4, 3, 64, 3, true>(a, st, scratch, mtps);
    }
}

}  // namespace ss
