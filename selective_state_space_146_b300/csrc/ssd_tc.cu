// ssd_tc.cu -- chunked Mamba-2 SSD scan on the tcgen05 tensor cores.
//
// What is computed (page "Mamba模型笔记" §5, the SSM / attention duality;
// state-spaces/mamba README §4.3): per batch row b and head h, steps are
// taken in blocks of QB = 128.  With cum_t = sum_{r <= t} dt_r A_h inside the
// block (log2 units below), S the state entering the block and w_t =
// exp(cum_last - cum_t) dt_t:
//
//   CB     = C B^T                                   (QB x QB, K = N)
//   M_ij   = CB_ij exp(cum_i - cum_j) dt_j  (j <= i), 0 above the diagonal
//   y      = M X  +  diag(exp(cum)) C S^T  +  D_h x   (the dual form inside the
//                                                     block, the carried state
//                                                     for everything before it)
//   S     <- exp(cum_last) S + (diag(w) X)^T B        (state passed on)
//
// M X runs on the tensor cores with M rounded to bf16, except M's diagonal
// (M_ii = CB_ii dt_i, the step's own input): that term stays in fp32 and joins
// the skip term, y_i += (D_h + M_ii) x_i, since on a short sequence one bf16
// M_ii can set the error of a whole row on its own.
//
// The dual form of a longer chunk splits into these 128-step diagonal blocks
// plus low-rank off-diagonal blocks, and the off-diagonal part is exactly the
// state term above, so every chunk length that is a multiple of 128 gives the
// same result; the blocks are always 128 steps here.
//
// One CTA per (b, h), blocks in sequence, warp-specialised:
//  * a control warp issues the TMA loads (x, B, C tiles with 128-byte swizzle;
//    dt) and the MMAs (tcgen05.mma kind::f16, bf16 operands from shared
//    memory, fp32 accumulators in tensor memory, M = 128), and prefetches the
//    next block's B, C, dt as soon as this block's MMAs are done:
//      CB   = C . B^T      A = C  (K-major)   B = B  (K-major)      TMEM [0, 128)
//      Yoff = C . S^T      A = C  (K-major)   B = S  (MN-major)     TMEM [192, 256)
//      Ydg  = M . X        A = M  (K-major)   B = X  (MN-major)     TMEM [128, 192)
//      dS^T = B^T . X~     A = B  (MN-major)  B = X~ (MN-major)     TMEM [0, 64)
//  * four compute warps: thread t owns row t of every accumulator (TMEM lane
//    t): it builds row t of M (over the C tiles), writes row t of X~ (over
//    the state copy, free once C S^T is done), finishes row t of y and keeps
//    row n = t of the fp32 state S^T in registers (a bf16 copy in shared
//    memory feeds the next block's Yoff).
// Off the diagonal 32-step chunk, exp(cum_i - cum_j) = exp(cum_i - cum_e) *
// exp(cum_e - cum_j) with e the chunk's last step: one exponential per row
// and chunk plus a column factor shared by all rows, both <= 1 for A <= 0.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>

#include "internal.h"
#include "ptx.cuh"
#include "ssscan.h"
#include "tc.cuh"

namespace ss {

namespace ssdtc {

constexpr int QB = 128;  // steps per block
constexpr int P = 64;    // head dimension
constexpr int N = 128;   // state size
constexpr int NCOMP = 128;           // compute threads (4 warps, one TMEM lane each)
constexpr int NTHREADS = NCOMP + 32;  // + control warp (TMA and MMA issue)

// shared-memory layout (bytes from a 1024-aligned base)
constexpr int OFF_X = 0;                 // [128 t][64 p] bf16, swizzled          16 KB
constexpr int OFF_B = OFF_X + 16384;     // 2 x [128 t][64 n]                      32 KB
constexpr int OFF_C = OFF_B + 32768;     // 2 x [128 t][64 n]; then M (K-major)    32 KB
constexpr int OFF_S = OFF_C + 32768;     // X~ [128 t][64 p]; then S^T copy [128 n][64 p]  16 KB
constexpr int OFF_DT = OFF_S + 16384;    // [128 t][8 h] bf16                       2 KB
constexpr int OFF_CUM = OFF_DT + 2048;   // cum (log2 units) [128] f32
constexpr int OFF_DTF = OFF_CUM + 512;   // dt [128] f32
constexpr int OFF_GF = OFF_DTF + 512;    // column factors of the decay matrix [128] f32
constexpr int OFF_WS = OFF_GF + 512;     // warp partial sums [4] f32
constexpr int OFF_DIAG = OFF_WS + 64;    // the diagonal of M per row [128] f32
constexpr int OFF_BAR = OFF_DIAG + 512;  // mbarriers + TMEM address
constexpr int SMEM_BYTES = OFF_BAR + 128 + 1024;
constexpr uint32_t TMEM_COLS = 256;
constexpr int BAR_COMP = 1;  // named barrier of the compute warps

struct Params {
    int Bsz, L, H, G;
    const float* A; int64_t sA;
    const float* Dv; int64_t sD;
    __nv_bfloat16* y; int64_t sy_b, sy_l, sy_h;
    float* last; int64_t sl_b, sl_h, sl_p, sl_n;
    const float* h0; int64_t sh_b, sh_h, sh_p, sh_n;  // initial state, may be null
    int late_cumsum;  // two-head kernel: never form the next cumulative decay early
    unsigned* err;
};

__device__ __forceinline__ int swz(int r, int c) { return (r << 7) + ((c ^ (r & 7)) << 4); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void unpack8(const uint4& r, float* o) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        o[2 * i] = __uint_as_float(w[i] << 16);
        o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Prefetch a tile of a 3-D / 4-D tensor map into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_3d(const void* tmap, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];"
                 ::"l"(tmap), "r"(c0), "r"(c1), "r"(c2) : "memory");
}
__device__ __forceinline__ void tma_prefetch_l2_4d(const void* tmap, int c0, int c1, int c2, int c3) {
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];"
                 ::"l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3) : "memory");
}

__global__ void __launch_bounds__(NTHREADS, 2)
ssd_chunk_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_B,
             const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_dt,
             const Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    uint64_t* bar_bc = bar + 0;     // B, C, dt of the block landed
    uint64_t* bar_x = bar + 1;      // x of the block landed
    uint64_t* bar_mma1 = bar + 2;   // C B^T and C S^T done
    uint64_t* bar_mma23 = bar + 3;  // M X and B^T X~ done
    uint64_t* bar_m = bar + 4;      // M and X~ written (compute -> control)
    uint64_t* bar_s = bar + 5;      // state copy written, x consumed (compute -> control)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_BAR + 64);
    float* cum = reinterpret_cast<float*>(sm + OFF_CUM);
    float* dtf = reinterpret_cast<float*>(sm + OFF_DTF);
    float* gf = reinterpret_cast<float*>(sm + OFF_GF);
    float* wsum = reinterpret_cast<float*>(sm + OFF_WS);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // M_ii of the thread's row, from its M build to its epilogue (in shared
    // memory rather than a register held across the block)
    const uint32_t sdiag = smem_u32(sm + OFF_DIAG) + tid * 4;
    const int b = blockIdx.x / p.H, h = blockIdx.x % p.H;
    const int g = h / (p.H / p.G);
    const float A2 = p.A[h * p.sA] * kLog2e;
    const float Dh = p.Dv ? p.Dv[h * p.sD] : 0.f;
    // off-diagonal decay factorisation needs non-increasing cum (A <= 0)
    const bool factor = A2 <= 0.f;
    const uint32_t sbase = smem_u32(sm);
    const int nblk = (p.L + QB - 1) / QB;

    if (tid == 0) {
        mbar_init(bar_bc, 1);
        mbar_init(bar_x, 1);
        mbar_init(bar_mma1, 1);
        mbar_init(bar_mma23, 1);
        mbar_init(bar_m, NCOMP);
        mbar_init(bar_s, NCOMP);
        fence_mbar_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_slot, TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 4) {
        // ================= control: TMA loads and MMA issue =================
        if (lane == 0) {
            constexpr uint32_t ID_CB = tc::idesc_bf16(QB, QB, false, false);
            constexpr uint32_t ID_YOFF = tc::idesc_bf16(QB, P, false, true);
            constexpr uint32_t ID_YDG = tc::idesc_bf16(QB, P, false, true);
            constexpr uint32_t ID_DS = tc::idesc_bf16(N, P, true, true);
            tma_prefetch_desc(&tm_x);
            tma_prefetch_desc(&tm_B);
            tma_prefetch_desc(&tm_C);
            tma_prefetch_desc(&tm_dt);
            auto load_bc = [&](int k) {
                const int t0 = k * QB;
                mbar_arrive_expect_tx(bar_bc, 32768 + 32768 + 2048);
                tma_load_4d(sm + OFF_B, &tm_B, bar_bc, 0, g, t0, b);
                tma_load_4d(sm + OFF_B + 16384, &tm_B, bar_bc, 64, g, t0, b);
                tma_load_4d(sm + OFF_C, &tm_C, bar_bc, 0, g, t0, b);
                tma_load_4d(sm + OFF_C + 16384, &tm_C, bar_bc, 64, g, t0, b);
                tma_load_3d(sm + OFF_DT, &tm_dt, bar_bc, (h / 8) * 8, k * QB, b);
            };
            auto load_x = [&](int k) {
                mbar_arrive_expect_tx(bar_x, 16384);
                tma_load_4d(sm + OFF_X, &tm_x, bar_x, 0, h, k * QB, b);
            };
            load_bc(0);
            load_x(0);
            for (int k = 0; k < nblk; ++k) {
                // B, C, dt and x of the next block into L2 now: their copies
                // into shared memory wait for this block's last reader, and
                // then come from L2
                if (k + 1 < nblk) {
                    const int t1 = (k + 1) * QB;
                    tma_prefetch_l2_4d(&tm_B, 0, g, t1, b);
                    tma_prefetch_l2_4d(&tm_B, 64, g, t1, b);
                    tma_prefetch_l2_4d(&tm_C, 0, g, t1, b);
                    tma_prefetch_l2_4d(&tm_C, 64, g, t1, b);
                    tma_prefetch_l2_3d(&tm_dt, (h / 8) * 8, t1, b);
                    tma_prefetch_l2_4d(&tm_x, 0, h, t1, b);
                }
                // C B^T and C S^T: needs B, C of block k and the state copy S(k)
                if (!mbar_wait(bar_bc, k & 1, p.err) || !mbar_wait(bar_s, k & 1, p.err)) break;
                tc::fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
                    const uint64_t dc = tc::smem_desc_sw128(sbase + OFF_C + koff, 0, 1024);
                    const uint64_t db = tc::smem_desc_sw128(sbase + OFF_B + koff, 0, 1024);
                    const uint64_t ds = tc::smem_desc_sw128(sbase + OFF_S + kk * 2048, 16384, 1024);
                    tc::mma_bf16(tmem + 0, dc, db, ID_CB, kk > 0);
                    tc::mma_bf16(tmem + 192, dc, ds, ID_YOFF, kk > 0);
                }
                tc::mma_commit(bar_mma1);
                // M X and B^T X~: needs M (over C) and X~ (over the state copy)
                if (!mbar_wait(bar_m, k & 1, p.err)) break;
                tc::fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
                    const uint64_t dm = tc::smem_desc_sw128(sbase + OFF_C + koff, 0, 1024);
                    const uint64_t dx = tc::smem_desc_sw128(sbase + OFF_X + kk * 2048, 16384, 1024);
                    const uint64_t db = tc::smem_desc_sw128(sbase + OFF_B + kk * 2048, 16384, 1024);
                    const uint64_t dxt = tc::smem_desc_sw128(sbase + OFF_S + kk * 2048, 16384, 1024);
                    tc::mma_bf16(tmem + 128, dm, dx, ID_YDG, kk > 0);
                    tc::mma_bf16(tmem + 0, db, dxt, ID_DS, kk > 0);
                }
                tc::mma_commit(bar_mma23);
                if (k + 1 < nblk) {
                    // B, C, dt free once both MMA groups are done
                    if (!mbar_wait(bar_mma23, k & 1, p.err)) break;
                    load_bc(k + 1);
                    // x free once the compute warps have finished block k
                    if (!mbar_wait(bar_s, (k + 1) & 1, p.err)) break;
                    load_x(k + 1);
                }
            }
        }
    } else {
        // ================= compute warps: one TMEM lane / row each =================
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        // state entering block 0 (row n = tid of S^T): the caller's or zero
        float S[P];
        const float* h0row = p.h0 ? p.h0 + (int64_t)b * p.sh_b + (int64_t)h * p.sh_h +
                                        (int64_t)tid * p.sh_n
                                  : nullptr;
#pragma unroll
        for (int i = 0; i < P; ++i) S[i] = h0row ? h0row[i * p.sh_p] : 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(sm + OFF_S + swz(tid, c)) =
                make_uint4(pack_bf16(S[c * 8 + 0], S[c * 8 + 1]), pack_bf16(S[c * 8 + 2], S[c * 8 + 3]),
                           pack_bf16(S[c * 8 + 4], S[c * 8 + 5]), pack_bf16(S[c * 8 + 6], S[c * 8 + 7]));
        fence_proxy_async_smem();
        mbar_arrive(bar_s);  // S(0) is ready

        bool ok = true;
        for (int k = 0; k < nblk; ++k) {
            const int t0 = k * QB;
            if (!named_sync_and(BAR_COMP, NCOMP, mbar_wait(bar_bc, k & 1, p.err))) { ok = false; break; }
            // ---- cumulative decay (log2 units) and the column factors
            const uint16_t raw = *reinterpret_cast<const uint16_t*>(sm + OFF_DT + tid * 16 + (h & 7) * 2);
            const float dtv = __uint_as_float((uint32_t)raw << 16);
            float v = dtv * A2;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (lane == 31) wsum[warp] = v;
            named_sync(BAR_COMP, NCOMP);
            for (int w = 0; w < warp; ++w) v += wsum[w];
            const float cum_t = v;
            cum[tid] = cum_t;
            dtf[tid] = dtv;
            // end of this thread's 32-step chunk: lane 31 of the same warp
            const float cum_end = __shfl_sync(0xffffffffu, cum_t, 31);
            gf[tid] = ex2_approx(cum_end - cum_t) * dtv;  // <= dt when A <= 0
            named_sync(BAR_COMP, NCOMP);
            const float cum_last = cum[QB - 1];

            if (!named_sync_and(BAR_COMP, NCOMP, mbar_wait(bar_mma1, k & 1, p.err))) { ok = false; break; }
            tc::fence_after_sync();

            // ---- row tid of M = C B^T o decay o dt (strictly lower triangle),
            //      bf16, K-major over the C tiles; the diagonal M_ii = (C B^T)_ii
            //      dt_i in fp32 (in shared memory, sdiag)
#pragma unroll 1
            for (int jc = 0; jc < 4; ++jc) {
                uint8_t* mt = sm + OFF_C + (jc >> 1) * 16384;
                if (jc <= warp) {
                    float cb[32];
                    tc::tmem_ld32(trow + jc * 32, cb);
                    tc::tmem_wait_ld();
                    float m[32];
                    if (jc < warp && factor) {
                        // rows after this chunk: exp(cum_i - cum_j) = f1 * exp(cum_end - cum_j)
                        const float f1 = ex2_approx(cum_t - cum[jc * 32 + 31]);
                        const float2 f11 = make_float2(f1, f1);
                        const float2* g2 = reinterpret_cast<const float2*>(gf + jc * 32);
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float2 v = __fmul2_rn(make_float2(cb[2 * e], cb[2 * e + 1]),
                                                        __fmul2_rn(f11, g2[e]));
                            m[2 * e] = v.x;
                            m[2 * e + 1] = v.y;
                        }
                    } else {
                        const float2* c2 = reinterpret_cast<const float2*>(cum + jc * 32);
                        const float2* d2 = reinterpret_cast<const float2*>(dtf + jc * 32);
                        const float2 ct = make_float2(cum_t, cum_t);
                        // the diagonal (j = i) stays out of the bf16 M: the pair
                        // holding it lane / 2 is kept in fp32 and the epilogue
                        // adds M_ii x_i with the skip term
                        const int ed = lane >> 1;
                        float2 pick = make_float2(0.f, 0.f);
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int j = jc * 32 + 2 * e;
                            const float2 arg = __ffma2_rn(c2[e], make_float2(-1.f, -1.f), ct);  // ct - c, exact negation
                            const float2 dec = make_float2(ex2_approx(arg.x), ex2_approx(arg.y));  // j > i: discarded
                            const float2 v = __fmul2_rn(__fmul2_rn(make_float2(cb[2 * e], cb[2 * e + 1]), dec), d2[e]);
                            if (e == ed) pick = v;
                            m[2 * e] = j < tid ? v.x : 0.f;
                            m[2 * e + 1] = j + 1 < tid ? v.y : 0.f;
                        }
                        if (jc == warp)
                            asm volatile("st.shared.f32 [%0], %1;" ::"r"(sdiag), "f"((lane & 1) ? pick.y : pick.x)
                                         : "memory");
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int c = (jc & 1) * 4 + q;
                        *reinterpret_cast<uint4*>(mt + swz(tid, c)) =
                            make_uint4(pack_bf16(m[q * 8 + 0], m[q * 8 + 1]), pack_bf16(m[q * 8 + 2], m[q * 8 + 3]),
                                       pack_bf16(m[q * 8 + 4], m[q * 8 + 5]), pack_bf16(m[q * 8 + 6], m[q * 8 + 7]));
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<uint4*>(mt + swz(tid, (jc & 1) * 4 + q)) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            // ---- X~ row tid = w_t x_t into the state-copy buffer
            if (!named_sync_and(BAR_COMP, NCOMP, mbar_wait(bar_x, k & 1, p.err))) { ok = false; break; }
            {
                const float wt = ex2_approx(cum_last - cum_t) * dtv;
                const float2 wt2 = make_float2(wt, wt);
                uint4 xr[8];  // all of the row first: the stores go to another buffer
#pragma unroll
                for (int c = 0; c < 8; ++c) xr[c] = *reinterpret_cast<const uint4*>(sm + OFF_X + swz(tid, c));
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float x8[8];
                    unpack8(xr[c], x8);
                    uint32_t w[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 v = __fmul2_rn(wt2, make_float2(x8[2 * i], x8[2 * i + 1]));
                        w[i] = pack_bf16(v.x, v.y);
                    }
                    *reinterpret_cast<uint4*>(sm + OFF_S + swz(tid, c)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            fence_proxy_async_smem();
            tc::fence_before_sync();
            mbar_arrive(bar_m);

            if (!named_sync_and(BAR_COMP, NCOMP, mbar_wait(bar_mma23, k & 1, p.err))) { ok = false; break; }
            tc::fence_after_sync();

            // ---- y row tid = Ydiag + exp(cum) Yoff + (D + M_ii) x
            {
                const float eoff = ex2_approx(cum_t);
                float mii;
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(mii) : "r"(sdiag) : "memory");
                const float dx = Dh + mii;
                const int t = t0 + tid;
                __nv_bfloat16* yrow = p.y + (int64_t)b * p.sy_b + (int64_t)t * p.sy_l + (int64_t)h * p.sy_h;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float yd[32], yo[32];
                    tc::tmem_ld32(trow + 128 + half * 32, yd);
                    tc::tmem_ld32(trow + 192 + half * 32, yo);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float x8[8];
                        unpack8(*reinterpret_cast<const uint4*>(sm + OFF_X + swz(tid, half * 4 + q)), x8);
                        uint32_t w[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int e = q * 8 + 2 * i;
                            const float2 o = __ffma2_rn(
                                make_float2(dx, dx), make_float2(x8[2 * i], x8[2 * i + 1]),
                                __ffma2_rn(make_float2(eoff, eoff), make_float2(yo[e], yo[e + 1]),
                                           make_float2(yd[e], yd[e + 1])));
                            w[i] = pack_bf16(o.x, o.y);
                        }
                        if (t < p.L)
                            *reinterpret_cast<uint4*>(yrow + half * 32 + q * 8) =
                                make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            // ---- S^T row tid <- exp(cum_last) S^T + dS^T; bf16 copy for block k+1
            {
                const float ablk = ex2_approx(cum_last);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float ds[32];
                    tc::tmem_ld32(trow + half * 32, ds);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const float2 v = __ffma2_rn(make_float2(ablk, ablk),
                                                    make_float2(S[half * 32 + i], S[half * 32 + i + 1]),
                                                    make_float2(ds[i], ds[i + 1]));
                        S[half * 32 + i] = v.x;
                        S[half * 32 + i + 1] = v.y;
                    }
                }
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4*>(sm + OFF_S + swz(tid, c)) =
                        make_uint4(pack_bf16(S[c * 8 + 0], S[c * 8 + 1]), pack_bf16(S[c * 8 + 2], S[c * 8 + 3]),
                                   pack_bf16(S[c * 8 + 4], S[c * 8 + 5]), pack_bf16(S[c * 8 + 6], S[c * 8 + 7]));
            }
            fence_proxy_async_smem();
            tc::fence_before_sync();
            mbar_arrive(bar_s);
        }
        if (ok && p.last) {
            float* ls = p.last + (int64_t)b * p.sl_b + (int64_t)h * p.sl_h + (int64_t)tid * p.sl_n;
#pragma unroll
            for (int i = 0; i < P; ++i) ls[i * p.sl_p] = S[i];
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace ssdtc

// ---------------------------------------------------------------------------
// Two heads of one group per CTA (one CTA per SM, all 512 TMEM columns).
//
// Same algebra as ssd_chunk_tc.  C B^T is shared by the heads of a group, so
// it is loaded and computed once for the pair.  Warps 0-3 compute head 0,
// warps 4-7 head 1 (warp w reads TMEM lanes 32 (w % 4) ..), warp 8 issues TMA
// loads and MMAs.  Differences from the one-head kernel:
//  * M stays in tensor memory: each thread writes its row of M (bf16, two per
//    32-bit column) into its head's dS^T columns, which are free from the
//    head's state update of the previous block until this block's B^T X~, and
//    M X reads its A operand from there (tcgen05.mma with A in TMEM).  B^T X~
//    of both heads is issued once both M X are done.  Shared memory holds no
//    M, which leaves room for two B buffers: B of block k+2 loads as soon as
//    B^T X~ of block k has read its buffer, so C B^T of block k+1 never waits
//    for B and runs under the epilogue.
//  * B, C, dt and x of the next block are prefetched into L2 at the top of
//    each block.
//  * Every compute warp forms the head's whole cumulative decay itself, so
//    the cumulative sum needs no barrier between the head's warps; it runs
//    while M X and B^T X~ do if the next block's dt has landed, else after the
//    state update.
namespace ssdtc2 {

using ssdtc::tma_prefetch_l2_3d;
using ssdtc::tma_prefetch_l2_4d;

// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return r != 0;
}

using ssdtc::N;
using ssdtc::P;
using ssdtc::QB;
using ssdtc::pack_bf16;
using ssdtc::swz;
using ssdtc::unpack8;

constexpr int NHEAD = 2;
constexpr int NCOMP = 128 * NHEAD;
constexpr int NTHREADS = NCOMP + 32;
constexpr int OFF_X = 0;                  // NHEAD x [128 t][64 p] bf16            32 KB
constexpr int OFF_B = OFF_X + 32768;      // 2 blocks x 2 x [128 t][64 n]          64 KB
constexpr int OFF_C = OFF_B + 65536;      // 2 x [128 t][64 n]                     32 KB
constexpr int OFF_S = OFF_C + 32768;      // NHEAD x (X~, then the S^T copy)       32 KB
constexpr int OFF_DT = OFF_S + 32768;     // 2 x [128 t][8 h] bf16 (block parity)   4 KB
constexpr int OFF_CUM = OFF_DT + 4096;    // [NHEAD][128] f32
constexpr int OFF_DTF = OFF_CUM + 1024;
constexpr int OFF_GF = OFF_DTF + 1024;
constexpr int OFF_DIAG = OFF_GF + 1024;   // [NHEAD][128] f32: the diagonal of M per row
constexpr int OFF_BAR = OFF_DIAG + 1024;  // 16 mbarriers, then the TMEM address
constexpr int SMEM_BYTES = OFF_BAR + 128 + 16 + 1024;
constexpr uint32_t TMEM_COLS = 512;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

// TMEM columns: C B^T 0..127, then per head pair M X, C S^T and B^T X~ with
// the two heads side by side (C S^T and B^T X~ of both heads are one MMA of
// N = 128 each: the heads' S buffers are 16 KB apart, the operand's stride
// between its two 64-column halves); a head's B^T X~ columns hold its M
// (bf16) from its M build until its M X is done
__device__ __forceinline__ uint32_t tm_ydg(int hh) { return 128u + 64u * hh; }
__device__ __forceinline__ uint32_t tm_yoff(int hh) { return 256u + 64u * hh; }
__device__ __forceinline__ uint32_t tm_ds(int hh) { return 384u + 64u * hh; }

__global__ void __launch_bounds__(NTHREADS, 1)
ssd_chunk_tc2(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_B,
              const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_dt,
              const __grid_constant__ CUtensorMap tm_y, const ssdtc::Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    uint64_t* bar_c = bar + 0;       // C and dt of the block landed
    uint64_t* bar_x = bar + 1;       // [hh] x of the block landed
    uint64_t* bar_cb = bar + 3;      // C B^T done
    uint64_t* bar_yoff = bar + 4;    // [hh] C S^T done
    uint64_t* bar_mma23 = bar + 6;   // [hh] M X done
    uint64_t* bar_m = bar + 8;       // [hh] M and X~ written (compute -> control)
    uint64_t* bar_s = bar + 10;      // [hh] state copy written, x consumed
    uint64_t* bar_b = bar + 12;      // [block parity] B of the block landed
    uint64_t* bar_cfree = bar + 14;  // C S^T of both heads done: C may be refilled
    uint64_t* bar_bfree = bar + 15;  // B^T X~ of both heads done: B may be refilled
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_BAR + 128);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hpairs = p.H / NHEAD;
    const int b = blockIdx.x / hpairs, h0 = (blockIdx.x % hpairs) * NHEAD;
    const int g = h0 / (p.H / p.G);
    const uint32_t sbase = smem_u32(sm);
    const int nblk = (p.L + QB - 1) / QB;

    if (tid == 0) {
        mbar_init(bar_c, 1);
        mbar_init(&bar_b[0], 1);
        mbar_init(&bar_b[1], 1);
        mbar_init(bar_cb, 1);
        mbar_init(bar_cfree, 1);
        mbar_init(bar_bfree, 1);
        for (int hh = 0; hh < NHEAD; ++hh) {
            mbar_init(&bar_x[hh], 1);
            mbar_init(&bar_yoff[hh], 1);
            mbar_init(&bar_mma23[hh], 1);
            mbar_init(&bar_m[hh], 128);
            mbar_init(&bar_s[hh], 128);
        }
        fence_mbar_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_slot, TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == NCOMP / 32) {
        // ================= control: TMA loads and MMA issue =================
        if (lane == 0) {
            constexpr uint32_t ID_CB = tc::idesc_bf16(QB, QB, false, false);
            constexpr uint32_t ID_YOFF = tc::idesc_bf16(QB, NHEAD * P, false, true);
            constexpr uint32_t ID_YDG = tc::idesc_bf16(QB, P, false, true);
            constexpr uint32_t ID_DS = tc::idesc_bf16(N, NHEAD * P, true, true);
            tma_prefetch_desc(&tm_x);
            tma_prefetch_desc(&tm_B);
            tma_prefetch_desc(&tm_C);
            tma_prefetch_desc(&tm_dt);
            // C (with dt) and B have their own barriers: C reloads (block
            // k+1) once both heads' C S^T of block k are done; B has two
            // buffers by block parity and reloads (block k+2) once both
            // heads' B^T X~ of block k are done, so block k+1's C B^T only
            // waits for C
            auto load_c = [&](int k) {
                const int t0 = k * QB;
                mbar_arrive_expect_tx(bar_c, 32768 + 2048);
                tma_load_4d(sm + OFF_C, &tm_C, bar_c, 0, g, t0, b);
                tma_load_4d(sm + OFF_C + 16384, &tm_C, bar_c, 64, g, t0, b);
                tma_load_3d(sm + OFF_DT + (k & 1) * 2048, &tm_dt, bar_c, (h0 / 8) * 8, t0, b);
            };
            auto load_b = [&](int k) {
                const int t0 = k * QB;
                uint64_t* bb = &bar_b[k & 1];
                uint8_t* dst = sm + OFF_B + (k & 1) * 32768;
                mbar_arrive_expect_tx(bb, 32768);
                tma_load_4d(dst, &tm_B, bb, 0, g, t0, b);
                tma_load_4d(dst + 16384, &tm_B, bb, 64, g, t0, b);
            };
            auto load_x = [&](int hh, int k) {
                mbar_arrive_expect_tx(&bar_x[hh], 16384);
                tma_load_4d(sm + OFF_X + hh * 16384, &tm_x, &bar_x[hh], 0, h0 + hh, k * QB, b);
            };
            // the last block whose load was issued, per barrier (for draining
            // loads still in flight if a wait gives up)
            int c_last = 0, b_last[2] = {0, -1}, x_last[NHEAD] = {};
            // C B^T of block k into TMEM columns 0..127 (read by both heads'
            // M build of block k)
            auto issue_cb = [&](int k) {
                tc::fence_after_sync();
                const uint32_t bbuf = sbase + OFF_B + (k & 1) * 32768;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
                    tc::mma_bf16(tmem + 0, tc::smem_desc_sw128(sbase + OFF_C + koff, 0, 1024),
                                 tc::smem_desc_sw128(bbuf + koff, 0, 1024), ID_CB, kk > 0);
                }
                tc::mma_commit(bar_cb);
            };
            load_c(0);
            load_b(0);
            if (nblk > 1) {
                load_b(1);
                b_last[1] = 1;
            }
            for (int hh = 0; hh < NHEAD; ++hh) load_x(hh, 0);
            bool go = mbar_wait(bar_c, 0, p.err) && mbar_wait(&bar_b[0], 0, p.err);
            if (go) issue_cb(0);
            for (int k = 0; k < nblk && go; ++k) {
                // both heads' state copies S(k) written and x tiles free (y of
                // block k-1 has left them): x of block k first, then C S^T
                for (int hh = 0; hh < NHEAD && go; ++hh) {
                    if (!mbar_wait(&bar_s[hh], k & 1, p.err)) { go = false; break; }
                    if (k > 0) {
                        load_x(hh, k);
                        x_last[hh] = k;
                    }
                }
                if (!go) break;
                // x of block k+1 into L2 now: its copy into shared memory (at
                // the top of the next block, once y of this block has left the
                // tile) then comes from L2 instead of DRAM
                if (k + 1 < nblk) {
                    for (int hh = 0; hh < NHEAD; ++hh)
                        tma_prefetch_l2_4d(&tm_x, 0, h0 + hh, (k + 1) * QB, b);
                    // and its B, C and dt: their copies into shared memory
                    // wait for this block's last reader of the buffer, and
                    // then come from L2
                    const int t1 = (k + 1) * QB;
                    tma_prefetch_l2_4d(&tm_C, 0, g, t1, b);
                    tma_prefetch_l2_4d(&tm_C, 64, g, t1, b);
                    tma_prefetch_l2_4d(&tm_B, 0, g, t1, b);
                    tma_prefetch_l2_4d(&tm_B, 64, g, t1, b);
                    tma_prefetch_l2_3d(&tm_dt, (h0 / 8) * 8, t1, b);
                }
                tc::fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
                    tc::mma_bf16(tmem + tm_yoff(0), tc::smem_desc_sw128(sbase + OFF_C + koff, 0, 1024),
                                 tc::smem_desc_sw128(sbase + OFF_S + kk * 2048, 16384, 1024),
                                 ID_YOFF, kk > 0);
                }
                for (int hh = 0; hh < NHEAD; ++hh) tc::mma_commit(&bar_yoff[hh]);
                tc::mma_commit(bar_cfree);
                if (k + 1 < nblk) {
                    if (!mbar_wait(bar_cfree, k & 1, p.err)) { go = false; break; }
                    load_c(k + 1);
                    c_last = k + 1;
                }
                // M X per head as soon as the head's M (in its dS^T columns)
                // and X~ are written
                for (int hh = 0; hh < NHEAD && go; ++hh) {
                    if (!mbar_wait(&bar_m[hh], k & 1, p.err)) { go = false; break; }
                    tc::fence_after_sync();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        tc::mma_bf16_ta(tmem + tm_ydg(hh), tmem + tm_ds(hh) + 8u * kk,
                                    tc::smem_desc_sw128(sbase + OFF_X + hh * 16384 + kk * 2048, 16384, 1024),
                                    ID_YDG, kk > 0);
                    tc::mma_commit(&bar_mma23[hh]);
                }
                if (!go) break;
                // B^T X~ of both heads (one MMA of N = 128) into the dS^T
                // columns once both M X have read M there
                if (!mbar_wait(&bar_mma23[NHEAD - 1], k & 1, p.err)) { go = false; break; }
                tc::fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc::mma_bf16(tmem + tm_ds(0),
                                 tc::smem_desc_sw128(sbase + OFF_B + (k & 1) * 32768 + kk * 2048, 16384, 1024),
                                 tc::smem_desc_sw128(sbase + OFF_S + kk * 2048, 16384, 1024), ID_DS, kk > 0);
                tc::mma_commit(bar_bfree);
                if (k + 1 < nblk) {
                    // C B^T of block k+1 (both heads' M builds have read this
                    // block's; its B landed a block ago): it runs under the
                    // epilogue; then B of block k+2 into this block's B
                    // buffer once B^T X~ has read it
                    if (!mbar_wait(bar_c, (k + 1) & 1, p.err) ||
                        !mbar_wait(&bar_b[(k + 1) & 1], ((k + 1) >> 1) & 1, p.err)) {
                        go = false;
                        break;
                    }
                    issue_cb(k + 1);
                    if (k + 2 < nblk) {
                        if (!mbar_wait(bar_bfree, k & 1, p.err)) { go = false; break; }
                        load_b(k + 2);
                        b_last[k & 1] = k + 2;
                    }
                }
            }
            if (!go) {
                // a wait gave up: let the loads still in flight land (bounded)
                mbar_wait(bar_c, c_last & 1, p.err);
                for (int j = 0; j < 2; ++j)
                    if (b_last[j] >= 0) mbar_wait(&bar_b[j], (b_last[j] >> 1) & 1, p.err);
                for (int hh = 0; hh < NHEAD; ++hh) mbar_wait(&bar_x[hh], x_last[hh] & 1, p.err);
            }
        }
    } else {
        // ================= compute warps: head hh, one TMEM lane / row each =================
        const int hh = warp / 4, wq = warp & 3, row = tid & 127;
        const int h = h0 + hh;
        const int nb = 1 + hh;  // named barrier of this head's 128 threads
        const uint32_t trow = tmem + ((uint32_t)(wq * 32) << 16);
        const float A2 = p.A[h * p.sA] * kLog2e;
        const float Dh = p.Dv ? p.Dv[h * p.sD] : 0.f;
        const bool factor = A2 <= 0.f;
        float* cum = reinterpret_cast<float*>(sm + OFF_CUM) + hh * 128;
        float* dtf = reinterpret_cast<float*>(sm + OFF_DTF) + hh * 128;
        float* gf = reinterpret_cast<float*>(sm + OFF_GF) + hh * 128;
        // M_ii of the thread's row, from its M build to its epilogue (in shared
        // memory rather than a register held across the block)
        const uint32_t sdiag = smem_u32(sm + OFF_DIAG) + (hh * 128 + row) * 4;
        uint8_t* xs = sm + OFF_X + hh * 16384;
        uint8_t* ss = sm + OFF_S + hh * 16384;

        float S[P];
        const float* h0row = p.h0 ? p.h0 + (int64_t)b * p.sh_b + (int64_t)h * p.sh_h +
                                        (int64_t)row * p.sh_n
                                  : nullptr;
#pragma unroll
        for (int i = 0; i < P; ++i) S[i] = h0row ? h0row[i * p.sh_p] : 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(ss + swz(row, c)) =
                make_uint4(pack_bf16(S[c * 8 + 0], S[c * 8 + 1]), pack_bf16(S[c * 8 + 2], S[c * 8 + 3]),
                           pack_bf16(S[c * 8 + 4], S[c * 8 + 5]), pack_bf16(S[c * 8 + 6], S[c * 8 + 7]));
        fence_proxy_async_smem();
        mbar_arrive(&bar_s[hh]);  // S(0) is ready

        // ---- cumulative decay of block k (log2 units) and the column factors:
        //      this row's step, cumulative decay and the block's total in
        //      registers, the head's columns in shared memory (read by the M
        //      build only, so the next block's may replace them once every
        //      thread of the head has built its row of M).  Every warp of the
        //      head forms all four 32-step chunks (lane l holds steps l,
        //      l + 32, l + 64, l + 96), so no barrier between the warps is
        //      needed: the same scan within each chunk, then the earlier
        //      chunks' totals in order, and the same values written by all.
        //      `landed`: the head already knows that dt of block k is here.
        auto cumsum = [&](int k, bool landed, float& cum_t, float& dtv, float& cum_last) -> bool {
            if (!landed && !named_sync_and(nb, 128, mbar_wait(bar_c, k & 1, p.err))) return false;
            const uint8_t* dts = sm + OFF_DT + (k & 1) * 2048 + (h & 7) * 2;
            float d[4], v[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint16_t raw = *reinterpret_cast<const uint16_t*>(dts + (c * 32 + lane) * 16);
                d[c] = __uint_as_float((uint32_t)raw << 16);
                v[c] = d[c] * A2;
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float u = __shfl_up_sync(0xffffffffu, v[c], o);
                    if (lane >= o) v[c] += u;
                }
            }
            float tot[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) tot[c] = __shfl_sync(0xffffffffu, v[c], 31);
#pragma unroll
            for (int c = 1; c < 4; ++c)
#pragma unroll
                for (int w = 0; w < c; ++w) v[c] += tot[w];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float cend = __shfl_sync(0xffffffffu, v[c], 31);
                const int r = c * 32 + lane;
                cum[r] = v[c];
                dtf[r] = d[c];
                gf[r] = ex2_approx(cend - v[c]) * d[c];  // <= dt when A <= 0
            }
            __syncwarp();
            cum_t = wq == 0 ? v[0] : wq == 1 ? v[1] : wq == 2 ? v[2] : v[3];
            dtv = wq == 0 ? d[0] : wq == 1 ? d[1] : wq == 2 ? d[2] : d[3];
            cum_last = __shfl_sync(0xffffffffu, v[3], 31);
            return true;
        };

        float cum_t = 0.f, dtv = 0.f, cum_last = 0.f;
        bool ok = cumsum(0, false, cum_t, dtv, cum_last);
        for (int k = 0; k < nblk && ok; ++k) {
            const int t0 = k * QB;
            if (!named_sync_and(nb, 128, mbar_wait(bar_cb, k & 1, p.err))) { ok = false; break; }
            tc::fence_after_sync();
            // ---- row `row` of M = C B^T o decay o dt (strictly lower
            //      triangle), bf16, into this head's dS^T columns of TMEM (free
            //      from the last state update to this block's B^T X~): chunk jc
            //      in columns tm_ds(hh) + 16 jc .. + 16; the diagonal
            //      M_ii = (C B^T)_ii dt_i in fp32 (in shared memory, sdiag)
#pragma unroll 1
            for (int jc = 0; jc < 4; ++jc) {
                uint32_t w[16];
                if (jc <= wq) {
                    float cb[32];
                    tc::tmem_ld32(trow + jc * 32, cb);
                    tc::tmem_wait_ld();
                    float m[32];
                    if (jc < wq && factor) {
                        const float f1 = ex2_approx(cum_t - cum[jc * 32 + 31]);
                        const float2 f11 = make_float2(f1, f1);
                        const float2* g2 = reinterpret_cast<const float2*>(gf + jc * 32);
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float2 v = __fmul2_rn(make_float2(cb[2 * e], cb[2 * e + 1]),
                                                        __fmul2_rn(f11, g2[e]));
                            m[2 * e] = v.x;
                            m[2 * e + 1] = v.y;
                        }
                    } else {
                        const float2* c2 = reinterpret_cast<const float2*>(cum + jc * 32);
                        const float2* d2 = reinterpret_cast<const float2*>(dtf + jc * 32);
                        const float2 ct = make_float2(cum_t, cum_t);
                        // the diagonal (j = row) stays out of the bf16 M: the pair
                        // holding it (row & 31) / 2 is kept in fp32 and the
                        // epilogue adds M_ii x_i with the skip term
                        const int ed = (row & 31) >> 1;
                        float2 pick = make_float2(0.f, 0.f);
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int j = jc * 32 + 2 * e;
                            const float2 arg = __ffma2_rn(c2[e], make_float2(-1.f, -1.f), ct);  // ct - c, exact negation
                            const float2 dec = make_float2(ex2_approx(arg.x), ex2_approx(arg.y));  // j > row: discarded
                            const float2 v = __fmul2_rn(__fmul2_rn(make_float2(cb[2 * e], cb[2 * e + 1]), dec), d2[e]);
                            if (e == ed) pick = v;
                            m[2 * e] = j < row ? v.x : 0.f;
                            m[2 * e + 1] = j + 1 < row ? v.y : 0.f;
                        }
                        if (jc == wq)
                            asm volatile("st.shared.f32 [%0], %1;" ::"r"(sdiag), "f"((row & 1) ? pick.y : pick.x)
                                         : "memory");
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e) w[e] = pack_bf16(m[2 * e], m[2 * e + 1]);
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) w[e] = 0u;
                }
                tc::tmem_st16(trow + tm_ds(hh) + 16 * jc, w);
            }
            tc::tmem_wait_st();
            // ---- X~ row = w_t x_t into the state-copy buffer, once C S^T has read it
            const bool got = mbar_wait(&bar_x[hh], k & 1, p.err) && mbar_wait(&bar_yoff[hh], k & 1, p.err);
            if (!named_sync_and(nb, 128, got)) { ok = false; break; }
            {
                const float wt = ex2_approx(cum_last - cum_t) * dtv;
                const float2 wt2 = make_float2(wt, wt);
                // all eight chunks of the x row first: the stores below go to
                // another buffer, but the compiler cannot tell
                uint4 xr[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) xr[c] = *reinterpret_cast<const uint4*>(xs + swz(row, c));
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float x8[8];
                    unpack8(xr[c], x8);
                    uint32_t w[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 v = __fmul2_rn(wt2, make_float2(x8[2 * i], x8[2 * i + 1]));
                        w[i] = pack_bf16(v.x, v.y);
                    }
                    *reinterpret_cast<uint4*>(ss + swz(row, c)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            fence_proxy_async_smem();
            tc::fence_before_sync();
            mbar_arrive(&bar_m[hh]);

            // ---- the next block's cumulative decay while this block's MMAs
            //      run if its dt has landed, else after the state update (a
            //      late dt must not hold up this block's epilogue)
            float n_cum_t = 0.f, n_dtv = 0.f, n_cum_last = 0.f;
            const bool early = k + 1 < nblk && !p.late_cumsum &&
                               named_sync_and(nb, 128, mbar_test(bar_c, (k + 1) & 1));
            if (early && !cumsum(k + 1, true, n_cum_t, n_dtv, n_cum_last)) { ok = false; break; }

            if (!named_sync_and(nb, 128, mbar_wait(&bar_mma23[hh], k & 1, p.err))) { ok = false; break; }
            tc::fence_after_sync();
            // ---- y row = Ydiag + exp(cum) Yoff + (D + M_ii) x, written over the
            //      row's x in shared memory; the tile leaves with one TMA store
            //      (rows past the end are clipped)
            {
                const float eoff = ex2_approx(cum_t);
                float mii;
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(mii) : "r"(sdiag) : "memory");
                const float dx = Dh + mii;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float yd[32], yo[32];
                    tc::tmem_ld32(trow + tm_ydg(hh) + half * 32, yd);
                    tc::tmem_ld32(trow + tm_yoff(hh) + half * 32, yo);
                    uint4 xr[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) xr[q] = *reinterpret_cast<const uint4*>(xs + swz(row, half * 4 + q));
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4* cell = reinterpret_cast<uint4*>(xs + swz(row, half * 4 + q));
                        float x8[8];
                        unpack8(xr[q], x8);
                        uint32_t w[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int e = q * 8 + 2 * i;
                            const float2 o = __ffma2_rn(
                                make_float2(dx, dx), make_float2(x8[2 * i], x8[2 * i + 1]),
                                __ffma2_rn(make_float2(eoff, eoff), make_float2(yo[e], yo[e + 1]),
                                           make_float2(yd[e], yd[e + 1])));
                            w[i] = pack_bf16(o.x, o.y);
                        }
                        *cell = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
                fence_proxy_async_smem();
                named_sync(nb, 128);
                if (row == 0) {
                    tma_store_4d(&tm_y, xs, 0, h, t0, b);
                    bulk_commit();
                }
            }
            // ---- S^T row <- exp(cum_last) S^T + dS^T; bf16 copy for block k+1
            if (!named_sync_and(nb, 128, mbar_wait(bar_bfree, k & 1, p.err))) { ok = false; break; }
            tc::fence_after_sync();
            {
                const float ablk = ex2_approx(cum_last);
                float ds[64];
                tc::tmem_ld32(trow + tm_ds(hh), ds);
                tc::tmem_ld32(trow + tm_ds(hh) + 32, ds + 32);
                tc::tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 64; i += 2) {
                    const float2 v = __ffma2_rn(make_float2(ablk, ablk), make_float2(S[i], S[i + 1]),
                                                make_float2(ds[i], ds[i + 1]));
                    S[i] = v.x;
                    S[i + 1] = v.y;
                }
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4*>(ss + swz(row, c)) =
                        make_uint4(pack_bf16(S[c * 8 + 0], S[c * 8 + 1]), pack_bf16(S[c * 8 + 2], S[c * 8 + 3]),
                                   pack_bf16(S[c * 8 + 4], S[c * 8 + 5]), pack_bf16(S[c * 8 + 6], S[c * 8 + 7]));
            }
            fence_proxy_async_smem();
            tc::fence_before_sync();
            if (row == 0) bulk_wait_read<0>();  // y has left the x tile: it may be refilled
            mbar_arrive(&bar_s[hh]);
            if (k + 1 < nblk && !early && !cumsum(k + 1, false, n_cum_t, n_dtv, n_cum_last)) { ok = false; break; }
            cum_t = n_cum_t;
            dtv = n_dtv;
            cum_last = n_cum_last;
        }
        if (row == 0) bulk_wait<0>();
        if (ok && p.last) {
            float* ls = p.last + (int64_t)b * p.sl_b + (int64_t)h * p.sl_h + (int64_t)row * p.sl_n;
#pragma unroll
            for (int i = 0; i < P; ++i) ls[i * p.sl_p] = S[i];
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace ssdtc2

// ---------------------------------------------------------------------------
// Host side.

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                              CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                              CUtensorMapFloatOOBfill);

static bool encode(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                   const cuuint64_t* strides_bytes, const cuuint32_t* box, bool swizzle) {
    auto enc = reinterpret_cast<EncodeFn>(tensor_map_encoder());
    if (!enc) return false;
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims,
               strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static bool tc_layout_ok(const SSDArgs& a) {
    if (a.dtype != SS_BF16 || a.P != ssdtc::P || a.N != ssdtc::N) return false;
    auto al16 = [](const void* ptr) { return reinterpret_cast<uintptr_t>(ptr) % 16 == 0; };
    auto m8 = [](int64_t s) { return s % 8 == 0 && s * 2 < (int64_t(1) << 40); };
    if (a.sx_p != 1 || !al16(a.x) || !m8(a.sx_l) || !m8(a.sx_h) || !m8(a.sx_b)) return false;
    if (a.sB_n != 1 || !al16(a.Bm) || !m8(a.sB_l) || !m8(a.sB_g) || !m8(a.sB_b)) return false;
    if (a.sC_n != 1 || !al16(a.Cm) || !m8(a.sC_l) || !m8(a.sC_g) || !m8(a.sC_b)) return false;
    if (a.sdt_h != 1 || !al16(a.dt) || !m8(a.sdt_l) || !m8(a.sdt_b)) return false;
    if (a.sy_p != 1 || !al16(a.y) || !m8(a.sy_l) || !m8(a.sy_h) || !m8(a.sy_b)) return false;
    return true;
}

// dt whose (b, l) rows of H values are not at a 16-byte pitch (H not a
// multiple of 8, for one) while everything else suits the tensor-core
// kernels: dt is copied into stream-ordered scratch with the pitch rounded up
// to 8 heads (B * L * H values, small beside x) and the kernels read it from
// there.  *taken stays false when that does not make the layout fit.
int launch_ssd_tc(const SSDArgs& a, cudaStream_t st, const Scratch& scratch, bool* taken);

static int run_dt_padded(const SSDArgs& a, cudaStream_t st, const Scratch& scratch, bool* taken) {
    *taken = false;
    if (a.dtype != SS_BF16 || a.sdt_h != 1 || a.H < 1 || scratch.limit != ~size_t(0)) return SS_OK;
    if (a.L > 1 && a.sdt_l < a.H) return SS_OK;  // rows overlap
    const int64_t Hp = padded_len(a.H, 2);
    SSDArgs c = a;
    c.dt = reinterpret_cast<const void*>(uintptr_t(256));  // stands in until the scratch exists
    c.sdt_l = Hp;
    c.sdt_b = (int64_t)a.L * Hp;
    if (!tc_layout_ok(c)) return SS_OK;
    void* pdt = scratch.alloc((size_t)a.Bsz * a.L * Hp * 2, st, scratch.ctx);
    if (!pdt) return SS_OK;
    RowPacker pk(SS_BF16, a.H, Hp, st);
    pk.add(pdt, a.dt, a.Bsz, a.sdt_b, a.L, a.sdt_l, true);
    int rc = pk.flush();
    *taken = true;
    if (rc == SS_OK) {
        c.dt = pdt;
        bool t2 = false;
        rc = launch_ssd_tc(c, st, scratch, &t2);
    }
    scratch.release(pdt, st, scratch.ctx);
    return rc;
}

// Path selection for tests: SS_DEBUG_SSD_PATH 0 forces the CUDA-core kernel.
int launch_ssd_tc(const SSDArgs& a, cudaStream_t st, const Scratch& scratch, bool* taken) {
    *taken = false;
    const int path = debug_path(SS_DEBUG_SSD_PATH);
    if (path == 0 || a.L < 1) return SS_OK;
    if (!tc_layout_ok(a)) return run_dt_padded(a, st, scratch, taken);
    *taken = true;

    CUtensorMap mx, mb, mc, mdt;
    {
        cuuint64_t dims[4] = {(cuuint64_t)a.P, (cuuint64_t)a.H, (cuuint64_t)a.L, (cuuint64_t)a.Bsz};
        cuuint64_t str[3] = {(cuuint64_t)(a.sx_h * 2), (cuuint64_t)(a.sx_l * 2), (cuuint64_t)(a.sx_b * 2)};
        cuuint32_t box[4] = {64, 1, ssdtc::QB, 1};
        if (!encode(&mx, a.x, 4, dims, str, box, true)) return SS_ERR_CUDA;
    }
    {
        cuuint64_t dims[4] = {(cuuint64_t)a.N, (cuuint64_t)a.G, (cuuint64_t)a.L, (cuuint64_t)a.Bsz};
        cuuint64_t sb[3] = {(cuuint64_t)(a.sB_g * 2), (cuuint64_t)(a.sB_l * 2), (cuuint64_t)(a.sB_b * 2)};
        cuuint64_t sc[3] = {(cuuint64_t)(a.sC_g * 2), (cuuint64_t)(a.sC_l * 2), (cuuint64_t)(a.sC_b * 2)};
        cuuint32_t box[4] = {64, 1, ssdtc::QB, 1};
        if (!encode(&mb, a.Bm, 4, dims, sb, box, true)) return SS_ERR_CUDA;
        if (!encode(&mc, a.Cm, 4, dims, sc, box, true)) return SS_ERR_CUDA;
    }
    {
        cuuint64_t dims[3] = {(cuuint64_t)a.H, (cuuint64_t)a.L, (cuuint64_t)a.Bsz};
        cuuint64_t str[2] = {(cuuint64_t)(a.sdt_l * 2), (cuuint64_t)(a.sdt_b * 2)};
        cuuint32_t box[3] = {8, ssdtc::QB, 1};
        if (!encode(&mdt, a.dt, 3, dims, str, box, false)) return SS_ERR_CUDA;
    }
    CUtensorMap my;
    {
        cuuint64_t dims[4] = {(cuuint64_t)a.P, (cuuint64_t)a.H, (cuuint64_t)a.L, (cuuint64_t)a.Bsz};
        cuuint64_t str[3] = {(cuuint64_t)(a.sy_h * 2), (cuuint64_t)(a.sy_l * 2), (cuuint64_t)(a.sy_b * 2)};
        cuuint32_t box[4] = {64, 1, ssdtc::QB, 1};
        if (!encode(&my, a.y, 4, dims, str, box, true)) return SS_ERR_CUDA;
    }
    ssdtc::Params p{};
    p.Bsz = a.Bsz; p.L = a.L; p.H = a.H; p.G = a.G;
    p.late_cumsum = debug_path(SS_DEBUG_SSD_LATE_CUMSUM) == 1;
    p.A = a.A; p.sA = a.sA; p.Dv = a.Dv; p.sD = a.sD;
    p.y = static_cast<__nv_bfloat16*>(a.y); p.sy_b = a.sy_b; p.sy_l = a.sy_l; p.sy_h = a.sy_h;
    p.last = a.last; p.sl_b = a.sl_b; p.sl_h = a.sl_h; p.sl_p = a.sl_p; p.sl_n = a.sl_n;
    p.h0 = a.h0; p.sh_b = a.sh_b; p.sh_h = a.sh_h; p.sh_p = a.sh_p; p.sh_n = a.sh_n;
    p.err = a.err;

    // two heads per CTA when every group holds an even number of heads
    // (SS_DEBUG_SSD_PATH 2 keeps one head per CTA, for tests)
    const bool pair = (a.H / a.G) % 2 == 0 && path != 2;
    static bool attr_set[2][64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[pair][dev]) {
        const cudaError_t e =
            pair ? cudaFuncSetAttribute(ssdtc2::ssd_chunk_tc2,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        ssdtc2::SMEM_BYTES)
                 : cudaFuncSetAttribute(ssdtc::ssd_chunk_tc,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        ssdtc::SMEM_BYTES);
        if (e != cudaSuccess) return SS_ERR_LAUNCH;
        if (dev >= 0 && dev < 64) attr_set[pair][dev] = true;
    }
    if (pair)
        ssdtc2::ssd_chunk_tc2<<<(unsigned)(a.Bsz * (a.H / 2)), ssdtc2::NTHREADS, ssdtc2::SMEM_BYTES,
                                st>>>(mx, mb, mc, mdt, my, p);
    else
        ssdtc::ssd_chunk_tc<<<(unsigned)(a.Bsz * a.H), ssdtc::NTHREADS, ssdtc::SMEM_BYTES, st>>>(
            mx, mb, mc, mdt, p);
    count_launch(1);
    return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_LAUNCH;
}

}  // namespace ss
