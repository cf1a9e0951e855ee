// selective_scan_grouped.cu -- the selective scan with B, C per channel
// group when the groups are smaller than the shared-B, C kernel's channel
// tile (down to one B, C per channel).  Same recurrence as selective_scan.cu
// (page "Mamba模型笔记" §2.2, §4.1: B and C depend on the input, one SSM per
// channel); only the way B and C reach the lanes differs.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <initializer_list>

#include "internal.h"
#include "ptx.cuh"
#include "scan_common.cuh"
#include "ssscan.h"

namespace ss {

// ---------------------------------------------------------------------------
// Per-channel B / C (groups smaller than a channel tile, e.g. one B, C per
// channel): every channel streams its own 2 N rows, 64 bytes per step in bf16,
// so the kernel is bound by HBM.  Sixteen lanes per channel, lane n keeping
// state n; rows are read 16 steps (32 or 64 bytes) at a time with vector
// loads.  delta is computed once per step (lane n takes step n of the chunk)
// and shared by shuffles; the 16 partial readouts of each lane are
// reduce-scattered so that lane n ends with y of step n and finishes it.

template <typename T>
__device__ __forceinline__ void load16_row(const T* p, float* v) {
    if constexpr (sizeof(T) == 2) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const uint4 w = __ldg(reinterpret_cast<const uint4*>(p) + q);
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[8 * q + 2 * i] = __uint_as_float(ww[i] << 16);
                v[8 * q + 2 * i + 1] = __uint_as_float(ww[i] & 0xffff0000u);
            }
        }
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 w = __ldg(reinterpret_cast<const float4*>(p) + q);
            v[4 * q] = w.x; v[4 * q + 1] = w.y; v[4 * q + 2] = w.z; v[4 * q + 3] = w.w;
        }
    }
}

template <typename T, bool HAS_Z>
__global__ void __launch_bounds__(256) scan_pc(ScanArgs a) {
    constexpr int TC = 16;
    const int lane = threadIdx.x & 31, n = lane & 15;
    const int64_t ch = (int64_t)blockIdx.x * 16 + (threadIdx.x >> 4);
    const bool valid = ch < (int64_t)a.Bsz * a.D;
    const int64_t chs = valid ? ch : 0;
    const int b = (int)(chs / a.D), d = (int)(chs % a.D);
    const int g = a.G > 1 ? d / (a.D / a.G) : 0;
    const float A2 = a.A[d * a.sA_d + n * a.sA_n] * kLog2e;
    float h = (valid && a.h0) ? a.h0[b * a.sh_b + d * a.sh_d + n * a.sh_n] : 0.f;
    const float Dd = a.Dv ? a.Dv[d * a.sD] : 0.f;
    const float bd = a.bias ? a.bias[d * a.sbias] : 0.f;
    const bool sp = a.softplus != 0;
    const T* u = static_cast<const T*>(a.u) + b * a.su_b + d * a.su_d;
    const T* dl = static_cast<const T*>(a.dl) + b * a.sdl_b + d * a.sdl_d;
    const T* z = HAS_Z ? static_cast<const T*>(a.z) + b * a.sz_b + d * a.sz_d : nullptr;
    T* y = static_cast<T*>(a.y) + b * a.sy_b + d * a.sy_d;
    const T* Bp = static_cast<const T*>(a.Bm) + b * a.sB_b + g * a.sB_g + n * a.sB_n;
    const T* Cp = static_cast<const T*>(a.Cm) + b * a.sC_b + g * a.sC_g + n * a.sC_n;
    const int src = lane & 16;  // first lane of this channel's group

    for (int t0 = 0; t0 < a.L; t0 += TC) {
        const int tn = min(TC, a.L - t0);
        float bv[TC], cv[TC], uv[TC];
        if (tn == TC) {
            load16_row<T>(Bp + t0, bv);
            load16_row<T>(Cp + t0, cv);
            load16_row<T>(u + t0, uv);
        } else {
#pragma unroll
            for (int j = 0; j < TC; ++j) {
                const bool in = j < tn;
                bv[j] = in ? Elem<T>::to_f(Bp[t0 + j]) : 0.f;
                cv[j] = in ? Elem<T>::to_f(Cp[t0 + j]) : 0.f;
                uv[j] = in ? Elem<T>::to_f(u[t0 + j]) : 0.f;
            }
        }
        float own = 0.f;
        if (n < tn) {
            const float x = Elem<T>::to_f(dl[t0 + n]) + bd;
            own = softplus_if(x, sp);
        }
        float yp[TC];
#pragma unroll
        for (int j = 0; j < TC; ++j) {
            const float dd = __shfl_sync(0xffffffffu, own, src + j);
            h = fmaf(ex2_approx(dd * A2), h, dd * uv[j] * bv[j]);
            yp[j] = cv[j] * h;
        }
        float y8[8], y4[4], y2[2], y1[1];
        reduce_half<16>(yp, y8, lane & 8, 8);
        reduce_half<8>(y8, y4, lane & 4, 4);
        reduce_half<4>(y4, y2, lane & 2, 2);
        reduce_half<2>(y2, y1, lane & 1, 1);
        // lane n now holds the readout of step t0 + n
        if (valid && n < tn) {
            const float uu = Elem<T>::to_f(u[t0 + n]);
            float out = fmaf(Dd, uu, y1[0]);
            if constexpr (HAS_Z) {
                const float zz = Elem<T>::to_f(z[t0 + n]);
                out *= zz * sigmoid_accurate(zz);
            }
            y[t0 + n] = Elem<T>::from_f(out);
        }
    }
    if (valid && a.last) a.last[b * a.sl_b + d * a.sl_d + n * a.sl_n] = h;
}

// Groups of 1, 2, 4 or 8 channels with TMA staging: the per-lane row loads
// above make a warp touch 32 rows per instruction, so L1 throughput, not HBM,
// bounds scan_pc.  Here a CTA takes 8 consecutive channels of one batch row; a
// producer warp streams, per tile of 128 bytes of t, the u / delta / z rows and
// the 16 B and 16 C rows of each group the tile's channels read
// ([group][n][t], 128-byte swizzle) into a 3-stage mbarrier ring, and 16 lanes
// per channel read their state's row 8 steps at a time from shared memory.
namespace pc2 {

template <typename T>
struct Cfg {
    static constexpr int ES = (int)sizeof(T);
    static constexpr int TT = 128 / ES;   // steps per tile
    static constexpr int CH = 8;          // channels per CTA
    static constexpr int STAGES = 3;
    static constexpr int ACT = CH * 128;  // one activation tile
    static constexpr int BC = CH * 16 * 128;  // B (or C) rows of the CTA's channels
    static constexpr int OFF_U = 0, OFF_DL = ACT, OFF_Z = 2 * ACT, OFF_B = 4 * ACT;
    static constexpr int OFF_C = OFF_B + BC;
    static constexpr int STAGE = OFF_C + BC;  // 4 KB + 32 KB
    static constexpr int NCONS = CH * 16;     // consumer threads
    static constexpr int NTHREADS = NCONS + 32;
    static constexpr int SMEM = STAGE * STAGES + 64 + 1024;
    static_assert(STAGE % 1024 == 0, "swizzled tiles 1024-aligned");
};

template <typename T, bool HAS_Z>
__global__ void __launch_bounds__(Cfg<T>::NTHREADS, 2)
scan_pc_tma(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_dl,
            const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_B,
            const __grid_constant__ CUtensorMap tm_C, const ScanArgs a) {
    using C = Cfg<T>;
    constexpr int ES = C::ES, TT = C::TT, S = C::STAGES;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGE * S);
    uint64_t* empty = full + S;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int dtiles = (a.D + C::CH - 1) / C::CH;
    const int b = blockIdx.x / dtiles, d0 = (blockIdx.x % dtiles) * C::CH;
    const int ntiles = (a.L + TT - 1) / TT;
    // channels per B / C group (1, 2, 4 or 8): the tile's 8 channels read
    // 8 / gsize group rows of B and C, starting at group d0 / gsize
    const int gsize = a.D / a.G;
    const int ngr = C::CH / gsize;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], C::NCONS);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == C::NCONS / 32) {
        if (lane == 0) {
            tma_prefetch_desc(&tm_u);
            tma_prefetch_desc(&tm_dl);
            tma_prefetch_desc(&tm_B);
            tma_prefetch_desc(&tm_C);
            if (HAS_Z) tma_prefetch_desc(&tm_z);
            for (int k = 0; k < ntiles; ++k) {
                const int s = k % S;
                if (k >= S && !mbar_wait(&empty[s], ((k / S) - 1) & 1, a.err)) break;
                uint8_t* st = smem + s * C::STAGE;
                const int t0 = k * TT;
                mbar_arrive_expect_tx(&full[s], (HAS_Z ? 3 : 2) * C::ACT + 2 * ngr * 16 * 128);
                tma_load_3d(st + C::OFF_U, &tm_u, &full[s], t0, d0, b);
                tma_load_3d(st + C::OFF_DL, &tm_dl, &full[s], t0, d0, b);
                if (HAS_Z) tma_load_3d(st + C::OFF_Z, &tm_z, &full[s], t0, d0, b);
                tma_load_4d(st + C::OFF_B, &tm_B, &full[s], t0, 0, d0 / gsize, b);
                tma_load_4d(st + C::OFF_C, &tm_C, &full[s], t0, 0, d0 / gsize, b);
            }
        }
        return;
    }

    const int ci = tid >> 4, n = tid & 15;  // channel row in the tile, state
    const int d = d0 + ci;
    const bool valid = d < a.D;
    const int dd_ = valid ? d : 0;
    const float A2 = a.A[dd_ * a.sA_d + n * a.sA_n] * kLog2e;
    float h = (valid && a.h0) ? a.h0[b * a.sh_b + dd_ * a.sh_d + n * a.sh_n] : 0.f;
    const float Dd = a.Dv ? a.Dv[dd_ * a.sD] : 0.f;
    const float bd = a.bias ? a.bias[dd_ * a.sbias] : 0.f;
    const bool sp = a.softplus != 0;
    T* y = static_cast<T*>(a.y) + b * a.sy_b + dd_ * a.sy_d;
    const int src = lane & 16;
    const int brow = (ci / gsize) * 16 + n;  // this lane's B / C row in the tile

    bool ok = true;
    for (int k = 0; k < ntiles; ++k) {
        const int s = k % S;
        if (!mbar_wait(&full[s], (k / S) & 1, a.err)) { ok = false; break; }
        const uint32_t st = smem_u32(smem + s * C::STAGE);
        const int t0 = k * TT, tn = min(TT, a.L - t0);
#pragma unroll 1
        for (int c16 = 0; c16 < TT / 16; ++c16) {
            const int j0 = c16 * 16;  // first step of this 16-step chunk in the tile
            // delta: lane n takes step j0 + n
            float own = 0.f;
            {
                const int j = j0 + n;
                const uint32_t off = (ci << 7) + ((((j * ES) >> 4) ^ (ci & 7)) << 4) + ((j * ES) & 15);
                const float x = (ES == 2 ? __uint_as_float(lds16(st + C::OFF_DL + off) << 16)
                                         : __uint_as_float(lds32(st + C::OFF_DL + off))) + bd;
                own = j < tn ? softplus_if(x, sp) : 0.f;
            }
            // this lane's B and C row, 16 steps, and the channel's u
            float bv[16], cv[16], uv[16];
#pragma unroll
            for (int q = 0; q < 16 * ES / 16; ++q) {
                const int chunk = (j0 * ES) / 16 + q;
                const uint32_t ob = brow * 128 + ((chunk ^ (brow & 7)) << 4);
                const uint32_t ou = (ci << 7) + ((chunk ^ (ci & 7)) << 4);
                constexpr int PER = 16 / ES;  // elements per 16 bytes
                lds_elems<T, PER>(st + C::OFF_B + ob, bv + q * PER);
                lds_elems<T, PER>(st + C::OFF_C + ob, cv + q * PER);
                lds_elems<T, PER>(st + C::OFF_U + ou, uv + q * PER);
            }
            float yp[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float dd = __shfl_sync(0xffffffffu, own, src + j);
                h = fmaf(ex2_approx(dd * A2), h, dd * uv[j] * bv[j]);
                yp[j] = cv[j] * h;
            }
            float y8[8], y4[4], y2[2], y1[1];
            reduce_half<16>(yp, y8, lane & 8, 8);
            reduce_half<8>(y8, y4, lane & 4, 4);
            reduce_half<4>(y4, y2, lane & 2, 2);
            reduce_half<2>(y2, y1, lane & 1, 1);
            // lane n holds the readout of step j0 + n
            const int j = j0 + n;
            if (valid && j < tn) {
                const uint32_t off = (ci << 7) + ((((j * ES) >> 4) ^ (ci & 7)) << 4) + ((j * ES) & 15);
                const float uu = ES == 2 ? __uint_as_float(lds16(st + C::OFF_U + off) << 16)
                                         : __uint_as_float(lds32(st + C::OFF_U + off));
                float out = fmaf(Dd, uu, y1[0]);
                if constexpr (HAS_Z) {
                    const float zz = ES == 2 ? __uint_as_float(lds16(st + C::OFF_Z + off) << 16)
                                             : __uint_as_float(lds32(st + C::OFF_Z + off));
                    out *= zz * sigmoid_accurate(zz);
                }
                y[t0 + j] = Elem<T>::from_f(out);
            }
        }
        mbar_arrive(&empty[s]);
    }
    if (ok && valid && a.last) a.last[b * a.sl_b + d * a.sl_d + n * a.sl_n] = h;
}

}  // namespace pc2

static bool pc_tma_ok(const ScanArgs& a) {
    if (a.G <= 1 || a.N != 16 || a.cw || a.L >= (1 << 30)) return false;
    const int gsize = a.D / a.G;  // channels per group: the tile's 8 must hold whole groups
    if (gsize != 1 && gsize != 2 && gsize != 4 && gsize != 8) return false;
    const int es = a.dtype == SS_BF16 ? 2 : 4;
    auto al = [&](const void* ptr, std::initializer_list<int64_t> outer, int64_t st) {
        if (!ptr) return true;
        if (st != 1 && a.L > 1) return false;
        if (reinterpret_cast<uintptr_t>(ptr) % 16) return false;
        for (int64_t o : outer)
            if ((o * es) % 16 || o * es >= (int64_t(1) << 40)) return false;
        return true;
    };
    return al(a.u, {a.su_b, a.su_d}, a.su_t) && al(a.dl, {a.sdl_b, a.sdl_d}, a.sdl_t) &&
           al(a.z, {a.sz_b, a.sz_d}, a.sz_t) && al(a.Bm, {a.sB_b, a.sB_g, a.sB_n}, a.sB_t) &&
           al(a.Cm, {a.sC_b, a.sC_g, a.sC_n}, a.sC_t) && (a.sy_t == 1 || a.L <= 1);
}

static bool make_map_bc4(CUtensorMap* m, const void* base, int dtype, int64_t L, int64_t G,
                         int64_t Bsz, int64_t sn, int64_t sg, int64_t sb, int box_t, int box_g) {
    auto enc = reinterpret_cast<EncodeFn>(tensor_map_encoder());
    if (!enc) return false;
    const int es = dtype == SS_BF16 ? 2 : 4;
    cuuint64_t dims[4] = {(cuuint64_t)L, 16, (cuuint64_t)G, (cuuint64_t)Bsz};
    cuuint64_t strides[3] = {(cuuint64_t)(sn * es), (cuuint64_t)(sg * es), (cuuint64_t)(sb * es)};
    cuuint32_t box[4] = {(cuuint32_t)box_t, 16, (cuuint32_t)box_g, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, dtype == SS_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
               4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T>
static int run_pc_tma(const ScanArgs& a, cudaStream_t st) {
    using C = pc2::Cfg<T>;
    CUtensorMap m[5];
    if (!make_map_3d(&m[0], a.u, a.dtype, a.L, a.D, a.Bsz, a.su_d, a.su_b, C::TT, C::CH) ||
        !make_map_3d(&m[1], a.dl, a.dtype, a.L, a.D, a.Bsz, a.sdl_d, a.sdl_b, C::TT, C::CH) ||
        !make_map_bc4(&m[3], a.Bm, a.dtype, a.L, a.G, a.Bsz, a.sB_n, a.sB_g, a.sB_b, C::TT,
                      C::CH / (a.D / a.G)) ||
        !make_map_bc4(&m[4], a.Cm, a.dtype, a.L, a.G, a.Bsz, a.sC_n, a.sC_g, a.sC_b, C::TT,
                      C::CH / (a.D / a.G)))
        return -1;
    if (a.z) {
        if (!make_map_3d(&m[2], a.z, a.dtype, a.L, a.D, a.Bsz, a.sz_d, a.sz_b, C::TT, C::CH)) return -1;
    } else {
        m[2] = m[0];
    }
    auto kern = a.z ? pc2::scan_pc_tma<T, true> : pc2::scan_pc_tma<T, false>;
    static bool attr_set[2][64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    const int zi = a.z ? 1 : 0;
    if (dev < 0 || dev >= 64 || !attr_set[zi][dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
            cudaSuccess)
            return SS_ERR_LAUNCH;
        if (dev >= 0 && dev < 64) attr_set[zi][dev] = true;
    }
    const int64_t ctas = (int64_t)a.Bsz * ((a.D + C::CH - 1) / C::CH);
    kern<<<(unsigned)ctas, C::NTHREADS, C::SMEM, st>>>(m[0], m[1], m[2], m[3], m[4], a);
    count_launch(1);
    return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_LAUNCH;
}

static bool pc_layout_ok(const ScanArgs& a) {
    if (a.N != 16 || a.cw) return false;
    const int es = a.dtype == SS_BF16 ? 2 : 4;
    auto row_ok = [&](const void* ptr, std::initializer_list<int64_t> outer, int64_t st) {
        if (!ptr) return true;
        if (st != 1 && a.L > 1) return false;
        if (reinterpret_cast<uintptr_t>(ptr) % 16) return false;
        for (int64_t o : outer)
            if ((o * es) % 16) return false;
        return true;
    };
    return row_ok(a.u, {a.su_b, a.su_d}, a.su_t) && row_ok(a.dl, {a.sdl_b, a.sdl_d}, a.sdl_t) &&
           row_ok(a.z, {a.sz_b, a.sz_d}, a.sz_t) && row_ok(a.y, {a.sy_b, a.sy_d}, a.sy_t) &&
           row_ok(a.Bm, {a.sB_b, a.sB_g, a.sB_n}, a.sB_t) &&
           row_ok(a.Cm, {a.sC_b, a.sC_g, a.sC_n}, a.sC_t);
}

template <typename T>
static int run_pc(const ScanArgs& a, cudaStream_t st) {
    const int64_t blocks = ((int64_t)a.Bsz * a.D + 15) / 16;
    if (a.z) scan_pc<T, true><<<(unsigned)blocks, 256, 0, st>>>(a);
    else scan_pc<T, false><<<(unsigned)blocks, 256, 0, st>>>(a);
    count_launch(1);
    return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_LAUNCH;
}

// Groups of 1, 2, 4 or 8 channels: the TMA kernel (SS_DEBUG_GROUPED_PATH 0 keeps the
// row-load kernel, for tests); other small groups: the row-load kernel.  *taken says
// whether a kernel was launched.
int launch_selective_grouped(const ScanArgs& a, cudaStream_t st, bool* taken) {
    *taken = false;
    const bool bf = a.dtype == SS_BF16;
    const bool rows = debug_path(SS_DEBUG_GROUPED_PATH) == 0;
    if (pc_tma_ok(a) && !rows) {
        const int rc = bf ? run_pc_tma<__nv_bfloat16>(a, st) : run_pc_tma<float>(a, st);
        if (rc != -1) {  // -1: no tensor map for this layout
            *taken = true;
            return rc;
        }
    }
    if (pc_layout_ok(a)) {
        *taken = true;
        return bf ? run_pc<__nv_bfloat16>(a, st) : run_pc<float>(a, st);
    }
    return SS_OK;
}

}  // namespace ss
