// selective_scan_wide.cu -- the selective scan for wider states, N in {32, 64,
// 128} (page "Mamba模型笔记" §2.2 recurrence, §4.3 gate; 0539edu paper talk
// §2.3 discretisation and §4.1: d_state 16 in Mamba-1, larger states for
// longer memory).  Same definition as selective_scan.cu; B, C shared by the
// channels of a batch row.
//
// N / 16 lanes per channel, 16 states per lane in registers.  A CTA of T
// threads (128 for N = 64, else 256) owns T / (N / 16) channels of one batch
// row.  Time runs in chunks
// of 32 steps: all threads load the chunk's B and C rows (16-byte loads, the
// next chunk's while the current one is scanned) and write them as an fp32
// table [t][state pair: B, B, C, C] in shared memory, double buffered.  Per
// 8-step sub-chunk, lane `part` computes delta (softplus) for its own steps and
// the channel's lanes exchange them by shuffles; each lane steps its 16 states
// with packed f32x2 arithmetic and keeps partial readouts, which are
// reduce-scattered so every lane finishes (skip, gate) and stores its own steps.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"
#include "scan_common.cuh"
#include "ssscan.h"

namespace ss {

namespace wide {

// Threads per CTA and CTAs per SM (the register budget), measured at the
// Mamba-130M layer shape (8 x 1536 x 2048, bf16).  N = 32 and 64: 128-thread
// CTAs, three per SM (up to 168 registers, no spills): 0.450 and 0.595 ms,
// against 0.583 ms (256 threads, two per SM, 128 registers and spills) and
// 0.643 ms (128 threads, four per SM, spills).  N = 128: 256-thread CTAs, two
// per SM: 1.20 ms, against 1.29 ms with three 128-thread CTAs (the fp32 B, C
// tables, 64 KB double-buffered, leave room for no more).
__host__ __device__ constexpr int threads_for(int N) { return N == 128 ? 256 : 128; }
__host__ __device__ constexpr int ctas_per_sm_for(int N) { return N == 128 ? 2 : 3; }
constexpr int TC = 32;  // steps per chunk
constexpr int VEC = 8;  // steps per sub-chunk

template <int N>
struct Cfg {
    static constexpr int NT = threads_for(N);     // threads per CTA
    static constexpr int NL = N / 16;             // lanes per channel
    static constexpr int CPB = NT / NL;           // channels per CTA
    static constexpr int K = VEC / NL;            // own steps per lane and sub-chunk
    static constexpr int ROW = 8 * N;             // table bytes per step
    static constexpr int TABLE = TC * ROW;        // one table buffer
    static constexpr int SEGS = 2 * N * (TC / 8) / NT;  // 8-step row pieces per thread
    static_assert(N % 16 == 0 && NL <= VEC, "16 states per lane, at least one own step");
    static_assert(SEGS >= 1 && 2 * N * (TC / 8) % NT == 0, "chunk pieces per thread");
};

// u, delta and z of the CTA's channels for one chunk: [tensor][channel][TC]
// elements, rows padded by 16 bytes so that the 8 channels a warp reads at
// once start on different banks.
template <typename T, int N>
struct ActCfg {
    static constexpr int ES = (int)sizeof(T);
    static constexpr int RB = TC * ES + 16;                 // row bytes
    static constexpr int TENSOR = Cfg<N>::CPB * RB;
    static constexpr int BYTES = 3 * TENSOR;                // one buffer
    static constexpr int PIECES_PER_ROW = TC * ES / 16;
    static constexpr int PIECES = 3 * Cfg<N>::CPB * PIECES_PER_ROW;
    static constexpr int PER_THREAD = (PIECES + Cfg<N>::NT - 1) / Cfg<N>::NT;
    static constexpr int SMEM = 2 * Cfg<N>::TABLE + 2 * BYTES;
};

// The chunk's u, delta, z rows of the CTA's channels, 16 bytes per piece,
// held in registers from the load to the store into the other buffer.
template <typename T, int N>
struct ActLoader {
    using AC = ActCfg<T, N>;
    uint4 w[AC::PER_THREAD];
    __device__ __forceinline__ void load(const T* r0, const T* r1, const T* r2, int64_t s0,
                                         int64_t s1, int64_t s2, int d0, int D, int t0, int L,
                                         int tid) {
#pragma unroll
        for (int q = 0; q < AC::PER_THREAD; ++q) {
            const int pc = tid + q * Cfg<N>::NT;
            w[q] = make_uint4(0u, 0u, 0u, 0u);
            if (pc >= AC::PIECES) continue;
            const int tensor = pc / (Cfg<N>::CPB * AC::PIECES_PER_ROW);
            const int rem = pc % (Cfg<N>::CPB * AC::PIECES_PER_ROW);
            const int ch = rem / AC::PIECES_PER_ROW, piece = rem % AC::PIECES_PER_ROW;
            const T* base = tensor == 0 ? r0 : (tensor == 1 ? r1 : r2);
            const int64_t sdt = tensor == 0 ? s0 : (tensor == 1 ? s1 : s2);
            if (!base || d0 + ch >= D) continue;
            constexpr int PE = 16 / (int)sizeof(T);  // elements per piece
            const int tp = t0 + piece * PE;
            const T* src = base + (int64_t)(d0 + ch) * sdt + tp;
            if (tp + PE <= L) {
                w[q] = __ldg(reinterpret_cast<const uint4*>(src));
            } else {
                T tmp[PE];
#pragma unroll
                for (int e = 0; e < PE; ++e) tmp[e] = tp + e < L ? src[e] : Elem<T>::from_f(0.f);
                uint32_t ww[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if constexpr (sizeof(T) == 2) {
                        ww[i] = (uint32_t)__bfloat16_as_ushort(tmp[2 * i]) |
                                ((uint32_t)__bfloat16_as_ushort(tmp[2 * i + 1]) << 16);
                    } else {
                        ww[i] = __float_as_uint(Elem<T>::to_f(tmp[i]));
                    }
                }
                w[q] = make_uint4(ww[0], ww[1], ww[2], ww[3]);
            }
        }
    }
    __device__ __forceinline__ void store(uint32_t act, int tid) const {
#pragma unroll
        for (int q = 0; q < AC::PER_THREAD; ++q) {
            const int pc = tid + q * Cfg<N>::NT;
            if (pc >= AC::PIECES) continue;
            const int tensor = pc / (Cfg<N>::CPB * AC::PIECES_PER_ROW);
            const int rem = pc % (Cfg<N>::CPB * AC::PIECES_PER_ROW);
            const int ch = rem / AC::PIECES_PER_ROW, piece = rem % AC::PIECES_PER_ROW;
            const uint32_t dst = act + tensor * AC::TENSOR + ch * AC::RB + piece * 16;
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(w[q].x),
                         "r"(w[q].y), "r"(w[q].z), "r"(w[q].w) : "memory");
        }
    }
};

// The chunk's B and C as fp32 table rows: piece s of a thread covers 8 steps
// of one row (tensor s / (4 N), state n = s % N, steps 8 * ((s / N) % 4) ..);
// the loads of the next chunk are held in registers while the current one is
// scanned.
template <typename T, int N>
struct ChunkLoader {
    using C = Cfg<N>;
    static constexpr int W = (int)sizeof(T) / 2;  // 16-byte words per 8-element piece
    uint4 raw[C::SEGS * W];                       // kept packed until the store
    __device__ __forceinline__ void load(const T* Bp, const T* Cp, int64_t sB_n, int64_t sC_n,
                                         int t0, int L, int tid) {
#pragma unroll
        for (int q = 0; q < C::SEGS; ++q) {
            const int s = tid + q * Cfg<N>::NT;
            const int tensor = s / (4 * N), n = s % N, seg = (s / N) % 4;
            const T* src = (tensor ? Cp + n * sC_n : Bp + n * sB_n) + t0 + seg * 8;
            const int left = L - (t0 + seg * 8);
            if (left >= 8) {
#pragma unroll
                for (int w = 0; w < W; ++w) raw[q * W + w] = __ldg(reinterpret_cast<const uint4*>(src) + w);
            } else {
                uint32_t ww[4 * W];
#pragma unroll
                for (int i = 0; i < 4 * W; ++i) {
                    if constexpr (sizeof(T) == 2) {
                        const uint32_t lo = 2 * i < left ? __bfloat16_as_ushort(src[2 * i]) : 0u;
                        const uint32_t hi = 2 * i + 1 < left ? __bfloat16_as_ushort(src[2 * i + 1]) : 0u;
                        ww[i] = lo | (hi << 16);
                    } else {
                        ww[i] = i < left ? __float_as_uint(Elem<T>::to_f(src[i])) : 0u;
                    }
                }
#pragma unroll
                for (int w = 0; w < W; ++w)
                    raw[q * W + w] = make_uint4(ww[4 * w], ww[4 * w + 1], ww[4 * w + 2], ww[4 * w + 3]);
            }
        }
    }
    __device__ __forceinline__ void store(uint32_t table, int tid) const {
#pragma unroll
        for (int q = 0; q < C::SEGS; ++q) {
            const int s = tid + q * Cfg<N>::NT;
            const int tensor = s / (4 * N), n = s % N, seg = (s / N) % 4;
            float v[8];
            if constexpr (sizeof(T) == 2) {
                const uint32_t w[4] = {raw[q].x, raw[q].y, raw[q].z, raw[q].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    v[2 * i] = __uint_as_float(w[i] << 16);
                    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
                }
            } else {
#pragma unroll
                for (int w = 0; w < W; ++w) {
                    v[4 * w] = __uint_as_float(raw[q * W + w].x);
                    v[4 * w + 1] = __uint_as_float(raw[q * W + w].y);
                    v[4 * w + 2] = __uint_as_float(raw[q * W + w].z);
                    v[4 * w + 3] = __uint_as_float(raw[q * W + w].w);
                }
            }
            // word of (n, tensor) in a table row: pair n / 2 holds B, B, C, C, at
            // position pair ^ (pair / 8) so that the channel's lanes, which read
            // pairs 8 part + j at the same time, hit different banks
            const int pr = n >> 1;
            const uint32_t col = ((pr ^ ((pr >> 3) & 7)) * 4 + tensor * 2 + (n & 1)) * 4;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                asm volatile("st.shared.b32 [%0], %1;"
                             ::"r"(table + (seg * 8 + e) * C::ROW + col), "r"(__float_as_uint(v[e]))
                             : "memory");
        }
    }
};

template <typename T, int N, bool HAS_Z>
__global__ void __launch_bounds__(Cfg<N>::NT, ctas_per_sm_for(N)) scan_wide(ScanArgs a) {
    using C = Cfg<N>;
    using AC = ActCfg<T, N>;
    constexpr int NL = C::NL, K = C::K, ES = (int)sizeof(T);
    extern __shared__ __align__(16) uint8_t smem[];
    const uint32_t tab0 = smem_u32(smem);
    const uint32_t act0 = tab0 + 2 * C::TABLE;

    const int tid = threadIdx.x, lane = tid & 31;
    const int ch = tid / NL, part = tid % NL;
    const int gbase = lane - part;
    const int dtiles = (a.D + C::CPB - 1) / C::CPB;
    const int b = blockIdx.x / dtiles;
    const int d = (blockIdx.x % dtiles) * C::CPB + ch;
    const bool valid = d < a.D;
    const int dd_ = valid ? d : 0;

    float2 A2[8], h2[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int n = part * 16 + 2 * j;
        A2[j] = make_float2(a.A[dd_ * a.sA_d + n * a.sA_n] * kLog2e,
                            a.A[dd_ * a.sA_d + (n + 1) * a.sA_n] * kLog2e);
        h2[j] = (valid && a.h0) ? make_float2(a.h0[b * a.sh_b + dd_ * a.sh_d + n * a.sh_n],
                                              a.h0[b * a.sh_b + dd_ * a.sh_d + (n + 1) * a.sh_n])
                                : make_float2(0.f, 0.f);
    }
    const float Dd = a.Dv ? a.Dv[dd_ * a.sD] : 0.f;
    const float biasd = a.bias ? a.bias[dd_ * a.sbias] : 0.f;
    const bool sp = a.softplus != 0;
    T* y = static_cast<T*>(a.y) + b * a.sy_b + dd_ * a.sy_d;
    const int d0 = (blockIdx.x % dtiles) * C::CPB;
    // batch row b of u, delta, z; rows unit-stride in t
    const T* ru = static_cast<const T*>(a.u) + b * a.su_b;
    const T* rd = static_cast<const T*>(a.dl) + b * a.sdl_b;
    const T* rz = HAS_Z ? static_cast<const T*>(a.z) + b * a.sz_b : nullptr;
    // this lane's channel rows in the activation buffer
    auto act_row = [&](int buf, int tensor) {
        return act0 + buf * AC::BYTES + tensor * AC::TENSOR + ch * AC::RB;
    };
    auto lds_elem = [&](uint32_t addr) {
        return ES == 2 ? __uint_as_float(lds16(addr) << 16) : __uint_as_float(lds32(addr));
    };
    const T* Bp = static_cast<const T*>(a.Bm) + b * a.sB_b;
    const T* Cp = static_cast<const T*>(a.Cm) + b * a.sC_b;
    const int L = a.L;
    const int nchunk = (L + TC - 1) / TC;

    ChunkLoader<T, N> ld;
    ActLoader<T, N> la;
    ld.load(Bp, Cp, a.sB_n, a.sC_n, 0, L, tid);
    la.load(ru, rd, rz, a.su_d, a.sdl_d, a.sz_d, d0, a.D, 0, L, tid);
    ld.store(tab0, tid);
    la.store(act0, tid);
    __syncthreads();

    for (int c = 0; c < nchunk; ++c) {
        const int t0 = c * TC;
        const int buf = c & 1;
        const uint32_t tab = tab0 + buf * C::TABLE;
        if (c + 1 < nchunk) {
            ld.load(Bp, Cp, a.sB_n, a.sC_n, t0 + TC, L, tid);
            la.load(ru, rd, rz, a.su_d, a.sdl_d, a.sz_d, d0, a.D, t0 + TC, L, tid);
        }
        const uint32_t ur = act_row(buf, 0), dr = act_row(buf, 1), zr = act_row(buf, 2);
#pragma unroll 1
        for (int sc = 0; sc < TC / VEC; ++sc) {
            const int ts = t0 + sc * VEC;  // first step of the sub-chunk
            if (ts >= L) break;
            // delta of the own steps, shared across the channel's lanes
            const int jo = sc * VEC + part * K;  // first own step in the chunk
            float own[K];
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int t = ts + part * K + k;
                float x = lds_elem(dr + (jo + k) * ES) + biasd;
                x = softplus_if(x, sp);
                own[k] = t < L ? x : 0.f;  // past the end: no update
            }
            float dd[VEC], uf[VEC];
            if constexpr (ES == 2) {
                lds_elems<T, VEC>(ur + sc * VEC * ES, uf);
            } else {  // 32 bytes: two vector loads
                lds_elems<T, 4>(ur + sc * VEC * ES, uf);
                lds_elems<T, 4>(ur + sc * VEC * ES + 16, uf + 4);
            }
#pragma unroll
            for (int j = 0; j < VEC; ++j) dd[j] = __shfl_sync(0xffffffffu, own[j % K], gbase + j / K);
            float yv[VEC];
            const uint32_t rowp = tab + (sc * VEC) * C::ROW + part * 8 * 16;
#pragma unroll
            for (int i = 0; i < VEC; ++i) {
                const float2 d2 = make_float2(dd[i], dd[i]);
                const float du = dd[i] * uf[i];
                const float2 du2 = make_float2(du, du);
                float2 acc = make_float2(0.f, 0.f);
                // the step's loads and exponentials first, then the state updates
                // and the readout, so no result is needed right after it is asked for
                float4 bc[8];
                float2 ab[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    bc[j] = lds128f(rowp + i * C::ROW + ((j ^ part) & 7) * 16);  // B, C pair
                    const float2 ar = __fmul2_rn(d2, A2[j]);
                    ab[j] = make_float2(ex2_approx(ar.x), ex2_approx(ar.y));
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    h2[j] = __ffma2_rn(ab[j], h2[j], __fmul2_rn(du2, make_float2(bc[j].x, bc[j].y)));
                    acc = __ffma2_rn(make_float2(bc[j].z, bc[j].w), h2[j], acc);
                }
                yv[i] = acc.x + acc.y;
            }
            // readouts summed over the channel's lanes; lane `part` keeps its K steps
            float yo[K];
            if constexpr (NL == 2) {
                reduce_half<VEC>(yv, yo, part & 1, 1);
            } else if constexpr (NL == 4) {
                float w4[VEC / 2];
                reduce_half<VEC>(yv, w4, (part >> 1) & 1, 2);
                reduce_half<VEC / 2>(w4, yo, part & 1, 1);
            } else {
                float w4[VEC / 2], w2[VEC / 4];
                reduce_half<VEC>(yv, w4, (part >> 2) & 1, 4);
                reduce_half<VEC / 2>(w4, w2, (part >> 1) & 1, 2);
                reduce_half<VEC / 4>(w2, yo, part & 1, 1);
            }
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int t = ts + part * K + k;
                if (valid && t < L) {
                    float o = fmaf(Dd, lds_elem(ur + (jo + k) * ES), yo[k]);
                    if constexpr (HAS_Z) {
                        const float zz = lds_elem(zr + (jo + k) * ES);
                        o *= zz * sigmoid_accurate(zz);
                    }
                    y[t * a.sy_t] = Elem<T>::from_f(o);
                }
            }
        }
        if (c + 1 < nchunk) {
            ld.store(tab0 + ((c + 1) & 1) * C::TABLE, tid);
            la.store(act0 + ((c + 1) & 1) * AC::BYTES, tid);
        }
        __syncthreads();
    }
    if (valid && a.last) {
        float* ls = a.last + b * a.sl_b + d * a.sl_d;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int n = part * 16 + 2 * j;
            ls[n * a.sl_n] = h2[j].x;
            ls[(n + 1) * a.sl_n] = h2[j].y;
        }
    }
}

template <typename T, int N>
static int run(const ScanArgs& a, cudaStream_t st) {
    using C = Cfg<N>;
    constexpr int SMEM = ActCfg<T, N>::SMEM;
    auto kern = a.z ? scan_wide<T, N, true> : scan_wide<T, N, false>;
    static bool attr_set[2][64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    const int zi = a.z ? 1 : 0;
    if (dev < 0 || dev >= 64 || !attr_set[zi][dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM) !=
            cudaSuccess)
            return SS_ERR_LAUNCH;
        if (dev >= 0 && dev < 64) attr_set[zi][dev] = true;
    }
    const int64_t ctas = (int64_t)a.Bsz * ((a.D + C::CPB - 1) / C::CPB);
    kern<<<(unsigned)ctas, C::NT, SMEM, st>>>(a);
    count_launch(1);
    return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_LAUNCH;
}

}  // namespace wide

// B, C shared per batch row, N in {32, 64, 128} (fp32: 64, 128), unit
// t-stride and 16-byte aligned rows of B, C, u, delta, z (the chunk loads are
// 16 bytes wide).
int launch_selective_wide(const ScanArgs& a, cudaStream_t st, bool* taken) {
    *taken = false;
    if (a.G > 1 || a.cw || a.L < 1) return SS_OK;
    if (a.N != 32 && a.N != 64 && a.N != 128) return SS_OK;
    const int es = a.dtype == SS_BF16 ? 2 : 4;
    auto rows_ok = [&](const void* p, int64_t sb, int64_t sn, int64_t stt) {
        return stt == 1 && reinterpret_cast<uintptr_t>(p) % 16 == 0 && (sb * es) % 16 == 0 &&
               (sn * es) % 16 == 0;
    };
    if (!rows_ok(a.Bm, a.sB_b, a.sB_n, a.sB_t) || !rows_ok(a.Cm, a.sC_b, a.sC_n, a.sC_t) ||
        !rows_ok(a.u, a.su_b, a.su_d, a.su_t) || !rows_ok(a.dl, a.sdl_b, a.sdl_d, a.sdl_t) ||
        (a.z && !rows_ok(a.z, a.sz_b, a.sz_d, a.sz_t)))
        return SS_OK;
    if (a.dtype != SS_BF16 && a.N == 32) return SS_OK;  // fp32 rows of 128 channels: too much shared memory
    *taken = true;
    const bool bf = a.dtype == SS_BF16;
    if (a.N == 32) return wide::run<__nv_bfloat16, 32>(a, st);  // bf16 only (checked above)
    if (a.N == 64) return bf ? wide::run<__nv_bfloat16, 64>(a, st) : wide::run<float, 64>(a, st);
    return bf ? wide::run<__nv_bfloat16, 128>(a, st) : wide::run<float, 128>(a, st);
}

}  // namespace ss
