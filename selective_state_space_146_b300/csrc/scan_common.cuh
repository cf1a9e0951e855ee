// scan_common.cuh -- device helpers shared by the selective-scan kernels
// (shared-memory element loads, branch-free selects, the lane reduce-scatter)
// and the signature of cuTensorMapEncodeTiled.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"

namespace ss {

// K consecutive elements of T (K * sizeof(T) in {2, 4, 8, 16} bytes) from
// shared memory, widened to float.
template <typename T, int K>
__device__ __forceinline__ void lds_elems(uint32_t a, float* out) {
    constexpr int BYTES = K * (int)sizeof(T);
    static_assert(BYTES == 2 || BYTES == 4 || BYTES == 8 || BYTES == 16, "one load of 2..16 bytes");
    uint32_t w[4];
    if constexpr (BYTES == 16) {
        const uint4 v = lds128(a);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if constexpr (BYTES == 8) {
        const uint2 v = lds64(a);
        w[0] = v.x; w[1] = v.y;
    } else if constexpr (BYTES == 4) {
        w[0] = lds32(a);
    } else {
        out[0] = __uint_as_float(lds16(a) << 16);  // one bf16
        return;
    }
    if constexpr (sizeof(T) == 2) {
#pragma unroll
        for (int i = 0; i < K / 2; ++i) {
            out[2 * i] = __uint_as_float(w[i] << 16);
            out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    } else {
#pragma unroll
        for (int i = 0; i < K; ++i) out[i] = __uint_as_float(w[i]);
    }
}

// on ? a : b as a select instruction, so that a flag fixed for the whole
// launch puts no branch into the caller's loop.
__device__ __forceinline__ float sel_f(bool on, float a, float b) {
    asm("{ .reg .pred q; setp.ne.s32 q, %2, 0; selp.f32 %0, %1, %0, q; }"
        : "+f"(b) : "f"(a), "r"((int)on));
    return b;
}

// softplus(x) when `on`, else x (both evaluated, then selected).
__device__ __forceinline__ float softplus_if(float x, bool on) {
    return sel_f(on, softplus_f(x), x);
}

// One round of the readout reduce-scatter across the lanes of a channel:
// keep one half of v (the upper half if `upper`), send the other half to the
// partner lane (lane ^ m) and add what the partner sends back.
template <int LEN>
__device__ __forceinline__ void reduce_half(const float* v, float* out, bool upper, int m) {
#pragma unroll
    for (int e = 0; e < LEN / 2; ++e) {
        const float lo = v[e], hi = v[LEN / 2 + e];
        const float send = upper ? lo : hi;
        const float keep = upper ? hi : lo;
        out[e] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
}

// Byte offset of 16-byte chunk c of row r in a 128-byte-swizzled tile.
__device__ __forceinline__ int swz(int r, int c) { return (r << 7) + ((c ^ (r & 7)) << 4); }

// Conversion of one tile's raw B / C ([n][t] as loaded by TMA) into the fp32
// table bc[t][32]: 16-byte chunk j holds (B[2j], B[2j+1], C[2j], C[2j+1]), so
// a lane keeping the state pairs [j0, j0 + m) reads m consecutive chunks, one
// ld.shared.v4 per pair, at offsets known at compile time.  Lane l writes rows
// 2l, 2l+1 (bf16) or row l (fp32); the chunk order is rotated by lane so the
// lanes of one store hit distinct banks.  Without C (summary pass) the C slots
// hold zeros.
// convert_bc_part does pass `it` of 8 (one chunk column per lane), so that
// the passes can be split over several warps.
template <typename T, bool WITH_C>
__device__ __forceinline__ void convert_bc_part(uint32_t rawB, uint32_t rawC, uint32_t bc, int lane, int it) {
    {
        const int j = (it + lane) & 7;
        const uint32_t rb = rawB + (2 * j) * 128, rc = rawC + (2 * j) * 128;
        if constexpr (sizeof(T) == 2) {
            // word `lane` of a 128-byte row holds the bf16 pair (t = 2 lane, 2 lane + 1)
            const uint32_t b0 = lds32(rb + lane * 4), b1 = lds32(rb + 128 + lane * 4);
            const uint32_t c0 = WITH_C ? lds32(rc + lane * 4) : 0u;
            const uint32_t c1 = WITH_C ? lds32(rc + 128 + lane * 4) : 0u;
            const float4 lo = make_float4(__uint_as_float(b0 << 16), __uint_as_float(b1 << 16),
                                          __uint_as_float(c0 << 16), __uint_as_float(c1 << 16));
            const float4 hi = make_float4(__uint_as_float(b0 & 0xffff0000u),
                                          __uint_as_float(b1 & 0xffff0000u),
                                          __uint_as_float(c0 & 0xffff0000u),
                                          __uint_as_float(c1 & 0xffff0000u));
            sts128f(bc + (2 * lane) * 128 + j * 16, lo);
            sts128f(bc + (2 * lane + 1) * 128 + j * 16, hi);
        } else {
            float4 v;
            v.x = __uint_as_float(lds32(rb + lane * 4));
            v.y = __uint_as_float(lds32(rb + 128 + lane * 4));
            v.z = WITH_C ? __uint_as_float(lds32(rc + lane * 4)) : 0.f;
            v.w = WITH_C ? __uint_as_float(lds32(rc + 128 + lane * 4)) : 0.f;
            sts128f(bc + lane * 128 + j * 16, v);
        }
    }
}

template <typename T, bool WITH_C>
__device__ __forceinline__ void convert_bc(uint32_t rawB, uint32_t rawC, uint32_t bc, int lane) {
#pragma unroll
    for (int it = 0; it < 8; ++it) convert_bc_part<T, WITH_C>(rawB, rawC, bc, lane, it);
}

// Byte offset of 16-byte chunk c of row r in a tile of ROWB-byte rows with
// the ROWB-byte TMA swizzle: within each 1024-byte (128-byte rows) or
// 512-byte (64-byte rows) atom, the chunk index is XORed with the row index
// (128) or with half the row index (64), so the rows a quarter-warp reads
// land on distinct banks.
template <int ROWB>
__device__ __forceinline__ int swz_rows(int r, int c) {
    static_assert(ROWB == 128 || ROWB == 64, "row of 64 or 128 bytes");
    if constexpr (ROWB == 128) return (r << 7) + ((c ^ (r & 7)) << 4);
    return (r << 6) + ((c ^ ((r >> 1) & 3)) << 4);
}

// convert_bc for raw tiles of 64-byte rows (32 bf16 or 16 fp32 steps): lanes
// 0..15 write the state pairs 0..3 of their step pair (bf16) or step (fp32),
// lanes 16..31 the pairs 4..7, chunk order rotated by lane; pass `it` of 4.
template <typename T, bool WITH_C>
__device__ __forceinline__ void convert_bc64_part(uint32_t rawB, uint32_t rawC, uint32_t bc, int lane, int it) {
    const int w = lane & 15, half = lane >> 4;
    {
        const int j = 4 * half + ((it + w) & 3);
        const uint32_t rb = rawB + (2 * j) * 64, rc = rawC + (2 * j) * 64;
        if constexpr (sizeof(T) == 2) {
            // word w of a 64-byte row holds the bf16 pair (t = 2 w, 2 w + 1)
            const uint32_t b0 = lds32(rb + w * 4), b1 = lds32(rb + 64 + w * 4);
            const uint32_t c0 = WITH_C ? lds32(rc + w * 4) : 0u;
            const uint32_t c1 = WITH_C ? lds32(rc + 64 + w * 4) : 0u;
            const float4 lo = make_float4(__uint_as_float(b0 << 16), __uint_as_float(b1 << 16),
                                          __uint_as_float(c0 << 16), __uint_as_float(c1 << 16));
            const float4 hi = make_float4(__uint_as_float(b0 & 0xffff0000u),
                                          __uint_as_float(b1 & 0xffff0000u),
                                          __uint_as_float(c0 & 0xffff0000u),
                                          __uint_as_float(c1 & 0xffff0000u));
            sts128f(bc + (2 * w) * 128 + j * 16, lo);
            sts128f(bc + (2 * w + 1) * 128 + j * 16, hi);
        } else {
            // word w of a 64-byte row holds step w
            float4 v;
            v.x = __uint_as_float(lds32(rb + w * 4));
            v.y = __uint_as_float(lds32(rb + 64 + w * 4));
            v.z = WITH_C ? __uint_as_float(lds32(rc + w * 4)) : 0.f;
            v.w = WITH_C ? __uint_as_float(lds32(rc + 64 + w * 4)) : 0.f;
            sts128f(bc + w * 128 + j * 16, v);
        }
    }
}

template <typename T, bool WITH_C>
__device__ __forceinline__ void convert_bc64(uint32_t rawB, uint32_t rawC, uint32_t bc, int lane) {
#pragma unroll
    for (int it = 0; it < 4; ++it) convert_bc64_part<T, WITH_C>(rawB, rawC, bc, lane, it);
}

// Store K floats as T to global memory: one aligned vector store, or (in the
// last chunk of the sequence) element by element up to `limit` elements.
template <typename T, int K>
__device__ __forceinline__ void stg_elems(T* p, const float* v, int limit) {
    constexpr int BYTES = K * (int)sizeof(T);
    if constexpr (BYTES == 2) {
        if (limit >= 1) p[0] = Elem<T>::from_f(v[0]);
        return;
    }
    if (limit >= K) {
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
        if constexpr (BYTES == 16) *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
        else if constexpr (BYTES == 8) *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
        else *reinterpret_cast<uint32_t*>(p) = w[0];
    } else {
#pragma unroll
        for (int i = 0; i < K; ++i)
            if (i < limit) p[i] = Elem<T>::from_f(v[i]);
    }
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                              CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                              CUtensorMapFloatOOBfill);

}  // namespace ss
