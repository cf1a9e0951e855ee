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

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                              CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                              CUtensorMapFloatOOBfill);

}  // namespace ss
