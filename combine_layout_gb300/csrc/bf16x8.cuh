// Eight bf16 values in one 16-byte vector: fp32 multiply-accumulate and the
// round-to-nearest-even packing back to bf16 (shared by the reductions).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace moeep {

// a[i] = fma(w, bf16 element i of v, a[i]), elements in memory order.
__device__ __forceinline__ void acc8(float (&a)[8], float w, const uint4& v)
{
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        a[2 * i] = fmaf(w, __uint_as_float(u[i] << 16), a[2 * i]);
        a[2 * i + 1] = fmaf(w, __uint_as_float(u[i] & 0xffff0000u), a[2 * i + 1]);
    }
}

// Eight fp32 values rounded to bf16 (nearest even), in memory order.
__device__ __forceinline__ uint4 pack8(const float (&a)[8])
{
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(a[2 * i], a[2 * i + 1]);
        o[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace moeep
