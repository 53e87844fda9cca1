// E4M3 encoding of 16-element runs, shared by the 8-bit scatter and the 8-bit
// decode with append so that both store the same codes for the same input.
//
// Element x becomes the code nearest to the float32 quotient x / scale (IEEE
// division, __fdiv_rn), rounded to nearest even and saturated to +-448 by the
// hardware conversion cvt.rn.satfinite.e4m3x2.f32.
#pragma once

#include "common.cuh"

namespace pa {
namespace fp8 {

// 16 consecutive source elements (16-byte aligned) as floats.
template <typename TS>
__device__ __forceinline__ void load16(const TS *src, float *f) {
    constexpr int kPer = Vec16<TS>::N;                 // elements per 16-byte vector
#pragma unroll
    for (int u = 0; u < 16 / kPer; ++u) {
        const uint4 w = __ldcs(reinterpret_cast<const uint4 *>(src) + u);
        Vec16<TS>::unpack(w, f + u * kPer);
    }
}

// Codes of x[0..15] / scale, code i in byte i of the result.
__device__ __forceinline__ uint4 encode16(const float *x, float scale) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint16_t lo, hi;
        const float a = __fdiv_rn(x[4 * i], scale), b = __fdiv_rn(x[4 * i + 1], scale);
        const float c = __fdiv_rn(x[4 * i + 2], scale), d = __fdiv_rn(x[4 * i + 3], scale);
        // the first source operand lands in the upper byte
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
        w[i] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace fp8
}  // namespace pa
