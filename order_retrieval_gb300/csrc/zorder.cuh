// zorder.cuh -- the grid cell of a coordinate and bit dilation for Morton codes,
// shared by the encode kernels and the fused projection + encode kernel.
//
// Passage: OpenReview discussion of "ZETA: Leveraging Z-order Curves for
// Efficient Top-k Attention", reply A2 "Clarification of Binary Expansion and
// Precision" (normalise to [0, 1], a grid of 2^bits cells, interleave the bits).
#pragma once

#include "common.cuh"

namespace zeta {

// Grid cell of one coordinate.  Float32, no contraction: (x + 1) rounded once,
// then an exact power-of-two scale.
__device__ __forceinline__ uint32_t quantise(float x, float scale, float umax) {
    float t = __fmul_rn(__fadd_rn(x, 1.0f), scale);
    float f = floorf(t);
    f = fmaxf(f, 0.0f);      // also maps NaN to 0
    f = fminf(f, umax);
    return static_cast<uint32_t>(f);
}

// Spread the low 21 bits of x so that bit j moves to bit 3j.
__device__ __forceinline__ uint64_t dilate3(uint64_t x) {
    x &= 0x1fffffull;
    x = (x | (x << 32)) & 0x001f00000000ffffull;
    x = (x | (x << 16)) & 0x001f0000ff0000ffull;
    x = (x | (x << 8)) & 0x100f00f00f00f00full;
    x = (x | (x << 4)) & 0x10c30c30c30c30c3ull;
    x = (x | (x << 2)) & 0x1249249249249249ull;
    return x;
}

// Spread the low 32 bits of x so that bit j moves to bit 2j.
__device__ __forceinline__ uint64_t dilate2(uint64_t x) {
    x &= 0xffffffffull;
    x = (x | (x << 16)) & 0x0000ffff0000ffffull;
    x = (x | (x << 8)) & 0x00ff00ff00ff00ffull;
    x = (x | (x << 4)) & 0x0f0f0f0f0f0f0f0full;
    x = (x | (x << 2)) & 0x3333333333333333ull;
    x = (x | (x << 1)) & 0x5555555555555555ull;
    return x;
}

// Morton code of three cells (coordinate 0 the most significant bit of each level).
__device__ __forceinline__ uint64_t morton3(uint32_t u0, uint32_t u1, uint32_t u2) {
    return (dilate3(u0) << 2) | (dilate3(u1) << 1) | dilate3(u2);
}

}  // namespace zeta
