// bwd_rec.cuh -- the per-query record the backward's query side hands to its
// key side.
#pragma once

#include "common.cuh"

namespace zeta {

// q (padded to 4), then {1/s, -gbar/s, m, gbar} (m: the softmax shift; 0 for
// the other weight kernels), so that dL/dw_ij = g_ij / s - gbar / s is one fma
// and the two scalars it needs are adjacent (one 8-byte load).
struct __align__(16) QRec {
    float4 q;
    float4 sg;
};

}  // namespace zeta
