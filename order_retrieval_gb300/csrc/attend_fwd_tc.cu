// attend_fwd_tc.cu -- launcher of the tensor-core forward (attend_fwd_tc.cuh) on
// the window indices made by the select step.
#include "attend_fwd_tc.cuh"

namespace zeta {

bool attend_fwd_tc_supported(const Prob &p) {
    return p.vdt == ZETA_BF16 && p.dV == DV && p.dK <= 4;
}

cudaError_t launch_attend_fwd_tc(const Prob &p, const float *q, const float *k, const void *v,
                                 const float *gamma, const int32_t *idx, void *out,
                                 float *rowsum, int32_t *status, cudaStream_t st) {
    const int tpc = (p.C + TQ - 1) / TQ;
    const dim3 grid((unsigned)(p.n * tpc), (unsigned)p.S);
    const __nv_bfloat16 *vb = static_cast<const __nv_bfloat16 *>(v);
    __nv_bfloat16 *ob = static_cast<__nv_bfloat16 *>(out);
#define ZETA_FWD_TC(D, WK)                                                                    \
    attend_fwd_tc<D, WK, NoSel><<<grid, THREADS, 0, st>>>(q, k, vb, gamma, idx, ob, rowsum,       \
                                                          status, p.N, p.H, p.k, p.C, tpc,     \
                                                          NoSel{})
#define ZETA_FWD_TC_D(WK)                        \
    switch (p.dK) {                              \
        case 1: ZETA_FWD_TC(1, WK); break;       \
        case 2: ZETA_FWD_TC(2, WK); break;       \
        case 3: ZETA_FWD_TC(3, WK); break;       \
        default: ZETA_FWD_TC(4, WK); break;      \
    }
    if (p.wk == kWSoftmax) {
        ZETA_FWD_TC_D(kWSoftmax);
    } else if (p.wk == kWInvEuclid) {
        ZETA_FWD_TC_D(kWInvEuclid);
    } else {
        ZETA_FWD_TC_D(kWCauchy);
    }
#undef ZETA_FWD_TC_D
#undef ZETA_FWD_TC
    return cudaGetLastError();
}

}  // namespace zeta
