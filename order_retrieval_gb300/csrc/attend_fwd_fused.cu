// attend_fwd_fused.cu -- select + attend in one launch: the tensor-core forward
// (attend_fwd_tc.cuh) with each query's window found inside the kernel (binary
// search of its code in its sorted prefix, OpenReview discussion of "ZETA:
// Leveraging Z-order Curves for Efficient Top-k Attention", reply A3
// "Chunking ... & Where efficiency is coming from"); the window rows are also
// written out for the backward.  Shapes the tensor-core kernel does not take
// run the select and the generic forward as two launches.
#include "attend_fwd_tc.cuh"

namespace zeta {
namespace {

template <typename K>
cudaError_t launch_fused(const Prob &p, const float *q, const float *k, const void *v,
                         const float *gamma, const void *q_codes, const void *prefix_codes,
                         const int32_t *prefix_idx, int32_t *idx, void *out, float *rowsum,
                         int32_t *status, cudaStream_t st) {
    const int tpc = (p.C + TQ - 1) / TQ;
    const dim3 grid((unsigned)(p.n * tpc), (unsigned)p.S);
    const __nv_bfloat16 *vb = static_cast<const __nv_bfloat16 *>(v);
    __nv_bfloat16 *ob = static_cast<__nv_bfloat16 *>(out);
    const FusedSel<K> sel{static_cast<const K *>(q_codes), static_cast<const K *>(prefix_codes),
                          prefix_idx, idx, p.T};
#define ZETA_FUSED(D, WK)                                                                     \
    attend_fwd_tc<D, WK, FusedSel<K>><<<grid, THREADS, 0, st>>>(                              \
        q, k, vb, gamma, nullptr, ob, rowsum, status, p.N, p.H, p.k, p.C, tpc, sel)
#define ZETA_FUSED_D(WK)                         \
    switch (p.dK) {                              \
        case 1: ZETA_FUSED(1, WK); break;        \
        case 2: ZETA_FUSED(2, WK); break;        \
        case 3: ZETA_FUSED(3, WK); break;        \
        default: ZETA_FUSED(4, WK); break;       \
    }
    if (p.wk == kWSoftmax) {
        ZETA_FUSED_D(kWSoftmax);
    } else if (p.wk == kWInvEuclid) {
        ZETA_FUSED_D(kWInvEuclid);
    } else {
        ZETA_FUSED_D(kWCauchy);
    }
#undef ZETA_FUSED_D
#undef ZETA_FUSED
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_select_attend_fwd(const Prob &p, const float *q, const float *k,
                                     const void *v, const float *gamma, const void *q_codes,
                                     const void *prefix_codes, const int32_t *prefix_idx,
                                     int32_t *idx, void *out, float *rowsum, int32_t *status,
                                     cudaStream_t st) {
    // the fused kernel is the tensor-core forward: value rows read 32 bytes at a time
    if (!attend_fwd_tc_supported(p) || (reinterpret_cast<uintptr_t>(v) & 31u) != 0) {
        cudaError_t e = launch_select(p, q_codes, prefix_codes, prefix_idx, idx, st);
        if (e != cudaSuccess) return e;
        return launch_attend_fwd(p, q, k, v, gamma, idx, out, rowsum, status, st);
    }
    if (p.code64)
        return launch_fused<uint64_t>(p, q, k, v, gamma, q_codes, prefix_codes, prefix_idx, idx,
                                      out, rowsum, status, st);
    return launch_fused<uint32_t>(p, q, k, v, gamma, q_codes, prefix_codes, prefix_idx, idx, out,
                                  rowsum, status, st);
}

}  // namespace zeta
