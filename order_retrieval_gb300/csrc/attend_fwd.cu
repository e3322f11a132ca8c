// attend_fwd.cu -- Adaptive Cauchy-softmax over each query's attended set.
//
// Passages (OpenReview discussion of "ZETA: Leveraging Z-order Curves for
// Efficient Top-k Attention"): reply A2 "Discussion on its robustness" (the
// Cauchy softmax with a trainable gamma acting as a temperature), reply A3
// "Justification for Euclidean Distance Claim" (Euclidean distance between
// query and key); atlas.scime.ai summary, "Approach".
//
// Attended set of query i in chunk c: the k window keys (idx row i, -1 = none)
// plus every own-chunk key j with cC <= j <= i.
//   w_ij = 1 / (1 + |q_i - k_j|^2 / gamma_h^2),  s_i = sum_j w_ij,
//   out_i = sum_j w_ij v_j / s_i,                rowsum_i = s_i.
// Other weight kernels (flags): softmax of -d2 / gamma^2 and inverse Euclidean
// (reply A3 "Justification for Euclidean Distance Claim"); the softmax takes
// its shift, the smallest d2 of the set, in a first pass over the keys.
//
// Generic path: one warp per query, one key per lane for the weights, then the
// warp walks the 32 keys with lanes spread over the value columns.  Any d_V up
// to 256, float32 or bf16 values.  bf16 values with d_V = 64 and d_K <= 4 take
// the tensor-core kernel in attend_fwd_tc.cu instead.
#include "common.cuh"

namespace zeta {
namespace {

template <typename V, int VPL>
struct FwdAcc {
    float acc[VPL];
    float s;
    __device__ void zero() {
#pragma unroll
        for (int e = 0; e < VPL; ++e) acc[e] = 0.f;
        s = 0.f;
    }
    // Lane holds (w, j) for one key (j < 0: none); the warp adds all 32 rows.
    __device__ void add32(float w, int j, const V *__restrict__ vb, int dV, int lane) {
        s += w;
        for (int u = 0; u < 32; ++u) {
            const float wu = __shfl_sync(kFull, w, u);
            const int ju = __shfl_sync(kFull, j, u);
            if (ju < 0) continue;
            const V *row = vb + (int64_t)ju * dV;
#pragma unroll
            for (int e = 0; e < VPL; ++e) {
                const int col = lane + 32 * e;
                if (col < dV) acc[e] = __fmaf_rn(wu, VT<V>::ld(row + col), acc[e]);
            }
        }
    }
};

__device__ __forceinline__ float dist2(const float *qi, const float *kj, int dK) {
    float d2 = 0.f;
#pragma unroll
    for (int d = 0; d < kMaxDK; ++d) {
        if (d < dK) {
            const float e = qi[d] - kj[d];
            d2 = __fmaf_rn(e, e, d2);
        }
    }
    return d2;
}

template <typename V, int VPL, int WK>
__global__ void __launch_bounds__(256)
attend_fwd_generic(const float *__restrict__ q, const float *__restrict__ kx,
                   const V *__restrict__ v, const float *__restrict__ gamma,
                   const int32_t *__restrict__ idx, V *__restrict__ out,
                   float *__restrict__ rowsum, int32_t *status, int64_t S, int N, int H, int dK,
                   int dV, int k, int C) {
    const int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    if (gw >= S * N) return;
    const int lane = threadIdx.x & 31;
    const int64_t seg = gw / N;
    const int i = (int)(gw % N);
    const float g = gamma[seg % H];
    const float inv_g2 = __frcp_rn(g * g);
    float qi[kMaxDK];
#pragma unroll
    for (int d = 0; d < kMaxDK; ++d) qi[d] = d < dK ? q[(seg * N + i) * dK + d] : 0.f;
    const float *kb = kx + seg * N * dK;
    const V *vb = v + seg * N * dV;
    const int cC = (i / C) * C;
    FwdAcc<V, VPL> a;
    a.zero();
    const int32_t *irow = idx + (seg * N + i) * (int64_t)k;
    float m = 0.f;                                 // softmax shift: min d2 of the set
    if constexpr (WK == kWSoftmax) {
        float mn = INFINITY;
        for (int t = lane; t < k; t += 32) {
            const int j = irow[t];
            if (j >= 0 && j < cC) mn = fminf(mn, dist2(qi, kb + (int64_t)j * dK, dK));
        }
        for (int j = cC + lane; j <= i; j += 32) mn = fminf(mn, dist2(qi, kb + (int64_t)j * dK, dK));
        for (int o = 16; o > 0; o >>= 1) mn = fminf(mn, __shfl_xor_sync(kFull, mn, o));
        m = mn;
    }
    for (int t0 = 0; t0 < k; t0 += 32) {
        const int t = t0 + lane;
        int j = -1;
        if (t < k) {
            j = irow[t];
            if (j != -1 && (j < 0 || j >= cC)) {
                set_status(status, ZETA_ERR_BOUNDS);
                j = -1;
            }
        }
        const float w = j >= 0 ? weight_of<WK>(dist2(qi, kb + (int64_t)j * dK, dK), m, inv_g2)
                               : 0.f;
        a.add32(w, j, vb, dV, lane);
    }
    for (int j0 = cC; j0 <= i; j0 += 32) {
        const int j = j0 + lane <= i ? j0 + lane : -1;
        const float w = j >= 0 ? weight_of<WK>(dist2(qi, kb + (int64_t)j * dK, dK), m, inv_g2)
                               : 0.f;
        a.add32(w, j, vb, dV, lane);
    }
    float s = a.s;
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
    V *orow = out + (seg * N + i) * dV;
#pragma unroll
    for (int e = 0; e < VPL; ++e) {
        const int col = lane + 32 * e;
        if (col < dV) VT<V>::st(orow + col, __fdiv_rn(a.acc[e], s));
    }
    if (lane == 0) rowsum[seg * N + i] = s;
}

template <typename V, int VPL>
cudaError_t fwd_generic(const Prob &p, const float *q, const float *k, const void *v,
                        const float *gamma, const int32_t *idx, void *out, float *rowsum,
                        int32_t *status, cudaStream_t st) {
    const int64_t warps = p.S * p.N;
    const int64_t blocks = (warps + 7) / 8;
#define ZETA_FWD_G(WK)                                                                        \
    attend_fwd_generic<V, VPL, WK><<<(unsigned)blocks, 256, 0, st>>>(                         \
        q, k, static_cast<const V *>(v), gamma, idx, static_cast<V *>(out), rowsum, status, p.S, \
        p.N, p.H, p.dK, p.dV, p.k, p.C)
    if (p.wk == kWSoftmax) ZETA_FWD_G(kWSoftmax);
    else if (p.wk == kWInvEuclid) ZETA_FWD_G(kWInvEuclid);
    else ZETA_FWD_G(kWCauchy);
#undef ZETA_FWD_G
    return cudaGetLastError();
}

template <typename V>
cudaError_t fwd_generic_dispatch(const Prob &p, const float *q, const float *k, const void *v,
                                 const float *gamma, const int32_t *idx, void *out,
                                 float *rowsum, int32_t *status, cudaStream_t st) {
    if (p.dV <= 32) return fwd_generic<V, 1>(p, q, k, v, gamma, idx, out, rowsum, status, st);
    if (p.dV <= 64) return fwd_generic<V, 2>(p, q, k, v, gamma, idx, out, rowsum, status, st);
    if (p.dV <= 128) return fwd_generic<V, 4>(p, q, k, v, gamma, idx, out, rowsum, status, st);
    return fwd_generic<V, 8>(p, q, k, v, gamma, idx, out, rowsum, status, st);
}

}  // namespace

cudaError_t launch_attend_fwd(const Prob &p, const float *q, const float *k, const void *v,
                              const float *gamma, const int32_t *idx, void *out, float *rowsum,
                              int32_t *status, cudaStream_t st) {
    // the tensor-core kernel reads value rows 32 bytes at a time
    if (attend_fwd_tc_supported(p) && (reinterpret_cast<uintptr_t>(v) & 31u) == 0)
        return launch_attend_fwd_tc(p, q, k, v, gamma, idx, out, rowsum, status, st);
    if (p.vdt == ZETA_BF16)
        return fwd_generic_dispatch<__nv_bfloat16>(p, q, k, v, gamma, idx, out, rowsum, status,
                                                   st);
    return fwd_generic_dispatch<float>(p, q, k, v, gamma, idx, out, rowsum, status, st);
}

}  // namespace zeta
