// attend_bwd.cu -- gradients of the Cauchy-softmax attention, selection fixed.
//
// The pages time a forward+backward pass (OpenReview discussion of "ZETA:
// Leveraging Z-order Curves for Efficient Top-k Attention", replies A3/A4 on
// time and memory; atlas.scime.ai summary, "Measured effects", whose table
// times a 65,536-token training pass), so the method is trained end to end.
// The window is not differentiated: idx is an input.
//
// With a_ij = w_ij / s_i, g_ij = dO_i . v_j, gbar_i = sum_j a_ij g_ij:
//   dL/dw_ij = (g_ij - gbar_i) / s_i,   dw/d(d^2) = -w^2 / gamma^2,
//   dw/dgamma = 2 w (1 - w) / gamma  (Cauchy; the other weight kernels swap in
//   their own dw/d(d^2) and dw/dgamma, common.cuh, and the softmax first finds
//   its shift, the smallest d^2 of the set, which the key side reads back).
// Query side (one warp per query): s_i, gbar_i, dq_i and the query's share
// of dgamma.  Key side (one warp per key): dv_j and dk_j, reducing over the
// queries that selected j.  Those are found through a transpose of idx built
// by a stable radix sort of (key, query) pairs, so every key reads its
// queries in ascending order and all sums run in a fixed order: the results
// are bit-reproducible, with no floating-point atomics.  dgamma is summed per
// head in double in a fixed order.
#include "common.cuh"

namespace zeta {
namespace {

__device__ __forceinline__ float dist2b(const float *a, const float *b, int dK) {
    float d2 = 0.f;
#pragma unroll
    for (int d = 0; d < kMaxDK; ++d) {
        if (d < dK) {
            const float e = a[d] - b[d];
            d2 = __fmaf_rn(e, e, d2);
        }
    }
    return d2;
}

template <typename V>
__device__ __forceinline__ float dot_row(const float *__restrict__ sm, const V *__restrict__ row,
                                         int dV) {
    float g = 0.f;
    for (int e = 0; e < dV; ++e) g = __fmaf_rn(sm[e], VT<V>::ld(row + e), g);
    return g;
}

__device__ __forceinline__ float warp_sum(float x) {
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
    return x;
}

// ---------------------------------------------------------- query side ---
// One pass over the attended set of query i.  With c_ij = 2 dw/d(d^2) and
// e_ij = dw/dgamma, and dL/dw_ij = (g_ij - gbar_i) / s_i:
//   s      = sum w,          G  = sum w g        -> gbar = G / s
//   A_d    = sum g c (q-k)_d, Bd = sum c (q-k)_d -> dq_d  = (A_d - gbar Bd) / s
//   E1     = sum g e,        E2 = sum e          -> dgamma_i = (E1 - gbar E2) / s
// so gbar is exact (from the values themselves, not the rounded output).

template <typename V, int VPL, int WK>
__global__ void __launch_bounds__(256)
bwd_query_generic(const float *__restrict__ q, const float *__restrict__ kx,
                  const V *__restrict__ v, const float *__restrict__ gamma,
                  const int32_t *__restrict__ idx, const V *__restrict__ dout,
                  float *__restrict__ dq, float *__restrict__ s_out, float *__restrict__ gbar_out,
                  float *__restrict__ m_out, float *__restrict__ dg_part, int32_t *status,
                  int64_t S, int N, int H, int dK, int dV, int k, int C) {
    __shared__ float sdo[8][kMaxDV];
    const int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    if (gw >= S * N) return;
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int64_t seg = gw / N;
    const int i = (int)(gw % N);
    const int64_t row = seg * N + i;
    const float g = gamma[seg % H];
    const float inv_g2 = __frcp_rn(g * g);
    const float inv_g = __frcp_rn(g);
    float qi[kMaxDK];
#pragma unroll
    for (int d = 0; d < kMaxDK; ++d) qi[d] = d < dK ? q[row * dK + d] : 0.f;
    for (int e = lane; e < dV; e += 32) sdo[wib][e] = VT<V>::ld(dout + row * dV + e);
    __syncwarp();
    const float *kb = kx + seg * N * dK;
    const V *vb = v + seg * N * dV;
    const int cC = (i / C) * C;
    float A[kMaxDK], Bd[kMaxDK];
#pragma unroll
    for (int d = 0; d < kMaxDK; ++d) A[d] = Bd[d] = 0.f;
    float sw = 0.f, G = 0.f, E1 = 0.f, E2 = 0.f;
    const int32_t *irow = idx + row * (int64_t)k;
    float m = 0.f;                                 // softmax shift: min d2 of the set
    if constexpr (WK == kWSoftmax) {
        float mn = INFINITY;
        for (int t = lane; t < k; t += 32) {
            const int j = irow[t];
            if (j >= 0 && j < cC) mn = fminf(mn, dist2b(qi, kb + (int64_t)j * dK, dK));
        }
        for (int j = cC + lane; j <= i; j += 32)
            mn = fminf(mn, dist2b(qi, kb + (int64_t)j * dK, dK));
        for (int o = 16; o > 0; o >>= 1) mn = fminf(mn, __shfl_xor_sync(kFull, mn, o));
        m = mn;
    }
    auto visit = [&](int j) {
        const float *kj = kb + (int64_t)j * dK;
        const float d2 = dist2b(qi, kj, dK);
        const float w = weight_of<WK>(d2, m, inv_g2);
        const float gij = dot_row<V>(sdo[wib], vb + (int64_t)j * dV, dV);
        const float c = -2.f * neg_dw_dd2<WK>(w, inv_g2);
        const float e = dw_dgamma<WK>(w, d2, m, inv_g2, inv_g);
        sw += w;
        G = __fmaf_rn(w, gij, G);
        E1 = __fmaf_rn(gij, e, E1);
        E2 += e;
#pragma unroll
        for (int d = 0; d < kMaxDK; ++d)
            if (d < dK) {
                const float t = c * (qi[d] - kj[d]);
                A[d] = __fmaf_rn(gij, t, A[d]);
                Bd[d] += t;
            }
    };
    for (int t = lane; t < k; t += 32) {
        int j = irow[t];
        if (j == -1) continue;
        if (j < 0 || j >= cC) { set_status(status, ZETA_ERR_BOUNDS); continue; }
        visit(j);
    }
    for (int j = cC + lane; j <= i; j += 32) visit(j);
    sw = warp_sum(sw);
    G = warp_sum(G);
    E1 = warp_sum(E1);
    E2 = warp_sum(E2);
    const float inv_s = __frcp_rn(sw);
    const float gb = G * inv_s;
#pragma unroll
    for (int d = 0; d < kMaxDK; ++d) {
        A[d] = warp_sum(A[d]);
        Bd[d] = warp_sum(Bd[d]);
    }
    if (lane == 0) {
        for (int d = 0; d < dK; ++d) dq[row * dK + d] = (A[d] - gb * Bd[d]) * inv_s;
        s_out[row] = sw;
        gbar_out[row] = gb;
        m_out[row] = m;
        dg_part[row] = (E1 - gb * E2) * inv_s;
    }
}

// ------------------------------------------------------------ key side ---

// off[seg][j] = first position of key j in the sorted (key, query) list; the
// key of a sorted word is word >> key_shift (0: plain keys, 16: packed words).
// A lane takes eight consecutive positions (two 16-byte loads where the
// segment's words are 16-byte aligned); the key before its first position
// comes from the previous lane, lane 0 reading it.  Warps stride over the
// segment together, so every lane of a warp takes part in each shuffle.
__global__ void csr_offsets(const uint32_t *__restrict__ skeys, const uint32_t *__restrict__ seglen,
                            int64_t stride, int N, int key_shift, uint32_t *__restrict__ off) {
    const int64_t seg = blockIdx.y;
    const int64_t L = seglen[seg];
    const uint32_t *K = skeys + seg * stride;
    uint32_t *o = off + seg * (int64_t)(N + 1);
    const bool vec = (reinterpret_cast<uintptr_t>(K) & 15u) == 0;
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t w0 = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5);
    for (int64_t wb = 256 * w0; wb <= L; wb += 256 * warps) {
        const int64_t p0 = wb + 8 * lane;
        // key[1 + e]: key at p0 + e (N at and past L); key[0]: the key before p0
        int key[9];
        if (vec && p0 + 8 <= L) {
            const uint4 a = *reinterpret_cast<const uint4 *>(K + p0);
            const uint4 b = *reinterpret_cast<const uint4 *>(K + p0 + 4);
            key[1] = (int)(a.x >> key_shift);
            key[2] = (int)(a.y >> key_shift);
            key[3] = (int)(a.z >> key_shift);
            key[4] = (int)(a.w >> key_shift);
            key[5] = (int)(b.x >> key_shift);
            key[6] = (int)(b.y >> key_shift);
            key[7] = (int)(b.z >> key_shift);
            key[8] = (int)(b.w >> key_shift);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) key[1 + e] = p0 + e < L ? (int)(K[p0 + e] >> key_shift) : N;
        }
        key[0] = __shfl_up_sync(kFull, key[8], 1);
        if (lane == 0) key[0] = p0 > 0 ? (int)(K[p0 - 1] >> key_shift) : -1;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int64_t p = p0 + e;
            if (p > L) break;
            for (int j = key[e] + 1; j <= key[e + 1]; ++j) o[j] = (uint32_t)p;
        }
    }
}

template <typename V, int VPL, int WK>
__global__ void __launch_bounds__(256)
bwd_key_generic(const float *__restrict__ q, const float *__restrict__ kx,
                const V *__restrict__ v, const float *__restrict__ gamma,
                const float *__restrict__ rowsum, const V *__restrict__ dout,
                const float *__restrict__ gbar, const float *__restrict__ shift,
                const uint32_t *__restrict__ csr_q,
                const uint32_t *__restrict__ off, int64_t csr_stride, float *__restrict__ dk,
                V *__restrict__ dv, int64_t S, int N, int H, int dK, int dV, int C) {
    __shared__ float sv[8][kMaxDV];
    const int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    if (gw >= S * N) return;
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int64_t seg = gw / N;
    const int j = (int)(gw % N);
    const int64_t row = seg * N + j;
    const float g = gamma[seg % H];
    const float inv_g2 = __frcp_rn(g * g);
    float kj[kMaxDK];
#pragma unroll
    for (int d = 0; d < kMaxDK; ++d) kj[d] = d < dK ? kx[row * dK + d] : 0.f;
    for (int e = lane; e < dV; e += 32) sv[wib][e] = VT<V>::ld(v + row * dV + e);
    __syncwarp();
    const float *qb = q + seg * N * dK;
    const V *dob = dout + seg * N * dV;
    const float *rs = rowsum + seg * N;
    const float *gbb = gbar + seg * N;
    float acc[VPL];
#pragma unroll
    for (int e = 0; e < VPL; ++e) acc[e] = 0.f;
    float dka[kMaxDK];
#pragma unroll
    for (int d = 0; d < kMaxDK; ++d) dka[d] = 0.f;
    // Lane handles query i (i < 0: none); then the warp adds a_ij dO_i rows.
    auto step = [&](int i) {
        float a = 0.f;
        if (i >= 0) {
            const float *qi = qb + (int64_t)i * dK;
            const float w = weight_of<WK>(dist2b(qi, kj, dK), shift[seg * N + i], inv_g2);
            const float inv_s = __frcp_rn(rs[i]);
            a = w * inv_s;
            const float gij = dot_row<V>(sv[wib], dob + (int64_t)i * dV, dV);
            const float dldw = (gij - gbb[i]) * inv_s;
            const float coef = dldw * (2.f * neg_dw_dd2<WK>(w, inv_g2));
#pragma unroll
            for (int d = 0; d < kMaxDK; ++d)
                if (d < dK) dka[d] = __fmaf_rn(coef, qi[d] - kj[d], dka[d]);
        }
        for (int u = 0; u < 32; ++u) {
            const float au = __shfl_sync(kFull, a, u);
            const int iu = __shfl_sync(kFull, i, u);
            if (iu < 0) continue;
            const V *drow = dob + (int64_t)iu * dV;
#pragma unroll
            for (int e = 0; e < VPL; ++e) {
                const int col = lane + 32 * e;
                if (col < dV) acc[e] = __fmaf_rn(au, VT<V>::ld(drow + col), acc[e]);
            }
        }
    };
    const uint32_t *o = off + seg * (int64_t)(N + 1);
    const int64_t b0 = o[j], b1 = o[j + 1];
    const uint32_t *lst = csr_q + seg * csr_stride;
    for (int64_t p0 = b0; p0 < b1; p0 += 32) {
        const int64_t p = p0 + lane;
        step(p < b1 ? (int)lst[p] : -1);
    }
    const int cend = (j / C + 1) * C;
    for (int i0 = j; i0 < cend; i0 += 32) step(i0 + lane < cend ? i0 + lane : -1);
#pragma unroll
    for (int d = 0; d < kMaxDK; ++d) dka[d] = warp_sum(dka[d]);
    if (lane == 0)
        for (int d = 0; d < dK; ++d) dk[row * dK + d] = dka[d];
#pragma unroll
    for (int e = 0; e < VPL; ++e) {
        const int col = lane + 32 * e;
        if (col < dV) VT<V>::st(dv + row * dV + col, acc[e]);
    }
}

// dgamma[h] = sum over b and i of the per-query partials, in double and in a
// fixed order: one CTA per slice sums its N contiguous partials (tree order),
// then one thread per head adds its B slice sums in b order.
__global__ void __launch_bounds__(1024)
dgamma_slices(const float *__restrict__ part, int N, double *__restrict__ slice_sum) {
    __shared__ double red[32];
    const float *p = part + (int64_t)blockIdx.x * N;
    double s = 0.0;
    for (int i = threadIdx.x; i < N; i += 1024) s += (double)p[i];
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x < 32) {
        s = red[threadIdx.x];
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
        if (threadIdx.x == 0) slice_sum[blockIdx.x] = s;
    }
}

__global__ void dgamma_heads(const double *__restrict__ slice_sum, int B, int H,
                             float *__restrict__ dgamma) {
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h >= H) return;
    double s = 0.0;
    for (int b = 0; b < B; ++b) s += slice_sum[(int64_t)b * H + h];
    dgamma[h] = (float)s;
}

struct BwdWs {
    float *s;
    float *gbar;
    float *m;
    float *dgp;
    void *rec;
    double *slice_sum;
    RadixWs rw;
    uint32_t *off;
    float *own_dv;       // key side's own-chunk sums (tcgen05 path), else null
    float *own_dk;
};

BwdWs carve_bwd(const Prob &p, void *base, size_t *bytes) {
    Carver cv(base);
    BwdWs w;
    const int64_t rows = p.S * p.N;
    const int64_t L = p.N * (int64_t)p.k;
    w.s = cv.take<float>(rows);
    w.gbar = cv.take<float>(rows);
    w.m = cv.take<float>(rows);
    w.dgp = cv.take<float>(rows);
    w.rec = cv.take<char>(bwd_tc_rec_bytes(p));
    w.slice_sum = cv.take<double>(p.S);
    w.rw.keys[0] = cv.take<uint32_t>(p.S * L);
    w.rw.keys[1] = cv.take<uint32_t>(p.S * L);
    w.rw.vals[0] = cv.take<uint32_t>(p.S * L);
    w.rw.vals[1] = cv.take<uint32_t>(p.S * L);
    w.rw.hist = cv.take<uint32_t>(p.S * radix_tiles(L) * 256);
    w.rw.seglen = cv.take<uint32_t>(p.S);
    w.off = cv.take<uint32_t>(p.S * (p.N + 1));
    w.own_dv = w.own_dk = nullptr;
    if (attend_bwd_tc_supported(p) && bwd_own_tc05_supported(p)) {
        w.own_dv = cv.take<float>(rows * 64);
        w.own_dk = cv.take<float>(rows * 4);
    }
    if (bytes) *bytes = cv.bytes();
    return w;
}

void dgamma_reduce(const Prob &p, const BwdWs &w, float *dgamma, cudaStream_t st) {
    dgamma_slices<<<(unsigned)p.S, 1024, 0, st>>>(w.dgp, p.N, w.slice_sum);
    dgamma_heads<<<(unsigned)((p.H + 127) / 128), 128, 0, st>>>(w.slice_sum, p.B, p.H, dgamma);
}

template <typename V, int VPL, int WK>
cudaError_t bwd_generic(const Prob &p, const float *q, const float *k, const void *v,
                        const float *gamma, const int32_t *idx, const void *dout, float *dq,
                        float *dk, void *dv, float *dgamma, void *ws, int32_t *status,
                        cudaStream_t st) {
    BwdWs w = carve_bwd(p, ws, nullptr);
    const int64_t warps = p.S * p.N;
    const unsigned blocks = (unsigned)((warps + 7) / 8);
    bwd_query_generic<V, VPL, WK><<<blocks, 256, 0, st>>>(
        q, k, static_cast<const V *>(v), gamma, idx, static_cast<const V *>(dout), dq, w.s,
        w.gbar, w.m, w.dgp, status, p.S, p.N, p.H, p.dK, p.dV, p.k, p.C);
    int ob = 0;
    cudaError_t e = radix_sort_idx(idx, p.S, p.N, p.k, p.C, w.rw, &ob, status, st);
    if (e != cudaSuccess) return e;
    const int64_t L = p.N * (int64_t)p.k;
    csr_offsets<<<dim3(64, (unsigned)p.S), 256, 0, st>>>(
        static_cast<const uint32_t *>(w.rw.keys[ob]), w.rw.seglen, L, p.N, 0, w.off);
    bwd_key_generic<V, VPL, WK><<<blocks, 256, 0, st>>>(
        q, k, static_cast<const V *>(v), gamma, w.s, static_cast<const V *>(dout), w.gbar, w.m,
        w.rw.vals[ob], w.off, L, dk, static_cast<V *>(dv), p.S, p.N, p.H, p.dK, p.dV, p.C);
    dgamma_reduce(p, w, dgamma, st);
    return cudaGetLastError();
}

template <typename V>
cudaError_t bwd_dispatch(const Prob &p, const float *q, const float *k, const void *v,
                         const float *gamma, const int32_t *idx, const void *dout, float *dq,
                         float *dk, void *dv, float *dgamma, void *ws, int32_t *status,
                         cudaStream_t st) {
#define ZETA_BWD(VPL)                                                                        \
    if (p.wk == kWSoftmax)                                                                   \
        return bwd_generic<V, VPL, kWSoftmax>(p, q, k, v, gamma, idx, dout, dq, dk, dv, dgamma, \
                                              ws, status, st);                               \
    if (p.wk == kWInvEuclid)                                                                 \
        return bwd_generic<V, VPL, kWInvEuclid>(p, q, k, v, gamma, idx, dout, dq, dk, dv,     \
                                                dgamma, ws, status, st);                     \
    return bwd_generic<V, VPL, kWCauchy>(p, q, k, v, gamma, idx, dout, dq, dk, dv, dgamma, ws, \
                                         status, st)
    if (p.dV <= 32) {
        ZETA_BWD(1);
    }
    if (p.dV <= 64) {
        ZETA_BWD(2);
    }
    if (p.dV <= 128) {
        ZETA_BWD(4);
    }
    ZETA_BWD(8);
#undef ZETA_BWD
}

}  // namespace

size_t bwd_ws_bytes(const Prob &p) {
    size_t b = 0;
    carve_bwd(p, nullptr, &b);
    return b;
}

cudaError_t launch_attend_bwd(const Prob &p, const float *q, const float *k, const void *v,
                              const float *gamma, const int32_t *idx, const void *dout, float *dq,
                              float *dk, void *dv, float *dgamma, void *ws, int32_t *status,
                              cudaStream_t st) {
    if (attend_bwd_tc_supported(p)) {
        BwdWs w = carve_bwd(p, ws, nullptr);
        cudaError_t e = launch_bwd_query_tc(p, q, k, v, gamma, idx, dout, dq, w.rec, w.dgp,
                                            status, st);
        if (e != cudaSuccess) return e;
        if (w.own_dv) {
            e = launch_bwd_key_own_tc05(p, k, v, gamma, dout, w.rec, w.own_dv, w.own_dk, status,
                                        st);
            if (e == cudaErrorNotSupported) {       // no tensor-map encoder: the key kernel
                w.own_dv = w.own_dk = nullptr;      // computes its own-chunk block itself
                e = cudaSuccess;
            }
            if (e != cudaSuccess) return e;
        }
        int ob = 0;
        // the key walk needs a warp's 16 keys contiguous, not ordered by key;
        // it skips the key half (8 keys) that none of 16 consecutive entries
        // belongs to.  With packed words and chunks a multiple of 8 long, a
        // sort by key / 8 keeps both (N, a multiple of C, is then one of 8 too,
        // so every group is whole).
        const bool packed = p.N <= 65536;
        const bool groups = packed && p.C % 8 == 0;
        e = packed ? radix_sort_idx_packed(idx, p.S, p.N, p.k, p.C, groups, w.rw, &ob, status, st)
                   : radix_sort_idx(idx, p.S, p.N, p.k, p.C, w.rw, &ob, status, st);
        if (e != cudaSuccess) return e;
        const int64_t L = p.N * (int64_t)p.k;
        const uint32_t *sorted = static_cast<const uint32_t *>(w.rw.keys[ob]);
        const int kgs = groups ? 3 : 0;
        csr_offsets<<<dim3(64, (unsigned)p.S), 256, 0, st>>>(sorted, w.rw.seglen, L, p.N >> kgs,
                                                              packed ? 16 + kgs : 0, w.off);
        e = launch_bwd_key_tc(p, k, v, gamma, dout, w.rec, packed ? sorted : w.rw.vals[ob],
                              packed ? nullptr : sorted, packed ? 0xffffu : 0xffffffffu, kgs,
                              w.off, L, dk, dv, w.own_dv, w.own_dk, st);
        if (e != cudaSuccess) return e;
        dgamma_reduce(p, w, dgamma, st);
        return cudaGetLastError();
    }
    if (p.vdt == ZETA_BF16)
        return bwd_dispatch<__nv_bfloat16>(p, q, k, v, gamma, idx, dout, dq, dk, dv, dgamma, ws,
                                           status, st);
    return bwd_dispatch<float>(p, q, k, v, gamma, idx, dout, dq, dk, dv, dgamma, ws, status, st);
}

}  // namespace zeta
